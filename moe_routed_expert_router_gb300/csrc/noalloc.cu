// moe_route_static: routing and grouping for callers that cannot allocate
// device memory (see include/moe_nvfp4.h).  It runs the same router and
// grouping kernels as moe_route; their scratch lives in one file-scope device
// array instead of a plan's workspace.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
cudaError_t configure_group_kernel();
}

namespace {

constexpr int64_t kStaticMaxLogits = 1 << 20;   // T * E
constexpr int64_t kStaticMaxPairs = 1 << 16;    // T * k
constexpr int kStaticMaxExperts = moe::kMaxExperts;
constexpr int64_t kStaticMaxRowsPad = kStaticMaxPairs + (int64_t)kStaticMaxExperts * (moe::kTileRows - 1);

struct StaticScratch {
    float logits[kStaticMaxLogits];
    moe::CallScratch scratch;            // followed directly by counts (cleared together)
    int32_t counts[kStaticMaxExperts];
    int32_t offsets[kStaticMaxExperts + 2];
    int32_t poff[kStaticMaxExperts + 2];
    int32_t sorted[kStaticMaxPairs];
    int32_t inv[kStaticMaxPairs];
    int32_t pad_pair[kStaticMaxRowsPad];
    int err[4];
};

// One copy per device that loads the library, kept until the process exits.
static __device__ __align__(256) StaticScratch g_route_scratch;

StaticScratch *g_addr[moe::kMaxDevices] = {};
int g_sms[moe::kMaxDevices] = {};
std::mutex g_mu;

// Device address of the array on the current device (looked up once per
// device; host code must not use the symbol itself as an address).
moe_status static_scratch(StaticScratch **out, int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= moe::kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::configure_group_kernel() != cudaSuccess) return MOE_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
        g_sms[dev] = n;
        g_addr[dev] = static_cast<StaticScratch *>(p);
    }
    *out = g_addr[dev];
    *sms = g_sms[dev];
    return MOE_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" moe_status moe_route_static(const void *x_bf16, int32_t T, int32_t hidden, const float *router_w,
                                       const float *router_bias, int32_t num_experts, int32_t top_k,
                                       int32_t router, int32_t renormalize, int32_t *topk_ids, float *topk_w,
                                       int32_t *expert_offsets, int32_t *sorted_rows, void *stream) {
    if (T < 0 || hidden < 256 || hidden % 256 || hidden > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (num_experts < 1 || num_experts > kStaticMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (top_k < 1 || top_k > num_experts || top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)T * num_experts > kStaticMaxLogits || (int64_t)T * top_k > kStaticMaxPairs)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((router != MOE_ROUTER_SOFTMAX && router != MOE_ROUTER_SIGMOID) || (renormalize != 0 && renormalize != 1))
        return MOE_ERR_INVALID_ARG;
    if (!expert_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x_bf16 || !router_w || !topk_ids || !topk_w || !sorted_rows)) return MOE_ERR_INVALID_ARG;
    if ((x_bf16 && !aligned(x_bf16, 16)) || (router_w && !aligned(router_w, 16)) ||
        (router_bias && !aligned(router_bias, 4)) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
        !aligned(expert_offsets, 4) || !aligned(sorted_rows, 4))
        return MOE_ERR_MISALIGNED;
    StaticScratch *S = nullptr;
    moe::Plan p;
    moe_status st = static_scratch(&S, &p.num_sms);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0)
        return cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (num_experts + 1), s) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    p.cfg = moe_config{hidden, 128, num_experts, top_k, T, router, renormalize, MOE_W4A16, 0, 0};
    cudaGetDevice(&p.device);
    p.pairs_max = (int64_t)T * top_k;
    p.rows_pad_max = kStaticMaxRowsPad;
    p.logits = S->logits;
    p.scratch = &S->scratch;
    p.counts = S->counts;
    p.offsets = S->offsets;
    p.poff = S->poff;
    p.sorted = S->sorted;
    p.inv = S->inv;
    p.pad_pair = S->pad_pair;
    p.err = S->err;
    // the per-call words and counts must start at zero; the error word too
    if (cudaMemsetAsync(&S->scratch, 0, sizeof(moe::CallScratch) + sizeof(int32_t) * num_experts, s) != cudaSuccess ||
        cudaMemsetAsync(S->err, 0, sizeof(int), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (moe::launch_router(p, x_bf16, T, router_w, router_bias, topk_ids, topk_w, s) != cudaSuccess) return MOE_ERR_CUDA;
    return moe::launch_group(p, T, topk_ids, expert_offsets, sorted_rows, false, s) == cudaSuccess ? MOE_OK
                                                                                                    : MOE_ERR_CUDA;
}
