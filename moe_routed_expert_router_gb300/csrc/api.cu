// C ABI of the MoE NVFP4 library: plan management, argument checks and the
// order of the device steps.  Every step of the path runs in this library's
// kernels; the host only validates arguments and launches.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
size_t group_smem_bytes(int E);
cudaError_t configure_group_kernel();
cudaError_t configure_tc(const Plan &p);
cudaError_t configure_simt();
bool tc_supported(const Plan &p);
bool warp_mma_supported(const Plan &p);
cudaError_t launch_ffn_tc(const Plan &p, const void *x, int T, const ExpertPtrs &routed, const ExpertPtrs *shared,
                          int part, cudaStream_t st, bool warp_mma);
}  // namespace moe

using moe::Plan;

struct moe_plan_s {
    Plan p;
    int path = MOE_PATH_AUTO;
    // per-stage timing (moe_plan_set_profiling)
    bool prof = false;
    std::vector<cudaEvent_t> pool;
    size_t next = 0;
    struct Rec { int stage; cudaEvent_t b, e; };
    std::vector<Rec> recs;
    int64_t launches[MOE_NUM_STAGES] = {};
    int64_t calls[MOE_NUM_STAGES] = {};
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_status check_config(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->router != MOE_ROUTER_SOFTMAX && c->router != MOE_ROUTER_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (c->mode != MOE_W4A16 && c->mode != MOE_W4A4) return MOE_ERR_INVALID_ARG;
    if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
    if (c->has_shared != 0 && c->has_shared != 1) return MOE_ERR_INVALID_ARG;
    if (c->router_dtype != MOE_ROUTER_F32 && c->router_dtype != MOE_ROUTER_BF16) return MOE_ERR_INVALID_ARG;
    if (c->weight_format != MOE_WEIGHTS_NVFP4 && c->weight_format != MOE_WEIGHTS_MXFP4) return MOE_ERR_INVALID_ARG;
    if (c->weight_format == MOE_WEIGHTS_MXFP4 &&
        (c->hidden % 512 || c->inter % 512 || (c->has_shared && c->shared_inter % 512)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return MOE_ERR_INVALID_ARG;
    if (c->hidden < 256 || c->hidden % 256 || c->hidden > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->inter < 128 || c->inter % 128 || c->inter > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->has_shared && (c->shared_inter < 128 || c->shared_inter % 128 || c->shared_inter > 8192))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->num_experts < 1 || c->num_experts > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)c->max_tokens * c->top_k > (1 << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

moe_status check_nvfp4(const moe_nvfp4 &w, bool mx) {
    if (!w.codes || !w.scales || (!mx && !w.tensor_scale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w.codes) || (!mx && !aligned4(w.tensor_scale))) return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

moe_status check_set(const moe_expert_set *s, bool mx) {
    if (!s) return MOE_ERR_INVALID_ARG;
    moe_status r;
    if ((r = check_nvfp4(s->gate, mx)) != MOE_OK) return r;
    if ((r = check_nvfp4(s->up, mx)) != MOE_OK) return r;
    return check_nvfp4(s->down, mx);
}

// MXFP4 weights have no tensor scale: the kernels read the plan's array of ones.
moe::ExpertPtrs ptrs(const moe_expert_set &s, const moe::Plan &p) {
    if (p.cfg.weight_format == MOE_WEIGHTS_MXFP4)
        return moe::ExpertPtrs{s.gate.codes, s.gate.scales, s.up.codes, s.up.scales, s.down.codes, s.down.scales,
                               p.ones, p.ones, p.ones};
    return moe::ExpertPtrs{s.gate.codes, s.gate.scales, s.up.codes, s.up.scales, s.down.codes, s.down.scales,
                           s.gate.tensor_scale, s.up.tensor_scale, s.down.tensor_scale};
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Carves 256-byte aligned slices out of one allocation.
struct Carver {
    size_t off = 0;
    char *base = nullptr;
    template <class T>
    T *take(size_t bytes) {
        size_t o = (off + 255) & ~size_t(255);
        off = o + bytes;
        return base ? reinterpret_cast<T *>(base + o) : nullptr;
    }
};

// Per-call scratch, cleared at the start of every call: the call's counters,
// the per-expert counts, and the arrival tickets of split gate/up items.
size_t scratch_bytes(const Plan &p) {
    return sizeof(moe::CallScratch) + sizeof(int32_t) * ((size_t)p.cfg.num_experts + 8 * (size_t)p.num_sms);
}

void carve(Plan &p, Carver &c) {
    const moe_config &k = p.cfg;
    const int64_t T = k.max_tokens, H = k.hidden, E = k.num_experts;
    const int64_t Imax = k.has_shared ? std::max(k.inter, k.shared_inter) : k.inter;
    p.logits = c.take<float>(sizeof(float) * T * E);
    p.ids = c.take<int32_t>(sizeof(int32_t) * p.pairs_max);
    p.wts = c.take<float>(sizeof(float) * p.pairs_max);
    p.scratch = c.take<moe::CallScratch>(scratch_bytes(p));
    p.counts = p.scratch ? reinterpret_cast<int32_t *>(p.scratch + 1) : nullptr;
    p.tail_tickets = p.counts ? p.counts + E : nullptr;
    p.offsets = c.take<int32_t>(sizeof(int32_t) * (E + 2));
    p.poff = c.take<int32_t>(sizeof(int32_t) * (E + 2));
    p.sorted = c.take<int32_t>(sizeof(int32_t) * p.pairs_max);
    p.inv = c.take<int32_t>(sizeof(int32_t) * p.pairs_max);
    p.pad_pair = c.take<int32_t>(sizeof(int32_t) * p.rows_pad_max);
    p.chunks = c.take<int4>(sizeof(int4) * p.chunks_max);
    p.tiles = c.take<int4>(sizeof(int4) * p.tiles_max);
    p.group_blk = c.take<int32_t>(sizeof(int32_t) * (size_t)((p.pairs_max + moe::kGroupSeg - 1) / moe::kGroupSeg) * E);
    if (k.mode == MOE_W4A4) {
        p.xp = c.take<uint8_t>(p.rows_pad_max * H / 2);
        p.xp_atoms = c.take<uint8_t>(p.rows_pad_max * H / 16);
        p.hq_atoms = c.take<uint8_t>(p.rows_pad_max * Imax / 16);
    } else {
        p.xp16 = c.take<__half>(p.rows_pad_max * H * 2);
        p.tail_part = c.take<float>(sizeof(float) * (size_t)p.num_sms * moe::kTailPartFloats);
    }
    p.xts = c.take<float>(64);
    p.xq = c.take<uint8_t>(T * H / 2);
    p.xsc = c.take<uint8_t>(T * H / 16);
    p.hbuf = c.take<float>(sizeof(float) * p.rows_pad_max * Imax);
    p.hq = c.take<uint8_t>(p.rows_pad_max * Imax / 2);
    p.hsc = c.take<uint8_t>(p.rows_pad_max * Imax / 16);
    p.hts = c.take<float>(64);
    p.acc = c.take<float>(sizeof(float) * T * H);
    p.err = c.take<int>(64);
    p.ones = c.take<float>(sizeof(float) * (E + 1));
    p.x_stage = c.take<void>(2 * T * H);
    p.out_stage = c.take<void>(2 * T * H);
}


moe_status check_call(moe_plan plan, const void *x, int32_t T, const void *rw, const float *bias) {
    if (!plan || T < 0 || T > plan->p.cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !rw)) return MOE_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (rw && !aligned16(rw)) || (bias && !aligned4(bias))) return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

// Event pair around one stage of a call, when profiling is on.
struct Stage {
    moe_plan pl;
    int stage;
    cudaStream_t st;
    cudaEvent_t b = nullptr, e = nullptr;
    Stage(moe_plan pl_, int stage_, cudaStream_t st_) : pl(pl_), stage(stage_), st(st_) {
        if (pl->prof && pl->next + 2 <= pl->pool.size()) {
            b = pl->pool[pl->next++];
            e = pl->pool[pl->next++];
            cudaEventRecord(b, st);
        }
    }
    cudaError_t done(cudaError_t err, int kernels) {
        pl->launches[stage] += kernels;
        pl->calls[stage] += 1;
        if (b) {
            cudaEventRecord(e, st);
            pl->recs.push_back({stage, b, e});
        }
        return err;
    }
};

moe_status forward_device(moe_plan plan, const void *x, int32_t T, const void *rw, const float *bias,
                          const moe_expert_set *routed, const moe_expert_set *shared, void *out, cudaStream_t st) {
    Plan &p = plan->p;
    cudaError_t e = cudaMemsetAsync(p.scratch, 0, scratch_bytes(p), st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // engine: CUDA-core streaming kernels, tcgen05 grouped GEMMs, or (W4A16)
    // warp-level MMAs fed from registers; AUTO takes the warp MMAs when the
    // batch leaves fewer than two rows an expert on average (decode)
    bool wm = plan->path == MOE_PATH_WARP_MMA;
    bool tc = wm || plan->path == MOE_PATH_TENSOR_CORE;
    if (plan->path == MOE_PATH_AUTO) {
        wm = moe::warp_mma_supported(p) && T * p.cfg.top_k < 2 * p.cfg.num_experts;
        tc = wm || (moe::tc_supported(p) && (p.cfg.mode == MOE_W4A16 || T * p.cfg.top_k >= 64));
        if (p.cfg.weight_format == MOE_WEIGHTS_MXFP4 && p.cfg.mode == MOE_W4A16) {   // warp MMAs or CUDA cores
            wm = moe::warp_mma_supported(p);
            tc = wm;
        }
    }
    // rows a tensor-core tile covers: 32 for the warp MMAs, 64 for the W4A16
    // tcgen05 GEMMs, 128 for the W4A4 ones
    p.tile_rows = p.cfg.mode == MOE_W4A4 ? moe::kTileRows : (wm ? 32 : 64);
    // decode-sized batches: the router's last block also groups the pairs
    const bool fused_group = moe::router_groups(T);
    {
        Stage s(plan, MOE_STAGE_ROUTE, st);
        if (s.done(moe::launch_router(p, x, T, rw, bias, p.ids, p.wts, st, fused_group), moe::router_launches(T)) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (!fused_group) {
        Stage s(plan, MOE_STAGE_GROUP, st);
        if (s.done(moe::launch_group(p, T, p.ids, nullptr, nullptr, true, st), moe::group_launches(p, T)) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (p.cfg.mode == MOE_W4A4) {
        Stage s(plan, MOE_STAGE_QUANT_X, st);
        if (s.done(moe::launch_quant_act(p, x, T, p.xq, p.xsc, p.xts, true, st), 1) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    moe::ExpertPtrs r = ptrs(*routed, p), sh{};
    if (shared) sh = ptrs(*shared, p);
    const moe::ExpertPtrs *shp = shared ? &sh : nullptr;
    {
        Stage s(plan, MOE_STAGE_GATE_UP, st);
        e = tc ? moe::launch_ffn_tc(p, x, T, r, shp, 0, st, wm) : moe::launch_ffn_simt(p, x, T, r, shp, 0, st);
        if (s.done(e, (tc && !wm) ? 2 : 1) != cudaSuccess) return MOE_ERR_CUDA;   // + the permute launch
    }
    // W4A4: the SwiGLU output's quantisation, a pass of its own except for
    // MXFP4 on the tensor cores, whose gate/up epilogue quantises h itself
    if (p.cfg.mode == MOE_W4A4 && !(tc && p.cfg.weight_format == MOE_WEIGHTS_MXFP4)) {
        Stage s(plan, MOE_STAGE_QUANT_H, st);
        if (s.done(moe::launch_quant_h(p, tc, st), 1) != cudaSuccess) return MOE_ERR_CUDA;
    }
    {
        Stage s(plan, MOE_STAGE_DOWN, st);
        e = tc ? moe::launch_ffn_tc(p, x, T, r, shp, 1, st, wm) : moe::launch_ffn_simt(p, x, T, r, shp, 1, st);
        if (s.done(e, 1) != cudaSuccess) return MOE_ERR_CUDA;
    }
    Stage s(plan, MOE_STAGE_FINALIZE, st);
    return cuda_status(s.done(moe::launch_finalize(p, T, out, st), 1));
}

}  // namespace

extern "C" {

const char *moe_version(void) { return "moe_nvfp4 0.1 (sm_103a)"; }

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MOE_ERR_NONFINITE: return "non-finite activation";
        case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_OOM: return "out of device memory";
        case MOE_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

moe_status moe_plan_create(const moe_config *cfg, moe_plan *out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    moe_plan plan = new (std::nothrow) moe_plan_s;
    if (!plan) return MOE_ERR_OOM;
    Plan &p = plan->p;
    p.cfg = *cfg;
    if (cudaGetDevice(&p.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess) {
        delete plan;
        return MOE_ERR_CUDA;
    }
    const int64_t T = cfg->max_tokens, E = cfg->num_experts;
    p.pairs_max = T * cfg->top_k;
    p.rows_pad_max = p.pairs_max + std::min<int64_t>(E, p.pairs_max) * (moe::kTileRows - 1) +
                     (cfg->has_shared ? (T + moe::kTileRows - 1) / moe::kTileRows * moe::kTileRows : 0);
    p.rows_pad_max = (p.rows_pad_max + moe::kTileRows - 1) / moe::kTileRows * moe::kTileRows;
    p.chunks_max = p.pairs_max / moe::kChunkRows + E + 2 + (cfg->has_shared ? T / moe::kChunkRows + 1 : 0);
    p.tile_rows = cfg->mode == MOE_W4A16 ? 32 : moe::kTileRows;   // the smallest tiles a call may use
    p.tiles_max = p.pairs_max / p.tile_rows + E + 2 + (cfg->has_shared ? T / p.tile_rows + 1 : 0);
    Carver dry;
    carve(p, dry);
    p.ws_bytes = dry.off + 256;
    if (cudaMalloc(&p.ws, p.ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete plan;
        return MOE_ERR_OOM;
    }
    Carver real;
    real.base = static_cast<char *>(p.ws);
    carve(p, real);
    cudaError_t e = cudaMemset(p.ws, 0, p.ws_bytes);
    if (e == cudaSuccess) {
        std::vector<float> ones((size_t)cfg->num_experts + 1, 1.0f);
        e = cudaMemcpy(p.ones, ones.data(), sizeof(float) * ones.size(), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = moe::configure_group_kernel();
    if (e == cudaSuccess) e = moe::configure_simt();
    if (e == cudaSuccess && moe::tc_supported(p)) e = moe::configure_tc(p);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(p.ws);
        delete plan;
        return MOE_ERR_CUDA;
    }
    *out = plan;
    return MOE_OK;
}

moe_status moe_plan_set_path(moe_plan plan, int32_t path) {
    if (!plan || path < MOE_PATH_AUTO || path > MOE_PATH_WARP_MMA) return MOE_ERR_INVALID_ARG;
    // MXFP4 takes the tcgen05 GEMMs for W4A4 only (kind::mxf4); its W4A16 runs on
    // the warp MMAs or the CUDA cores
    if (path == MOE_PATH_TENSOR_CORE &&
        (!moe::tc_supported(plan->p) ||
         (plan->p.cfg.weight_format == MOE_WEIGHTS_MXFP4 && plan->p.cfg.mode == MOE_W4A16)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (path == MOE_PATH_WARP_MMA && !moe::warp_mma_supported(plan->p)) return MOE_ERR_UNSUPPORTED_SHAPE;
    plan->path = path;
    return MOE_OK;
}

moe_status moe_plan_keep_h(moe_plan plan, int32_t keep) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    plan->p.keep_h = keep != 0;
    return MOE_OK;
}

moe_status moe_plan_set_profiling(moe_plan plan, int32_t enable) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (enable && plan->pool.empty()) {
        plan->pool.resize(8192);
        for (auto &ev : plan->pool)
            if (cudaEventCreate(&ev) != cudaSuccess) return MOE_ERR_CUDA;
    }
    plan->prof = enable != 0;
    return MOE_OK;
}

moe_status moe_plan_read_profile(moe_plan plan, float *ms, int64_t *launches, int64_t *calls) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    for (const auto &r : plan->recs) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.b, r.e) != cudaSuccess) return MOE_ERR_CUDA;
        if (ms) ms[r.stage] += t;
    }
    for (int i = 0; i < MOE_NUM_STAGES; ++i) {
        if (launches) launches[i] += plan->launches[i];
        if (calls) calls[i] += plan->calls[i];
        plan->launches[i] = plan->calls[i] = 0;
    }
    plan->recs.clear();
    plan->next = 0;
    return MOE_OK;
}

moe_status moe_plan_destroy(moe_plan plan) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    for (auto &ev : plan->pool) cudaEventDestroy(ev);
    cudaError_t e = cudaFree(plan->p.ws);
    delete plan;
    return cuda_status(e);
}

moe_status moe_route(moe_plan plan, const void *x_bf16, int32_t T, const void *router_w, const float *router_bias,
                     int32_t *topk_ids, float *topk_w, int32_t *expert_offsets, int32_t *sorted_rows, void *stream) {
    moe_status st = check_call(plan, x_bf16, T, router_w, router_bias);
    if (st != MOE_OK) return st;
    if (!topk_ids || !topk_w || !expert_offsets || !sorted_rows) return MOE_ERR_INVALID_ARG;
    if (!aligned4(topk_ids) || !aligned4(topk_w) || !aligned4(expert_offsets) || !aligned4(sorted_rows))
        return MOE_ERR_MISALIGNED;
    Plan &p = plan->p;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.scratch, 0, scratch_bytes(p), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) {
        return cuda_status(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (p.cfg.num_experts + 1), s));
    }
    if (moe::launch_router(p, x_bf16, T, router_w, router_bias, topk_ids, topk_w, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_status(moe::launch_group(p, T, topk_ids, expert_offsets, sorted_rows, false, s));
}

moe_status moe_forward(moe_plan plan, const void *x_bf16, int32_t T, const void *router_w, const float *router_bias,
                       const moe_expert_set *routed, const moe_expert_set *shared, void *out_bf16, void *stream) {
    moe_status st = check_call(plan, x_bf16, T, router_w, router_bias);
    if (st != MOE_OK) return st;
    const bool mx = plan->p.cfg.weight_format == MOE_WEIGHTS_MXFP4;
    if ((st = check_set(routed, mx)) != MOE_OK) return st;
    if (plan->p.cfg.has_shared) {
        if ((st = check_set(shared, mx)) != MOE_OK) return st;
    } else if (shared) {
        return MOE_ERR_INVALID_ARG;
    }
    if (T > 0 && !out_bf16) return MOE_ERR_INVALID_ARG;
    if (out_bf16 && !aligned16(out_bf16)) return MOE_ERR_MISALIGNED;
    if (T == 0) return MOE_OK;
    return forward_device(plan, x_bf16, T, router_w, router_bias, routed, shared, out_bf16,
                          static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_host(moe_plan plan, const void *x_bf16_host, int32_t T, const void *router_w,
                            const float *router_bias, const moe_expert_set *routed, const moe_expert_set *shared,
                            void *out_bf16_host, void *stream) {
    if (!plan || T < 0 || T > plan->p.cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x_bf16_host || !out_bf16_host)) return MOE_ERR_INVALID_ARG;
    Plan &p = plan->p;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)T * p.cfg.hidden * 2;
    moe_status st = check_call(plan, p.x_stage, T, router_w, router_bias);
    if (st != MOE_OK) return st;
    const bool mx = p.cfg.weight_format == MOE_WEIGHTS_MXFP4;
    if ((st = check_set(routed, mx)) != MOE_OK) return st;
    if (p.cfg.has_shared && (st = check_set(shared, mx)) != MOE_OK) return st;
    if (!p.cfg.has_shared && shared) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (cudaMemcpyAsync(p.x_stage, x_bf16_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
    st = forward_device(plan, p.x_stage, T, router_w, router_bias, routed, shared, p.out_stage, s);
    if (st != MOE_OK) return st;
    return cuda_status(cudaMemcpyAsync(out_bf16_host, p.out_stage, bytes, cudaMemcpyDeviceToHost, s));
}

moe_status moe_quantize_act(moe_plan plan, const void *x_bf16, int32_t T, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, void *stream) {
    if (!plan || T < 0 || T > plan->p.cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !codes || !scales || !tensor_scale) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_bf16)) return MOE_ERR_MISALIGNED;
    if (!aligned16(codes) || !aligned4(tensor_scale)) return MOE_ERR_MISALIGNED;
    Plan &p = plan->p;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.scratch, 0, scratch_bytes(p), s) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(moe::launch_quant_act(p, x_bf16, T, codes, scales, tensor_scale, false, s));
}

moe_status moe_quantize_nvfp4(const float *w, int32_t batch, int32_t rows, int32_t cols, uint8_t *codes,
                              uint8_t *scales, float *tensor_scale, void *stream) {
    if (batch < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
    if (cols % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (batch == 0 || rows == 0 || cols == 0) return MOE_OK;
    if (!w || !codes || !scales || !tensor_scale) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(codes) || !aligned4(tensor_scale)) return MOE_ERR_MISALIGNED;
    return cuda_status(moe::launch_quant_nvfp4(w, batch, rows, cols, codes, scales, tensor_scale,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_mxfp4(const float *w, int64_t rows, int32_t cols, uint8_t *codes, uint8_t *scales,
                              void *stream) {
    if (rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
    if (cols % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!w || !codes || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(codes)) return MOE_ERR_MISALIGNED;
    return cuda_status(moe::launch_quant_mxfp4(w, rows, cols, codes, scales, static_cast<cudaStream_t>(stream)));
}

moe_status moe_convert_f32(const float *src, int64_t n, int32_t format, uint8_t *dst, void *stream) {
    if (n < 0 || (format != MOE_FMT_E4M3 && format != MOE_FMT_E2M1)) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!src || !dst) return MOE_ERR_INVALID_ARG;
    if (!aligned16(src)) return MOE_ERR_MISALIGNED;
    return cuda_status(moe::launch_convert(src, n, format, dst, static_cast<cudaStream_t>(stream)));
}

moe_status moe_plan_sync_status(moe_plan plan, void *stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, plan->p.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(plan->p.err, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (err & moe::kErrNonFinite) return MOE_ERR_NONFINITE;
    if (err & moe::kErrTimeout) return MOE_ERR_TIMEOUT;
    if (err) return MOE_ERR_DEVICE;
    return MOE_OK;
}

moe_status moe_plan_check_timeout(moe_plan plan, int64_t wait_ns, void *stream) {
    if (!plan || wait_ns < 0 || wait_ns > 1000000000LL) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_wait_check(plan->p.err, (uint64_t)wait_ns, static_cast<cudaStream_t>(stream)));
}

moe_status moe_plan_debug_buffer(moe_plan plan, const char *name, void **ptr, size_t *bytes) {
    if (!plan || !name || !ptr) return MOE_ERR_INVALID_ARG;
    const Plan &p = plan->p;
    const int64_t Imax = p.cfg.has_shared ? std::max(p.cfg.inter, p.cfg.shared_inter) : p.cfg.inter;
    struct Item { const char *n; void *p; size_t b; } items[] = {
        {"h_codes", p.hq, (size_t)(p.rows_pad_max * Imax / 2)},
        {"h_scales", p.hsc, (size_t)(p.rows_pad_max * Imax / 16)},
        {"h_scale_atoms", p.hq_atoms, p.hq_atoms ? (size_t)(p.rows_pad_max * Imax / 16) : 0},
        {"h_ts", p.hts, 2 * sizeof(float)},
        {"x_ts", p.xts, sizeof(float)},
        {"acc", p.acc, sizeof(float) * (size_t)p.cfg.max_tokens * p.cfg.hidden},
        {"counts", p.counts, sizeof(int32_t) * (size_t)p.cfg.num_experts},
        {"padded_offsets", p.poff, sizeof(int32_t) * (size_t)(p.cfg.num_experts + 2)},
        {"offsets", p.offsets, sizeof(int32_t) * (size_t)(p.cfg.num_experts + 1)},
        {"sorted", p.sorted, sizeof(int32_t) * (size_t)p.pairs_max},
        {"tiles", p.tiles, sizeof(int4) * (size_t)p.tiles_max},
        {"pad_pair", p.pad_pair, sizeof(int32_t) * (size_t)p.rows_pad_max},
        {"h", p.hbuf, sizeof(float) * (size_t)(p.rows_pad_max * Imax)},
    };
    for (const Item &it : items) {
        if (std::strcmp(it.n, name) == 0) {
            *ptr = it.p;
            if (bytes) *bytes = it.b;
            return MOE_OK;
        }
    }
    return MOE_ERR_INVALID_ARG;
}

}  // extern "C"
