// Internal declarations of the GB300 MoE NVFP4 library (device side and plan).
// Nothing here is part of the C ABI; see include/moe_nvfp4.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"

namespace moe {

// Rows of every expert's segment in the permuted activation / SwiGLU buffers
// are padded to this multiple, so a 128-row tensor-core tile never mixes experts.
constexpr int kTileRows = 128;
// Tokens of one expert handled together by the CUDA-core (decode-shaped) kernels.
constexpr int kChunkRows = 4;
// The warp-MMA engine may split the items of its grid's last, partial round
// along K (at most kMaxTailParts pieces); a gate/up piece leaves its partial
// sums for 8 row groups x 4 token tiles x 32 lanes x (4 gate + 4 up) values.
constexpr int kMaxTailParts = 4;
// Pairs a block of the multi-block grouping takes.
constexpr int kGroupSeg = 1024;
constexpr int kTailPartFloats = 8 * 4 * 32 * 8;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
// Devices a process may use (per-device one-time set-up tables).
constexpr int kMaxDevices = 64;

// Device error bits (plan error word).
constexpr int kErrNonFinite = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrDevice = 4;

// Per-call scratch words, cleared by one memset at the start of every call.
struct CallScratch {
    unsigned int x_amax;        // fp32 bits of amax|x| (W4A4)
    unsigned int h_amax;        // fp32 bits of amax|h| over routed rows (W4A4)
    unsigned int hs_amax;       // same for the shared expert's rows
    int n_chunks;               // CUDA-core work chunks
    int n_tiles;                // tensor-core tiles (gate/up)
    int route_done;             // router blocks finished (the last one runs top-k)
    int n_chunks_routed;        // chunks of routed experts (the shared expert's follow)
    int pad;
};

struct Plan {
    moe_config cfg;
    int device = 0;
    int num_sms = 0;
    int keep_h = 0;             // also store the fp32 SwiGLU output where the gate/up launch quantises it
    int64_t pairs_max = 0;      // max_tokens * k
    int64_t rows_pad_max = 0;   // padded permuted rows (routed + shared)
    int64_t chunks_max = 0;

    void *ws = nullptr;
    size_t ws_bytes = 0;

    float *logits = nullptr;        // [Tmax][E]
    int32_t *ids = nullptr;         // [P]
    float *wts = nullptr;           // [P]
    int32_t *counts = nullptr;      // [E]
    int32_t *offsets = nullptr;     // [E+2]
    int32_t *poff = nullptr;        // [E+2] padded offsets; index E = shared segment
    int32_t *sorted = nullptr;      // [P]
    int32_t *inv = nullptr;         // [P] pair -> padded row
    int32_t *pad_pair = nullptr;    // [rows_pad] pair at a padded row (-1 pad, >= P shared token)
    int4 *chunks = nullptr;         // [chunks_max] {expert, first padded row, rows, 0}
    int4 *tiles = nullptr;          // [tiles_max] {expert, first padded row, valid rows, 0}
    int64_t tiles_max = 0;
    int tile_rows = kTileRows;      // rows a tensor-core tile covers: 128 (W4A4) or 64 (W4A16)
    uint8_t *xp = nullptr;          // [rows_pad][H/2] permuted x codes (tensor-core path)
    uint8_t *xp_atoms = nullptr;    // [rows_pad/128][H/64][512] their scales, tensor-core layout
    uint8_t *hq_atoms = nullptr;    // [rows_pad/128][Imax/64][512] SwiGLU scales, tensor-core layout
    __half *xp16 = nullptr;         // [rows_pad][H] permuted x as f16 (W4A16 tensor-core path)
    CallScratch *scratch = nullptr;
    float *xts = nullptr;           // [2] x tensor scale, spare
    uint8_t *xq = nullptr;          // [Tmax][H/2]
    uint8_t *xsc = nullptr;         // [Tmax][H/16]
    float *hbuf = nullptr;          // [rows_pad][Imax] fp32 (W4A4) or bf16 (W4A16)
    uint8_t *hq = nullptr;          // [rows_pad][Imax/2]
    uint8_t *hsc = nullptr;         // [rows_pad][Imax/16]
    float *hts = nullptr;           // [2] h tensor scales (routed, shared)
    float *acc = nullptr;           // [Tmax][H] fp32 combine accumulator, kept zero between calls
    int32_t *group_blk = nullptr;      // [ceil(pairs_max / kGroupSeg)][E] per-block expert counts / first slots
    int32_t *tail_tickets = nullptr;   // [8 * num_sms] arrivals per split gate/up item and row group (per-call scratch)
    float *tail_part = nullptr;        // [num_sms][8192] partial gate/up sums of split items (W4A16 warp MMAs)
    int *err = nullptr;             // device error word
    float *ones = nullptr;          // [E + 1] 1.0f: the tensor scales of MXFP4 weights, which have none
    void *x_stage = nullptr;        // [Tmax][H] bf16 (moe_forward_host)
    void *out_stage = nullptr;      // [Tmax][H] bf16
};

// ------------------------------------------------------------- conversions

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Two E2M1 codes (one byte; element 0 in the low nibble) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(out) : "r"(byte));
    return out;
}

// Four E2M1x2 bytes of a word -> four f16x2 words (exact).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// Two E4M3 bytes (low byte = first) -> f16x2 (exact: E4M3 fits f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t out;
    asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(out) : "r"(two_bytes));
    return out;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// fp32 -> E4M3 byte (sign kept), round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float v) {
    uint32_t out;
    asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
        : "=r"(out) : "f"(v), "f"(0.0f));
    return out & 0xFFu;
}

// Two fp32 -> one byte of two E2M1 codes (lo -> bits 0..3, hi -> bits 4..7),
// round to nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(out) : "f"(lo), "f"(hi));
    return out & 0xFFu;
}

// NVFP4 quantisation of one 16-value block with tensor scale ts, in the
// fixed fp32 order: s = E4M3((amax/6)/ts); den = E4M3(s)*ts; code = E2M1(v/den).
__device__ __forceinline__ void quant_block16(const float (&v)[16], float ts, uint2 &codes, uint32_t &scale) {
    float bamax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
    uint32_t s = 0;
    if (ts != 0.0f) s = f32_to_e4m3_sat(__fdiv_rn(__fdiv_rn(bamax, 6.0f), ts));
    const float den = __fmul_rn(e4m3_to_f32(s), ts);
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        b[i] = (den == 0.0f) ? 0u : f32x2_to_e2m1x2(__fdiv_rn(v[2 * i], den), __fdiv_rn(v[2 * i + 1], den));
    }
    codes.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    codes.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    scale = s;
}

// MXFP4 (OCP MX) conversion of one 32-value block: E8M0 scale byte
// s = clamp(floor(log2(amax)) - 2 + 127, 0, 254) (0 for an all-zero block),
// codes = E2M1_rne_sat(v * 2^(127 - s)), a multiplication by a power of two
// that is exact.  For a normal amax floor(log2(amax)) + 127 is its biased
// exponent field, so s = max(field - 2, 0); a subnormal amax gives s = 0.
__device__ __forceinline__ void quant_block32_mx(const float (&v)[32], uint4 &codes, uint32_t &scale) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int field = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    const int s = field > 2 ? field - 2 : 0;
    const float inv = __uint_as_float((uint32_t)(254 - s) << 23);   // 2^(127 - s), s <= 252
    uint32_t b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = f32x2_to_e2m1x2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv));
    codes.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    codes.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    codes.z = b[8] | (b[9] << 8) | (b[10] << 16) | (b[11] << 24);
    codes.w = b[12] | (b[13] << 8) | (b[14] << 16) | (b[15] << 24);
    scale = (uint32_t)s;
}

// E8M0 byte -> fp32 2^(byte - 127) (byte 0: the subnormal 2^-127; 255: NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte) {
    byte &= 0xFFu;
    if (byte == 0) return __uint_as_float(0x00400000u);
    if (byte == 255) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(byte << 23);
}

__device__ __forceinline__ void atomic_max_nonneg(unsigned int *addr, float v) {
    atomicMax(addr, __float_as_uint(v));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// ------------------------------------------------- mbarrier / bulk copies

constexpr uint64_t kWaitNs = 1000000000ull;  // bound on any single mbarrier wait

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Explicit shared-memory accesses (32-bit shared addresses), for buffers whose
// pointer the compiler cannot trace back to shared memory.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity; false (and the timeout
// bit set) if it has not completed within `limit_ns` (kWaitNs by default).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err, uint64_t limit_ns = kWaitNs) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!mbar_test(bar, parity)) {
        if (now_ns() - t0 > limit_ns) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the previous kernel in the stream is finishing; it calls pdl_wait()
// before it reads anything that kernel wrote (the wait returns once that
// kernel has completed and its writes are visible; without the launch
// attribute it returns at once), then pdl_trigger() so that the next kernel's
// launch can overlap this one in turn.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------ launchers

struct ExpertPtrs {
    const uint8_t *gc, *gs, *uc, *us, *dc, *ds;
    const float *gts, *uts, *dts;
};

int router_launches(int T);
bool router_groups(int T);
cudaError_t launch_router(const Plan &p, const void *x, int T, const void *rw, const float *bias,
                          int32_t *ids, float *wts, cudaStream_t st, bool with_group = false);
int group_launches(const Plan &p, int T);
cudaError_t launch_group(const Plan &p, int T, const int32_t *ids, int32_t *offsets_out,
                         int32_t *sorted_out, bool build_work, cudaStream_t st);
cudaError_t launch_quant_act(const Plan &p, const void *x, int T, uint8_t *codes, uint8_t *scales,
                             float *ts_out, bool amax_ready, cudaStream_t st);
cudaError_t launch_quant_nvfp4(const float *w, int batch, int rows, int cols, uint8_t *codes, uint8_t *scales,
                               float *ts, cudaStream_t st);
cudaError_t launch_quant_mxfp4(const float *w, int64_t rows, int cols, uint8_t *codes, uint8_t *scales,
                               cudaStream_t st);
// part 0: gate + up + SwiGLU; part 1: down + routing weight + scatter-add.
cudaError_t launch_ffn_simt(const Plan &p, const void *x, int T, const ExpertPtrs &routed,
                            const ExpertPtrs *shared, int part, cudaStream_t st);
cudaError_t launch_quant_h(const Plan &p, bool tc_layout, cudaStream_t st);
cudaError_t launch_convert(const float *src, int64_t n, int format, uint8_t *dst, cudaStream_t st);
cudaError_t launch_finalize(const Plan &p, int T, void *out, cudaStream_t st);
cudaError_t launch_wait_check(int *err, uint64_t limit_ns, cudaStream_t st);

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
