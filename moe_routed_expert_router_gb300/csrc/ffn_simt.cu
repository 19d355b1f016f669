// Decode-shaped expert FFN on the CUDA cores: each expert's NVFP4 (or MXFP4) weight rows
// are streamed once (128-bit loads of codes, 16-bit loads of scale pairs) for
// all the rows routed to it, E2M1 is decoded in registers, and the dot products
// run in fp32.  Work is a list of chunks (up to kChunkRows rows of one expert)
// built by the grouping kernel.
//
// "NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4 Round 1:
// routed NVFP4 experts on the card in decode with one tensor scale an expert
// (#517); a run of several tokens dots each selected expert's rows for all its
// slots (#808); E4M3 scales decoded in pairs (#884); several chunks' loads kept
// in flight (section 9, #511); the combine folded into the card sum (#701).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kFeatGroup = 128;  // features (gate/up) or output rows (down) per work item

// Activation tile in shared memory: kChunkRows rows of K fp32 values, each row
// stored chunk-major -- the 4-value chunk j (0..7) of 32-value unit u sits at
// float offset (j * (K / 32) + u) * 4 -- so a warp reading one unit per lane
// (u = lane + 32m) touches consecutive 16-byte words, with no per-load index
// arithmetic beyond a constant stride.
__device__ __forceinline__ int tile_pos(int k, int K) { return (((k & 31) >> 2) * (K >> 5) + (k >> 5)) * 4 + (k & 3); }

struct FfnArgs {
    const int4 *chunks;
    const CallScratch *scratch;
    int E, H, I, Is, P, k;
    const uint16_t *x;          // W4A16 activations [T][H]
    const uint8_t *xq;          // W4A4 codes [T][H/2]
    const uint8_t *xsc;         // W4A4 scales [T][H/16]
    const int32_t *pad_pair;
    const float *wts;           // routing weights [P]
    void *hbuf;                 // [rows][hstride]: bf16 (W4A16) or fp32 (W4A4)
    int hstride;
    const uint8_t *hq;          // W4A4 quantised h codes [rows][hstride/2]
    const uint8_t *hsc;         // [rows][hstride/16]
    const float *hts;           // [2] h tensor scales
    unsigned int *h_amax, *hs_amax;
    float *acc;                 // [T][H]
    int *err;                   // plan error word (bounded waits)
    ExpertPtrs r, s;
};

__device__ __forceinline__ int token_of(int pair, int P, int k) { return pair >= P ? pair - P : pair / k; }

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

// Dot of one 32-value unit (16 code bytes + 2 scale bytes) with NR activation
// rows held in shared memory (swizzled), accumulated into acc[].  The unit is
// decoded once (E2M1 -> f16x2 -> fp32 pairs) and used for all NR rows; the 16
// products of a scale block are summed in fp32 pairs, then scaled.
// MX (MXFP4 weights): one E8M0 scale byte for the whole 32-value unit.
template <int NR, int MX = 0>
__device__ __forceinline__ void unit_dot(const uint4 &c, uint32_t sp, const float *xs, int K, int u,
                                         float (&acc)[kChunkRows]) {
    const float2 scf = MX ? make_float2(e8m0_to_f32(sp), e8m0_to_f32(sp)) : f16x2_to_f32x2(e4m3x2_to_f16x2(sp));
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    const int cs = K >> 3;   // floats between chunk j and chunk j+1 of a unit (K/32 units x 4)
    const float *xu = xs + u * 4;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float2 w[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(words[blk * 2 + q], h);
#pragma unroll
            for (int j = 0; j < 4; ++j) w[q * 4 + j] = f16x2_to_f32x2(h[j]);
        }
        const float sc = blk ? scf.y : scf.x;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float *row = xu + r * K + blk * 4 * cs;
            float2 p = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 xv = *reinterpret_cast<const float4 *>(row + j * cs);
                p = ffma2(w[2 * j], make_float2(xv.x, xv.y), p);
                p = ffma2(w[2 * j + 1], make_float2(xv.z, xv.w), p);
            }
            acc[r] = fmaf(p.x + p.y, sc, acc[r]);
        }
    }
}

template <int MODE, int MX>
__device__ void stage_x(const FfnArgs &a, const int4 &ch, float *xs) {
    const int H = a.H;
    for (int idx = threadIdx.x; idx < ch.z * (H / 16); idx += blockDim.x) {
        const int r = idx / (H / 16), b = idx % (H / 16);
        float v[16];
        {
            const int tok = token_of(a.pad_pair[ch.y + r], a.P, a.k);
            if (MODE == MOE_W4A16) {
                const uint4 *p = reinterpret_cast<const uint4 *>(a.x + (size_t)tok * H + b * 16);
                uint4 q0 = p[0], q1 = p[1];
                uint32_t u[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[2 * j] = __uint_as_float(u[j] << 16);
                    v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            } else {
                const uint2 cw = *reinterpret_cast<const uint2 *>(a.xq + (size_t)tok * (H / 2) + b * 8);
                const float sc = MX ? e8m0_to_f32(a.xsc[(size_t)tok * (H / 32) + b / 2])
                                    : e4m3_to_f32(a.xsc[(size_t)tok * (H / 16) + b]);
                uint32_t h[8];
                e2m1x8_to_f16x8(cw.x, *reinterpret_cast<uint32_t(*)[4]>(h));
                e2m1x8_to_f16x8(cw.y, *reinterpret_cast<uint32_t(*)[4]>(h + 4));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float2 f = f16x2_to_f32x2(h[j]);
                    v[2 * j] = f.x * sc;
                    v[2 * j + 1] = f.y * sc;
                }
            }
        }
        float *row = xs + r * H;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4 *>(row + tile_pos(b * 16 + 4 * j, H)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

// Each warp streams its own contiguous weight rows into a ring of `slots`
// shared-memory slots with bulk copies (one mbarrier per slot, bounded
// waits); lanes then read one 32-value unit at a time from shared memory, so
// the bytes in flight do not depend on registers.
struct Ring {
    uint8_t *base;      // this warp's slots
    uint64_t *bars;     // this warp's slot barriers
    int slot_bytes, slots;
    __device__ __forceinline__ uint8_t *slot(int q) const { return base + (size_t)(q % slots) * slot_bytes; }
    __device__ __forceinline__ uint64_t *bar(int q) const { return bars + q % slots; }
    __device__ __forceinline__ uint32_t parity(int q) const { return (uint32_t)((q / slots) & 1); }
};

// Item of the gate/up kernel: (chunk, group of 128 features).  Routed chunks
// come first (I/128 groups each), then the shared expert's (Is/128 groups).
__device__ __forceinline__ int4 gateup_item(const FfnArgs &a, int item, int &fg) {
    const int nr = a.scratch->n_chunks_routed, gi = a.I / 128;
    if (item < nr * gi) {
        fg = item % gi;
        return a.chunks[item / gi];
    }
    const int j = item - nr * gi, gs = a.Is / 128;
    fg = j % gs;
    return a.chunks[nr + j / gs];
}

__device__ __forceinline__ int gateup_items(const FfnArgs &a) {
    const int nr = a.scratch->n_chunks_routed, ns = a.scratch->n_chunks - nr;
    return nr * (a.I / 128) + (a.Is ? ns * (a.Is / 128) : 0);
}

// Issue step q of a warp's gate/up stream (lane 0): feature
// fg*128 + warp*16 + (q % 16) of item q / 16's chunk, i.e. one gate row and one
// up row (codes + scales) into slot q.  Returns false past the last item.
template <int MX>
__device__ __forceinline__ bool gateup_issue(const FfnArgs &a, const Ring &rg, int q, int n_items, int nw, int warp) {
    const int per_warp = 128 / nw;
    const int item = blockIdx.x + (q / per_warp) * gridDim.x;
    if (item >= n_items) return false;
    int fg;
    const int4 ch = gateup_item(a, item, fg);
    const bool sh = (ch.x == a.E);
    const ExpertPtrs &W = sh ? a.s : a.r;
    const int I = sh ? a.Is : a.I, e = sh ? 0 : ch.x, H = a.H;
    const size_t row = (size_t)e * I + fg * 128 + warp * per_warp + q % per_warp;
    uint8_t *dst = rg.slot(q);
    uint64_t *bar = rg.bar(q);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int sb = MX ? H / 32 : H / 16;   // scale bytes a row
    mbar_expect_tx(bar, 2 * (H / 2) + 2 * sb);
    bulk_copy(dst, W.gc + row * (H / 2), H / 2, bar);
    bulk_copy(dst + H / 2, W.uc + row * (H / 2), H / 2, bar);
    bulk_copy(dst + H, W.gs + row * sb, sb, bar);
    bulk_copy(dst + H + sb, W.us + row * sb, sb, bar);
    return true;
}

template <int MODE, int NR, int MX>
__device__ __forceinline__ void gateup_compute(const FfnArgs &a, const uint8_t *slot, const int4 &ch, int i,
                                               const float *xs, float tsg, float tsu, float &lmax) {
    const int lane = threadIdx.x & 31;
    const int H = a.H, units = H / 32;
    float ag[kChunkRows], au[kChunkRows];
#pragma unroll
    for (int r = 0; r < kChunkRows; ++r) ag[r] = au[r] = 0.0f;
    for (int u = lane; u < units; u += 32) {
        const uint4 cg = *reinterpret_cast<const uint4 *>(slot + u * 16);
        const uint4 cu = *reinterpret_cast<const uint4 *>(slot + H / 2 + u * 16);
        uint32_t sg, su;
        if (MX) {
            sg = slot[H + u];
            su = slot[H + H / 32 + u];
        } else {
            sg = *reinterpret_cast<const unsigned short *>(slot + H + u * 2);
            su = *reinterpret_cast<const unsigned short *>(slot + H + H / 16 + u * 2);
        }
        unit_dot<NR, MX>(cg, sg, xs, H, u, ag);
        unit_dot<NR, MX>(cu, su, xs, H, u, au);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        ag[r] = warp_sum(ag[r]);
        au[r] = warp_sum(au[r]);
    }
    if (lane < NR) {
        float g = 0.f, uu = 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r)
            if (r == lane) { g = ag[r]; uu = au[r]; }
        g *= tsg;
        uu *= tsu;
        const float h = g / (1.0f + expf(-g)) * uu;
        const size_t hrow = (size_t)(ch.y + lane) * a.hstride + i;
        if (MODE == MOE_W4A16) {
            static_cast<__nv_bfloat16 *>(a.hbuf)[hrow] = __float2bfloat16_rn(h);
        } else {
            static_cast<float *>(a.hbuf)[hrow] = h;
            lmax = fmaxf(lmax, fabsf(h));
        }
    }
}

// Gate + up + SwiGLU.  Dynamic shared memory: x tile [kChunkRows][H] fp32,
// then nw warps x `slots` slots of (2 code rows + 2 scale rows), then the
// slot barriers.
template <int MODE, int MX>
__global__ void __launch_bounds__(512) k_gateup_stream(FfnArgs a, int slots) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int H = a.H;
    float *xs = reinterpret_cast<float *>(smem);
    const int slot_bytes = H + (MX ? H / 16 : H / 8);
    uint8_t *rings = smem + (size_t)kChunkRows * H * 4;
    uint64_t *bars = reinterpret_cast<uint64_t *>(rings + (size_t)nw * slots * slot_bytes);
    Ring rg{rings + (size_t)warp * slots * slot_bytes, bars + warp * slots, slot_bytes, slots};
    if (lane == 0)
        for (int s = 0; s < slots; ++s) mbar_init(rg.bars + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    const int n_items = gateup_items(a);
    const int per_warp = 128 / nw;
    // W4A4 activation tensor scale (MXFP4 activations have none)
    const float xscale = (MODE == MOE_W4A4 && !MX) ? __fdiv_rn(__uint_as_float(a.scratch->x_amax), 2688.0f) : 1.0f;
    int issued = 0;
    if (lane == 0)
        while (issued < slots && gateup_issue<MX>(a, rg, issued, n_items, nw, warp)) ++issued;
    issued = __shfl_sync(0xffffffffu, issued, 0);
    bool ok = true;
    int q = 0, done = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        int fg;
        const int4 ch = gateup_item(a, item, fg);
        const bool sh = (ch.x == a.E);
        const ExpertPtrs &W = sh ? a.s : a.r;
        const int e = sh ? 0 : ch.x;
        __syncthreads();
        stage_x<MODE, MX>(a, ch, xs);
        __syncthreads();
        const float tsg = W.gts[e] * xscale, tsu = W.uts[e] * xscale;
        float lmax = 0.0f;
        for (int f = 0; f < per_warp; ++f, ++q) {
            if (ok && !mbar_wait(rg.bar(q), rg.parity(q), a.err)) ok = false;
            if (ok) {
                done = q + 1;
                const uint8_t *slot = rg.slot(q);
                const int i = fg * 128 + warp * per_warp + f;
                switch (ch.z) {
                    case 1: gateup_compute<MODE, 1, MX>(a, slot, ch, i, xs, tsg, tsu, lmax); break;
                    case 2: gateup_compute<MODE, 2, MX>(a, slot, ch, i, xs, tsg, tsu, lmax); break;
                    case 3: gateup_compute<MODE, 3, MX>(a, slot, ch, i, xs, tsg, tsu, lmax); break;
                    default: gateup_compute<MODE, 4, MX>(a, slot, ch, i, xs, tsg, tsu, lmax); break;
                }
            }
            __syncwarp();
            if (lane == 0 && ok && issued == q + slots && gateup_issue<MX>(a, rg, issued, n_items, nw, warp)) ++issued;
            issued = __shfl_sync(0xffffffffu, issued, 0);
        }
        if (MODE == MOE_W4A4) {
            lmax = warp_max(lmax);
            if (lane == 0 && lmax > 0.0f) atomic_max_nonneg(sh ? a.hs_amax : a.h_amax, lmax);
        }
    }
    // after a timeout, wait (bounded) for copies still landing in this warp's slots
    for (int d = done; d < issued; ++d) mbar_wait(rg.bar(d), rg.parity(d), a.err);
}

template <int MODE, int MX>
__device__ void stage_h(const FfnArgs &a, const int4 &ch, int I, float *hs) {
    for (int idx = threadIdx.x; idx < ch.z * (I / 16); idx += blockDim.x) {
        const int r = idx / (I / 16), b = idx % (I / 16);
        float v[16];
        {
            const size_t row = (size_t)(ch.y + r);
            if (MODE == MOE_W4A16) {
                const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.hbuf) +
                                                                 row * a.hstride + b * 16);
                uint4 q0 = p[0], q1 = p[1];
                uint32_t u[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[2 * j] = __uint_as_float(u[j] << 16);
                    v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            } else {
                const uint2 cw = *reinterpret_cast<const uint2 *>(a.hq + row * (a.hstride / 2) + b * 8);
                const float sc = MX ? e8m0_to_f32(a.hsc[row * (a.hstride / 32) + b / 2])
                                    : e4m3_to_f32(a.hsc[row * (a.hstride / 16) + b]);
                uint32_t h[8];
                e2m1x8_to_f16x8(cw.x, *reinterpret_cast<uint32_t(*)[4]>(h));
                e2m1x8_to_f16x8(cw.y, *reinterpret_cast<uint32_t(*)[4]>(h + 4));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float2 f = f16x2_to_f32x2(h[j]);
                    v[2 * j] = f.x * sc;
                    v[2 * j + 1] = f.y * sc;
                }
            }
        }
        float *rowp = hs + r * I;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4 *>(rowp + tile_pos(b * 16 + 4 * j, I)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

// Down: item = (chunk, group of 128 output rows); warp w owns rows
// og*128 + w*rpw .. +rpw, streamed kDownRows rows per slot.
constexpr int kDownRows = 8;

template <int MX>
__device__ __forceinline__ bool down_issue(const FfnArgs &a, const Ring &rg, int q, int n_items, int nw, int warp) {
    const int steps = 128 / nw / kDownRows;
    const int item = blockIdx.x + (q / steps) * gridDim.x;
    if (item >= n_items) return false;
    const int groups = a.H / 128;
    const int4 ch = a.chunks[item / groups];
    const int og = item % groups;
    const bool sh = (ch.x == a.E);
    const ExpertPtrs &W = sh ? a.s : a.r;
    const int I = sh ? a.Is : a.I, e = sh ? 0 : ch.x;
    const size_t row = (size_t)e * a.H + og * 128 + warp * (128 / nw) + (q % steps) * kDownRows;
    uint8_t *dst = rg.slot(q);
    uint64_t *bar = rg.bar(q);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int sb = MX ? I / 32 : I / 16;   // scale bytes a row
    mbar_expect_tx(bar, kDownRows * (I / 2 + sb));
    bulk_copy(dst, W.dc + row * (I / 2), kDownRows * (I / 2), bar);
    bulk_copy(dst + kDownRows * (I / 2), W.ds + row * sb, kDownRows * sb, bar);
    return true;
}

template <int NR, int MX>
__device__ __forceinline__ void down_compute(const FfnArgs &a, const uint8_t *slot, int I, int j0, const float *hs,
                                             float scale, float wrow, int tok) {
    const int lane = threadIdx.x & 31;
    const int units = I / 32;
    float acc[kDownRows][kChunkRows];
#pragma unroll
    for (int q = 0; q < kDownRows; ++q)
#pragma unroll
        for (int r = 0; r < kChunkRows; ++r) acc[q][r] = 0.0f;
    for (int u = lane; u < units; u += 32) {
#pragma unroll
        for (int q = 0; q < kDownRows; ++q) {
            const uint4 c = *reinterpret_cast<const uint4 *>(slot + q * (I / 2) + u * 16);
            const uint32_t s = MX ? (uint32_t)slot[kDownRows * (I / 2) + q * (I / 32) + u]
                                  : *reinterpret_cast<const unsigned short *>(slot + kDownRows * (I / 2) + q * (I / 16) + u * 2);
            unit_dot<NR, MX>(c, s, hs, I, u, acc[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < kDownRows; ++q)
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[q][r] = warp_sum(acc[q][r]);
    const int q = lane / NR, r = lane % NR;
    float y = 0.f;
#pragma unroll
    for (int qq = 0; qq < kDownRows; ++qq)
#pragma unroll
        for (int rr = 0; rr < NR; ++rr)
            if (qq == q && rr == r) y = acc[qq][rr];
    const float wr = __shfl_sync(0xffffffffu, wrow, r);
    const int tk = __shfl_sync(0xffffffffu, tok, r);
    if (q < kDownRows) atomicAdd(a.acc + (size_t)tk * a.H + j0 + q, y * scale * wr);
}

template <int MODE, int MX>
__global__ void __launch_bounds__(256) k_down_stream(FfnArgs a, int slots) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int Imax = max(a.I, a.Is);
    float *hs = reinterpret_cast<float *>(smem);
    const int slot_bytes = kDownRows * (Imax / 2 + (MX ? Imax / 32 : Imax / 16));
    uint8_t *rings = smem + (size_t)kChunkRows * Imax * 4;
    uint64_t *bars = reinterpret_cast<uint64_t *>(rings + (size_t)nw * slots * slot_bytes);
    Ring rg{rings + (size_t)warp * slots * slot_bytes, bars + warp * slots, slot_bytes, slots};
    if (lane == 0)
        for (int s = 0; s < slots; ++s) mbar_init(rg.bars + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    const int groups = a.H / 128;
    const int n_items = a.scratch->n_chunks * groups;
    const int steps = 128 / nw / kDownRows;
    int issued = 0;
    if (lane == 0)
        while (issued < slots && down_issue<MX>(a, rg, issued, n_items, nw, warp)) ++issued;
    issued = __shfl_sync(0xffffffffu, issued, 0);
    bool ok = true;
    int q = 0, done = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int4 ch = a.chunks[item / groups];
        const int og = item % groups;
        const bool sh = (ch.x == a.E);
        const int I = sh ? a.Is : a.I;
        __syncthreads();
        stage_h<MODE, MX>(a, ch, I, hs);
        __syncthreads();
        const ExpertPtrs &W = sh ? a.s : a.r;
        const int e = sh ? 0 : ch.x;
        float scale = W.dts[e];
        if (MODE == MOE_W4A4) scale *= a.hts[sh ? 1 : 0];
        float wrow = 0.f;
        int tok = 0;
        if (lane < ch.z) {
            const int pair = a.pad_pair[ch.y + lane];
            tok = token_of(pair, a.P, a.k);
            wrow = sh ? 1.0f : a.wts[pair];
        }
        for (int st = 0; st < steps; ++st, ++q) {
            if (ok && !mbar_wait(rg.bar(q), rg.parity(q), a.err)) ok = false;
            if (ok) {
                done = q + 1;
                const uint8_t *slot = rg.slot(q);
                const int j0 = og * 128 + warp * (128 / nw) + st * kDownRows;
                switch (ch.z) {
                    case 1: down_compute<1, MX>(a, slot, I, j0, hs, scale, wrow, tok); break;
                    case 2: down_compute<2, MX>(a, slot, I, j0, hs, scale, wrow, tok); break;
                    case 3: down_compute<3, MX>(a, slot, I, j0, hs, scale, wrow, tok); break;
                    default: down_compute<4, MX>(a, slot, I, j0, hs, scale, wrow, tok); break;
                }
            }
            __syncwarp();
            if (lane == 0 && ok && issued == q + slots && down_issue<MX>(a, rg, issued, n_items, nw, warp)) ++issued;
            issued = __shfl_sync(0xffffffffu, issued, 0);
        }
    }
    for (int d = done; d < issued; ++d) mbar_wait(rg.bar(d), rg.parity(d), a.err);
}

constexpr size_t kSmemBudget = 227 * 1024;

// Largest (warps, slots) whose shared memory fits, preferring more warps
// (up to max_warps) and then deeper rings.
bool pick_config(size_t fixed, size_t slot_bytes, int max_warps, int &nw, int &slots) {
    for (int w : {16, 8, 4, 2}) {
        if (w > max_warps) continue;
        for (int s : {3, 2}) {
            const size_t need = fixed + (size_t)w * s * slot_bytes + (size_t)w * s * 8 + 128;
            if (need <= kSmemBudget) {
                nw = w;
                slots = s;
                return true;
            }
        }
    }
    return false;
}

// Fallback for wide rows: 8, 4 or 2 warps with a single slot each.
bool pick_config1(size_t fixed, size_t slot_bytes, int &nw, int &slots) {
    for (int w : {8, 4, 2}) {
        const size_t need = fixed + (size_t)w * slot_bytes + (size_t)w * 8 + 128;
        if (need <= kSmemBudget) {
            nw = w;
            slots = 1;
            return true;
        }
    }
    return false;
}

template <int MODE, int MX>
cudaError_t run_mode(const FfnArgs &a, const Plan &p, int part, cudaStream_t st) {
    int nw = 0, slots = 0;
    if (part == 0) {
        const size_t fixed = (size_t)kChunkRows * a.H * 4, slot = (size_t)a.H + (MX ? a.H / 16 : a.H / 8);
        if (!pick_config(fixed, slot, 16, nw, slots) && !pick_config1(fixed, slot, nw, slots))
            return cudaErrorInvalidValue;
        const size_t smem = fixed + (size_t)nw * slots * slot + (size_t)nw * slots * 8 + 128;
        k_gateup_stream<MODE, MX><<<p.num_sms, nw * 32, smem, st>>>(a, slots);
        return cudaGetLastError();
    }
    const int Imax = max(a.I, a.Is);
    const size_t fixed = (size_t)kChunkRows * Imax * 4,
                 slot = (size_t)kDownRows * (Imax / 2 + (MX ? Imax / 32 : Imax / 16));
    if (!pick_config(fixed, slot, 8, nw, slots) && !pick_config1(fixed, slot, nw, slots)) return cudaErrorInvalidValue;
    const size_t smem = fixed + (size_t)nw * slots * slot + (size_t)nw * slots * 8 + 128;
    k_down_stream<MODE, MX><<<p.num_sms, nw * 32, smem, st>>>(a, slots);
    return cudaGetLastError();
}

}  // namespace

// Shared-memory limits of the streamed kernels, set once (plan creation) so
// that moe_forward makes no configuration call and can be graph-captured.
cudaError_t configure_simt() {
    const int lim = (int)kSmemBudget;
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(k_gateup_stream<MOE_W4A16, 0>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gateup_stream<MOE_W4A4, 0>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_down_stream<MOE_W4A16, 0>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_down_stream<MOE_W4A4, 0>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gateup_stream<MOE_W4A16, 1>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gateup_stream<MOE_W4A4, 1>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_down_stream<MOE_W4A16, 1>, at, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_down_stream<MOE_W4A4, 1>, at, lim);
    return e;
}

cudaError_t launch_ffn_simt(const Plan &p, const void *x, int T, const ExpertPtrs &routed, const ExpertPtrs *shared,
                            int part, cudaStream_t st) {
    FfnArgs a{};
    a.chunks = p.chunks;
    a.scratch = p.scratch;
    a.E = p.cfg.num_experts;
    a.H = p.cfg.hidden;
    a.I = p.cfg.inter;
    a.Is = p.cfg.has_shared ? p.cfg.shared_inter : 0;
    a.P = T * p.cfg.top_k;
    a.k = p.cfg.top_k;
    a.x = static_cast<const uint16_t *>(x);
    a.xq = p.xq;
    a.xsc = p.xsc;
    a.pad_pair = p.pad_pair;
    a.wts = p.wts;
    a.hbuf = p.hbuf;
    a.hstride = max(a.I, a.Is);
    a.hq = p.hq;
    a.hsc = p.hsc;
    a.hts = p.hts;
    a.h_amax = &p.scratch->h_amax;
    a.hs_amax = &p.scratch->hs_amax;
    a.acc = p.acc;
    a.err = p.err;
    a.r = routed;
    if (shared) a.s = *shared;
    else a.s = routed;
    if (p.cfg.weight_format == MOE_WEIGHTS_MXFP4)
        return p.cfg.mode == MOE_W4A4 ? run_mode<MOE_W4A4, 1>(a, p, part, st) : run_mode<MOE_W4A16, 1>(a, p, part, st);
    return p.cfg.mode == MOE_W4A4 ? run_mode<MOE_W4A4, 0>(a, p, part, st) : run_mode<MOE_W4A16, 0>(a, p, part, st);
}

}  // namespace moe
