// Decode-shaped expert FFN on the CUDA cores: each expert's NVFP4 weight rows
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

// Row-major [kChunkRows][K] fp32 tile in shared memory with 16-byte chunks
// xor-swizzled inside each group of 8, so a warp reading one 32-value unit per
// lane (unit u = lane + 32m) hits distinct banks.
__device__ __forceinline__ int swz(int k) {
    int q = k >> 2;
    q = (q & ~7) | ((q ^ (q >> 3)) & 7);
    return (q << 2) | (k & 3);
}

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
template <int NR>
__device__ __forceinline__ void unit_dot(const uint4 &c, uint32_t sp, const float *xs, int K, int u,
                                         float (&acc)[kChunkRows]) {
    const float2 scf = f16x2_to_f32x2(e4m3x2_to_f16x2(sp));
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
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
        const int kbase = u * 32 + blk * 16;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float *row = xs + r * K;
            float2 p = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 xv = *reinterpret_cast<const float4 *>(row + swz(kbase + 4 * j));
                p = ffma2(w[2 * j], make_float2(xv.x, xv.y), p);
                p = ffma2(w[2 * j + 1], make_float2(xv.z, xv.w), p);
            }
            acc[r] = fmaf(p.x + p.y, sc, acc[r]);
        }
    }
}

template <int MODE>
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
                const float sc = e4m3_to_f32(a.xsc[(size_t)tok * (H / 16) + b]);
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
            *reinterpret_cast<float4 *>(row + swz(b * 16 + 4 * j)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

// Rows of one weight-row pair (gate i, up i) for FPW features at a time: all
// loads of the wave are issued before any arithmetic.
template <int MODE, int UPL, int FPW, int NR>
__device__ __forceinline__ void gateup_rows(const FfnArgs &a, const ExpertPtrs &W, int e, int I, int i0, int i_end,
                                            const int4 &ch, const float *xs, float tsg, float tsu, float &lmax) {
    const int lane = threadIdx.x & 31;
    const int H = a.H, units = H / 32;
    for (int i = i0; i < i_end; i += FPW) {
        uint4 cg[FPW][UPL], cu[FPW][UPL];
        uint32_t sg[FPW][UPL], su[FPW][UPL];
#pragma unroll
        for (int f = 0; f < FPW; ++f) {
            const size_t row = (size_t)e * I + i + f;
            const uint8_t *gc = W.gc + row * (H / 2), *uc = W.uc + row * (H / 2);
            const uint8_t *gs = W.gs + row * (H / 16), *us = W.us + row * (H / 16);
#pragma unroll
            for (int m = 0; m < UPL; ++m) {
                const int u = lane + 32 * m;
                if (u < units) {
                    cg[f][m] = ldg_stream(gc + u * 16);
                    cu[f][m] = ldg_stream(uc + u * 16);
                    sg[f][m] = __ldg(reinterpret_cast<const unsigned short *>(gs + u * 2));
                    su[f][m] = __ldg(reinterpret_cast<const unsigned short *>(us + u * 2));
                }
            }
        }
#pragma unroll
        for (int f = 0; f < FPW; ++f) {
            float ag[kChunkRows], au[kChunkRows];
#pragma unroll
            for (int r = 0; r < kChunkRows; ++r) ag[r] = au[r] = 0.0f;
#pragma unroll
            for (int m = 0; m < UPL; ++m) {
                const int u = lane + 32 * m;
                if (u < units) {
                    unit_dot<NR>(cg[f][m], sg[f][m], xs, H, u, ag);
                    unit_dot<NR>(cu[f][m], su[f][m], xs, H, u, au);
                }
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
                const size_t hrow = (size_t)(ch.y + lane) * a.hstride + i + f;
                if (MODE == MOE_W4A16) {
                    static_cast<__nv_bfloat16 *>(a.hbuf)[hrow] = __float2bfloat16_rn(h);
                } else {
                    static_cast<float *>(a.hbuf)[hrow] = h;
                    lmax = fmaxf(lmax, fabsf(h));
                }
            }
        }
    }
}

// Gate + up + SwiGLU.  Item = (chunk, group of kFeatGroup features); each warp
// takes kFeatGroup / kWarps consecutive features.
template <int MODE, int UPL>
__global__ void __launch_bounds__(kWarps * 32) k_gateup_simt(FfnArgs a) {
    extern __shared__ float xs[];
    constexpr int FPW = UPL <= 4 ? 2 : 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Imax = max(a.I, a.Is);
    const int groups = (Imax + kFeatGroup - 1) / kFeatGroup;
    const int n_items = a.scratch->n_chunks * groups;
    const float xscale = (MODE == MOE_W4A4) ? __fdiv_rn(__uint_as_float(a.scratch->x_amax), 2688.0f) : 1.0f;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int4 ch = a.chunks[item / groups];
        const int fg = item % groups;
        const bool sh = (ch.x == a.E);
        const int I = sh ? a.Is : a.I;
        if (fg * kFeatGroup >= I) continue;
        __syncthreads();
        stage_x<MODE>(a, ch, xs);
        __syncthreads();
        const ExpertPtrs &W = sh ? a.s : a.r;
        const int e = sh ? 0 : ch.x;
        const float tsg = W.gts[e] * xscale, tsu = W.uts[e] * xscale;
        float lmax = 0.0f;
        const int i0 = fg * kFeatGroup + warp * (kFeatGroup / kWarps);
        const int i_end = min(i0 + kFeatGroup / kWarps, I);
        switch (ch.z) {
            case 1: gateup_rows<MODE, UPL, FPW, 1>(a, W, e, I, i0, i_end, ch, xs, tsg, tsu, lmax); break;
            case 2: gateup_rows<MODE, UPL, FPW, 2>(a, W, e, I, i0, i_end, ch, xs, tsg, tsu, lmax); break;
            case 3: gateup_rows<MODE, UPL, FPW, 3>(a, W, e, I, i0, i_end, ch, xs, tsg, tsu, lmax); break;
            default: gateup_rows<MODE, UPL, FPW, 4>(a, W, e, I, i0, i_end, ch, xs, tsg, tsu, lmax); break;
        }
        if (MODE == MOE_W4A4) {
            lmax = warp_max(lmax);
            if (lane == 0 && lmax > 0.0f) atomic_max_nonneg(sh ? a.hs_amax : a.h_amax, lmax);
        }
    }
}

template <int MODE>
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
                const float sc = e4m3_to_f32(a.hsc[row * (a.hstride / 16) + b]);
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
            *reinterpret_cast<float4 *>(rowp + swz(b * 16 + 4 * j)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

// Down rows j0 .. j0+RPW-1 for NR tokens: loads first, then arithmetic, then one
// atomic add per (row, token) of y * tensor scales * routing weight.
template <int UPL, int RPW, int NR>
__device__ __forceinline__ void down_rows(const FfnArgs &a, const ExpertPtrs &W, int e, int I, int j0,
                                          const float *hs, float scale, float wrow, int tok) {
    const int lane = threadIdx.x & 31;
    const int H = a.H, units = I / 32;
    uint4 c[RPW][UPL];
    uint32_t s[RPW][UPL];
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
        const size_t row = (size_t)e * H + j0 + q;
        const uint8_t *dc = W.dc + row * (I / 2), *ds = W.ds + row * (I / 16);
#pragma unroll
        for (int m = 0; m < UPL; ++m) {
            const int u = lane + 32 * m;
            if (u < units) {
                c[q][m] = ldg_stream(dc + u * 16);
                s[q][m] = __ldg(reinterpret_cast<const unsigned short *>(ds + u * 2));
            }
        }
    }
    float acc[RPW][kChunkRows];
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int r = 0; r < kChunkRows; ++r) acc[q][r] = 0.0f;
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int m = 0; m < UPL; ++m) {
            const int u = lane + 32 * m;
            if (u < units) unit_dot<NR>(c[q][m], s[q][m], hs, I, u, acc[q]);
        }
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[q][r] = warp_sum(acc[q][r]);
    // lane (q * NR + r) adds one value
    const int q = lane / NR, r = lane % NR;
    float y = 0.f;
#pragma unroll
    for (int qq = 0; qq < RPW; ++qq)
#pragma unroll
        for (int rr = 0; rr < NR; ++rr)
            if (qq == q && rr == r) y = acc[qq][rr];
    const float wr = __shfl_sync(0xffffffffu, wrow, r);
    const int tk = __shfl_sync(0xffffffffu, tok, r);
    if (q < RPW) atomicAdd(a.acc + (size_t)tk * H + j0 + q, y * scale * wr);
}

// Down + routing weight + scatter-add.  Item = (chunk, group of kFeatGroup
// output rows); a warp takes kFeatGroup / kWarps rows, RPW at a time.
template <int MODE, int UPL>
__global__ void __launch_bounds__(kWarps * 32) k_down_simt(FfnArgs a) {
    extern __shared__ float hs[];
    constexpr int RPW = UPL <= 2 ? 8 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H;
    const int groups = H / kFeatGroup;
    const int n_items = a.scratch->n_chunks * groups;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int4 ch = a.chunks[item / groups];
        const int og = item % groups;
        const bool sh = (ch.x == a.E);
        const int I = sh ? a.Is : a.I;
        __syncthreads();
        stage_h<MODE>(a, ch, I, hs);
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
        for (int q0 = 0; q0 < kFeatGroup / kWarps; q0 += RPW) {
            const int j0 = og * kFeatGroup + warp * (kFeatGroup / kWarps) + q0;
            switch (ch.z) {
                case 1: down_rows<UPL, RPW, 1>(a, W, e, I, j0, hs, scale, wrow, tok); break;
                case 2: down_rows<UPL, RPW, 2>(a, W, e, I, j0, hs, scale, wrow, tok); break;
                case 3: down_rows<UPL, RPW, 3>(a, W, e, I, j0, hs, scale, wrow, tok); break;
                default: down_rows<UPL, RPW, 4>(a, W, e, I, j0, hs, scale, wrow, tok); break;
            }
        }
    }
}

template <int MODE, int UPL>
cudaError_t launch_gateup(const FfnArgs &a, int grid, cudaStream_t st) {
    const size_t smem = sizeof(float) * kChunkRows * a.H;
    cudaError_t e = cudaFuncSetAttribute(k_gateup_simt<MODE, UPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_gateup_simt<MODE, UPL><<<grid, kWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

template <int MODE, int UPL>
cudaError_t launch_down(const FfnArgs &a, int grid, cudaStream_t st) {
    const size_t smem = sizeof(float) * kChunkRows * max(a.I, a.Is);
    cudaError_t e = cudaFuncSetAttribute(k_down_simt<MODE, UPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_down_simt<MODE, UPL><<<grid, kWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t run_mode(const FfnArgs &a, const Plan &p, int part, cudaStream_t st) {
    const int grid = p.num_sms * 4;
    if (part == 0) {
        const int upl_h = (a.H / 32 + 31) / 32;
        if (upl_h <= 1) return launch_gateup<MODE, 1>(a, grid, st);
        if (upl_h <= 2) return launch_gateup<MODE, 2>(a, grid, st);
        if (upl_h <= 4) return launch_gateup<MODE, 4>(a, grid, st);
        return launch_gateup<MODE, 8>(a, grid, st);
    }
    const int upl_i = (max(a.I, a.Is) / 32 + 31) / 32;
    if (upl_i <= 1) return launch_down<MODE, 1>(a, grid, st);
    if (upl_i <= 2) return launch_down<MODE, 2>(a, grid, st);
    if (upl_i <= 4) return launch_down<MODE, 4>(a, grid, st);
    return launch_down<MODE, 8>(a, grid, st);
}

}  // namespace

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
    a.r = routed;
    if (shared) a.s = *shared;
    else a.s = routed;
    return p.cfg.mode == MOE_W4A4 ? run_mode<MOE_W4A4>(a, p, part, st) : run_mode<MOE_W4A16>(a, p, part, st);
}

}  // namespace moe
