// Router and grouping kernels.
//
// Router ("NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4
// Round 1: router logits in fp32 on a shared tile, #763; "bloomery 0.3.9",
// From our contributors: normalisation policy as a named value, #772).
// Grouping (same page and section, #740: a whole batch is routed in one run so
// each routed expert's weights are read once).
#include "moe_internal.cuh"

namespace moe {
namespace {

// Logits in the fixed order: lane l of a warp owns the 8-value chunks c of H
// with c mod 32 == l and sums fmaf over them in increasing h; the lane sums are
// combined with an xor butterfly (16, 8, 4, 2, 1); the bias is added last.
// A warp computes a TT x TE tile (tokens x experts); the block holds 4 warps
// side by side along the experts.  The blocks with blockIdx.x == 0 also check
// that x is finite and, for W4A4, fold x into the batch amax.
template <int TT, int TE>
__global__ void __launch_bounds__(128) k_router_logits(const uint16_t *__restrict__ x, int T, int H,
                                                       const float *__restrict__ rw, const float *__restrict__ bias,
                                                       int E, float *__restrict__ logits, int *err,
                                                       unsigned int *x_amax) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int e0 = (blockIdx.x * 4 + warp) * TE;
    const int t0 = blockIdx.y * TT;
    const bool check = (blockIdx.x == 0);
    float acc[TT][TE];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int e = 0; e < TE; ++e) acc[t][e] = 0.0f;
    bool bad = false;
    float amax = 0.0f;
    const int nchunk = H >> 3;
    for (int c = lane; c < nchunk; c += 32) {
        float w[TE][8];
#pragma unroll
        for (int e = 0; e < TE; ++e) {
            if (e0 + e < E) {
                const float4 *p = reinterpret_cast<const float4 *>(rw + (size_t)(e0 + e) * H + c * 8);
                float4 a = __ldg(p), b = __ldg(p + 1);
                w[e][0] = a.x; w[e][1] = a.y; w[e][2] = a.z; w[e][3] = a.w;
                w[e][4] = b.x; w[e][5] = b.y; w[e][6] = b.z; w[e][7] = b.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) w[e][j] = 0.0f;
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            if (t0 + t >= T) continue;
            uint4 q = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + t) * H + c * 8));
            uint32_t u[4] = {q.x, q.y, q.z, q.w};
            float xv[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xv[2 * j] = __uint_as_float(u[j] << 16);
                xv[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                if (check) {
                    bad |= ((u[j] & 0x7F80u) == 0x7F80u) | ((u[j] & 0x7F800000u) == 0x7F800000u);
                    amax = fmaxf(amax, fmaxf(fabsf(xv[2 * j]), fabsf(xv[2 * j + 1])));
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < TE; ++e) acc[t][e] = fmaf(xv[j], w[e][j], acc[t][e]);
        }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int e = 0; e < TE; ++e) {
            float v = acc[t][e];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
            acc[t][e] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < TE; ++e)
                if (t0 + t < T && e0 + e < E) {
                    float v = acc[t][e];
                    if (bias) v = v + bias[e0 + e];
                    logits[(size_t)(t0 + t) * E + e0 + e] = v;
                }
    }
    if (check && warp == 0) {
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kErrNonFinite);
        if (x_amax) {
            amax = warp_max(amax);
            if (lane == 0) atomic_max_nonneg(x_amax, amax);
        }
    }
}

// One warp per token: top-k by logit (ties -> lower id), then the weights.
// NPL logits per lane (expert lane + 32*i).
template <int NPL>
__global__ void __launch_bounds__(128) k_router_topk(const float *__restrict__ logits, int T, int E, int k,
                                                     int kind, int renorm, int32_t *__restrict__ ids,
                                                     float *__restrict__ wts, int32_t *__restrict__ counts,
                                                     int *err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t >= T) return;
    const float NEG = -__int_as_float(0x7f800000);
    float v[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? logits[(size_t)t * E + e] : NEG;
    }
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        if (lane + 32 * i >= E) taken |= 1u << i;
    float mine = 0.0f;  // lane j keeps the logit of slot j
    for (int j = 0; j < k; ++j) {
        float bv = NEG;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if (taken & (1u << i)) continue;
            int e = lane + 32 * i;
            if (bi == 0x7fffffff || v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            bool take = (oi != 0x7fffffff) && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
            if (take) { bv = ov; bi = oi; }
        }
        if (bi == 0x7fffffff || bi >= E) {  // only NaN logits left
            if (lane == 0) atomicOr(err, kErrDevice);
            bi = 0;
            bv = 0.0f;
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) mine = bv;
        if (lane == 0) {
            ids[(size_t)t * k + j] = bi;
            if (counts) atomicAdd(counts + bi, 1);
        }
    }
    float num = 0.0f, den;
    if (kind == MOE_ROUTER_SOFTMAX) {
        float m = NEG;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (lane + 32 * i < E) m = fmaxf(m, v[i]);
        m = warp_max(m);
        num = (lane < k) ? expf(mine - m) : 0.0f;
        if (renorm) {
            den = warp_sum(num);
        } else {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (lane + 32 * i < E) s += expf(v[i] - m);
            den = warp_sum(s);
        }
    } else {
        num = (lane < k) ? 1.0f / (1.0f + expf(-mine)) : 0.0f;
        den = renorm ? warp_sum(num) : 1.0f;
    }
    if (lane < k) wts[(size_t)t * k + lane] = num / den;
}

// Single-block grouping (1024 threads).  Stable counting sort of the pairs
// p = t*k + j by expert: each of the 32 warps owns a contiguous segment of
// pairs, counts it per expert, the per-(warp, expert) bases are scanned, and a
// second walk places every pair (ranks within a warp come from match_any, so
// the order inside an expert is increasing p).  Also writes the padded row
// layout used by the expert kernels and their work lists.
__global__ void __launch_bounds__(1024) k_group(const int32_t *__restrict__ ids, int P, int E, int T, int k,
                                                int has_shared, const int32_t *__restrict__ counts,
                                                int32_t *__restrict__ offsets, int32_t *__restrict__ poff,
                                                int32_t *__restrict__ sorted, int32_t *__restrict__ inv,
                                                int32_t *__restrict__ pad_pair, int4 *__restrict__ chunks,
                                                int4 *__restrict__ tiles,
                                                CallScratch *scratch, int32_t *__restrict__ offsets_out,
                                                int32_t *__restrict__ sorted_out, int build_work, int rows_cap,
                                                int *err) {
    extern __shared__ int smem[];
    int *wc = smem;                        // [32][E]
    int *s_off = smem + 32 * E;            // [E+1]
    int *s_poff = s_off + (E + 1);         // [E+2]
    int *s_cb = s_poff + (E + 2);          // [E+2] chunk bases
    int *s_tb = s_cb + (E + 2);            // [E+2] tile bases
    __shared__ int s_warp[32][3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int i = tid; i < 32 * E; i += 1024) wc[i] = 0;
    // exclusive scans over experts of (count, padded count, chunks)
    int c = 0, pc = 0, nc = 0;
    if (tid < E) {
        c = counts[tid];
        pc = (c + kTileRows - 1) / kTileRows * kTileRows;
        nc = (c + kChunkRows - 1) / kChunkRows;
    }
    int a = c, b = pc, d = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o),
            yd = __shfl_up_sync(0xffffffffu, d, o);
        if (lane >= o) { a += ya; b += yb; d += yd; }
    }
    if (lane == 31) { s_warp[warp][0] = a; s_warp[warp][1] = b; s_warp[warp][2] = d; }
    __syncthreads();
    if (warp == 0) {
        int wa = s_warp[lane][0], wb = s_warp[lane][1], wd = s_warp[lane][2];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int ya = __shfl_up_sync(0xffffffffu, wa, o), yb = __shfl_up_sync(0xffffffffu, wb, o),
                yd = __shfl_up_sync(0xffffffffu, wd, o);
            if (lane >= o) { wa += ya; wb += yb; wd += yd; }
        }
        s_warp[lane][0] = wa; s_warp[lane][1] = wb; s_warp[lane][2] = wd;
    }
    __syncthreads();
    const int ba = warp ? s_warp[warp - 1][0] : 0, bb = warp ? s_warp[warp - 1][1] : 0,
              bd = warp ? s_warp[warp - 1][2] : 0;
    if (tid < E) {
        s_off[tid] = ba + a - c;
        s_poff[tid] = bb + b - pc;
        s_cb[tid] = bd + d - nc;
        s_tb[tid] = (bb + b - pc) / kTileRows;   // a padded segment holds count/128 (rounded up) tiles
    }
    if (tid == 0) {
        int tot_a = s_warp[31][0], tot_b = s_warp[31][1], tot_d = s_warp[31][2];
        s_off[E] = tot_a;
        s_poff[E] = tot_b;
        s_poff[E + 1] = tot_b + (has_shared ? (T + kTileRows - 1) / kTileRows * kTileRows : 0);
        s_cb[E] = tot_d;
        s_cb[E + 1] = tot_d + (has_shared ? (T + kChunkRows - 1) / kChunkRows : 0);
        s_tb[E] = tot_b / kTileRows;
        s_tb[E + 1] = s_poff[E + 1] / kTileRows;
        if (tot_a != P) atomicOr(err, kErrDevice);
    }
    __syncthreads();
    for (int i = tid; i <= E; i += 1024) {
        offsets[i] = s_off[i];
        if (offsets_out) offsets_out[i] = s_off[i];
    }
    for (int i = tid; i <= E + 1; i += 1024) poff[i] = s_poff[i];

    // pass 1: per-warp segment counts
    const int seg = ((P + 31) / 32 + 31) / 32 * 32;
    const int p_beg = warp * seg, p_end = min(P, p_beg + seg);
    for (int base = p_beg; base < p_end; base += 32) {
        int p = base + lane;
        int e = (p < p_end) ? ids[p] : -1 - lane;
        if (p < p_end && (e < 0 || e >= E)) { atomicOr(err, kErrDevice); e = -1 - lane; }
        unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wc[warp * E + e] += __popc(peers);
    }
    __syncthreads();
    // per-expert scan over warps
    for (int e = tid; e < E; e += 1024) {
        int run = s_off[e];
        for (int w = 0; w < 32; ++w) {
            int t = wc[w * E + e];
            wc[w * E + e] = run;
            run += t;
        }
    }
    __syncthreads();
    // pass 2: place
    for (int base = p_beg; base < p_end; base += 32) {
        int p = base + lane;
        int e = (p < p_end) ? ids[p] : -1 - lane;
        if (e >= E) e = -1 - lane;
        unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = wc[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) wc[warp * E + e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            int prow = s_poff[e] + (pos - s_off[e]);
            if (pos >= P || prow >= rows_cap) {  // inconsistent counts: refuse, never write out of range
                atomicOr(err, kErrDevice);
                continue;
            }
            sorted[pos] = p;
            if (sorted_out) sorted_out[pos] = p;
            inv[p] = prow;
            pad_pair[prow] = p;
        }
    }
    if (!build_work) return;
    if (s_poff[E + 1] > rows_cap) {
        if (tid == 0) atomicOr(err, kErrDevice);
        return;
    }
    // padding rows and the shared expert's rows
    for (int e = warp; e < E; e += 32) {
        int cnt = s_off[e + 1] - s_off[e];
        int pend = s_poff[e + 1] - s_poff[e];
        for (int q = cnt + lane; q < pend; q += 32) pad_pair[s_poff[e] + q] = -1;
    }
    if (has_shared) {
        int sh_rows = s_poff[E + 1] - s_poff[E];
        for (int q = tid; q < sh_rows; q += 1024) pad_pair[s_poff[E] + q] = (q < T) ? P + q : -1;
    }
    // CUDA-core work chunks: up to kChunkRows rows of one expert each
    for (int e = tid; e <= E; e += 1024) {
        int cnt = (e < E) ? s_off[e + 1] - s_off[e] : (has_shared ? T : 0);
        int cb = s_cb[e];
        for (int q = 0; q * kChunkRows < cnt; ++q)
            chunks[cb + q] = make_int4(e, s_poff[e] + q * kChunkRows, min(kChunkRows, cnt - q * kChunkRows), 0);
    }
    // tensor-core tiles: 128 padded rows of one expert each
    for (int e = tid; e <= E; e += 1024) {
        int cnt = (e < E) ? s_off[e + 1] - s_off[e] : (has_shared ? T : 0);
        int tb = s_tb[e];
        for (int q = 0; q * kTileRows < cnt; ++q)
            tiles[tb + q] = make_int4(e, s_poff[e] + q * kTileRows, min(kTileRows, cnt - q * kTileRows), 0);
    }
    if (tid == 0) {
        scratch->n_tiles = s_tb[E + 1];
        scratch->n_chunks = s_cb[E + 1];
        int na = 0;
        for (int e = 0; e < E; ++e) na += (s_off[e + 1] > s_off[e]);
        scratch->n_active = na;
    }
}

}  // namespace

cudaError_t launch_router(const Plan &p, const void *x, int T, const float *rw, const float *bias, int32_t *ids,
                          float *wts, cudaStream_t st) {
    const int H = p.cfg.hidden, E = p.cfg.num_experts;
    unsigned int *amax = (p.cfg.mode == MOE_W4A4) ? &p.scratch->x_amax : nullptr;
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    if (T <= 4) {
        dim3 g((E + 3) / 4, (T + 3) / 4);
        k_router_logits<4, 1><<<g, 128, 0, st>>>(xb, T, H, rw, bias, E, p.logits, p.err, amax);
    } else if (T <= 16) {
        dim3 g((E + 3) / 4, (T + 15) / 16);
        k_router_logits<16, 1><<<g, 128, 0, st>>>(xb, T, H, rw, bias, E, p.logits, p.err, amax);
    } else {
        dim3 g((E + 31) / 32, (T + 7) / 8);
        k_router_logits<8, 8><<<g, 128, 0, st>>>(xb, T, H, rw, bias, E, p.logits, p.err, amax);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int k = p.cfg.top_k;
    const int npl = (E + 31) / 32;
    dim3 g((T + 3) / 4);
#define MOE_TOPK(N) k_router_topk<N><<<g, 128, 0, st>>>(p.logits, T, E, k, p.cfg.router, p.cfg.renormalize, ids, wts, p.counts, p.err)
    if (npl <= 1) MOE_TOPK(1);
    else if (npl <= 2) MOE_TOPK(2);
    else if (npl <= 4) MOE_TOPK(4);
    else if (npl <= 8) MOE_TOPK(8);
    else if (npl <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    return cudaGetLastError();
}

size_t group_smem_bytes(int E) { return sizeof(int) * (32 * (size_t)E + 4 * (size_t)E + 8); }

cudaError_t configure_group_kernel(int E) {
    return cudaFuncSetAttribute(k_group, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)group_smem_bytes(E));
}

cudaError_t launch_group(const Plan &p, int T, const int32_t *ids, int32_t *offsets_out, int32_t *sorted_out,
                         bool build_work, cudaStream_t st) {
    const int E = p.cfg.num_experts, k = p.cfg.top_k;
    size_t smem = group_smem_bytes(E);
    k_group<<<1, 1024, smem, st>>>(ids, T * k, E, T, k, p.cfg.has_shared, p.counts, p.offsets, p.poff, p.sorted,
                                   p.inv, p.pad_pair, p.chunks, p.tiles, p.scratch, offsets_out, sorted_out,
                                   build_work ? 1 : 0, (int)p.rows_pad_max, p.err);
    return cudaGetLastError();
}

}  // namespace moe
