// Router and grouping kernels.
//
// Router ("NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4
// Round 1: router logits in fp32 on a shared tile, #763; "bloomery 0.3.9",
// From our contributors: normalisation policy as a named value, #772).
// Grouping (same page and section, #740: a whole batch is routed in one run so
// each routed expert's weights are read once).
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Logits in the fixed order: position h of H belongs to lane h mod 32 of a
// warp, which sums fmaf over its positions in increasing h starting from +0;
// the 32 lane sums are combined with an xor butterfly (16, 8, 4, 2, 1); the
// bias is added last.  Every kernel below keeps exactly this order, whatever
// its tiling: x and the router weight are staged in shared memory so that lane
// l reads position 32j + l of every 32-position group.

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ bool bf16x2_bad(uint32_t u) {
    return ((u & 0x7F80u) == 0x7F80u) | ((u & 0x7F800000u) == 0x7F800000u);
}

// Two independent IEEE fp32 FMAs (round to nearest) in one instruction:
// (a.x*b.x + c.x, a.y*b.y + c.y), each exactly fmaf.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    const uint32_t d = smem_u32(dst);
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}

// Large batches: a block computes 16 tokens x 32 experts with 8 warps (2 x 4
// sub-tiles of 8 x 8).  Slabs of 128 positions of x (bf16) and of the router
// rows (fp32) stream through a 4-deep cp.async ring in their natural layout;
// in slab j lane l reads position 32i + l (i < 4) of each of its 8 tokens and
// 8 experts, so every lane still walks h = l, l+32, l+64, ... in increasing
// order, and a warp's reads are 32 consecutive elements (no bank conflicts).
constexpr int kRT = 16, kRE = 32, kRSlab = 128, kRStages = 4;
constexpr int kRXBytes = kRT * kRSlab * 2;          // 4 KB
constexpr int kRWBytes = kRE * kRSlab * 4;          // 16 KB (fp32 router words; bf16 words use half)
constexpr int kRouterTiledSmem = kRStages * (kRXBytes + kRWBytes);

// A router weight word as fp32: fp32 as it is, bf16 widened (exact), so the
// logits keep the same fixed order and fp32 arithmetic whatever the word type.
__device__ __forceinline__ float rw_f32(float w) { return w; }
__device__ __forceinline__ float rw_f32(__nv_bfloat16 w) { return __uint_as_float((uint32_t)__bfloat16_as_ushort(w) << 16); }

template <typename W>
__global__ void __launch_bounds__(256, 2) k_router_tiled(const uint16_t *__restrict__ x, int T, int H,
                                                         const W *__restrict__ rw, const float *__restrict__ bias,
                                                         int E, float *__restrict__ logits, int *err,
                                                         unsigned int *x_amax) {
    extern __shared__ __align__(16) uint8_t rsmem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.y * kRT, e0 = blockIdx.x * kRE;
    const int tw = (warp >> 2) * 8, ew = (warp & 3) * 8;
    const int slabs = H / kRSlab;
    const bool check = (blockIdx.x == 0);
    constexpr int kWPer16 = 16 / sizeof(W);   // router words a 16-byte copy moves
    auto xs = [&](int b) { return reinterpret_cast<uint16_t *>(rsmem + b * (kRXBytes + kRWBytes)); };
    auto ws = [&](int b) { return reinterpret_cast<W *>(rsmem + b * (kRXBytes + kRWBytes) + kRXBytes); };
    auto load = [&](int s) {
        if (s < slabs) {
            const int b = s % kRStages;
            {   // x: 16 rows x 16 chunks of 8 bf16
                const int row = tid >> 4, c = tid & 15;
                const bool v = t0 + row < T;
                cp_async16(xs(b) + row * kRSlab + c * 8, x + (size_t)(v ? t0 + row : 0) * H + s * kRSlab + c * 8, v);
            }
            constexpr int kChunks = kRSlab / kWPer16;   // 16-byte chunks a router row of the slab
#pragma unroll
            for (int i = 0; i < kRE * kChunks / 256; ++i) {   // weights: 32 rows x kChunks chunks
                const int idx = tid + 256 * i, row = idx / kChunks, c = idx % kChunks;
                const bool v = e0 + row < E;
                cp_async16(ws(b) + row * kRSlab + c * kWPer16,
                           rw + (size_t)(v ? e0 + row : 0) * H + s * kRSlab + c * kWPer16, v);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float2 acc2[8][4];   // (token t, experts 2p and 2p+1): two chains in one packed FMA
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc2[t][p] = make_float2(0.0f, 0.0f);
    bool bad = false;
    float amax = 0.0f;
#pragma unroll
    for (int s = 0; s < kRStages - 1; ++s) load(s);
    for (int s = 0; s < slabs; ++s) {
        load(s + kRStages - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kRStages - 1) : "memory");
        __syncthreads();
        const uint16_t *xb = xs(s % kRStages);
        const W *wb = ws(s % kRStages);
        if (check && (warp & 3) == 0) {   // warps of expert sub-tile 0 check their tokens once
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (t0 + tw + t >= T) break;
#pragma unroll
                for (int i = 0; i < kRSlab / 32; ++i) {
                    const uint32_t u = xb[(tw + t) * kRSlab + 32 * i + lane];
                    bad |= (u & 0x7F80u) == 0x7F80u;
                    amax = fmaxf(amax, fabsf(__uint_as_float(u << 16)));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRSlab / 32; ++i) {
            const int h = 32 * i + lane;
            float xv[8];
            float2 wv[4];
#pragma unroll
            for (int t = 0; t < 8; ++t) xv[t] = __uint_as_float((uint32_t)xb[(tw + t) * kRSlab + h] << 16);
#pragma unroll
            for (int p = 0; p < 4; ++p)
                wv[p] = make_float2(rw_f32(wb[(ew + 2 * p) * kRSlab + h]), rw_f32(wb[(ew + 2 * p + 1) * kRSlab + h]));
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
                for (int p = 0; p < 4; ++p) acc2[t][p] = ffma2(make_float2(xv[t], xv[t]), wv[p], acc2[t][p]);
        }
        __syncthreads();
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    float acc[8][8];
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v = (e & 1) ? acc2[t][e >> 1].y : acc2[t][e >> 1].x;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
            acc[t][e] = v;
        }
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
        const int j = lane + 32 * k2, t = j >> 3, e = j & 7;
        float v = 0.f;
#pragma unroll
        for (int tt = 0; tt < 8; ++tt)
#pragma unroll
            for (int ee = 0; ee < 8; ++ee)
                if (tt == t && ee == e) v = acc[tt][ee];
        const int tg = t0 + tw + t, eg = e0 + ew + e;
        if (tg < T && eg < E) logits[(size_t)tg * E + eg] = bias ? v + bias[eg] : v;
    }
    if (check && (warp & 3) == 0) {
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kErrNonFinite);
        if (x_amax) {
            amax = warp_max(amax);
            if (lane == 0) atomic_max_nonneg(x_amax, amax);
        }
    }
}

// Order-preserving map of an fp32 logit to an unsigned key (larger logit ->
// larger key); NaN maps to 0, below every other value, and is never chosen.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t b = __float_as_uint(v);
    if (v != v) return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The logit a non-zero key came from (logit_key is a bijection off NaN).
__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Top-k of token t by logit (ties -> lower id), then the weights; one warp,
// NPL logits per lane (expert lane + 32*i).  Each round every lane offers its
// best remaining (key, id); redux.sync takes the warp's largest key, then the
// smallest id among the lanes offering it.  Logits are read through L2 (they
// may come from other blocks of the same launch).
template <int NPL>
__device__ __forceinline__ void topk_token(const float *__restrict__ logits, int t, int E, int k, int kind, int renorm,
                                           int32_t *__restrict__ ids, float *__restrict__ wts,
                                           int32_t *__restrict__ counts, int *err, int *s_ids_out = nullptr) {
    const int lane = threadIdx.x & 31;
    const float NEG = -__int_as_float(0x7f800000);
    float v[NPL];
    uint32_t key[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? __ldcg(logits + (size_t)t * E + e) : NEG;
        key[i] = (e < E) ? logit_key(v[i]) : 0u;
    }
    float mine = 0.0f;  // lane j keeps the logit and the expert of slot j
    int mine_id = 0;
    bool nan_left = false;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (key[i] > bk) { bk = key[i]; bi = lane + 32 * i; }   // i ascending: ties keep the lower id
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        int wi = (int)__reduce_min_sync(0xffffffffu, (bk == wk && wk != 0u) ? (uint32_t)bi : 0x7fffffffu);
        float wv;
        if (wk == 0u || wi >= E) {  // only NaN logits left
            nan_left = true;
            wi = 0;
            wv = 0.0f;
        } else {
            wv = key_logit(wk);   // the winner's logit, exactly
            if ((wi & 31) == lane) {
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if ((wi >> 5) == i) key[i] = 0u;
            }
        }
        if (lane == j) { mine = wv; mine_id = wi; }
    }
    if (nan_left && lane == 0) atomicOr(err, kErrDevice);
    if (lane < k) {
        ids[(size_t)t * k + lane] = mine_id;
        if (s_ids_out) s_ids_out[t * k + lane] = mine_id;   // the same block groups the pairs next
        if (counts) atomicAdd(counts + mine_id, 1);
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

// One warp per token.
template <int NPL>
__global__ void __launch_bounds__(128) k_router_topk(const float *__restrict__ logits, int T, int E, int k,
                                                     int kind, int renorm, int32_t *__restrict__ ids,
                                                     float *__restrict__ wts, int32_t *__restrict__ counts,
                                                     int *err) {
    const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_token<NPL>(logits, t, E, k, kind, renorm, ids, wts, counts, err);
}

// Outputs of the grouping step when it runs inside the decode router.
struct GroupArgs {
    int active;
    int32_t *offsets, *poff, *sorted, *inv, *pad_pair;
    int4 *chunks, *tiles;
    int rows_cap, tile_rows, has_shared;
};

__host__ __device__ __forceinline__ size_t group_small_smem(int E, int P) {
    return sizeof(int) * (5 * (size_t)(E + 2) + (size_t)P + 4 * 32);
}

// Grouping of the pairs of at most 32 tokens by one block (the decode
// router's last block), with the outputs of k_group: offsets, padded
// offsets, the stable order, the padded row map and the work lists. A token's
// top-k experts are distinct, so each expert gets a bit mask of its tokens:
// its population is the expert's count and the bits below token t give the
// rank of t's pair inside the expert (the stable order, increasing p). Every
// step is then one thread a pair or an expert. The padding rows of the map
// were set to -1 by every block of the launch before this one started.
__device__ __forceinline__ int *group_small_ids(int *sm, int E) { return sm + 5 * (E + 2); }

// ids == nullptr: the pairs' experts are already in group_small_ids(sm, E).
__device__ void group_small(const GroupArgs &g, const int32_t *__restrict__ ids, int P, int E, int T, int k,
                            int *sm, CallScratch *sc, int *err) {
    unsigned *s_mask = reinterpret_cast<unsigned *>(sm);
    int *s_off = sm + (E + 2), *s_poff = s_off + (E + 2), *s_cb = s_poff + (E + 2), *s_tb = s_cb + (E + 2),
        *s_ids = s_tb + (E + 2), *s_warp = s_ids + P;   // s_warp: [32][4] scan of the warp totals
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x, nwarps = nthr >> 5;
    if (T > 32) {   // masks hold 32 tokens; the decode router never groups more
        if (tid == 0) atomicOr(err, kErrDevice);
        return;
    }
    for (int i = tid; i < E; i += nthr) s_mask[i] = 0u;
    __syncthreads();
    for (int q = tid; q < P; q += nthr) {
        int e = ids ? ids[q] : s_ids[q];
        if (e < 0 || e >= E) { atomicOr(err, kErrDevice); e = -1; }
        s_ids[q] = e;
        if (e >= 0) atomicOr(&s_mask[e], 1u << (q / k));
    }
    __syncthreads();
    // exclusive scans over experts of (count, padded count, chunks, tiles):
    // thread tid sums experts [tid * per, tid * per + per), then warp and block scans
    const int per = (E + nthr - 1) / nthr, e0 = tid * per;
    int va = 0, vb = 0, vd = 0, vf = 0;
    for (int j = 0; j < per; ++j) {
        const int e = e0 + j;
        if (e < E) {
            const int c = __popc(s_mask[e]);
            va += c;
            vb += (c + kTileRows - 1) / kTileRows * kTileRows;
            vd += (c + kChunkRows - 1) / kChunkRows;
            vf += (c + g.tile_rows - 1) / g.tile_rows;
        }
    }
    int a = va, b = vb, d = vd, f = vf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o),
                  yd = __shfl_up_sync(0xffffffffu, d, o), yf = __shfl_up_sync(0xffffffffu, f, o);
        if (lane >= o) { a += ya; b += yb; d += yd; f += yf; }
    }
    if (lane == 31) { s_warp[4 * warp] = a; s_warp[4 * warp + 1] = b; s_warp[4 * warp + 2] = d; s_warp[4 * warp + 3] = f; }
    __syncthreads();
    if (warp == 0) {
        int wa = lane < nwarps ? s_warp[4 * lane] : 0, wb = lane < nwarps ? s_warp[4 * lane + 1] : 0,
            wd = lane < nwarps ? s_warp[4 * lane + 2] : 0, wf = lane < nwarps ? s_warp[4 * lane + 3] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, wa, o), yb = __shfl_up_sync(0xffffffffu, wb, o),
                      yd = __shfl_up_sync(0xffffffffu, wd, o), yf = __shfl_up_sync(0xffffffffu, wf, o);
            if (lane >= o) { wa += ya; wb += yb; wd += yd; wf += yf; }
        }
        __syncwarp();
        if (lane < nwarps) { s_warp[4 * lane] = wa; s_warp[4 * lane + 1] = wb; s_warp[4 * lane + 2] = wd; s_warp[4 * lane + 3] = wf; }
    }
    __syncthreads();
    {
        int ra = (warp ? s_warp[4 * (warp - 1)] : 0) + a - va, rb = (warp ? s_warp[4 * (warp - 1) + 1] : 0) + b - vb,
            rd = (warp ? s_warp[4 * (warp - 1) + 2] : 0) + d - vd, rf = (warp ? s_warp[4 * (warp - 1) + 3] : 0) + f - vf;
        for (int j = 0; j < per; ++j) {
            const int e = e0 + j;
            if (e < E) {
                const int c = __popc(s_mask[e]);
                s_off[e] = ra;
                s_poff[e] = rb;
                s_cb[e] = rd;
                s_tb[e] = rf;
                ra += c;
                rb += (c + kTileRows - 1) / kTileRows * kTileRows;
                rd += (c + kChunkRows - 1) / kChunkRows;
                rf += (c + g.tile_rows - 1) / g.tile_rows;
            }
        }
        if (tid == 0) {
            const int ta = s_warp[4 * (nwarps - 1)], tb = s_warp[4 * (nwarps - 1) + 1],
                      td = s_warp[4 * (nwarps - 1) + 2], tf = s_warp[4 * (nwarps - 1) + 3];
            s_off[E] = ta;
            s_poff[E] = tb;
            s_poff[E + 1] = tb + (g.has_shared ? (T + kTileRows - 1) / kTileRows * kTileRows : 0);
            s_cb[E] = td;
            s_cb[E + 1] = td + (g.has_shared ? (T + kChunkRows - 1) / kChunkRows : 0);
            s_tb[E] = tf;
            s_tb[E + 1] = tf + (g.has_shared ? (T + g.tile_rows - 1) / g.tile_rows : 0);
            if (ta != P) atomicOr(err, kErrDevice);
        }
    }
    __syncthreads();
    for (int i = tid; i <= E; i += nthr) g.offsets[i] = s_off[i];
    for (int i = tid; i <= E + 1; i += nthr) g.poff[i] = s_poff[i];
    if (s_poff[E + 1] > g.rows_cap) {   // inconsistent counts: refuse, never write out of range
        if (tid == 0) atomicOr(err, kErrDevice);
        return;
    }
    for (int q = tid; q < P; q += nthr) {   // placement: rank of the pair's token among the expert's tokens
        const int e = s_ids[q];
        if (e < 0) continue;
        const int r = __popc(s_mask[e] & ((1u << (q / k)) - 1u));
        const int pos = s_off[e] + r, prow = s_poff[e] + r;
        if (pos >= P || prow >= g.rows_cap) {
            atomicOr(err, kErrDevice);
        } else {
            g.sorted[pos] = q;
            g.inv[q] = prow;
            g.pad_pair[prow] = q;
        }
    }
    if (g.has_shared)
        for (int q = tid; q < T; q += nthr) g.pad_pair[s_poff[E] + q] = P + q;
    for (int e = tid; e <= E; e += nthr) {   // work lists, one thread an expert (at most 32 rows each)
        const int cnt = (e < E) ? __popc(s_mask[e]) : (g.has_shared ? T : 0);
        const int cb = s_cb[e], tb = s_tb[e];
        for (int q = 0; q * kChunkRows < cnt; ++q)
            g.chunks[cb + q] = make_int4(e, s_poff[e] + q * kChunkRows, min(kChunkRows, cnt - q * kChunkRows), 0);
        for (int q = 0; q * g.tile_rows < cnt; ++q)
            g.tiles[tb + q] = make_int4(e, s_poff[e] + q * g.tile_rows, min(g.tile_rows, cnt - q * g.tile_rows), 0);
    }
    if (tid == 0) {
        sc->n_tiles = s_tb[E + 1];
        sc->n_chunks = s_cb[E + 1];
        sc->n_chunks_routed = s_cb[E];
    }
}

// Decode-sized batches (T <= 16), router and top-k in one launch: a block
// computes the logits of one expert (two for T > 8 and an even E, so the x
// rows streamed through the block serve two experts and half as many blocks
// read them) for every token.  The router rows (H fp32 each) are staged in
// shared memory once; warp t streams token t's x row through its own 4-deep
// cp.async ring of 1024-position slabs (512 for T > 8; the last slab ragged;
// 16-byte copies, no block barrier), lane l taking positions 32j + l in
// increasing j, one fma chain an expert.  Each block also checks a slice of x
// (non-finite values, amax).  The last block to finish (a ticket in
// the per-call scratch) runs the top-k for all tokens, one warp a token, and,
// in moe_forward, groups the pairs (group_small).
constexpr int kDecodeRouterThreads = 512;
constexpr int kDSlab = 1024, kDStages = 4;

__host__ __device__ __forceinline__ int decode_slab(int T) { return T <= 8 ? kDSlab : kDSlab / 2; }

// Experts a block of the decode router takes.
__host__ __device__ __forceinline__ int decode_epb(int T, int E) { return (T > 8 && E % 2 == 0) ? 2 : 1; }

// wbytes: bytes of a router weight word (4 fp32, 2 bf16)
__host__ __device__ __forceinline__ size_t decode_router_smem(int H, int T, int E, int wbytes) {
    return (size_t)wbytes * H * decode_epb(T, E) + (size_t)kDStages * T * decode_slab(T) * 2;
}

template <int NPL, typename W>
__global__ void __launch_bounds__(kDecodeRouterThreads) k_router_decode(
    const uint16_t *__restrict__ x, int T, int H, const W *__restrict__ rw, const float *__restrict__ bias,
    int E, int k, int kind, int renorm, float *__restrict__ logits, int32_t *__restrict__ ids,
    float *__restrict__ wts, int32_t *__restrict__ counts, CallScratch *sc, int *err, GroupArgs grp) {
    pdl_trigger();   // the next kernel may be scheduled on free SMs (it waits for this one to finish)
    extern __shared__ __align__(16) uint8_t dsmem[];  // router rows [epb][H], per-token x rings [T][kDStages][slab] bf16, grouping
    W *wrow = reinterpret_cast<W *>(dsmem);
    constexpr int kWPer16 = 16 / sizeof(W);
    __shared__ float s_amax[kDecodeRouterThreads / 32];
    __shared__ int s_bad[kDecodeRouterThreads / 32];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int epb = decode_epb(T, E), e = blockIdx.x * epb;   // this block's experts: e .. e + epb - 1
    const int slab = decode_slab(T);
    const int slabs = (H + slab - 1) / slab;
    for (int c = tid; c < epb * H / kWPer16; c += kDecodeRouterThreads)
        cp_async16(wrow + kWPer16 * c, rw + (size_t)e * H + kWPer16 * c, true);
    asm volatile("cp.async.commit_group;" ::: "memory");
    uint16_t *ring = reinterpret_cast<uint16_t *>(wrow + (size_t)epb * H) + (size_t)warp * kDStages * slab;
    const uint16_t *xr = x + (size_t)warp * H;
    auto load_x = [&](int sl) {   // warp-private: lane l copies 16-byte chunks lane + 32i of the slab
        if (sl < slabs) {
            for (int i = 0; i < slab / 256; ++i) {
                const int c = lane + 32 * i;
                if (sl * slab + 8 * c < H) cp_async16(ring + (sl % kDStages) * slab + 8 * c, xr + sl * slab + 8 * c, true);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (warp < T) {
#pragma unroll
        for (int sl = 0; sl < kDStages - 1; ++sl) load_x(sl);
    }
    {   // this block's slice of x: non-finite check and amax
        const int nchunks = T * H / 8;
        const int per = (nchunks + gridDim.x - 1) / gridDim.x;
        const int c0 = blockIdx.x * per, c1 = min(nchunks, c0 + per);
        bool bad = false;
        float amax = 0.0f;
        for (int c = c0 + tid; c < c1; c += kDecodeRouterThreads) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(x) + c);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                bad |= bf16x2_bad(u[i]);
                amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        amax = warp_max(amax);
        if (lane == 0) { s_amax[warp] = amax; s_bad[warp] = bad; }
    }
    // the router row is the oldest commit group of every thread
    if (warp < T) asm volatile("cp.async.wait_group %0;" ::"n"(kDStages - 1) : "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        float m = lane < kDecodeRouterThreads / 32 ? s_amax[lane] : 0.0f;
        int b = lane < kDecodeRouterThreads / 32 ? s_bad[lane] : 0;
        m = warp_max(m);
        b = __any_sync(0xffffffffu, b);
        if (lane == 0) {
            if (b) atomicOr(err, kErrNonFinite);
            if (m > 0.0f) atomic_max_nonneg(&sc->x_amax, m);
        }
    }
    if (warp < T) {
        float acc = 0.0f, acc1 = 0.0f;   // experts e and e + 1 (the second when epb == 2)
        for (int sl = 0; sl < slabs; ++sl) {
            load_x(sl + kDStages - 1);
            asm volatile("cp.async.wait_group %0;" ::"n"(kDStages - 1) : "memory");
            __syncwarp();
            const uint16_t *xs = ring + (sl % kDStages) * slab;
            const W *wr = wrow + sl * slab, *wr1 = wr + H;
            const int len = min(slab, H - sl * slab);   // a multiple of 256
            if (epb == 2) {
#pragma unroll 2
                for (int j0 = 0; j0 < len / 32; j0 += 8) {   // loads of the group issue ahead of its FMA chains
                    uint32_t xv[8];
                    float wv[8], wv1[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        xv[j] = xs[32 * (j0 + j) + lane];
                        wv[j] = rw_f32(wr[32 * (j0 + j) + lane]);
                        wv1[j] = rw_f32(wr1[32 * (j0 + j) + lane]);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc = fmaf(__uint_as_float(xv[j] << 16), wv[j], acc);
                        acc1 = fmaf(__uint_as_float(xv[j] << 16), wv1[j], acc1);
                    }
                }
            } else {
#pragma unroll 4
                for (int j0 = 0; j0 < len / 32; j0 += 8) {   // loads of the group issue ahead of its FMA chain
                    uint32_t xv[8];
                    float wv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        xv[j] = xs[32 * (j0 + j) + lane];
                        wv[j] = rw_f32(wr[32 * (j0 + j) + lane]);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc = fmaf(__uint_as_float(xv[j] << 16), wv[j], acc);
                }
            }
            __syncwarp();   // every lane is done with the slot before it is refilled
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
            acc1 = acc1 + __shfl_xor_sync(0xffffffffu, acc1, o);
        }
        if (lane == 0) {
            logits[(size_t)warp * E + e] = bias ? acc + bias[e] : acc;
            if (epb == 2) logits[(size_t)warp * E + e + 1] = bias ? acc1 + bias[e + 1] : acc1;
        }
    }
    if (grp.active) {   // every row of the padded map starts as padding; the last block fills in the pairs
        const int per = (grp.rows_cap + (int)gridDim.x - 1) / (int)gridDim.x;
        const int r0 = (int)blockIdx.x * per, r1 = min(grp.rows_cap, r0 + per);
        for (int r = r0 + tid; r < r1; r += kDecodeRouterThreads) grp.pad_pair[r] = -1;
    }
    // release this block's logits and padding rows before its ticket; the last
    // block's acquire makes every block's visible to it
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&sc->route_done, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    // with the grouping in this block, the pairs' experts go to its shared
    // memory too (and no expert counts: the grouping counts from bit masks)
    int *gsm = reinterpret_cast<int *>(dsmem + decode_router_smem(H, T, E, (int)sizeof(W)));
    for (int t = warp; t < T; t += kDecodeRouterThreads / 32)
        topk_token<NPL>(logits, t, E, k, kind, renorm, ids, wts, grp.active ? nullptr : counts, err,
                        grp.active ? group_small_ids(gsm, E) : nullptr);
    if (grp.active) {
        __syncthreads();   // the block's ids are visible to all its threads
        group_small(grp, nullptr, T * k, E, T, k, gsm, sc, err);
    }
}

// Per-expert layout of a grouping, computed by one 1024-thread block from the
// expert counts (thread e < E holds count c of expert e): exclusive scans over
// experts of (count, count padded to kTileRows, CUDA-core chunks, tensor-core
// tiles) into s_off, s_poff, s_cb, s_tb, with the totals (and the shared
// expert's segment) at E and E + 1.
__device__ void group_scan_experts(int c, int E, int T, int P, int has_shared, int tile_rows, int *s_off,
                                   int *s_poff, int *s_cb, int *s_tb, int (*s_warp)[4], int *err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pc = (c + kTileRows - 1) / kTileRows * kTileRows, nc = (c + kChunkRows - 1) / kChunkRows,
              nt = (c + tile_rows - 1) / tile_rows;
    int a = c, b = pc, d = nc, f = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o),
            yd = __shfl_up_sync(0xffffffffu, d, o), yf = __shfl_up_sync(0xffffffffu, f, o);
        if (lane >= o) { a += ya; b += yb; d += yd; f += yf; }
    }
    if (lane == 31) { s_warp[warp][0] = a; s_warp[warp][1] = b; s_warp[warp][2] = d; s_warp[warp][3] = f; }
    __syncthreads();
    if (warp == 0) {
        int wa = s_warp[lane][0], wb = s_warp[lane][1], wd = s_warp[lane][2], wf = s_warp[lane][3];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int ya = __shfl_up_sync(0xffffffffu, wa, o), yb = __shfl_up_sync(0xffffffffu, wb, o),
                yd = __shfl_up_sync(0xffffffffu, wd, o), yf = __shfl_up_sync(0xffffffffu, wf, o);
            if (lane >= o) { wa += ya; wb += yb; wd += yd; wf += yf; }
        }
        s_warp[lane][0] = wa; s_warp[lane][1] = wb; s_warp[lane][2] = wd; s_warp[lane][3] = wf;
    }
    __syncthreads();
    const int ba = warp ? s_warp[warp - 1][0] : 0, bb = warp ? s_warp[warp - 1][1] : 0,
              bd = warp ? s_warp[warp - 1][2] : 0, bf = warp ? s_warp[warp - 1][3] : 0;
    if (tid < E) {
        s_off[tid] = ba + a - c;
        s_poff[tid] = bb + b - pc;
        s_cb[tid] = bd + d - nc;
        s_tb[tid] = bf + f - nt;
    }
    if (tid == 0) {
        int tot_a = s_warp[31][0], tot_b = s_warp[31][1], tot_d = s_warp[31][2], tot_f = s_warp[31][3];
        s_off[E] = tot_a;
        s_poff[E] = tot_b;
        s_poff[E + 1] = tot_b + (has_shared ? (T + kTileRows - 1) / kTileRows * kTileRows : 0);
        s_cb[E] = tot_d;
        s_cb[E + 1] = tot_d + (has_shared ? (T + kChunkRows - 1) / kChunkRows : 0);
        s_tb[E] = tot_f;
        s_tb[E + 1] = tot_f + (has_shared ? (T + tile_rows - 1) / tile_rows : 0);
        if (tot_a != P) atomicOr(err, kErrDevice);
    }
    __syncthreads();
}

// The expert (0..E, E = shared) whose entries [base[e], base[e + 1]) hold entry
// i: the largest e with base[e] <= i (experts without entries are skipped).
__device__ __forceinline__ int group_owner(const int *base, int E, int i) {
    int lo = 0, hi = E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (base[mid] <= i) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The padded row map's padding rows and the shared expert's rows, the
// CUDA-core work chunks (up to kChunkRows rows of one expert) and the
// tensor-core tiles (tile_rows padded rows of one expert, inside its
// 128-row-aligned segment), from a block's s_off / s_poff / s_cb / s_tb.
// Padding: one warp an expert, its lanes writing consecutive rows (fewer than
// kTileRows each); chunks and tiles: one thread an entry, its expert found by
// binary search, so a heavily routed expert's thousands of entries spread over
// the block (both keep the stores coalesced).
__device__ void group_build_work(int E, int T, int P, int has_shared, int tile_rows, const int *s_off,
                                 const int *s_poff, const int *s_cb, const int *s_tb, int32_t *__restrict__ pad_pair,
                                 int4 *__restrict__ chunks, int4 *__restrict__ tiles, CallScratch *scratch) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    for (int e = warp; e < E; e += nwarps) {
        const int cnt = s_off[e + 1] - s_off[e], pend = s_poff[e + 1] - s_poff[e];
        for (int q = cnt + lane; q < pend; q += 32) pad_pair[s_poff[e] + q] = -1;
    }
    if (has_shared) {
        int sh_rows = s_poff[E + 1] - s_poff[E];
        for (int q = tid; q < sh_rows; q += nthr) pad_pair[s_poff[E] + q] = (q < T) ? P + q : -1;
    }
    for (int i = tid; i < s_cb[E + 1]; i += nthr) {
        const int e = group_owner(s_cb, E, i), q = i - s_cb[e];
        const int cnt = (e < E) ? s_off[e + 1] - s_off[e] : T;
        chunks[i] = make_int4(e, s_poff[e] + q * kChunkRows, min(kChunkRows, cnt - q * kChunkRows), 0);
    }
    for (int i = tid; i < s_tb[E + 1]; i += nthr) {
        const int e = group_owner(s_tb, E, i), q = i - s_tb[e];
        const int cnt = (e < E) ? s_off[e + 1] - s_off[e] : T;
        tiles[i] = make_int4(e, s_poff[e] + q * tile_rows, min(tile_rows, cnt - q * tile_rows), 0);
    }
    if (tid == 0) {
        scratch->n_tiles = s_tb[E + 1];
        scratch->n_chunks = s_cb[E + 1];
        scratch->n_chunks_routed = s_cb[E];
    }
}

// Stable placement of the pairs [p_beg, p_end) of one block, split among its
// 32 warps in order: each warp counts its segment per expert (shared atomics),
// the per-(warp, expert) starts are scanned from base[e] (the block's first
// slot of expert e), and a second walk places every pair (ranks within a warp
// from match_any, so the order inside an expert is increasing p). match_any
// has a low throughput an SM, so rounds past the warp's segment are skipped.
// wc: [32][E] shared words.
__device__ void group_place(const int32_t *__restrict__ ids, int p_beg, int p_end, int P, int E, int *wc,
                            const int *base, const int *s_off, const int *s_poff, int32_t *__restrict__ sorted,
                            int32_t *__restrict__ sorted_out, int32_t *__restrict__ inv,
                            int32_t *__restrict__ pad_pair, int rows_cap, int *err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kPre = 8;   // rounds whose ids are loaded together (one L2 round trip for kPre rounds)
    const int n = p_end - p_beg, seg = ((n + 31) / 32 + 31) / 32 * 32;
    const int w_beg = p_beg + warp * seg, w_end = min(p_end, w_beg + seg);
    for (int base0 = w_beg; base0 < w_end; base0 += 32 * kPre) {
        int ev[kPre];
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int p = base0 + 32 * u + lane;
            ev[u] = (p < w_end) ? __ldg(ids + p) : -1 - lane;
        }
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int p = base0 + 32 * u + lane;
            const int e = ev[u];
            if (p < w_end) {
                if (e < 0 || e >= E) atomicOr(err, kErrDevice);
                else atomicAdd(&wc[warp * E + e], 1);
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {   // per-expert scan over warps
        int run = base[e];
        for (int w = 0; w < 32; ++w) {
            int t = wc[w * E + e];
            wc[w * E + e] = run;
            run += t;
        }
    }
    __syncthreads();
    for (int base0 = w_beg; base0 < w_end; base0 += 32 * kPre) {
        int ev[kPre];
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int p = base0 + 32 * u + lane;
            ev[u] = (p < w_end) ? __ldg(ids + p) : -1 - lane;
        }
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            if (base0 + 32 * u >= w_end) break;   // warp-uniform
            const int p = base0 + 32 * u + lane;
            int e = ev[u];
            if (e >= E) e = -1 - lane;
            unsigned peers = __match_any_sync(0xffffffffu, e);
            int pos = 0;
            if (e >= 0) pos = wc[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) wc[warp * E + e] += __popc(peers);
            __syncwarp();
            if (e >= 0) {
                const int prow = s_poff[e] + (pos - s_off[e]);
                if (pos >= P || prow >= rows_cap) {  // inconsistent counts: refuse, never write out of range
                    atomicOr(err, kErrDevice);
                } else {
                    sorted[pos] = p;
                    if (sorted_out) sorted_out[pos] = p;
                    inv[p] = prow;
                    pad_pair[prow] = p;
                }
            }
        }
    }
}

// Single-block grouping (1024 threads), for small batches and callers without
// the per-block count buffer: stable counting sort of the pairs p = t*k + j by
// expert (group_place over all pairs), plus the padded row layout used by the
// expert kernels and their work lists.
__global__ void __launch_bounds__(1024) k_group(const int32_t *__restrict__ ids, int P, int E, int T, int k,
                                                int has_shared, const int32_t *__restrict__ counts,
                                                int32_t *__restrict__ offsets, int32_t *__restrict__ poff,
                                                int32_t *__restrict__ sorted, int32_t *__restrict__ inv,
                                                int32_t *__restrict__ pad_pair, int4 *__restrict__ chunks,
                                                int4 *__restrict__ tiles,
                                                CallScratch *scratch, int32_t *__restrict__ offsets_out,
                                                int32_t *__restrict__ sorted_out, int build_work, int rows_cap,
                                                int tile_rows, int *err) {
    extern __shared__ int smem[];
    int *wc = smem;                        // [32][E]
    int *s_off = smem + 32 * E;            // [E+1]
    int *s_poff = s_off + (E + 1);         // [E+2]
    int *s_cb = s_poff + (E + 2);          // [E+2] chunk bases
    int *s_tb = s_cb + (E + 2);            // [E+2] tile bases
    __shared__ int s_warp[32][4];
    const int tid = threadIdx.x;
    for (int i = tid; i < 32 * E; i += 1024) wc[i] = 0;
    group_scan_experts(tid < E ? counts[tid] : 0, E, T, P, has_shared, tile_rows, s_off, s_poff, s_cb, s_tb,
                       s_warp, err);
    for (int i = tid; i <= E; i += 1024) {
        offsets[i] = s_off[i];
        if (offsets_out) offsets_out[i] = s_off[i];
    }
    for (int i = tid; i <= E + 1; i += 1024) poff[i] = s_poff[i];
    group_place(ids, 0, P, P, E, wc, s_off, s_off, s_poff, sorted, sorted_out, inv, pad_pair, rows_cap, err);
    if (!build_work) return;
    if (s_poff[E + 1] > rows_cap) {
        if (tid == 0) atomicOr(err, kErrDevice);
        return;
    }
    group_build_work(E, T, P, has_shared, tile_rows, s_off, s_poff, s_cb, s_tb, pad_pair, chunks, tiles, scratch);
}

// Multi-block grouping of large batches, three launches over blocks of
// kGroupSeg pairs: per-block expert counts; one block scanning them into the
// per-expert layout (and each block's first slot of every expert) and building
// the work lists; per-block placement. The order is the single-block one.
__global__ void __launch_bounds__(1024) k_group_count(const int32_t *__restrict__ ids, int P, int E,
                                                      int32_t *__restrict__ blk, int *err) {
    pdl_trigger();   // the scan launch may be scheduled now (it waits for this one)
    extern __shared__ int hist[];   // [E]
    for (int i = threadIdx.x; i < E; i += 1024) hist[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * kGroupSeg + threadIdx.x;
    if (p < P) {
        const int e = ids[p];
        if (e < 0 || e >= E) atomicOr(err, kErrDevice);
        else atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += 1024) blk[(size_t)blockIdx.x * E + i] = hist[i];
}

// blk[b][e] (counts in, each block's first slot of expert e out)
__global__ void __launch_bounds__(1024) k_group_scan(int nb, int P, int E, int T, int has_shared,
                                                     int32_t *__restrict__ blk, int32_t *__restrict__ offsets,
                                                     int32_t *__restrict__ poff, int4 *__restrict__ chunks,
                                                     int4 *__restrict__ tiles, CallScratch *scratch,
                                                     int32_t *__restrict__ offsets_out, int32_t *__restrict__ pad_pair,
                                                     int build_work, int rows_cap, int tile_rows, int *err) {
    pdl_wait();      // the per-block counts are complete
    pdl_trigger();
    extern __shared__ int smem[];
    int *s_off = smem, *s_poff = s_off + (E + 1), *s_cb = s_poff + (E + 2), *s_tb = s_cb + (E + 2);
    __shared__ int s_warp[32][4];
    const int tid = threadIdx.x;
    int c = 0;
    if (tid < E) {   // the expert's count over all blocks (loads issued eight at a time)
        for (int b0 = 0; b0 < nb; b0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = b0 + u < nb ? blk[(size_t)(b0 + u) * E + tid] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) c += v[u];
        }
    }
    group_scan_experts(c, E, T, P, has_shared, tile_rows, s_off, s_poff, s_cb, s_tb, s_warp, err);
    if (tid < E) {   // each block's first slot of this expert (counts loaded eight at a time, then stored)
        int run = s_off[tid];
        for (int b0 = 0; b0 < nb; b0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = b0 + u < nb ? blk[(size_t)(b0 + u) * E + tid] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b0 + u < nb) blk[(size_t)(b0 + u) * E + tid] = run;
                run += v[u];
            }
        }
    }
    for (int i = tid; i <= E; i += 1024) {
        offsets[i] = s_off[i];
        if (offsets_out) offsets_out[i] = s_off[i];
    }
    for (int i = tid; i <= E + 1; i += 1024) poff[i] = s_poff[i];
    if (!build_work) return;
    if (s_poff[E + 1] > rows_cap) {
        if (tid == 0) atomicOr(err, kErrDevice);
        return;
    }
    group_build_work(E, T, P, has_shared, tile_rows, s_off, s_poff, s_cb, s_tb, pad_pair, chunks, tiles, scratch);
}

__global__ void __launch_bounds__(1024) k_group_place(const int32_t *__restrict__ ids, int P, int E,
                                                      const int32_t *__restrict__ blk,
                                                      const int32_t *__restrict__ offsets,
                                                      const int32_t *__restrict__ poff, int32_t *__restrict__ sorted,
                                                      int32_t *__restrict__ sorted_out, int32_t *__restrict__ inv,
                                                      int32_t *__restrict__ pad_pair, int rows_cap, int *err) {
    pdl_wait();      // the layout and the per-block first slots are complete
    pdl_trigger();
    extern __shared__ int smem[];
    int *wc = smem, *s_base = wc + 32 * E, *s_off = s_base + E, *s_poff = s_off + E;
    for (int i = threadIdx.x; i < 32 * E; i += 1024) wc[i] = 0;
    for (int i = threadIdx.x; i < E; i += 1024) {
        s_base[i] = blk[(size_t)blockIdx.x * E + i];
        s_off[i] = offsets[i];
        s_poff[i] = poff[i];
    }
    __syncthreads();
    const int p_beg = blockIdx.x * kGroupSeg, p_end = min(P, p_beg + kGroupSeg);
    group_place(ids, p_beg, p_end, P, E, wc, s_base, s_off, s_poff, sorted, sorted_out, inv, pad_pair, rows_cap, err);
}

}  // namespace

namespace {

template <typename W>
cudaError_t launch_router_w(const Plan &p, const void *x, int T, const W *rw, const float *bias, int32_t *ids,
                            float *wts, cudaStream_t st, bool with_group) {
    const int H = p.cfg.hidden, E = p.cfg.num_experts, k = p.cfg.top_k;
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    const int npl = (E + 31) / 32;
    if (T <= kDecodeRouterThreads / 32 && H % 256 == 0) {
        GroupArgs grp{};
        if (with_group) {
            grp = GroupArgs{1, p.offsets, p.poff, p.sorted, p.inv, p.pad_pair, p.chunks, p.tiles,
                            (int)p.rows_pad_max, p.tile_rows, p.cfg.has_shared};
        }
        const size_t smem = decode_router_smem(H, T, E, (int)sizeof(W)) + (with_group ? group_small_smem(E, T * k) : 0);
#define MOE_DEC(N)                                                                                           \
    k_router_decode<N, W><<<E / decode_epb(T, E), kDecodeRouterThreads, smem, st>>>(xb, T, H, rw, bias, E, k, p.cfg.router, \
                                                              p.cfg.renormalize, p.logits, ids, wts, p.counts, \
                                                              p.scratch, p.err, grp)
        if (npl <= 1) MOE_DEC(1);
        else if (npl <= 2) MOE_DEC(2);
        else if (npl <= 4) MOE_DEC(4);
        else if (npl <= 8) MOE_DEC(8);
        else if (npl <= 16) MOE_DEC(16);
        else MOE_DEC(32);
#undef MOE_DEC
        return cudaGetLastError();
    }
    unsigned int *amax = &p.scratch->x_amax;   // batch amax of x (W4A4 quantiser, f16 range of W4A16)
    dim3 gt((E + kRE - 1) / kRE, (T + kRT - 1) / kRT);
    k_router_tiled<W><<<gt, 256, kRouterTiledSmem, st>>>(xb, T, H, rw, bias, E, p.logits, p.err, amax);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
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

}  // namespace

// The router weight's word type comes from the plan: fp32, or bf16 words
// (MOE_ROUTER_BF16) widened to fp32 as they are read.
cudaError_t launch_router(const Plan &p, const void *x, int T, const void *rw, const float *bias, int32_t *ids,
                          float *wts, cudaStream_t st, bool with_group) {
    if (p.cfg.router_dtype == MOE_ROUTER_BF16)
        return launch_router_w(p, x, T, static_cast<const __nv_bfloat16 *>(rw), bias, ids, wts, st, with_group);
    return launch_router_w(p, x, T, static_cast<const float *>(rw), bias, ids, wts, st, with_group);
}

// Kernels launch_router issues for T tokens (hidden is always a multiple of 256).
int router_launches(int T) { return T <= kDecodeRouterThreads / 32 ? 1 : 2; }

// Whether launch_router(..., with_group = true) also groups the pairs.
bool router_groups(int T) { return T <= kDecodeRouterThreads / 32; }

size_t group_smem_bytes(int E) { return sizeof(int) * (32 * (size_t)E + 4 * (size_t)E + 8); }

// The routing kernels' dynamic shared-memory limits are per-function, per-device
// attributes shared by every plan and by moe_route_static.  They are set once
// a device, for the largest sizes any call may ask for (kMaxExperts experts,
// the decode router at H = 8192), so a later call can never lower a limit that
// an earlier plan or a static call still relies on.
cudaError_t configure_group_kernel() {
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(k_router_tiled<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterTiledSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_router_tiled<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRouterTiledSmem);
    if (e != cudaSuccess) return e;
    const int dec = (int)(decode_router_smem(8192, kDecodeRouterThreads / 32, 2, 4) +
                          group_small_smem(kMaxExperts, kDecodeRouterThreads / 32 * kMaxTopK));
    for (auto f : {k_router_decode<1, float>, k_router_decode<2, float>, k_router_decode<4, float>,
                   k_router_decode<8, float>, k_router_decode<16, float>, k_router_decode<32, float>}) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dec);
        if (e != cudaSuccess) return e;
    }
    for (auto f : {k_router_decode<1, __nv_bfloat16>, k_router_decode<2, __nv_bfloat16>,
                   k_router_decode<4, __nv_bfloat16>, k_router_decode<8, __nv_bfloat16>,
                   k_router_decode<16, __nv_bfloat16>, k_router_decode<32, __nv_bfloat16>}) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dec);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(k_group_place, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(int) * 35 * (size_t)kMaxExperts));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_group, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)group_smem_bytes(kMaxExperts));
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

// Launches of launch_group: three (count, scan, place) for batches larger than
// two segments when the plan holds the per-block count buffer, else one.
int group_launches(const Plan &p, int T) {
    return (p.group_blk && (int64_t)T * p.cfg.top_k > 2 * kGroupSeg) ? 3 : 1;
}

cudaError_t launch_group(const Plan &p, int T, const int32_t *ids, int32_t *offsets_out, int32_t *sorted_out,
                         bool build_work, cudaStream_t st) {
    const int E = p.cfg.num_experts, k = p.cfg.top_k, P = T * k;
    if (group_launches(p, T) == 3) {
        const int nb = (P + kGroupSeg - 1) / kGroupSeg;
        k_group_count<<<nb, 1024, sizeof(int) * E, st>>>(ids, P, E, p.group_blk, p.err);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess)
            e = launch_pdl(k_group_scan, dim3(1), dim3(1024), sizeof(int) * (4 * (size_t)E + 8), st, nb, P, E, T,
                           (int)p.cfg.has_shared, p.group_blk, p.offsets, p.poff, p.chunks, p.tiles, p.scratch,
                           offsets_out, p.pad_pair, build_work ? 1 : 0, (int)p.rows_pad_max, p.tile_rows, p.err);
        if (e == cudaSuccess)
            e = launch_pdl(k_group_place, dim3(nb), dim3(1024), sizeof(int) * 35 * (size_t)E, st, (const int32_t *)ids,
                           P, E, (const int32_t *)p.group_blk, (const int32_t *)p.offsets, (const int32_t *)p.poff,
                           p.sorted, sorted_out, p.inv, p.pad_pair, (int)p.rows_pad_max, p.err);
        return e;
    }
    size_t smem = group_smem_bytes(E);
    k_group<<<1, 1024, smem, st>>>(ids, P, E, T, k, p.cfg.has_shared, p.counts, p.offsets, p.poff, p.sorted,
                                   p.inv, p.pad_pair, p.chunks, p.tiles, p.scratch, offsets_out, sorted_out,
                                   build_work ? 1 : 0, (int)p.rows_pad_max, p.tile_rows, p.err);
    return cudaGetLastError();
}

}  // namespace moe
