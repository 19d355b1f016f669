// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05), NVFP4 x
// NVFP4 with E4M3 block scales (kind::mxf4nvf4, 16-value scale blocks), fp32
// accumulators in tensor memory, operands brought in by TMA.
//
// "NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4 Round 1:
// the routed NVFP4 prompt GEMM runs on the FP4 tensor cores with 4-bit
// activations (#687); gate, up and SwiGLU run as one launch (#766); the GEMM
// store scales each slot by its expert's tensor scale (#545); the operands are
// copied through a multi-stage pipeline in K steps (#822); the combine is folded
// into the down product's store (#701).
//
// Layout (swap-AB): A = expert weight rows (M = 128 features per MMA), B = the
// expert's token rows (N = 128), K along the hidden / intermediate dimension.
// One work item = (tile of 128 padded token rows of one expert, 256 weight
// rows): gate+up (two 128-row MMAs sharing B, SwiGLU epilogue) or down (two
// 128-row MMAs, weighted scatter-add epilogue).
//
// Warp roles (one CTA per SM, persistent over the items):
//   warp 0   TMA producer (one lane)
//   MMA warps: one lane each issues tcgen05.mma. A thread issuing tcgen05.mma
//            stalls about as long as the MMA runs, so whatever else it does
//            between MMAs (barrier waits, fences, descriptors, copies, commits)
//            idles the tensor pipe.
//     gate/up: warp 1 drives both accumulators; its stages wait on data
//              (weights and token rows from L2) more than on issue;
//     down:    warps 1 and 2, one accumulator each (the first and second 128
//              weight rows), so one lane's bookkeeping runs under the other's
//              MMAs.
//            Warp 1 owns the TMEM allocation.
//   scale warps, which put the stage's E4M3 scale factors into tensor memory:
//     gate/up: warps 2-5, each writing its own 32-lane quadrant with tcgen05.st,
//              so the tensor pipe spends no time on scales (448 threads);
//     down:    warp 3, which re-lays the weight scale tiles in shared memory into
//              512-byte atoms that each MMA lane copies with tcgen05.cp (the
//              atoms its MMAs read; 384 threads). The down epilogue keeps 128
//              accumulator values a thread in registers and needs the 168
//              registers a thread that a 12-warp block allows; at 14 warps it
//              would spill.
//   the last 8 warps: epilogue (tcgen05.ld of their 32-lane quadrant of the
//              accumulators)
// Every mbarrier wait is bounded (about one second); on expiry the kernel sets
// the plan's timeout bit and every role leaves its loop.
#include <cuda.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kBK = 256;                  // K values per pipeline stage
constexpr int kRowBytes = kBK / 2;        // 128 code bytes per row per stage
constexpr int kTile = 128 * kRowBytes;    // 16 KB operand tile
constexpr int kSf = 128 * 16;             // 2 KB: 128 rows x 16 scale bytes
constexpr int kStageBytes = 3 * kTile + 3 * kSf;   // A0, A1, B codes; A0, A1 scales (plain rows); B scales (atoms)
constexpr int kEpiWarps = 8;                      // two per 32-lane TMEM quadrant
constexpr uint32_t kSfCol0 = 256;                 // scale-factor TMEM columns, after the two 128-column accumulators

enum Epi { kSwiGLU = 0, kScatter = 1 };

// Warps by role: MMA issuers (gate/up one, down two) and scale warps (gate/up
// four tcgen05.st writers, down one shared-memory re-layout warp), after the
// producer warp; the 8 epilogue warps follow them.
__host__ __device__ constexpr int mma_warps(int epi) { return epi == kSwiGLU ? 1 : 2; }
__host__ __device__ constexpr int scale_warps(int epi) { return epi == kSwiGLU ? 4 : 1; }
__host__ __device__ constexpr int epi_warp0(int epi) { return 1 + mma_warps(epi) + scale_warps(epi); }
// TMEM scale columns a stage slot owns: A0, A1, B (gate/up, written by the
// scale warps and read by the MMA lane); A0, A1, B for MMA lane 0, B for MMA
// lane 1 (down: each lane copies the atoms its own MMAs read, since copies and
// MMAs issued by different threads are not ordered)
__host__ __device__ constexpr int sf_stride(int epi) { return epi == kSwiGLU ? 48 : 64; }
static_assert(kSfCol0 + kStages * 64 <= 512, "FP4 TMEM plan exceeds 512 columns");
__host__ __device__ constexpr int fp4_threads(int epi) { return 32 * (epi_warp0(epi) + kEpiWarps); }

struct TcArgs {
    CUtensorMap a0[2];      // [routed, shared]: gate codes (G1) / down codes (G2)
    CUtensorMap a1[2];      // up codes (G1) / unused (G2: second half of down rows from a0)
    CUtensorMap s0[2];      // plain scale tiles matching a0
    CUtensorMap s1[2];      // matching a1
    CUtensorMap b[3];       // token rows: Xp codes (G1) / SwiGLU codes (G2), boxes of 32, 64, 128 rows
    const uint8_t *b_atoms; // token-row scales in the tensor-core layout
    int b_atoms_per_block;  // 512-byte atoms per 128-row block (= row length / 64)
    const int4 *tiles;      // {expert (E = shared), first padded row, valid rows, 0}
    const CallScratch *scratch;
    int E, H, I, Is;
    int nf;                 // 256-row weight groups per item row (G1: Imax/128, G2: H/256)
    // epilogue
    const float *ts_a0[2], *ts_a1[2];  // tensor scales of the A operands
    const float *b_ts;      // SwiGLU tensor scales [routed, shared] (G2)
    float *hbuf;            // G1 output [rows][hstride] fp32
    int hstride;
    unsigned int *h_amax, *hs_amax;
    const int32_t *pad_pair;
    const float *wts;
    int P, k;
    float *acc;             // G2 output [T][H]
    int *err;
    int colfirst;           // down items: column groups a chunk (large T; 0: tile by tile; see decode_item)
    // MXFP4 gate/up: the SwiGLU output quantised in the epilogue (single pass)
    uint8_t *hq;            // codes [rows][hstride / 2]
    uint8_t *hq_atoms;      // E8M0 scales in the tensor-core layout (hstride / 128 atoms a 128-row block)
    float *hts_out;         // [2] SwiGLU tensor scales: 1 (MXFP4 has none)
    int keep_h;             // also store the fp32 h (stage-by-stage checks)
};

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Descriptor of one 512-byte scale-factor atom (32 rows x 16 bytes, no swizzle)
// for tcgen05.cp .32x128b.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1, UE4M3 scales, K-major,
// M = 128, N = n (a multiple of 16).
__device__ __forceinline__ uint32_t idesc_fp4(uint32_t n) {
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (0u << 23) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
}

// MXFP4 (kind::mxf4, UE8M0 scales, one a 32-value block): a K = 64 MMA takes
// two scale bytes a row.  A 32-bit scale cell of tensor memory holds four
// (K = 128, two MMAs); the descriptor's scale-factor ids (A: bits 29-30, B:
// bits 4-5) pick bytes 0-1 (id 0) or 2-3 (id 2) of the cell.
__device__ __forceinline__ uint32_t idesc_mx4(uint32_t n, int kk) {
    const uint32_t id = 2u * (uint32_t)(kk & 1);
    return idesc_fp4(n) | (1u << 23) | (id << 29) | (id << 4);
}

__device__ __forceinline__ void mma_mx4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
}

// One block-scaled FP4 MMA of K chunk kk: NVFP4 (cell = four 16-value blocks =
// one K chunk) or MXFP4 (cell = four 32-value blocks = two K chunks).
// sfa0 / sfb0: the stage's first scale column of the A / B operand.
template <int MX>
__device__ __forceinline__ void mma_blk(uint32_t d, uint64_t a, uint64_t b, uint32_t n, int kk, uint32_t sfa0,
                                        uint32_t sfb0, uint32_t acc) {
    if (MX)
        mma_mx4(d, a, b, idesc_mx4(n, kk), sfa0 + 4 * (kk >> 1), sfb0 + 4 * (kk >> 1), acc);
    else
        mma_fp4(d, a, b, idesc_fp4(n), sfa0 + 4 * kk, sfb0 + 4 * kk, acc);
}

// Token rows a tile loads and multiplies: 32, 64 or 128 (index into TcArgs::b).
__device__ __forceinline__ int rows_class(int valid) { return valid <= 32 ? 0 : (valid <= 64 ? 1 : 2); }

__device__ __forceinline__ void sf_copy(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 columns from v[0..15] (each thread: its lane).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// 32 lanes x 16 columns of fp32 into v[0..15] (each thread: its lane); the
// caller waits with tcgen05.wait::ld before reading v.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float *v) {
    uint32_t *r = reinterpret_cast<uint32_t *>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

struct Item {
    int e, row0, valid, f, sh, K;
    int kc0, kc1;   // code stages [kc0, kc1) of K this item covers (split-K down items)
    int part = 0, parts = 1, slot = -1;   // K piece of a split item (warp-MMA engine), its index among split items
};

// Items run tile by tile (one tile's token rows against every weight group).
// For many tokens the down items run in chunks of C = colfirst column groups
// instead, tile by tile within a chunk: the scatter-add into the fp32
// accumulator then touches a [T][256 C] slice of it at a time, which stays in
// L2, and the token rows of a tile are read once a chunk (C = 1 would read
// every tile's SwiGLU codes once per 256 output columns).  For few tokens the
// chunked order would make the CTAs running at the same time add into the same
// few addresses.
__device__ __forceinline__ bool decode_item(const TcArgs &a, int item, int epi, Item &it) {
    const int nt = a.scratch->n_tiles;
    int tile;
    if (epi == kScatter && a.colfirst) {
        const int C = a.colfirst;
        const int q = item / (nt * C);             // chunk
        const int cq = min(C, a.nf - q * C);       // its column groups (the last may be short)
        const int rem = item - q * nt * C;
        tile = rem / cq;
        it.f = q * C + (rem - tile * cq);
    } else {
        tile = item / a.nf;
        it.f = item % a.nf;
    }
    const int4 t = a.tiles[tile];
    it.e = t.x;
    it.row0 = t.y;
    it.valid = t.z;
    it.sh = (t.x == a.E);
    const int I = it.sh ? a.Is : a.I;
    if (epi == kSwiGLU) {
        it.K = a.H;
        return it.f * 128 < I;
    }
    it.K = I;
    return true;
}

// MX: MXFP4 operands (weights and token rows): E8M0 scales, a cell of four
// 32-value blocks, so a 256-value stage has two scale cells an operand; the
// weights' 16-byte scale box a row covers a pair of stages.
template <int EPI, int MX>
__global__ void __launch_bounds__(fp4_threads(EPI), 1) k_gemm_fp4(const __grid_constant__ TcArgs a) {
    constexpr int kMmaWarps = mma_warps(EPI), kScaleWarps = scale_warps(EPI), kEpiWarp0 = epi_warp0(EPI);
    pdl_wait();      // routing, permute or gate/up results come from the previous kernel
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *sf_ready = full + kStages;
    uint64_t *empty = sf_ready + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.scratch->n_tiles * a.nf;
    if (EPI == kSwiGLU && MX && blockIdx.x == 0 && threadIdx.x == 0) { a.hts_out[0] = 1.0f; a.hts_out[1] = 1.0f; }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(sf_ready + s, kScaleWarps);
            mbar_init(empty + s, kMmaWarps);   // every MMA lane commits every stage
        }
        mbar_init(acc_full, kMmaWarps);
        mbar_init(acc_empty, kEpiWarps);
        mbar_init(drain, kMmaWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t used = 0, last_ph = 0;  // stages loaded at least once, parity of their last load
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item(a, item, EPI, it)) continue;
                const int m = it.sh ? 1 : 0;
                int r0, r1;
                if (EPI == kSwiGLU) {
                    r0 = r1 = (it.sh ? 0 : it.e * a.I) + it.f * 128;
                } else {
                    r0 = (it.sh ? 0 : it.e * a.H) + it.f * 256;
                    r1 = r0 + 128;
                }
                const CUtensorMap *A1 = (EPI == kSwiGLU) ? &a.a1[m] : &a.a0[m];
                const CUtensorMap *S1 = (EPI == kSwiGLU) ? &a.s1[m] : &a.s0[m];
                const int rc = rows_class(it.valid);
                const uint32_t b_bytes = (32u << rc) * kRowBytes;
                const uint8_t *batoms = a.b_atoms + (size_t)(it.row0 / 128) * a.b_atoms_per_block * 512;
                const int ks_n = it.K / kBK;
                constexpr uint32_t kBSf = MX ? kSf / 2 : kSf;   // token-row scale atoms a stage
                for (int ks = 0; ks < ks_n; ++ks) {
                    if (!mbar_wait(empty + s, ph ^ 1, a.err)) { ok = false; break; }
                    uint8_t *st = smem + s * kStageBytes;
                    mbar_expect_tx(full + s, 2 * kTile + b_bytes + 2 * kSf + kBSf);
                    tma_2d(st, &a.a0[m], full + s, ks * kRowBytes, r0);
                    tma_2d(st + kTile, A1, full + s, ks * kRowBytes, r1);
                    tma_2d(st + 2 * kTile, &a.b[rc], full + s, ks * kRowBytes, it.row0);
                    const int sx = MX ? (ks >> 1) * 16 : ks * 16;
                    tma_2d(st + 3 * kTile, &a.s0[m], full + s, sx, r0);
                    tma_2d(st + 3 * kTile + kSf, S1, full + s, sx, r1);
                    bulk_copy(st + 3 * kTile + 2 * kSf, batoms + (size_t)ks * kBSf, kBSf, full + s);
                    used |= 1u << s;
                    last_ph = (last_ph & ~(1u << s)) | (ph << s);
                    if (++s == kStages) { s = 0; ph ^= 1; }
                }
            }
            // every load has landed before the block exits (already true unless a wait ran out)
            for (int t = 0; t < kStages; ++t)
                if (used & (1u << t)) mbar_wait(full + t, (last_ph >> t) & 1u, a.err);
        }
    } else if (warp >= 1 && warp <= kMmaWarps) {
        // ------------------------------------------------ MMA issue (one lane a warp)
        if (lane == 0) {
            // accumulators this lane drives: h0 .. h0 + nh - 1 (0: weight rows 0-127,
            // i.e. gate / first down half; 1: rows 128-255)
            const int h0 = warp - 1, nh = kMmaWarps == 1 ? 2 : 1;
            int s = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item(a, item, EPI, it)) continue;
                if (!mbar_wait(acc_empty, aph ^ 1, a.err)) break;
                aph ^= 1;
                tc_fence_after();
                const uint32_t nrows = 32u << rows_class(it.valid);
                const int ks_n = it.K / kBK;
#pragma unroll 2
                for (int ks = 0; ks < ks_n; ++ks) {
                    // sf_ready completes after every scale warp saw the stage's loads
                    // land (each waits on full first), so it covers full as well: one
                    // wait, not two (a satisfied wait still costs ~60 cycles here)
                    if (!mbar_wait(sf_ready + s, ph, a.err)) { ok = false; break; }
                    tc_fence_after();
                    // descriptors of the stage's operands: built once, then stepped by
                    // their 16-byte address units (the smem window is below 256 KB, so
                    // adding to the start-address field never carries out of it)
                    const uint32_t base = smem_u32(smem + s * kStageBytes);
                    const uint64_t dA = desc_sw128(base), dB = desc_sw128(base + 2 * kTile);
                    // scale factors of this stage slot: accumulator h's A at +16 h, its
                    // B at +32 (gate/up) or +32 + 16 h (down), four columns a K chunk
                    const uint32_t sf = tmem + kSfCol0 + s * sf_stride(EPI);
                    if (EPI == kScatter) {
                        const uint64_t dS = desc_sf(base + 3 * kTile);
                        for (int h = h0; h < h0 + nh; ++h) {
#pragma unroll
                            for (int c = 0; c < (MX ? 2 : 4); ++c) {   // the stage's scale cells
                                sf_copy(sf + 16 * h + 4 * c, dS + h * (kSf >> 4) + 32 * c);
                                sf_copy(sf + 32 + 16 * h + 4 * c, dS + (2 * kSf >> 4) + 32 * c);
                            }
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (ks | kk) ? 1u : 0u;
                        if (kMmaWarps == 1) {
                            mma_blk<MX>(tmem, dA + 2 * kk, dB + 2 * kk, nrows, kk, sf, sf + 32, accum);
                            mma_blk<MX>(tmem + 128, dA + (kTile >> 4) + 2 * kk, dB + 2 * kk, nrows, kk, sf + 16,
                                        sf + 32, accum);
                        } else {
                            mma_blk<MX>(tmem + 128 * h0, dA + h0 * (kTile >> 4) + 2 * kk, dB + 2 * kk, nrows, kk,
                                        sf + 16 * h0, sf + 32 + 16 * h0, accum);
                        }
                    }
                    mma_commit(empty + s);
                    if (++s == kStages) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(acc_full);
            }
            // all issued MMAs / copies complete before the accumulators are freed
            mma_commit(drain);
            mbar_wait(drain, 0, a.err);
        }
    } else if (warp > kMmaWarps && warp < kEpiWarp0 && EPI == kScatter) {
        // ------------------------------------------------ weight scale re-layout (down)
        // plain [128 rows][16 B] scale tiles -> four 512-byte atoms each, in place:
        // the 4 scale bytes of row r for K chunk c go to word (r % 32) * 4 + r / 32
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            Item it;
            if (!decode_item(a, item, EPI, it)) continue;
            const int ks_n = it.K / kBK;
            for (int ks = 0; ks < ks_n; ++ks) {
                if (!mbar_wait(full + s, ph, a.err)) { ok = false; break; }
                uint8_t *st = smem + s * kStageBytes;
#pragma unroll
                for (int op = 0; op < 2; ++op) {
                    // every lane reads its 4 rows, then (after the warp has read
                    // everything) writes its 4 atom words
                    const uint32_t tile = smem_u32(st + 3 * kTile + op * kSf);
                    uint4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = lds128(tile + 16 * (lane + 32 * q));
                    __syncwarp();
                    if (MX) {   // this stage's two cells: words 2 (ks & 1) and 2 (ks & 1) + 1 of a row
                        if (ks & 1) {
                            sts128(tile + 16 * (0 * 32 + lane), make_uint4(v[0].z, v[1].z, v[2].z, v[3].z));
                            sts128(tile + 16 * (1 * 32 + lane), make_uint4(v[0].w, v[1].w, v[2].w, v[3].w));
                        } else {
                            sts128(tile + 16 * (0 * 32 + lane), make_uint4(v[0].x, v[1].x, v[2].x, v[3].x));
                            sts128(tile + 16 * (1 * 32 + lane), make_uint4(v[0].y, v[1].y, v[2].y, v[3].y));
                        }
                    } else {
                        sts128(tile + 16 * (0 * 32 + lane), make_uint4(v[0].x, v[1].x, v[2].x, v[3].x));
                        sts128(tile + 16 * (1 * 32 + lane), make_uint4(v[0].y, v[1].y, v[2].y, v[3].y));
                        sts128(tile + 16 * (2 * 32 + lane), make_uint4(v[0].z, v[1].z, v[2].z, v[3].z));
                        sts128(tile + 16 * (3 * 32 + lane), make_uint4(v[0].w, v[1].w, v[2].w, v[3].w));
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(sf_ready + s);
                if (++s == kStages) { s = 0; ph ^= 1; }
            }
        }
        mbar_wait(drain, 0, a.err);
    } else if (warp > kMmaWarps && warp < kEpiWarp0) {
        // ------------------------------------------------ scale factors -> TMEM
        // Scale-factor layout (scale_vec::4X, M = N = 128), 4 columns per K chunk
        // kk of 64 values, as a 32x128b.warpx4 copy of a 512-byte atom lays it
        // out: lane l of each 32-lane quadrant, column 4 * kk + j holds the 4
        // scale bytes of row l + 32 * j.
        //   A (weight rows): the MMA reads row r's scales only from its own lane
        //     r (column 4 * kk + r / 32), so the warp of quadrant q loads just
        //     rows 32 q + l (one 16-byte row: its 4 chunk words) and writes each
        //     word to all four columns of its chunk.
        //   B (token rows): every quadrant reads all 128 rows, so each warp
        //     writes the full atoms (word j of atom kk, row l).
        // A0 and A1 arrive as plain [128 rows][16 B] tiles, B as four atoms.
        // Stage slot s owns columns kSfCol0 + 48 s ..: they are free again once
        // the slot's next TMA load has landed, because the producer reloads a
        // slot only after the MMAs that read it have completed.
        const int quad = warp & 3;
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + kSfCol0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            Item it;
            if (!decode_item(a, item, EPI, it)) continue;
            const int ks_n = it.K / kBK;
            for (int ks = 0; ks < ks_n; ++ks) {
                if (!mbar_wait(full + s, ph, a.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sfb = smem_u32(smem + s * kStageBytes + 3 * kTile);
                uint32_t o[16];
#pragma unroll
                for (int op = 0; op < 2; ++op) {
                    const uint4 v = lds128(sfb + op * kSf + 16 * (lane + 32 * quad));
                    // NVFP4: cells 0-3 are words x, y, z, w; MXFP4: the row's 16 bytes
                    // cover a pair of stages, this stage's two cells are words
                    // 2 (ks & 1) and 2 (ks & 1) + 1 (cells 2, 3 unused)
                    const uint32_t c0 = (MX && (ks & 1)) ? v.z : v.x, c1 = (MX && (ks & 1)) ? v.w : v.y;
                    const uint32_t c2 = MX ? 0u : v.z, c3 = MX ? 0u : v.w;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        o[j] = c0;
                        o[4 + j] = c1;
                        o[8 + j] = c2;
                        o[12 + j] = c3;
                    }
                    tmem_st16(t_lane + s * sf_stride(EPI) + 16 * op, o);
                }
                {
                    uint4 v[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        v[kk] = (MX && kk >= 2) ? make_uint4(0u, 0u, 0u, 0u) : lds128(sfb + 2 * kSf + 512 * kk + 16 * lane);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        o[4 * kk] = v[kk].x;
                        o[4 * kk + 1] = v[kk].y;
                        o[4 * kk + 2] = v[kk].z;
                        o[4 * kk + 3] = v[kk].w;
                    }
                    tmem_st16(t_lane + s * sf_stride(EPI) + 32, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sf_ready + s);
                if (++s == kStages) { s = 0; ph ^= 1; }
            }
        }
        mbar_wait(drain, 0, a.err);
    } else {
        // ------------------------------------------------ epilogue (8 warps)
        // Each warp copies its 32 lanes x 64 columns of both accumulators into
        // registers, releases the accumulators to the MMA warp, and only then
        // does the arithmetic and the global writes, so the next item's MMAs
        // overlap them.
        const int quad = warp & 3;                 // TMEM lanes this warp may read
        const int col0 = ((warp - kEpiWarp0) >> 2) * 64;   // its half of the token columns
        uint32_t aph = 0;
        float lmax = 0.0f, lmax_s = 0.0f;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            Item it;
            if (!decode_item(a, item, EPI, it)) continue;
            if (!mbar_wait(acc_full, aph, a.err)) break;
            aph ^= 1;
            tc_fence_after();
            const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
            const int m = it.sh ? 1 : 0;
            const int e = it.sh ? 0 : it.e;
            const int n_end = min(col0 + 64, it.valid);
            float v0[64], v1[64];
            if (col0 < n_end) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tmem_ld16_nowait(lane_base + col0 + 16 * c, v0 + 16 * c);
                    tmem_ld16_nowait(lane_base + 128 + col0 + 16 * c, v1 + 16 * c);
                }
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (col0 >= n_end) continue;
            if (EPI == kSwiGLU && MX) {
                // MXFP4: every 32-value block of h has its own scale and no batch
                // amax is needed, so h is quantised here, in one pass. The
                // warp's 32 lanes hold 32 consecutive features of a token row,
                // one MX block: the warp maximum of |h| gives the E8M0 byte
                // (clamp(floor(log2 amax) - 2 + 127, 0, 254), 0 for a zero
                // block), each lane its E2M1 code of h * 2^(127 - byte), and lane
                // pairs / quadruples assemble the block's 16 code bytes.
                const float sg = a.ts_a0[m][e], su = a.ts_a1[m][e];
                const int fb = it.f * 128 + quad * 32;   // the block's first feature
                const int blk = fb >> 5;
                float *hrow = a.hbuf + (size_t)(it.row0 + col0) * a.hstride + fb + lane;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    if (col0 + j < n_end) {   // the same for every lane
                        const float gv = v0[j] * sg, uv = v1[j] * su;
                        const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                        if (a.keep_h) hrow[(size_t)j * a.hstride] = h;
                        const uint32_t ab = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
                        const int field = (int)((ab >> 23) & 0xFFu);
                        const int sx = field > 2 ? field - 2 : 0;
                        const float inv = __uint_as_float((uint32_t)(254 - sx) << 23);   // 2^(127 - sx)
                        const uint32_t nib = f32x2_to_e2m1x2(__fmul_rn(h, inv), 0.0f) & 0xFu;
                        const uint32_t b = nib | (__shfl_down_sync(0xffffffffu, nib, 1) << 4);   // even lanes
                        const uint32_t w = b | (__shfl_down_sync(0xffffffffu, b, 2) << 8) |
                                           (__shfl_down_sync(0xffffffffu, b, 4) << 16) |
                                           (__shfl_down_sync(0xffffffffu, b, 6) << 24);   // lanes 8 q: word q
                        const int r = it.row0 + col0 + j, rr = r & 127;
                        if ((lane & 7) == 0)
                            *reinterpret_cast<uint32_t *>(a.hq + (size_t)r * (a.hstride / 2) + (fb >> 1) + (lane >> 1)) = w;
                        if (lane == 0)
                            a.hq_atoms[((size_t)(r >> 7) * (a.hstride / 128) + (blk >> 2)) * 512 + (rr & 31) * 16 +
                                       (rr >> 5) * 4 + (blk & 3)] = (uint8_t)sx;
                    }
                }
            } else if (EPI == kSwiGLU) {
                // NVFP4: the activation tensor scale from the batch amax
                const float xts = __fdiv_rn(__uint_as_float(a.scratch->x_amax), 2688.0f);
                const float sg = a.ts_a0[m][e] * xts, su = a.ts_a1[m][e] * xts;
                const int feat = it.f * 128 + quad * 32 + lane;
                float mx = 0.0f;
                float *hrow = a.hbuf + (size_t)(it.row0 + col0) * a.hstride + feat;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    if (col0 + j < n_end) {
                        const float gv = v0[j] * sg, uv = v1[j] * su;
                        const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                        hrow[(size_t)j * a.hstride] = h;
                        mx = fmaxf(mx, fabsf(h));
                    }
                }
                if (it.sh) lmax_s = fmaxf(lmax_s, mx);
                else lmax = fmaxf(lmax, mx);
            } else {
                const float ds = a.ts_a0[m][e] * a.b_ts[m];
                // columns col0 + lane and col0 + 32 + lane: token and routing weight
                int tok[2];
                float wgt[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = col0 + lane + 32 * q;
                    tok[q] = 0;
                    wgt[q] = 0.0f;
                    if (n < it.valid) {
                        const int pair = a.pad_pair[it.row0 + n];
                        tok[q] = pair >= a.P ? pair - a.P : pair / a.k;
                        wgt[q] = pair >= a.P ? 1.0f : a.wts[pair];
                    }
                }
                const int j0 = it.f * 256 + quad * 32 + lane;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int t = __shfl_sync(0xffffffffu, tok[j >> 5], j & 31);
                    const float wv = __shfl_sync(0xffffffffu, wgt[j >> 5], j & 31) * ds;
                    if (col0 + j < n_end) {
                        float *dst = a.acc + (size_t)t * a.H + j0;
                        atomicAdd(dst, v0[j] * wv);
                        atomicAdd(dst + 128, v1[j] * wv);
                    }
                }
            }
        }
        if (EPI == kSwiGLU) {
            lmax = warp_max(lmax);
            lmax_s = warp_max(lmax_s);
            if (lane == 0) {
                if (lmax > 0.0f) atomic_max_nonneg(a.h_amax, lmax);
                if (lmax_s > 0.0f) atomic_max_nonneg(a.hs_amax, lmax_s);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
    }
}

// ------------------------------------------------------------------ W4A16
// W4A16 on the tensor cores (tcgen05 kind::f16, fp32 accumulators), with the
// widened weights held in tensor memory: the MMA takes its A operand (128
// weight rows x 16 K) from TMEM and its B operand (token rows) from shared
// memory.  Shared memory then carries only the 4-bit codes and the f16 token
// rows, so its bandwidth no longer bounds the weight stream.
//   code ring  (4 x 36 KB, shared): NVFP4 codes of both A operands (128-byte
//              swizzle) + their plain scale tiles, 256 K values a stage;
//   B ring     (4 x 16 KB, shared): f16 token rows, 128-byte swizzle, in
//              boxes of 64 K values; a stage holds 512, 256 or 128 K values
//              for tiles of up to 16, 32 or 64 rows (MMA N = 16, 32, 64);
//   A ring     (2 x 128 TMEM columns): both operands widened to f16, 128 K
//              values a stage (row r in lane r, two K values a column);
//   accumulators (2 x 128 TMEM columns): gate / up (or the two down-row
//              halves), N <= 64 token columns each, double-buffered so an
//              item's epilogue overlaps the next item's MMAs.
// Sixteen converter warps, four per 32-lane quarter (operand x half of the
// stage's K values), widen E2M1 -> f16 (cvt.rn.f16x2.e2m1x2) and multiply by
// the E4M3 block scale in f16; code x scale has at most 6 significant bits, so
// the f16 weights are exact.  The activations are f16 rows: the permute kernel
// writes x * 2^-s, with s the smallest power of two keeping the batch amax
// inside f16 (s = 0 for ordinary activations); the epilogue multiplies 2^s
// back.  A work item is (tile of up to 64 token rows of one expert, 128 weight
// rows of each operand); the grouping kernel cuts W4A16 tiles at 64 rows.
constexpr int kHCK = 256;                        // K values per code stage
constexpr int kHCodeTile = 128 * 128;            // 16 KB: 128 rows x 128 code bytes
constexpr int kHCodeStage = 2 * kHCodeTile + 2 * 2048;   // A0, A1 codes + A0, A1 scales
constexpr int kHCStages = 4;
constexpr int kHBK = 64;                         // K values per MMA step
constexpr int kHBRows = 64;                      // token rows per tile (MMA N <= 64)
constexpr int kHBTile = 16384;                   // B stage: 16 KB of f16 token rows
constexpr int kHBStages = 4;
// The A ring's stages are 128 K values (8 MMAs an accumulator half): the MMA
// lanes' waits, commits and loop overhead come once per 8 MMAs (64 K values
// a stage measured ~850 cycles a stage against ~340 of MMA issue).
constexpr int kHAK = 128;                        // K values per A stage
constexpr int kHAStages = 2;                     // TMEM A ring
constexpr uint32_t kHACol0 = 256;                // first TMEM column of the A ring
constexpr int kConvSplit = 2;                    // converter warps per (operand, 32-lane quarter)
constexpr int kConvWarps = 8 * kConvSplit;
constexpr int kConvCols = kHAK / 2 / kConvSplit; // TMEM columns (2 K values each) a converter fills per A stage
static_assert(kConvSplit == 2, "the converter loop below is written for two K halves");
constexpr int kHEpiWarps = 4;
// the second MMA lane's warp, after the epilogue warps (warp 1 drives the
// first accumulator half, this one the second: a thread issuing tcgen05.mma
// stalls about as long as the MMA runs, so one issuer idles the pipe during
// its own barrier waits and commits)
constexpr int kHMma2 = 2 + kConvWarps + kHEpiWarps;
constexpr int kHThreads = 32 * (kHMma2 + 1);
constexpr size_t kHRingBytes = (size_t)kHCStages * kHCodeStage + (size_t)kHBStages * kHBTile;
constexpr size_t kHSmemBytes = kHRingBytes + 512 + 1024;
static_assert(kHSmemBytes <= 227 * 1024, "W4A16 pipeline exceeds shared memory");
static_assert(kHACol0 + kHAStages * kHAK <= 512, "W4A16 TMEM plan exceeds 512 columns");
static_assert(kHAK == 128 && kConvCols == 32, "the converter and MMA loops below are written for 128-K A stages");

struct HcArgs {
    CUtensorMap a0[2], a1[2];   // NVFP4 codes [rows][K/2], box 128 B x 128 rows, 128-byte swizzle
    CUtensorMap s0[2], s1[2];   // scales [rows][K/16], box 16 B x 128 rows
    CUtensorMap b[3];           // f16 token rows [rows_pad][Kdim], box 64 x (16/32/64), 128-byte swizzle
    const int4 *tiles;
    const CallScratch *scratch;
    int E, H, I, Is, nf;
    const float *ts_a0[2], *ts_a1[2];
    __half *hout;               // gate/up output (f16) [rows][hstride]
    int hstride;
    const int32_t *pad_pair;
    const float *wts;
    int P, k;
    float *acc;
    int *err;
    int colfirst;           // down items column group first (large T; see decode_item_h)
    // warp-MMA engine: ring geometry chosen per launch, and the raw activations
    // the gate/up launch gathers its token rows from (no separate permute)
    int rcst, rbst, rbslot;
    const uint16_t *x;
    int xres;               // gate/up: tokens whose activations sit resident in shared memory (0: token-row ring)
    int mx;                 // MXFP4 weights (selects the k_gemm_reg instantiation)
    // split last round (warp-MMA engine): arrival tickets and partial sums
    int tail_split;
    int *tickets;
    float *tail_part;
};

// f16 scale exponent s of the activations: x * 2^-s keeps amax below 2^15.
__device__ __forceinline__ int f16_shift(unsigned int amax_bits) {
    const int e = (int)((amax_bits >> 23) & 0xFF) - 127;   // floor(log2(amax)) for normal amax
    return e > 14 ? e - 14 : 0;
}

__device__ __forceinline__ uint32_t idesc_f16(uint32_t n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// D[tmem] (+)= A[tmem] x B[smem descriptor]
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Token-row class of a tile: 0, 1, 2 for up to 16, 32, 64 rows; the MMA N is
// 16 << class and a B stage holds (8 >> class) boxes of 64 K values.
__device__ __forceinline__ int hrows_class(int valid) { return valid <= 16 ? 0 : (valid <= 32 ? 1 : 2); }

// Item = kh * (n_tiles * nf) + tile * nf + f: the tile's token rows against
// weight-row group f, part kh of K when the caller splits K (ks parts; the
// kernels here use ks = 1: a split of the down items measured slower at
// decode).  For many tokens the down items run column group first,
// (kh * nf + f) * n_tiles + tile, so the accumulator slice being added into
// stays in L2 (see decode_item).  Returns false for a group past the expert's
// intermediate size or an empty part of K.
__device__ __forceinline__ bool decode_item_h(const HcArgs &a, int item, int epi, int ks, Item &it) {
    const int nt = a.scratch->n_tiles;
    int tile, kh = 0;
    if (epi == kScatter && a.colfirst) {
        tile = item % nt;
        const int rest = item / nt;
        it.f = rest % a.nf;
        kh = rest / a.nf;
    } else {
        const int per = nt * a.nf;
        kh = item / per;
        tile = (item % per) / a.nf;
        it.f = (item % per) % a.nf;
    }
    const int4 t = a.tiles[tile];
    it.e = t.x;
    it.row0 = t.y;
    it.valid = min(t.z, kHBRows);
    it.sh = (t.x == a.E);
    const int I = it.sh ? a.Is : a.I;
    it.K = epi == kSwiGLU ? a.H : I;
    const int stages = it.K / kHCK, per = (stages + ks - 1) / ks;
    it.kc0 = kh * per;
    it.kc1 = min(stages, it.kc0 + per);
    if (epi == kSwiGLU) return it.f * 128 < I;
    return it.kc0 < it.kc1;
}

__device__ __forceinline__ void h_rows(const HcArgs &a, const Item &it, int epi, int &r0, int &r1) {
    if (epi == kSwiGLU) {
        r0 = r1 = (it.sh ? 0 : it.e * a.I) + it.f * 128;
    } else {
        r0 = (it.sh ? 0 : it.e * a.H) + it.f * 256;
        r1 = r0 + 128;
    }
}

// Item order of the warp-MMA engine. The grid (one CTA an SM) takes items in
// rounds; when the last round would leave most SMs idle, each of its items is
// split along K into `parts` pieces (2 to kMaxTailParts, as many as the grid
// holds), so the round runs parts x as many shorter pieces. Down pieces add
// into the fp32 accumulator like whole items; gate/up pieces leave partial
// sums, and the last piece of each to finish adds them in piece order and
// applies SwiGLU.
struct RegSplit {
    int n_whole;   // items before the split round
    int parts;     // pieces a split item is cut into (1: no split)
    int n_items;   // flat items, pieces counted one by one
};

__device__ __forceinline__ RegSplit reg_split(const HcArgs &a) {
    const int n_full = a.scratch->n_tiles * a.nf;
    const int W = gridDim.x, r = n_full % W;
    RegSplit s;
    s.parts = (a.tail_split && r > 0 && 2 * r <= W) ? min(kMaxTailParts, W / r) : 1;
    s.n_whole = s.parts > 1 ? n_full - r : n_full;
    s.n_items = s.n_whole + (n_full - s.n_whole) * s.parts;
    return s;
}

__device__ __forceinline__ bool decode_item_r(const HcArgs &a, const RegSplit &rs, int item, int epi, Item &it) {
    int base = item, part = 0, parts = 1, slot = -1;
    if (item >= rs.n_whole) {
        const int j = item - rs.n_whole;
        slot = j / rs.parts;
        base = rs.n_whole + slot;
        part = j % rs.parts;
        parts = rs.parts;
    }
    if (!decode_item_h(a, base, epi, 1, it)) return false;
    if (parts > 1) {
        // pieces of `per` stages; as many pieces as that takes (never an empty one)
        const int stages = it.kc1 - it.kc0, per = (stages + parts - 1) / parts;
        parts = (stages + per - 1) / per;
        if (part >= parts) return false;
        it.kc1 = min(it.kc1, it.kc0 + (part + 1) * per);
        it.kc0 += part * per;
        it.part = part;
        it.parts = parts;
        it.slot = slot;
    }
    return true;
}

// One ring position: index in the ring and the parity of its current use.
struct RingPos {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) { s = 0; ph ^= 1; }
    }
};

template <int EPI>
__global__ void __launch_bounds__(kHThreads, 1) k_gemm_f16(const __grid_constant__ HcArgs a) {
    pdl_wait();      // routing, permute or gate/up results come from the previous kernel
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *code_ring = smem;
    uint8_t *b_ring = code_ring + kHCStages * kHCodeStage;
    uint64_t *cfull = reinterpret_cast<uint64_t *>(b_ring + kHBStages * kHBTile);
    uint64_t *cempty = cfull + kHCStages;
    uint64_t *bfull = cempty + kHCStages;
    uint64_t *bempty = bfull + kHBStages;
    uint64_t *afull = bempty + kHBStages;
    uint64_t *aempty = afull + kHAStages;
    uint64_t *acc_full = aempty + kHAStages;     // [2]
    uint64_t *acc_empty = acc_full + 2;          // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = 1;   // no split of K here
    const int n_items = a.scratch->n_tiles * a.nf;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kHCStages; ++i) { mbar_init(cfull + i, 1); mbar_init(cempty + i, kConvWarps); }
        for (int i = 0; i < kHBStages; ++i) { mbar_init(bfull + i, 1); mbar_init(bempty + i, 2); }
        for (int i = 0; i < kHAStages; ++i) { mbar_init(afull + i, kConvWarps); mbar_init(aempty + i, 2); }
        for (int i = 0; i < 2; ++i) { mbar_init(acc_full + i, 2); mbar_init(acc_empty + i, kHEpiWarps); }
        mbar_init(drain, 2);                // both MMA lanes commit
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------- producer of the code ring
            RingPos c;
            bool ok = true;
            uint32_t used = 0, last_ph = 0;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item_h(a, item, EPI, ks, it)) continue;
                const int m = it.sh ? 1 : 0;
                int r0, r1;
                h_rows(a, it, EPI, r0, r1);
                const CUtensorMap *A1 = (EPI == kSwiGLU) ? &a.a1[m] : &a.a0[m];
                const CUtensorMap *S1 = (EPI == kSwiGLU) ? &a.s1[m] : &a.s0[m];
                for (int kc = it.kc0; kc < it.kc1; ++kc) {
                    if (!mbar_wait(cempty + c.s, c.ph ^ 1, a.err)) { ok = false; break; }
                    uint8_t *st = code_ring + c.s * kHCodeStage;
                    mbar_expect_tx(cfull + c.s, kHCodeStage);
                    tma_2d(st, &a.a0[m], cfull + c.s, kc * 128, r0);
                    tma_2d(st + kHCodeTile, A1, cfull + c.s, kc * 128, r1);
                    tma_2d(st + 2 * kHCodeTile, &a.s0[m], cfull + c.s, kc * 16, r0);
                    tma_2d(st + 2 * kHCodeTile + 2048, S1, cfull + c.s, kc * 16, r1);
                    used |= 1u << c.s;
                    last_ph = (last_ph & ~(1u << c.s)) | (c.ph << c.s);
                    c.next(kHCStages);
                }
            }
            for (int t = 0; t < kHCStages; ++t)
                if (used & (1u << t)) mbar_wait(cfull + t, (last_ph >> t) & 1u, a.err);
        } else if (lane == 1) {
            // ---------------------------------------- producer of the B ring
            RingPos b;
            bool ok = true;
            uint32_t used = 0, last_ph = 0;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item_h(a, item, EPI, ks, it)) continue;
                const int rc = hrows_class(it.valid);
                const int rows = 16 << rc, boxes = 8 >> rc, nq = it.K / kHBK;
                for (int q0 = 0; q0 < nq; q0 += boxes) {
                    const int nb = min(boxes, nq - q0);   // the item's last stage may hold fewer boxes
                    if (!mbar_wait(bempty + b.s, b.ph ^ 1, a.err)) { ok = false; break; }
                    mbar_expect_tx(bfull + b.s, (uint32_t)(nb * rows * 128));
                    for (int bx = 0; bx < nb; ++bx)
                        tma_2d(b_ring + b.s * kHBTile + bx * rows * 128, &a.b[rc], bfull + b.s,
                               (q0 + bx) * kHBK, it.row0);
                    used |= 1u << b.s;
                    last_ph = (last_ph & ~(1u << b.s)) | (b.ph << b.s);
                    b.next(kHBStages);
                }
            }
            for (int t = 0; t < kHBStages; ++t)
                if (used & (1u << t)) mbar_wait(bfull + t, (last_ph >> t) & 1u, a.err);
        }
    } else if (warp >= 2 && warp < 2 + kConvWarps) {
        // ------------------------------------------------ NVFP4 -> f16 converters
        // warp (operand op, K half hf, lane quarter q): thread row c = 32 q +
        // lane of operand op.  Per code stage it loads its row's code chunks
        // 2j + hf (j < 4) and scale bytes, then per A stage j widens those 32 K
        // values (two scale blocks) into 16 TMEM columns of its lane.
        const int cw = (warp - 2) >> 2;
        const int op = cw & 1, hf = cw >> 1;
        const int q = warp & 3;
        const int c = q * 32 + lane;
        const uint32_t sw = (uint32_t)(c & 7);
        const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + kHACol0 + op * (kHAK / 2) + hf * kConvCols;
        const uint32_t ring0 = smem_u32(code_ring);
        RingPos cs, as;
        bool ok = true;
        // The TMEM store of A stage j completes (tcgen05.wait::st, then afull)
        // only after stage j + 1 is widened in registers, so the store's
        // latency overlaps the conversion work instead of adding to it.
        int pend = -1;   // A slot whose store is in flight
        auto finish_pending = [&]() {
            if (pend >= 0) {
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull + pend);
                pend = -1;
            }
        };
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            Item it;
            if (!decode_item_h(a, item, EPI, ks, it)) continue;
            for (int kc = it.kc0; ok && kc < it.kc1; ++kc) {
                if (!mbar_wait(cfull + cs.s, cs.ph, a.err)) { ok = false; break; }
                const uint32_t st = ring0 + cs.s * kHCodeStage;
                const uint32_t row = st + op * kHCodeTile + c * 128;
                // A stage j (K 128 j .. 128 j + 127): this warp's half hf is the
                // code chunks 4 j + 2 hf and 4 j + 2 hf + 1 (32 K values each)
                uint4 cq[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cq[j] = lds128(row + (((uint32_t)(4 * (j >> 1) + 2 * hf + (j & 1)) ^ sw) << 4));
                const uint4 scv = lds128(st + 2 * kHCodeTile + op * 2048 + c * 16);
                const uint32_t scw[4] = {scv.x, scv.y, scv.z, scv.w};
                __syncwarp();
                if (lane == 0) mbar_arrive(cempty + cs.s);   // this warp's bytes are in registers
                cs.next(kHCStages);
#pragma unroll
                for (int j = 0; j < kHCK / kHAK; ++j) {
                    uint32_t o[kConvCols];
                    // its scale blocks 8 j + 4 hf .. + 3: word 2 j + hf of the row's 16 bytes
                    const uint32_t sw4 = scw[2 * j + hf];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 cc = cq[2 * j + i];
                        const uint32_t cw4[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
                            const uint32_t sb = (sw4 >> (8 * (2 * i + blk))) & 0xFFu;
                            const uint32_t sc2 = e4m3x2_to_f16x2(sb * 0x101u);
                            uint32_t h[8];
                            e2m1x8_to_f16x8(cw4[2 * blk], *reinterpret_cast<uint32_t(*)[4]>(h));
                            e2m1x8_to_f16x8(cw4[2 * blk + 1], *reinterpret_cast<uint32_t(*)[4]>(h + 4));
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&h[e]),
                                                    *reinterpret_cast<const __half2 *>(&sc2));
                                o[i * 16 + blk * 8 + e] = *reinterpret_cast<uint32_t *>(&v);
                            }
                        }
                    }
                    finish_pending();
                    if (ok && !mbar_wait(aempty + as.s, as.ph ^ 1, a.err)) ok = false;
                    if (ok) {
                        tmem_st16(t_lane + as.s * kHAK, *reinterpret_cast<const uint32_t(*)[16]>(o));
                        tmem_st16(t_lane + as.s * kHAK + 16, *reinterpret_cast<const uint32_t(*)[16]>(o + 16));
                        pend = as.s;
                    }
                    as.next(kHAStages);
                }
            }
        }
        finish_pending();
    } else if (warp == 1 || warp == kHMma2) {
        // ------------------------------------------------ MMA issue: one lane an accumulator half
        if (lane == 0) {
            const int hs = warp == 1 ? 0 : 1;   // columns +64 hs of the accumulator, A columns +32 hs
            RingPos as, bs;
            int buf = 0;
            uint32_t aph = 0;   // bit b: parity of accumulator buffer b
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item_h(a, item, EPI, ks, it)) continue;
                if (!mbar_wait(acc_empty + buf, ((aph >> buf) & 1u) ^ 1u, a.err)) break;
                aph ^= 1u << buf;
                tc_fence_after();
                const uint32_t d = tmem + buf * 128 + 64 * hs;
                const int rc = hrows_class(it.valid);
                const int rows = 16 << rc, boxes = 8 >> rc, nqa = it.K / kHAK;
                constexpr int kBoxesA = kHAK / kHBK;   // B boxes (64 K values each) an A stage takes
                const uint32_t idesc = idesc_f16((uint32_t)rows);
                for (int qa = 0; qa < nqa; ++qa) {
                    const int b0 = (qa * kBoxesA) % boxes;   // the A stage's first box in its B stage
                    if (!mbar_wait(afull + as.s, as.ph, a.err) || (b0 == 0 && !mbar_wait(bfull + bs.s, bs.ph, a.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + kHACol0 + as.s * kHAK + (kHAK / 2) * hs;
                    const uint64_t bd0 = desc_sw128(smem_u32(b_ring + bs.s * kHBTile) + b0 * rows * 128);
                    const uint32_t box_units = (uint32_t)(rows * 128) >> 4;   // a box in descriptor address units
#pragma unroll
                    for (int kk = 0; kk < kHAK / 16; ++kk) {
                        const uint32_t accum = (qa | kk) ? 1u : 0u;
                        const uint64_t bd = bd0 + (uint64_t)((kk >> 2) * box_units + 2 * (kk & 3));
                        mma_f16_ts(d, at + 8 * kk, bd, idesc, accum);
                    }
                    mma_commit(aempty + as.s);
                    as.next(kHAStages);
                    if (b0 + kBoxesA == boxes || qa == nqa - 1) {
                        mma_commit(bempty + bs.s);
                        bs.next(kHBStages);
                    }
                }
                if (!ok) break;
                mma_commit(acc_full + buf);
                buf ^= 1;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, a.err);
        }
    } else {
        // ------------------------------------------------ epilogue (4 warps)
        const int quad = warp & 3;
        int buf = 0;
        uint32_t aph = 0;   // bit b: parity of accumulator buffer b
        const int xs = f16_shift(a.scratch->x_amax);
        const float xunscale = __uint_as_float((uint32_t)(127 + xs) << 23);   // 2^s
        bool range_bad = false;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            Item it;
            if (!decode_item_h(a, item, EPI, ks, it)) continue;
            if (!mbar_wait(acc_full + buf, (aph >> buf) & 1u, a.err)) break;
            aph ^= 1u << buf;
            tc_fence_after();
            const uint32_t lane_base = tmem + buf * 128 + ((uint32_t)(quad * 32) << 16);
            const int m = it.sh ? 1 : 0;
            const int e = it.sh ? 0 : it.e;
            const int n_end = it.valid;
            if (EPI == kSwiGLU) {
                const float sg = a.ts_a0[m][e] * xunscale, su = a.ts_a1[m][e] * xunscale;
                const int feat = it.f * 128 + quad * 32 + lane;
                for (int n0 = 0; n0 < n_end; n0 += 16) {
                    float g[16], u[16];
                    tmem_ld16_nowait(lane_base + n0, g);
                    tmem_ld16_nowait(lane_base + 64 + n0, u);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (n0 + j < n_end) {
                            const float gv = g[j] * sg, uv = u[j] * su;
                            // SwiGLU output rounded to bf16 (W4A16), then held as f16 for the down MMA
                            const float hb = __bfloat162float(__float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv));
                            range_bad |= fabsf(hb) > 65504.0f;
                            a.hout[(size_t)(it.row0 + n0 + j) * a.hstride + feat] = __float2half_rn(hb);
                        }
                    }
                }
            } else {
                const float ds = a.ts_a0[m][e];
                int tok[2];
                float wgt[2];
#pragma unroll
                for (int qd = 0; qd < 2; ++qd) {
                    const int n = lane + 32 * qd;
                    tok[qd] = 0;
                    wgt[qd] = 0.0f;
                    if (n < it.valid) {
                        const int pair = a.pad_pair[it.row0 + n];
                        tok[qd] = pair >= a.P ? pair - a.P : pair / a.k;
                        wgt[qd] = pair >= a.P ? 1.0f : a.wts[pair];
                    }
                }
                const int j0 = it.f * 256 + quad * 32 + lane;
                for (int n0 = 0; n0 < n_end; n0 += 16) {
                    float y0[16], y1[16];
                    tmem_ld16_nowait(lane_base + n0, y0);
                    tmem_ld16_nowait(lane_base + 64 + n0, y1);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int cc = n0 + j;
                        const int t = __shfl_sync(0xffffffffu, (cc >> 5) ? tok[1] : tok[0], cc & 31);
                        const float wv = __shfl_sync(0xffffffffu, (cc >> 5) ? wgt[1] : wgt[0], cc & 31) * ds;
                        if (cc < n_end) {
                            float *dst = a.acc + (size_t)t * a.H + j0;
                            atomicAdd(dst, y0[j] * wv);
                            atomicAdd(dst + 128, y1[j] * wv);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + buf);
            buf ^= 1;
        }
        if (__any_sync(0xffffffffu, range_bad) && lane == 0) atomicOr(a.err, kErrDevice);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
    }
}

// ------------------------------------------------------------------ W4A16, register path
// W4A16 for tiles of up to 32 token rows (decode and short prompts): E2M1
// codes are widened in registers straight into the A fragments of warp-level
// f16 MMAs (m16n8k16, fp32 accumulation), so no widened copy of the weights
// is ever stored.  The weight codes and scales arrive through the same TMA
// code ring as the tcgen05 kernel (4 x 36 KB, 128 weight rows of two operands,
// 256 K values a stage); the f16 token rows through a 3-stage ring (256 K
// values a stage).  Sixteen compute warps: warp (row group rg, operand op)
// owns 16 rows of one operand and all K.
//
// K order inside a 128-value group: lane quad q (lane & 3) holds the 32
// consecutive K values 32q .. 32q+31, i.e. exactly two scale blocks, so a lane
// scales each of its codes with one E4M3 value a row and block; MMA m (0..3)
// of block b takes K values 32q + 16b + 4m + {0,1} as fragment columns 2q,
// 2q+1 and 32q + 16b + 4m + {2,3} as 2q+8, 2q+9.  The token-row fragments use
// the same map, so the sum is the same dot product in another order.
constexpr int kRThreads = 32 * (2 + 16);          // TMA producer, token-row gatherer, 16 compute warps
constexpr int kRXchg = 8 * 4 * 32 * 4 * 4;        // 16 KB: up-operand accumulators handed to the gate warps
// Ring geometry a launch picks: with at most 16 tokens every tile has at most
// 16 rows, token-row slots of 8 KB suffice and the token-row ring gets a
// fourth stage (a fifth weight stage measured no faster).
struct RegRings { int cst, bst, bslot; };
constexpr RegRings kRegSmall{4, 4, 16 * 512}, kRegLarge{4, 3, 32 * 512};
// Per-CTA table of the launch's items, filled once by warp 1 at the start with
// all their global reads in flight together (the work list, the token and the
// routing weight of every row, the tensor scales), so the compute warps start
// each item from shared memory instead of a chain of dependent global loads.
// A CTA with more items than the table holds decodes the rest as it goes.
constexpr int kMetaItems = 32;
struct RegMeta {
    int e, row0, valid, f, sh, kc0, kc1, part, parts, slot, ok, pad;
    float ts0, ts1, pad2[2];
    int tok[32];      // token of row n (rows < valid)
    float w[32];      // routing weight of row n (1 for the shared expert)
};
constexpr size_t kMetaBytes = sizeof(RegMeta) * kMetaItems;
constexpr size_t reg_smem(RegRings r) {
    return (size_t)r.cst * kHCodeStage + (size_t)r.bst * r.bslot + kRXchg + kMetaBytes + 512 + 1024;
}
constexpr size_t kRSmemBytes = reg_smem(kRegSmall) > reg_smem(kRegLarge) ? reg_smem(kRegSmall) : reg_smem(kRegLarge);
static_assert(kRSmemBytes <= 227 * 1024, "register-path pipeline exceeds shared memory");

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 256-value K stage of a compute warp.  Token rows come from the token-row
// ring slot `bst` (RES = false), or (RES = true, one 8-row token tile) from the
// resident activations: `bst` is then the shared-memory address of this lane's
// token row, `xsw` its 16-byte chunk swizzle and `kc` the stage index.
// E8M0 scale byte -> f16 bits of 2^(byte - 127), for MXFP4 weights on the f16
// MMAs: code x scale is exact in f16 for byte 104 .. 140 (2^-23 .. 2^13); byte
// 0 (an all-zero block) gives 0; any other byte gives 0 and sets `bad`.
__device__ __forceinline__ uint32_t e8m0_f16_bits(uint32_t e, bool &bad) {
    if (e >= 113 && e <= 140) return (e - 112) << 10;   // normal f16
    if (e >= 104 && e < 113) return 1u << (e - 103);    // subnormal f16
    bad |= e != 0;
    return 0;
}

template <int NT, bool RES = false, int MX = 0>
__device__ __forceinline__ void reg_stage(uint32_t st, uint32_t bst, int op, int rg, int lane, float (&acc)[4][4],
                                          int kc = 0, uint32_t xsw = 0, bool *bad = nullptr) {
    const int g = lane >> 2, q = lane & 3;
    const int r0 = rg * 16 + g, r1 = r0 + 8;
    const uint32_t crow0 = st + op * kHCodeTile + r0 * 128, crow1 = st + op * kHCodeTile + r1 * 128;
    const uint4 sv0 = lds128(st + 2 * kHCodeTile + op * 2048 + r0 * 16);
    const uint4 sv1 = lds128(st + 2 * kHCodeTile + op * 2048 + r1 * 16);
    const uint32_t sw0[4] = {sv0.x, sv0.y, sv0.z, sv0.w}, sw1[4] = {sv1.x, sv1.y, sv1.z, sv1.w};
    const uint32_t ssel = (uint32_t)q | ((uint32_t)(4 + q) << 4);   // byte q of the r0 word, then of the r1 word
#pragma unroll
    for (int sb = 0; sb < 4; ++sb) {
        const uint32_t ch = (uint32_t)(2 * sb + (q >> 1));
        uint2 c0, c1;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(c0.x), "=r"(c0.y) : "r"(crow0 + ((ch ^ (uint32_t)(r0 & 7)) << 4) + (q & 1) * 8) : "memory");
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(c1.x), "=r"(c1.y) : "r"(crow1 + ((ch ^ (uint32_t)(r1 & 7)) << 4) + (q & 1) * 8) : "memory");
        // scale bytes of block 4 sb + q for rows r0 (low byte) and r1 (next byte);
        // MXFP4: the slot's 16 scale bytes a row cover this stage and its pair
        // (stage kc & 1 of them), block 2 sb + q / 2 of the stage
        uint32_t sc;
        if (MX) {
            const int w = 2 * (kc & 1) + (sb >> 1), bsel = 2 * (sb & 1) + (q >> 1);
            const uint32_t two = __byte_perm(sw0[w], sw1[w], (uint32_t)bsel | ((uint32_t)(4 + bsel) << 4));
            bool b = false;
            sc = e8m0_f16_bits(two & 0xFFu, b) | (e8m0_f16_bits((two >> 8) & 0xFFu, b) << 16);
            if (b) *bad = true;
        } else {
            sc = e4m3x2_to_f16x2(__byte_perm(sw0[sb], sw1[sb], ssel));
        }
        __half2 sc0 = __low2half2(*reinterpret_cast<const __half2 *>(&sc));
        __half2 sc1 = __high2half2(*reinterpret_cast<const __half2 *>(&sc));
        uint32_t h0[8], h1[8];
        e2m1x8_to_f16x8(c0.x, *reinterpret_cast<uint32_t(*)[4]>(h0));
        e2m1x8_to_f16x8(c0.y, *reinterpret_cast<uint32_t(*)[4]>(h0 + 4));
        e2m1x8_to_f16x8(c1.x, *reinterpret_cast<uint32_t(*)[4]>(h1));
        e2m1x8_to_f16x8(c1.y, *reinterpret_cast<uint32_t(*)[4]>(h1 + 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            __half2 v0 = __hmul2(*reinterpret_cast<const __half2 *>(&h0[i]), sc0);
            __half2 v1 = __hmul2(*reinterpret_cast<const __half2 *>(&h1[i]), sc1);
            h0[i] = *reinterpret_cast<uint32_t *>(&v0);
            h1[i] = *reinterpret_cast<uint32_t *>(&v1);
        }
        // token-row fragments: row n = 8 nt + g, K values 64 sb + 16 q .. +16 (box sb of the stage)
        uint4 bx[NT][2];
        if (RES) {
            // K values kc*256 + 64 sb + 16 q .. +16 of the token: 16-byte chunks c0, c0 + 1
            const uint32_t c0 = (uint32_t)(kc * 32 + sb * 8 + 2 * q);
            bx[0][0] = lds128(bst + ((c0 ^ xsw) << 4));
            bx[0][1] = lds128(bst + (((c0 + 1) ^ xsw) << 4));
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int n = nt * 8 + g;
                const uint32_t brow = bst + (uint32_t)sb * (NT > 2 ? 32 : 16) * 128 + n * 128;
                bx[nt][0] = lds128(brow + (((uint32_t)(2 * q) ^ (uint32_t)(n & 7)) << 4));
                bx[nt][1] = lds128(brow + (((uint32_t)(2 * q + 1) ^ (uint32_t)(n & 7)) << 4));
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t a[4] = {h0[2 * m], h1[2 * m], h0[2 * m + 1], h1[2 * m + 1]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 &b = bx[nt][m >> 1];
                mma16816(acc[nt], a, (m & 1) ? b.z : b.x, (m & 1) ? b.w : b.y);
            }
        }
    }
}

// Items of this CTA: blockIdx.x + j * gridDim.x for j < cta_items.
__device__ __forceinline__ int cta_items(int n_items) {
    return n_items > (int)blockIdx.x ? (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

// Warp 1: fill the item table.  Lane j decodes item j; then the token and
// routing weight of every row of every item are read, four items' reads in
// flight at a time.  Returns the number of entries.
template <int EPI>
__device__ __forceinline__ int reg_fill_meta(const HcArgs &a, const RegSplit &rs, RegMeta *meta, int lane) {
    const int n_tab = min(cta_items(rs.n_items), kMetaItems);
    if (lane < n_tab) {
        Item it;
        RegMeta &m = meta[lane];
        const bool ok = decode_item_r(a, rs, (int)blockIdx.x + lane * (int)gridDim.x, EPI, it);
        m.ok = ok;
        if (ok) {
            m.e = it.e;
            m.row0 = it.row0;
            m.valid = it.valid;
            m.f = it.f;
            m.sh = it.sh;
            m.kc0 = it.kc0;
            m.kc1 = it.kc1;
            m.part = it.part;
            m.parts = it.parts;
            m.slot = it.slot;
            const int mm = it.sh ? 1 : 0, e = it.sh ? 0 : it.e;
            m.ts0 = a.ts_a0[mm][e];
            m.ts1 = EPI == kSwiGLU ? a.ts_a1[mm][e] : 0.0f;
        }
    }
    __syncwarp();
    for (int j0 = 0; j0 < n_tab; j0 += 4) {
        int pr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u;
            pr[u] = -1;
            if (j < n_tab && meta[j].ok && lane < meta[j].valid) pr[u] = a.pad_pair[meta[j].row0 + lane];
        }
        float wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) wv[u] = (EPI == kScatter && pr[u] >= 0 && pr[u] < a.P) ? a.wts[pr[u]] : 1.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u;
            if (j < n_tab) {
                meta[j].tok[lane] = pr[u] < 0 ? 0 : (pr[u] >= a.P ? pr[u] - a.P : pr[u] / a.k);
                meta[j].w[lane] = wv[u];
            }
        }
    }
    return n_tab;
}

// Compute warps of k_gemm_reg (warps 2..17).
template <int EPI, int MX>
__device__ __forceinline__ void reg_compute(const HcArgs &a, int warp, int lane, uint8_t *code_ring, uint8_t *b_ring,
                                            float *xchg, uint64_t *cfull, uint64_t *cempty, uint64_t *bfull,
                                            uint64_t *bempty, uint64_t *xfull, uint64_t *xempty,
                                            const RegMeta *meta, uint64_t *meta_ready, uint64_t *x_full) {
    const RegSplit rs = reg_split(a);
    const int n_items = rs.n_items;
    const int cw = warp - 2, rg = cw & 7, op = cw >> 3;
    const int g = lane >> 2, q = lane & 3;
    const uint32_t ring0 = smem_u32(code_ring), bring0 = smem_u32(b_ring);
    const int xs = f16_shift(a.scratch->x_amax);
    const float xunscale = __uint_as_float((uint32_t)(127 + xs) << 23);   // 2^s
    const bool res = EPI == kSwiGLU && a.xres > 0;
    bool ok = true, range_bad = false;
    if (res) {
        // resident activations: the raw bf16 rows (copied at launch) -> f16 x 2^-s
        // in place, each 128-byte group of a row written with its 16-byte chunks
        // permuted by the token's row index (c -> c ^ (t & 7)), so the lanes
        // reading different tokens' rows hit different banks
        ok = mbar_wait(x_full, 0, a.err);
        const float scale = __uint_as_float((uint32_t)(127 - xs) << 23);   // 2^-s
        const int gpr = a.H * 2 / 128;                                       // groups a row
        for (int gi = cw * 32 + lane; ok && gi < a.xres * gpr; gi += 16 * 32) {
            const uint32_t base = bring0 + (uint32_t)gi * 128, sw = (uint32_t)((gi / gpr) & 7);
            uint4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = lds128(base + 16 * c);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t u[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    __half2 hh = __floats2half2_rn(__uint_as_float(u[h] << 16) * scale,
                                                   __uint_as_float(u[h] & 0xFFFF0000u) * scale);
                    u[h] = *reinterpret_cast<uint32_t *>(&hh);
                }
                v[c] = make_uint4(u[0], u[1], u[2], u[3]);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) sts128(base + 16 * ((uint32_t)c ^ sw), v[c]);
        }
        asm volatile("bar.sync 1, 512;" ::: "memory");   // the 16 compute warps
        ok = __all_sync(0xffffffffu, ok);
    }
    const int n_tab = min(cta_items(n_items), kMetaItems);
    if (ok && n_tab > 0) ok = mbar_wait(meta_ready, 0, a.err);
    RingPos cs, bs;
    uint32_t xph = 0;
    int ji = -1;   // index of the item among this CTA's
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        ++ji;
        Item it;
        float ts0, ts1;
        // epilogue inputs: tensor scales and the (token, weight) of this lane's
        // first two columns (from the item table, or read now so their latency
        // hides behind the K loop)
        int tk[2] = {0, 0};
        float wt[2] = {0.0f, 0.0f};
        int xtok = 0;   // resident activations: this lane's token row (row g; padding rows read row 0's)
        if (ji < n_tab) {
            const RegMeta &m = meta[ji];
            if (!m.ok) continue;
            it.e = m.e;
            it.row0 = m.row0;
            it.valid = m.valid;
            it.f = m.f;
            it.sh = m.sh;
            it.kc0 = m.kc0;
            it.kc1 = m.kc1;
            it.part = m.part;
            it.parts = m.parts;
            it.slot = m.slot;
            ts0 = m.ts0;
            ts1 = m.ts1;
            if (EPI == kScatter) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int n = 2 * q + c;
                    if (n < it.valid) { tk[c] = m.tok[n]; wt[c] = m.w[n]; }
                }
            }
            if (res) xtok = m.tok[g < it.valid ? g : 0];
        } else {
            if (!decode_item_r(a, rs, item, EPI, it)) continue;
            const int mm = it.sh ? 1 : 0;
            const int e = it.sh ? 0 : it.e;
            ts0 = a.ts_a0[mm][e];
            ts1 = EPI == kSwiGLU ? a.ts_a1[mm][e] : 0.0f;
            if (EPI == kScatter) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int n = 2 * q + c;
                    if (n < it.valid) {
                        const int pair = a.pad_pair[it.row0 + n];
                        tk[c] = pair >= a.P ? pair - a.P : pair / a.k;
                        wt[c] = pair >= a.P ? 1.0f : a.wts[pair];
                    }
                }
            }
            if (res) {
                const int pair = a.pad_pair[it.row0 + (g < it.valid ? g : 0)];
                xtok = pair >= a.P ? pair - a.P : pair / a.k;
            }
        }
        const int nt_n = (it.valid + 7) >> 3;
        const uint32_t xrow = bring0 + (uint32_t)xtok * (uint32_t)a.H * 2u, xsw = (uint32_t)(xtok & 7);
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[i][jj] = 0.0f;
        for (int kc = it.kc0; kc < it.kc1; ++kc) {
            if (!mbar_wait(cfull + cs.s, cs.ph, a.err) || (!res && !mbar_wait(bfull + bs.s, bs.ph, a.err))) {
                ok = false;
                break;
            }
            const uint32_t st = ring0 + cs.s * kHCodeStage, bst = bring0 + bs.s * a.rbslot;
            if (res) {
                reg_stage<1, true, MX>(st, xrow, op, rg, lane, acc, kc, xsw, &range_bad);
            } else {
                switch (nt_n) {
                    case 1: reg_stage<1, false, MX>(st, bst, op, rg, lane, acc, kc, 0, &range_bad); break;
                    case 2: reg_stage<2, false, MX>(st, bst, op, rg, lane, acc, kc, 0, &range_bad); break;
                    case 3: reg_stage<3, false, MX>(st, bst, op, rg, lane, acc, kc, 0, &range_bad); break;
                    default: reg_stage<4, false, MX>(st, bst, op, rg, lane, acc, kc, 0, &range_bad); break;
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(cempty + cs.s);
                if (!res) mbar_arrive(bempty + bs.s);
            }
            cs.next(a.rcst);
            if (!res) bs.next(a.rbst);
        }
        if (!ok) break;
        if (EPI == kSwiGLU) {
            float *slot = xchg + (size_t)rg * (4 * 32 * 4);
            if (op == 1) {   // up warp: hand the accumulators to the gate warp of the same rows
                if (!mbar_wait(xempty + rg, xph ^ 1, a.err)) { ok = false; break; }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    if (nt < nt_n)
                        *reinterpret_cast<float4 *>(slot + (nt * 32 + lane) * 4) =
                            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(xfull + rg);
            } else {
                if (!mbar_wait(xfull + rg, xph, a.err)) { ok = false; break; }
                float up[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    float4 u4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (nt < nt_n) u4 = *reinterpret_cast<const float4 *>(slot + (nt * 32 + lane) * 4);
                    up[nt][0] = u4.x;
                    up[nt][1] = u4.y;
                    up[nt][2] = u4.z;
                    up[nt][3] = u4.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xempty + rg);
                bool last = true;
                if (it.parts > 1) {
                    // a K piece: leave this piece's partial sums, then take the
                    // (item, row group) ticket; the last piece to arrive adds all
                    // pieces in piece order (the same sum whichever finishes last)
                    // and goes on to SwiGLU
                    const size_t stride = 4 * 32 * 8;
                    float *mine = a.tail_part + ((size_t)(it.slot * rs.parts + it.part) * 8 + rg) * stride;
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        if (nt >= nt_n) break;
                        float4 *dst = reinterpret_cast<float4 *>(mine + (nt * 32 + lane) * 8);
                        __stcg(dst, make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]));
                        __stcg(dst + 1, make_float4(up[nt][0], up[nt][1], up[nt][2], up[nt][3]));
                    }
                    __threadfence();
                    __syncwarp();
                    int arrived = 0;
                    if (lane == 0) arrived = atomicAdd(a.tickets + it.slot * 8 + rg, 1);
                    last = __shfl_sync(0xffffffffu, arrived, 0) == it.parts - 1;
                    if (last) {
                        __threadfence();
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            if (nt >= nt_n) break;
                            float gs[4] = {0.0f, 0.0f, 0.0f, 0.0f}, us[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            for (int pc = 0; pc < it.parts; ++pc) {
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    a.tail_part + ((size_t)(it.slot * rs.parts + pc) * 8 + rg) * stride + (nt * 32 + lane) * 8);
                                const float4 g4 = __ldcg(src), u4 = __ldcg(src + 1);
                                gs[0] += g4.x; gs[1] += g4.y; gs[2] += g4.z; gs[3] += g4.w;
                                us[0] += u4.x; us[1] += u4.y; us[2] += u4.z; us[3] += u4.w;
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                acc[nt][i] = gs[i];
                                up[nt][i] = us[i];
                            }
                        }
                    }
                }
                if (last) {
                    const float sg = ts0 * xunscale, su = ts1 * xunscale;
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        if (nt >= nt_n) break;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int n = nt * 8 + 2 * q + (i & 1);
                            const int feat = it.f * 128 + rg * 16 + g + (i >> 1) * 8;
                            if (n < it.valid) {
                                const float gv = acc[nt][i] * sg, uv = up[nt][i] * su;
                                // SwiGLU output rounded to bf16 (W4A16), held as f16 for the down product
                                const float hb = __bfloat162float(__float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv));
                                range_bad |= fabsf(hb) > 65504.0f;
                                a.hout[(size_t)(it.row0 + n) * a.hstride + feat] = __float2half_rn(hb);
                            }
                        }
                    }
                }
            }
            xph ^= 1;
        } else {
            const float ds = ts0;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                if (nt >= nt_n) break;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int n = nt * 8 + 2 * q + (i & 1);
                    if (n < it.valid) {
                        int t;
                        float wv;
                        if (nt == 0) {
                            t = tk[i & 1];
                            wv = wt[i & 1] * ds;
                        } else {
                            const int pair = a.pad_pair[it.row0 + n];
                            t = pair >= a.P ? pair - a.P : pair / a.k;
                            wv = (pair >= a.P ? 1.0f : a.wts[pair]) * ds;
                        }
                        const int j = it.f * 256 + op * 128 + rg * 16 + g + (i >> 1) * 8;
                        atomicAdd(a.acc + (size_t)t * a.H + j, acc[nt][i] * wv);
                    }
                }
            }
        }
    }
    if (__any_sync(0xffffffffu, range_bad) && lane == 0) atomicOr(a.err, kErrDevice);
}

// Token-row gatherer of the gate/up launch (one warp): builds each 256-value
// K stage of the tile's f16 token rows straight from x (bf16 -> f16 x 2^-s,
// exact), in the 128-byte-swizzled box layout the compute warps read.
template <int EPI>
__device__ __forceinline__ void reg_gather(const HcArgs &a, int lane, uint8_t *b_ring, uint64_t *bfull,
                                           uint64_t *bempty, const RegSplit &rs) {
    const int n_items = rs.n_items;
    const float scale = __uint_as_float((uint32_t)(127 - f16_shift(a.scratch->x_amax)) << 23);   // 2^-s
    RingPos b;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        Item it;
        if (!decode_item_r(a, rs, item, EPI, it)) continue;
        const int rows = it.valid <= 16 ? 16 : 32;
        int tok = 0;   // lane n < valid: token of row n
        if (lane < it.valid) {
            const int pair = a.pad_pair[it.row0 + lane];
            tok = pair >= a.P ? pair - a.P : pair / a.k;
        }
        // lane c copies chunk c (8 K values kc*256 + 8c .. +8) of every row, 512
        // contiguous bytes a row.  The first four rows (all of a decode tile) of
        // the next stage are loaded while the current one is converted.
        uint4 nx[4];
        auto load8 = [&](int kc, int n0, uint4 (&v)[4]) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = __shfl_sync(0xffffffffu, tok, (n0 + j) & 31);
                if (n0 + j < it.valid)
                    v[j] = __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kc * kHCK + 8 * lane));
            }
        };
        auto store8 = [&](uint32_t slot, int n0, const uint4 (&v)[4]) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + j;
                if (n < it.valid) {
                    const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        __half2 h = __floats2half2_rn(__uint_as_float(u[q] << 16) * scale,
                                                      __uint_as_float(u[q] & 0xFFFF0000u) * scale);
                        o[q] = *reinterpret_cast<uint32_t *>(&h);
                    }
                    const uint32_t box = (uint32_t)(lane >> 3), ch = (uint32_t)(lane & 7) ^ (uint32_t)(n & 7);
                    sts128(slot + box * rows * 128 + n * 128 + (ch << 4), make_uint4(o[0], o[1], o[2], o[3]));
                }
            }
        };
        load8(it.kc0, 0, nx);
        for (int kc = it.kc0; kc < it.kc1; ++kc) {
            uint4 cur[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) cur[j] = nx[j];
            if (kc + 1 < it.kc1) load8(kc + 1, 0, nx);
            if (!mbar_wait(bempty + b.s, b.ph ^ 1, a.err)) ok = false;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint32_t slot = smem_u32(b_ring + b.s * a.rbslot);
            store8(slot, 0, cur);
            for (int n0 = 4; n0 < it.valid; n0 += 4) {   // rows beyond four: loaded in place
                uint4 v[4];
                load8(kc, n0, v);
                store8(slot, n0, v);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bfull + b.s);
            b.next(a.rbst);
        }
    }
}

// MX: MXFP4 weights (E8M0 scales, a 16-byte scale box a row for a pair of stages).
template <int EPI, int MX>
__global__ void __launch_bounds__(kRThreads, 1) k_gemm_reg(const __grid_constant__ HcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *code_ring = smem;
    uint8_t *b_ring = code_ring + (size_t)a.rcst * kHCodeStage;   // token-row ring, or the resident activations
    float *xchg = reinterpret_cast<float *>(b_ring + (size_t)a.rbst * a.rbslot);
    RegMeta *meta = reinterpret_cast<RegMeta *>(reinterpret_cast<uint8_t *>(xchg) + kRXchg);
    uint64_t *cfull = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(meta) + kMetaBytes);
    uint64_t *cempty = cfull + a.rcst;
    uint64_t *bfull = cempty + a.rcst;
    uint64_t *bempty = bfull + a.rbst;
    uint64_t *xfull = bempty + a.rbst;           // [8] up accumulators written (SwiGLU)
    uint64_t *xempty = xfull + 8;                // [8] and read
    uint64_t *meta_ready = xempty + 8;           // item table filled
    uint64_t *x_full = meta_ready + 1;           // resident activations copied

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.rcst; ++i) { mbar_init(cfull + i, 1); mbar_init(cempty + i, 16); }
        for (int i = 0; i < a.rbst; ++i) { mbar_init(bfull + i, 1); mbar_init(bempty + i, 16); }
        for (int i = 0; i < 8; ++i) { mbar_init(xfull + i, 1); mbar_init(xempty + i, 1); }
        mbar_init(meta_ready, 1);
        mbar_init(x_full, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Resident activations (gate/up, a.xres tokens): the raw bf16 rows of x are
    // this launch's input, not the previous kernel's output, so their copy is
    // issued before the dependency wait and overlaps the router's tail.
    if (EPI == kSwiGLU && a.xres > 0 && threadIdx.x == 32) {
        mbar_expect_tx(x_full, (uint32_t)(a.xres * a.H * 2));
        for (int t = 0; t < a.xres; ++t)
            bulk_copy(b_ring + (size_t)t * a.H * 2, a.x + (size_t)t * a.H, (uint32_t)(a.H * 2), x_full);
    }
    // gate/up: the routing results come from the previous kernel. down: only
    // its token rows (h) do, so only their producer waits (below); the weights,
    // the work list and the routing weights were complete before the gate/up
    // kernel passed its own wait, and the weight stream starts at once.
    if (EPI != kScatter) pdl_wait();
    pdl_trigger();
    const RegSplit rs = reg_split(a);
    const int n_items = rs.n_items;
    const bool gather = EPI == kSwiGLU && a.x != nullptr && a.xres == 0;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------- producer of the code ring
            RingPos c;
            bool ok = true;
            uint32_t used = 0, last_ph = 0;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item_r(a, rs, item, EPI, it)) continue;
                const int m = it.sh ? 1 : 0;
                int r0, r1;
                h_rows(a, it, EPI, r0, r1);
                const CUtensorMap *A1 = (EPI == kSwiGLU) ? &a.a1[m] : &a.a0[m];
                const CUtensorMap *S1 = (EPI == kSwiGLU) ? &a.s1[m] : &a.s0[m];
                for (int kc = it.kc0; kc < it.kc1; ++kc) {
                    if (!mbar_wait(cempty + c.s, c.ph ^ 1, a.err)) { ok = false; break; }
                    uint8_t *st = code_ring + c.s * kHCodeStage;
                    mbar_expect_tx(cfull + c.s, kHCodeStage);
                    tma_2d(st, &a.a0[m], cfull + c.s, kc * 128, r0);
                    tma_2d(st + kHCodeTile, A1, cfull + c.s, kc * 128, r1);
                    const int sx = MX ? (kc >> 1) * 16 : kc * 16;   // MXFP4: the stage pair's 16 scale bytes
                    tma_2d(st + 2 * kHCodeTile, &a.s0[m], cfull + c.s, sx, r0);
                    tma_2d(st + 2 * kHCodeTile + 2048, S1, cfull + c.s, sx, r1);
                    used |= 1u << c.s;
                    last_ph = (last_ph & ~(1u << c.s)) | (c.ph << c.s);
                    c.next(a.rcst);
                }
            }
            for (int t = 0; t < a.rcst; ++t)
                if (used & (1u << t)) mbar_wait(cfull + t, (last_ph >> t) & 1u, a.err);
        }
    } else if (warp == 1) {
        // ---------------------------------------- item table, then the token rows
        const int n_tab = reg_fill_meta<EPI>(a, rs, meta, lane);
        __syncwarp();
        if (lane == 0 && n_tab > 0) mbar_arrive(meta_ready);
        if (gather) {
            reg_gather<EPI>(a, lane, b_ring, bfull, bempty, rs);
        } else if (EPI == kScatter && lane == 0) {
            // TMA producer of the token-row ring, in a warp of its own: its
            // dependency wait must not hold up the weight stream of warp 0
            pdl_wait();   // the token rows are the previous kernel's output
            RingPos b;
            bool ok = true;
            uint32_t used = 0, last_ph = 0;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                Item it;
                if (!decode_item_r(a, rs, item, EPI, it)) continue;
                const int rc = it.valid <= 16 ? 0 : 1;
                const int rows = 16 << rc;
                for (int kc = it.kc0; kc < it.kc1; ++kc) {
                    if (!mbar_wait(bempty + b.s, b.ph ^ 1, a.err)) { ok = false; break; }
                    mbar_expect_tx(bfull + b.s, (uint32_t)(4 * rows * 128));
                    for (int bx = 0; bx < 4; ++bx)
                        tma_2d(b_ring + b.s * a.rbslot + bx * rows * 128, &a.b[rc], bfull + b.s, kc * kHCK + bx * 64,
                               it.row0);
                    used |= 1u << b.s;
                    last_ph = (last_ph & ~(1u << b.s)) | (b.ph << b.s);
                    b.next(a.rbst);
                }
            }
            for (int t = 0; t < a.rbst; ++t)
                if (used & (1u << t)) mbar_wait(bfull + t, (last_ph >> t) & 1u, a.err);
        }
    } else {
        reg_compute<EPI, MX>(a, warp, lane, code_ring, b_ring, xchg, cfull, cempty, bfull, bempty, xfull, xempty, meta,
                         meta_ready, x_full);
    }
}

// x rows (bf16) -> padded per-expert f16 rows, times 2^-s (exact; s from the
// batch amax so the values fit f16).
__global__ void __launch_bounds__(256) k_permute_f16(const uint16_t *__restrict__ x, const int32_t *__restrict__ pad_pair,
                                                     const int32_t *__restrict__ poff, const CallScratch *__restrict__ sc,
                                                     int E, int H, int P, int k, __half *__restrict__ xp) {
    const int rows = poff[E + 1];
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const float scale = __uint_as_float((uint32_t)(127 - f16_shift(sc->x_amax)) << 23);   // 2^-s
    for (int r = warp; r < rows; r += nwarps) {
        const int pair = pad_pair[r];
        if (pair < 0) continue;
        const int t = pair >= P ? pair - P : pair / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        uint4 *dst = reinterpret_cast<uint4 *>(xp + (size_t)r * H);
        for (int i = lane; i < H / 8; i += 32) {
            const uint4 q = src[i];
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 h = __floats2half2_rn(__uint_as_float(u[j] << 16) * scale, __uint_as_float(u[j] & 0xFFFF0000u) * scale);
                o[j] = *reinterpret_cast<uint32_t *>(&h);
            }
            dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Gather x's NVFP4 codes into the padded per-expert rows and its scales into
// the tensor-core scale layout (512-byte atoms of 128 rows x 4 scale bytes:
// byte (r % 32) * 16 + (r / 32 % 4) * 4 + j of atom (r / 128, c)).
// sbk: K values a scale byte covers (16 NVFP4, 32 MXFP4); a scale word (one
// tensor-core scale cell) holds four consecutive scale bytes.
__global__ void __launch_bounds__(256) k_permute_fp4(const uint8_t *__restrict__ xq, const uint8_t *__restrict__ xsc,
                                                     const int32_t *__restrict__ pad_pair,
                                                     const int32_t *__restrict__ poff, int E, int H, int P, int k,
                                                     uint8_t *__restrict__ xp, uint8_t *__restrict__ xp_atoms, int sbk) {
    const int rows = poff[E + 1];
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int cb = H / 2 / 16;    // uint4 per code row
    const int sw = H / sbk / 4;   // scale words per row
    for (int r = warp; r < rows; r += nwarps) {
        const int pair = pad_pair[r];
        if (pair < 0) continue;
        const int t = pair >= P ? pair - P : pair / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(xq + (size_t)t * (H / 2));
        uint4 *dst = reinterpret_cast<uint4 *>(xp + (size_t)r * (H / 2));
        for (int i = lane; i < cb; i += 32) dst[i] = src[i];
        const uint32_t *ss = reinterpret_cast<const uint32_t *>(xsc + (size_t)t * (H / sbk));
        const int rb = r >> 7, rr = r & 127;
        uint8_t *ab = xp_atoms + (size_t)rb * sw * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
        for (int c = lane; c < sw; c += 32) *reinterpret_cast<uint32_t *>(ab + (size_t)c * 512) = ss[c];
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D tensor map of 1-byte (or, with u16, 2-byte) elements: `rows` rows of
// `row_elems` elements (row stride `stride` bytes), box = box_elems x box_rows.
bool make_map(CUtensorMap *m, const void *base, uint64_t row_elems, uint64_t rows, uint64_t stride,
              uint32_t box_elems, uint32_t box_rows, bool swizzle, bool u16 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_elems, rows};
    cuuint64_t strides[1] = {stride};
    cuuint32_t box[2] = {box_elems, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, u16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                    const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

constexpr size_t kSmemBytes = kStages * kStageBytes + 512 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "FP4 pipeline exceeds shared memory");

}  // namespace

// Shapes the tensor-core path takes: W4A4, H a multiple of 256, I (and the
// shared I) multiples of 256, scale rows 16-byte aligned.
bool tc_supported(const Plan &p) {
    const moe_config &c = p.cfg;
    if (c.hidden % 256 || c.inter % 256) return false;
    if (c.has_shared && c.shared_inter % 256) return false;
    return encode_fn() != nullptr;
}

cudaError_t configure_tc(const Plan &) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_fp4<kSwiGLU, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_fp4<kScatter, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_fp4<kSwiGLU, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_fp4<kScatter, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_f16<kSwiGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_f16<kScatter>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_reg<kSwiGLU, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_reg<kSwiGLU, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_reg<kScatter, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_reg<kScatter, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemBytes);
    return e;
}

// Shapes the register-path W4A16 kernels take: those of the tcgen05 kernels
// (the caller cuts their tiles at 32 token rows).
bool warp_mma_supported(const Plan &p) { return p.cfg.mode == MOE_W4A16 && tc_supported(p); }

namespace {

// Column groups (256 output columns each) of a chunk of the W4A4 down items
// for T tokens: as many as keep the accumulator slice a chunk adds into,
// T x 256 C fp32, within 16 MB of L2.
int down_col_chunk(int T, int H) {
    const int64_t per_group = (int64_t)T * 256 * 4;
    int64_t c = ((int64_t)16 << 20) / per_group;
    if (c < 1) c = 1;
    if (c > H / 256) c = H / 256;
    return (int)c;
}

// W4A16 on the tensor cores (see k_gemm_f16).
cudaError_t launch_ffn_tc_f16(const Plan &p, const void *x, int T, const ExpertPtrs &r, const ExpertPtrs *s, int part,
                              cudaStream_t st, bool warp_mma) {
    const moe_config &c = p.cfg;
    const int H = c.hidden, I = c.inter, E = c.num_experts;
    const int Is = c.has_shared ? c.shared_inter : 0;
    const int Imax = std::max(I, Is);
    const ExpertPtrs &sp = s ? *s : r;
    const int Is_ = s ? Is : I;
    HcArgs a{};
    a.tiles = p.tiles;
    a.scratch = p.scratch;
    a.E = E;
    a.H = H;
    a.I = I;
    a.Is = Is;
    a.hout = reinterpret_cast<__half *>(p.hbuf);
    a.hstride = Imax;
    a.pad_pair = p.pad_pair;
    a.wts = p.wts;
    a.P = T * c.top_k;
    a.colfirst = T >= 128;
    a.k = c.top_k;
    a.acc = p.acc;
    a.err = p.err;
    a.tail_split = (p.tail_part && p.tail_tickets) ? 1 : 0;
    a.tickets = p.tail_tickets;
    a.tail_part = p.tail_part;
    a.mx = c.weight_format == MOE_WEIGHTS_MXFP4 ? 1 : 0;
    const int sbk = a.mx ? 32 : 16;   // K values a scale byte covers
    const RegRings rr = T <= 16 ? kRegSmall : kRegLarge;   // T <= 16: every tile has at most 16 rows
    a.rcst = rr.cst;
    a.rbst = rr.bst;
    a.rbslot = rr.bslot;
    const size_t rsmem = reg_smem(rr);
    bool ok = true;
    if (part == 0) {
        if (warp_mma) {
            a.x = static_cast<const uint16_t *>(x);   // the gate/up launch gathers its token rows itself
            // few tokens (every tile within one 8-row MMA tile): the whole of x
            // fits the token-row ring's space and stays resident for the launch
            if (T <= 8 && (size_t)T * H * 2 <= (size_t)rr.bst * rr.bslot) a.xres = T;
        } else {
            k_permute_f16<<<p.num_sms * 4, 256, 0, st>>>(static_cast<const uint16_t *>(x), p.pad_pair, p.poff,
                                                         p.scratch, E, H, a.P, c.top_k, p.xp16);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        ok &= make_map(&a.a0[0], r.gc, H / 2, (uint64_t)E * I, H / 2, 128, 128, true);
        ok &= make_map(&a.a1[0], r.uc, H / 2, (uint64_t)E * I, H / 2, 128, 128, true);
        ok &= make_map(&a.s0[0], r.gs, H / sbk, (uint64_t)E * I, H / sbk, 16, 128, false);
        ok &= make_map(&a.s1[0], r.us, H / sbk, (uint64_t)E * I, H / sbk, 16, 128, false);
        ok &= make_map(&a.a0[1], sp.gc, H / 2, Is_, H / 2, 128, 128, true);
        ok &= make_map(&a.a1[1], sp.uc, H / 2, Is_, H / 2, 128, 128, true);
        ok &= make_map(&a.s0[1], sp.gs, H / sbk, Is_, H / sbk, 16, 128, false);
        ok &= make_map(&a.s1[1], sp.us, H / sbk, Is_, H / sbk, 16, 128, false);
        for (int k2 = 0; k2 < 3; ++k2)
            ok &= make_map(&a.b[k2], p.xp16, H, p.rows_pad_max, (uint64_t)H * 2, 64, 16u << k2, true, true);
        a.nf = Imax / 128;
        a.ts_a0[0] = r.gts;
        a.ts_a1[0] = r.uts;
        a.ts_a0[1] = sp.gts;
        a.ts_a1[1] = sp.uts;
        if (!ok) return cudaErrorInvalidValue;
        cudaError_t e0;
        if (warp_mma)
            e0 = a.mx ? launch_pdl(k_gemm_reg<kSwiGLU, 1>, dim3(p.num_sms), dim3(kRThreads), rsmem, st, a)
                      : launch_pdl(k_gemm_reg<kSwiGLU, 0>, dim3(p.num_sms), dim3(kRThreads), rsmem, st, a);
        else
            e0 = launch_pdl(k_gemm_f16<kSwiGLU>, dim3(p.num_sms), dim3(kHThreads), kHSmemBytes, st, a);
        if (e0 != cudaSuccess) return e0;
        return cudaGetLastError();
    }
    ok &= make_map(&a.a0[0], r.dc, I / 2, (uint64_t)E * H, I / 2, 128, 128, true);
    ok &= make_map(&a.s0[0], r.ds, I / sbk, (uint64_t)E * H, I / sbk, 16, 128, false);
    ok &= make_map(&a.a0[1], sp.dc, Is_ / 2, H, Is_ / 2, 128, 128, true);
    ok &= make_map(&a.s0[1], sp.ds, Is_ / sbk, H, Is_ / sbk, 16, 128, false);
    a.a1[0] = a.a0[0];
    a.a1[1] = a.a0[1];
    a.s1[0] = a.s0[0];
    a.s1[1] = a.s0[1];
    for (int k2 = 0; k2 < 3; ++k2)
        ok &= make_map(&a.b[k2], p.hbuf, Imax, p.rows_pad_max, (uint64_t)Imax * 2, 64, 16u << k2, true, true);
    a.nf = H / 256;
    a.ts_a0[0] = r.dts;
    a.ts_a0[1] = sp.dts;
    a.ts_a1[0] = r.dts;
    a.ts_a1[1] = sp.dts;
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e0;
    if (warp_mma)
        e0 = a.mx ? launch_pdl(k_gemm_reg<kScatter, 1>, dim3(p.num_sms), dim3(kRThreads), rsmem, st, a)
                  : launch_pdl(k_gemm_reg<kScatter, 0>, dim3(p.num_sms), dim3(kRThreads), rsmem, st, a);
    else
        e0 = launch_pdl(k_gemm_f16<kScatter>, dim3(p.num_sms), dim3(kHThreads), kHSmemBytes, st, a);
    if (e0 != cudaSuccess) return e0;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_tc(const Plan &p, const void *x, int T, const ExpertPtrs &r, const ExpertPtrs *s, int part,
                          cudaStream_t st, bool warp_mma) {
    if (p.cfg.mode == MOE_W4A16) return launch_ffn_tc_f16(p, x, T, r, s, part, st, warp_mma);
    const moe_config &c = p.cfg;
    const int H = c.hidden, I = c.inter, E = c.num_experts;
    const int Is = c.has_shared ? c.shared_inter : 0;
    const int Imax = std::max(I, Is);
    const ExpertPtrs &sp = s ? *s : r;
    const int Is_ = s ? Is : I;
    TcArgs a{};
    a.tiles = p.tiles;
    a.scratch = p.scratch;
    a.E = E;
    a.H = H;
    a.I = I;
    a.Is = Is;
    a.hbuf = p.hbuf;
    a.hstride = Imax;
    a.h_amax = &p.scratch->h_amax;
    a.hs_amax = &p.scratch->hs_amax;
    a.pad_pair = p.pad_pair;
    a.wts = p.wts;
    a.P = T * c.top_k;
    a.colfirst = T >= 128 ? down_col_chunk(T, H) : 0;
    a.k = c.top_k;
    a.acc = p.acc;
    a.err = p.err;
    a.b_ts = p.hts;
    const bool mx = c.weight_format == MOE_WEIGHTS_MXFP4;
    const int sbk = mx ? 32 : 16;   // K values a scale byte covers
    if (mx) {   // the gate/up epilogue quantises the SwiGLU output itself
        a.hq = p.hq;
        a.hq_atoms = p.hq_atoms;
        a.hts_out = p.hts;
        a.keep_h = p.keep_h;
    }
    bool ok = true;
    if (part == 0) {
        // permute x codes/scales into the padded rows first
        k_permute_fp4<<<p.num_sms * 4, 256, 0, st>>>(p.xq, p.xsc, p.pad_pair, p.poff, E, H, a.P, c.top_k, p.xp,
                                                     p.xp_atoms, sbk);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ok &= make_map(&a.a0[0], r.gc, H / 2, (uint64_t)E * I, H / 2, 128, 128, true);
        ok &= make_map(&a.a1[0], r.uc, H / 2, (uint64_t)E * I, H / 2, 128, 128, true);
        ok &= make_map(&a.s0[0], r.gs, H / sbk, (uint64_t)E * I, H / sbk, 16, 128, false);
        ok &= make_map(&a.s1[0], r.us, H / sbk, (uint64_t)E * I, H / sbk, 16, 128, false);
        ok &= make_map(&a.a0[1], sp.gc, H / 2, Is_, H / 2, 128, 128, true);
        ok &= make_map(&a.a1[1], sp.uc, H / 2, Is_, H / 2, 128, 128, true);
        ok &= make_map(&a.s0[1], sp.gs, H / sbk, Is_, H / sbk, 16, 128, false);
        ok &= make_map(&a.s1[1], sp.us, H / sbk, Is_, H / sbk, 16, 128, false);
        for (int c = 0; c < 3; ++c) ok &= make_map(&a.b[c], p.xp, H / 2, p.rows_pad_max, H / 2, 128, 32u << c, true);
        a.b_atoms = p.xp_atoms;
        a.b_atoms_per_block = H / sbk / 4;
        a.nf = Imax / 128;
        a.ts_a0[0] = r.gts;
        a.ts_a1[0] = r.uts;
        a.ts_a0[1] = sp.gts;
        a.ts_a1[1] = sp.uts;
        if (!ok) return cudaErrorInvalidValue;
        cudaError_t e0 = launch_pdl(mx ? k_gemm_fp4<kSwiGLU, 1> : k_gemm_fp4<kSwiGLU, 0>, dim3(p.num_sms),
                                     dim3(fp4_threads(kSwiGLU)), kSmemBytes, st, a);
        if (e0 != cudaSuccess) return e0;
        return cudaGetLastError();
    }
    ok &= make_map(&a.a0[0], r.dc, I / 2, (uint64_t)E * H, I / 2, 128, 128, true);
    ok &= make_map(&a.s0[0], r.ds, I / sbk, (uint64_t)E * H, I / sbk, 16, 128, false);
    ok &= make_map(&a.a0[1], sp.dc, Is_ / 2, H, Is_ / 2, 128, 128, true);
    ok &= make_map(&a.s0[1], sp.ds, Is_ / sbk, H, Is_ / sbk, 16, 128, false);
    a.a1[0] = a.a0[0];
    a.a1[1] = a.a0[1];
    a.s1[0] = a.s0[0];
    a.s1[1] = a.s0[1];
    for (int c = 0; c < 3; ++c) ok &= make_map(&a.b[c], p.hq, Imax / 2, p.rows_pad_max, Imax / 2, 128, 32u << c, true);
    a.b_atoms = p.hq_atoms;
    a.b_atoms_per_block = Imax / sbk / 4;
    a.nf = H / 256;
    a.ts_a0[0] = r.dts;
    a.ts_a0[1] = sp.dts;
    a.ts_a1[0] = r.dts;
    a.ts_a1[1] = sp.dts;
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e0 = launch_pdl(mx ? k_gemm_fp4<kScatter, 1> : k_gemm_fp4<kScatter, 0>, dim3(p.num_sms),
                                 dim3(fp4_threads(kScatter)), kSmemBytes, st, a);
    if (e0 != cudaSuccess) return e0;
    return cudaGetLastError();
}

}  // namespace moe
