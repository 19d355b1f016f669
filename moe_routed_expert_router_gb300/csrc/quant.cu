// NVFP4 quantisers (weights, W4A4 activations, W4A4 SwiGLU output) and the
// final bf16 write of the combine.
//
// "NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4 Round 1:
// NVFP4 = U8 codes + F8_E4M3 block scales + one fp32 tensor scale (#489, #517);
// 4-bit activations in the routed prompt GEMM (#687); the SwiGLU output
// quantised for the down product (#760); activation quantisation folded into
// its producer (remaining Round 1 items).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0f;
        v = warp_max(v);
    }
    return v;
}

// amax |x| of bf16 data (n multiple of 8) into *out (fp32 bits, atomicMax).
__global__ void __launch_bounds__(kThreads) k_amax_bf16(const uint4 *__restrict__ x, int64_t n8, unsigned int *out) {
    __shared__ float red[32];
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        uint4 q = x[i];
        uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[j] << 16)), fabsf(__uint_as_float(u[j] & 0xFFFF0000u))));
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) atomic_max_nonneg(out, m);
}

// amax |w| per batch item of fp32 data; grid.y = item.
__global__ void __launch_bounds__(kThreads) k_amax_f32(const float4 *__restrict__ w, int64_t n4_per_item,
                                                      unsigned int *out) {
    __shared__ float red[32];
    const float4 *base = w + (int64_t)blockIdx.y * n4_per_item;
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4_per_item;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = base[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) atomic_max_nonneg(out + blockIdx.y, m);
}

// One thread per 16-value block of fp32 weights; item b's amax is in ts_bits[b].
__global__ void __launch_bounds__(kThreads) k_quant_f32(const float *__restrict__ w, int64_t blocks_per_item,
                                                       int batch, const unsigned int *__restrict__ ts_bits,
                                                       uint2 *__restrict__ codes, uint8_t *__restrict__ scales) {
    const int64_t total = blocks_per_item * batch;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / blocks_per_item);
        const float ts = __fdiv_rn(__uint_as_float(ts_bits[b]), 2688.0f);
        const float4 *p = reinterpret_cast<const float4 *>(w + i * 16);
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 q = p[j];
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        }
        uint2 c;
        uint32_t s;
        quant_block16(v, ts, c, s);
        codes[i] = c;
        scales[i] = (uint8_t)s;
    }
}

__global__ void k_ts_finalize(float *ts, int batch) {
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) ts[b] = __fdiv_rn(ts[b], 2688.0f);  // ts[b] held amax as fp32 bits
}

// W4A4 activations: one thread per 16-value block of bf16 x; amax in *amax_bits.
__global__ void __launch_bounds__(kThreads) k_quant_act(const uint16_t *__restrict__ x, int64_t nblocks,
                                                       const unsigned int *__restrict__ amax_bits,
                                                       uint2 *__restrict__ codes, uint8_t *__restrict__ scales,
                                                       float *ts_out) {
    const float ts = __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0 && ts_out) *ts_out = ts;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 *p = reinterpret_cast<const uint4 *>(x + i * 16);
        uint4 a = p[0], b = p[1];
        uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float v[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[2 * j] = __uint_as_float(u[j] << 16);
            v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
        }
        uint2 c;
        uint32_t s;
        quant_block16(v, ts, c, s);
        codes[i] = c;
        scales[i] = (uint8_t)s;
    }
}

// MXFP4 weights: one thread per 32-value block of fp32 rows (any number of rows).
__global__ void __launch_bounds__(kThreads) k_quant_mx_f32(const float *__restrict__ w, int64_t nblocks,
                                                          uint4 *__restrict__ codes, uint8_t *__restrict__ scales) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 *p = reinterpret_cast<const float4 *>(w + i * 32);
        float v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 q = p[j];
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        }
        uint4 c;
        uint32_t s;
        quant_block32_mx(v, c, s);
        codes[i] = c;
        scales[i] = (uint8_t)s;
    }
}

// MXFP4 activations (W4A4 with MXFP4 weights): one thread per 32-value block of
// bf16 x; no tensor scale (ts_out, when given, receives 1).
__global__ void __launch_bounds__(kThreads) k_quant_act_mx(const uint16_t *__restrict__ x, int64_t nblocks,
                                                          uint4 *__restrict__ codes, uint8_t *__restrict__ scales,
                                                          float *ts_out) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && ts_out) *ts_out = 1.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 *p = reinterpret_cast<const uint4 *>(x + i * 32);
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 q = p[j];
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * j + 2 * h] = __uint_as_float(u[h] << 16);
                v[8 * j + 2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u);
            }
        }
        uint4 c;
        uint32_t s;
        quant_block32_mx(v, c, s);
        codes[i] = c;
        scales[i] = (uint8_t)s;
    }
}

// MXFP4 SwiGLU output (W4A4 with MXFP4 weights): fp32 h rows -> codes
// [row][stride/2] and scales, plain [row][stride/32] or (atoms != null) in the
// tensor-core layout: 512-byte atoms of 128 rows x 4 blocks, stride/128 atoms
// a 128-row block.  Every block on its own, no tensor scale (hts receives 1, 1).
__global__ void __launch_bounds__(kThreads) k_quant_h_mx(const float *__restrict__ h, int stride,
                                                        const int32_t *__restrict__ poff, int E, int I, int Is,
                                                        const int32_t *__restrict__ pad_pair, uint4 *__restrict__ codes,
                                                        uint8_t *__restrict__ scales, uint8_t *__restrict__ atoms,
                                                        float *hts) {
    if (blockIdx.x == 0 && threadIdx.x == 0) { hts[0] = 1.0f; hts[1] = 1.0f; }
    const int shared_row0 = poff[E];
    const int rows = poff[E + 1];
    const int bpr = stride / 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)rows * bpr;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int row = (int)(i / bpr), blk = (int)(i % bpr);
        if (pad_pair[row] < 0) continue;
        if (blk >= (row >= shared_row0 ? Is : I) / 32) continue;
        const float4 *p = reinterpret_cast<const float4 *>(h + (int64_t)row * stride + blk * 32);
        float v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 q = p[j];
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        }
        uint4 c;
        uint32_t s;
        quant_block32_mx(v, c, s);
        codes[(int64_t)row * (stride / 32) + blk] = c;
        if (atoms) {
            const int rr = row & 127;
            atoms[((int64_t)(row >> 7) * (stride / 128) + (blk >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 +
                  (blk & 3)] = (uint8_t)s;
        } else {
            scales[(int64_t)row * bpr + blk] = (uint8_t)s;
        }
    }
}

// W4A4 SwiGLU output: fp32 h rows (padded layout, row stride `stride` values)
// -> NVFP4 codes [row][stride/2] and scales [row][stride/16].  Rows of the
// routed segment use the routed amax, rows of the shared segment the shared one.
__global__ void __launch_bounds__(kThreads) k_quant_h(const float *__restrict__ h, int stride,
                                                     const int32_t *__restrict__ poff, int E, int I, int Is,
                                                     const int32_t *__restrict__ pad_pair,
                                                     const CallScratch *__restrict__ sc, uint2 *__restrict__ codes,
                                                     uint8_t *__restrict__ scales, uint8_t *__restrict__ atoms,
                                                     float *hts) {
    const float ts_r = __fdiv_rn(__uint_as_float(sc->h_amax), 2688.0f);
    const float ts_s = __fdiv_rn(__uint_as_float(sc->hs_amax), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) { hts[0] = ts_r; hts[1] = ts_s; }
    const int shared_row0 = poff[E];
    const int rows = poff[E + 1];
    const int bpr = stride / 16;
    // one warp an item of 32 consecutive 16-value blocks of a row (a lane a
    // block); an item of a padding row is skipped whole
    const int lane = threadIdx.x & 31;
    const int warps = (int)(gridDim.x * blockDim.x) >> 5;
    const int nch = (bpr + 31) / 32;
    for (int item = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); item < rows * nch; item += warps) {
        const int row = item / nch, blk = (item - row * nch) * 32 + lane;
        if (pad_pair[row] < 0) continue;   // warp-uniform
        const bool sh = row >= shared_row0;
        if (blk < (sh ? Is : I) / 16) {
            const float4 *p = reinterpret_cast<const float4 *>(h + (int64_t)row * stride + blk * 16);
            float v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float4 q = p[j];
                v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
            }
            uint2 c;
            uint32_t s;
            quant_block16(v, sh ? ts_s : ts_r, c, s);
            codes[(int64_t)row * (stride / 16) + blk] = c;
            if (atoms) {  // tensor-core scale layout: 512-byte atoms of 128 rows x 4 scales
                const int rr = row & 127;
                atoms[((int64_t)(row >> 7) * (stride / 64) + (blk >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (blk & 3)] =
                    (uint8_t)s;
            } else {
                scales[(int64_t)row * bpr + blk] = (uint8_t)s;
            }
        }
    }
}

// The element conversions of quant_block16 on their own (moe_convert_f32):
// format 0 E4M3 byte, format 1 E2M1 code (low nibble).
__global__ void __launch_bounds__(kThreads) k_convert(const float *__restrict__ src, int64_t n, int format,
                                                     uint8_t *__restrict__ dst) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = src[i];
        dst[i] = (uint8_t)(format == 0 ? f32_to_e4m3_sat(v) : (f32x2_to_e2m1x2(v, 0.0f) & 0xFu));
    }
}

// out = bf16_rne(acc); acc = 0 (so the next call starts from zero).
__global__ void __launch_bounds__(kThreads) k_finalize(float4 *__restrict__ acc, uint2 *__restrict__ out, int64_t n4) {
    pdl_wait();      // the down GEMM's scatter-adds are complete
    pdl_trigger();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = acc[i];
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&a);
        o.y = *reinterpret_cast<uint32_t *>(&b);
        out[i] = o;
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// One block waits on an mbarrier that nothing arrives on, through the same
// bounded wait the pipelined kernels use: the bound runs out and the timeout
// bit is set.
__global__ void k_wait_check(int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    mbar_wait(&bar, 0, err, limit_ns);
}

int grid_for(int64_t work, int num_sms) {
    int64_t g = (work + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)num_sms * 8;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

int device_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_quant_act(const Plan &p, const void *x, int T, uint8_t *codes, uint8_t *scales, float *ts_out,
                             bool amax_ready, cudaStream_t st) {
    const int64_t n = (int64_t)T * p.cfg.hidden;
    if (p.cfg.weight_format == MOE_WEIGHTS_MXFP4) {
        k_quant_act_mx<<<grid_for(n / 32, p.num_sms), kThreads, 0, st>>>(static_cast<const uint16_t *>(x), n / 32,
                                                                         reinterpret_cast<uint4 *>(codes), scales,
                                                                         ts_out);
        return cudaGetLastError();
    }
    if (!amax_ready) {
        k_amax_bf16<<<grid_for(n / 8, p.num_sms), kThreads, 0, st>>>(static_cast<const uint4 *>(x), n / 8,
                                                                     &p.scratch->x_amax);
    }
    k_quant_act<<<grid_for(n / 16, p.num_sms), kThreads, 0, st>>>(static_cast<const uint16_t *>(x), n / 16,
                                                                  &p.scratch->x_amax, reinterpret_cast<uint2 *>(codes),
                                                                  scales, ts_out);
    return cudaGetLastError();
}

cudaError_t launch_quant_h(const Plan &p, bool tc_layout, cudaStream_t st) {
    const int Imax = p.cfg.has_shared ? max(p.cfg.inter, p.cfg.shared_inter) : p.cfg.inter;
    if (p.cfg.weight_format == MOE_WEIGHTS_MXFP4) {
        k_quant_h_mx<<<p.num_sms * 8, kThreads, 0, st>>>(p.hbuf, Imax, p.poff, p.cfg.num_experts, p.cfg.inter,
                                                         p.cfg.shared_inter, p.pad_pair, reinterpret_cast<uint4 *>(p.hq),
                                                         p.hsc, tc_layout ? p.hq_atoms : nullptr, p.hts);
        return cudaGetLastError();
    }
    k_quant_h<<<p.num_sms * 8, kThreads, 0, st>>>(p.hbuf, Imax, p.poff, p.cfg.num_experts, p.cfg.inter,
                                                  p.cfg.shared_inter, p.pad_pair, p.scratch,
                                                  reinterpret_cast<uint2 *>(p.hq), p.hsc,
                                                  tc_layout ? p.hq_atoms : nullptr, p.hts);
    return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4(const float *w, int64_t rows, int cols, uint8_t *codes, uint8_t *scales,
                               cudaStream_t st) {
    const int64_t nb = rows * (cols / 32);
    k_quant_mx_f32<<<grid_for(nb, device_sms()), kThreads, 0, st>>>(w, nb, reinterpret_cast<uint4 *>(codes), scales);
    return cudaGetLastError();
}

cudaError_t launch_convert(const float *src, int64_t n, int format, uint8_t *dst, cudaStream_t st) {
    k_convert<<<grid_for(n, device_sms()), kThreads, 0, st>>>(src, n, format, dst);
    return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4(const float *w, int batch, int rows, int cols, uint8_t *codes, uint8_t *scales,
                               float *ts, cudaStream_t st) {
    const int sms = device_sms();
    const int64_t per = (int64_t)rows * cols;
    cudaError_t e = cudaMemsetAsync(ts, 0, sizeof(float) * batch, st);
    if (e != cudaSuccess) return e;
    int gx = grid_for(per / 4, sms);
    gx = max(1, gx / max(1, batch / 8));
    dim3 g(gx, batch);
    k_amax_f32<<<g, kThreads, 0, st>>>(reinterpret_cast<const float4 *>(w), per / 4,
                                       reinterpret_cast<unsigned int *>(ts));
    k_quant_f32<<<grid_for(per / 16 * batch, sms), kThreads, 0, st>>>(
        w, per / 16, batch, reinterpret_cast<const unsigned int *>(ts), reinterpret_cast<uint2 *>(codes), scales);
    k_ts_finalize<<<(batch + 255) / 256, 256, 0, st>>>(ts, batch);
    return cudaGetLastError();
}

cudaError_t launch_wait_check(int *err, uint64_t limit_ns, cudaStream_t st) {
    k_wait_check<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const Plan &p, int T, void *out, cudaStream_t st) {
    const int64_t n4 = (int64_t)T * p.cfg.hidden / 4;
    return launch_pdl(k_finalize, dim3(grid_for(n4, p.num_sms)), dim3(kThreads), 0, st, reinterpret_cast<float4 *>(p.acc),
                      static_cast<uint2 *>(out), n4);
}

}  // namespace moe
