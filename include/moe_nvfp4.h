/*
 * moe_nvfp4.h -- C ABI of the routed mixture-of-experts FFN over NVFP4
 * weights, for one NVIDIA GB300 (sm_103a).
 *
 * What it computes, for every token t of a batch x[T][H]:
 *
 *   out[t] = sum_{j<k} w[t][j] * FFN_{id[t][j]}(x_t)   (+ FFN_shared(x_t))
 *   FFN_e(v) = Wd_e ( silu(Wg_e v) * (Wu_e v) ),   silu(z) = z / (1 + e^-z)
 *
 * with the router choosing id[t][*] and w[t][*] (softmax or sigmoid, top-k,
 * renormalised) and every weight W = E2M1(code) * E4M3(block scale) *
 * tensor_scale.  Sources (page title, section):
 *   "NVIDIA FP4-Local checkpoints on DGX Spark (TP=1, TP=2) ... #565",
 *   section 4 Round 1: NVFP4 weights as U8 codes and F8_E4M3 scales held as
 *   stored (#489); routed experts with a gate, up and down product and one
 *   tensor scale an expert (#517, #545); a whole batch routed in one run so
 *   each expert is read once (#740); gate, up and SwiGLU in one launch (#766);
 *   W4A16 / W4A4 activation formats (#687, list of formats at the end of the
 *   section); the SwiGLU output quantised for the down product (#760); down
 *   rows in BF16 rounded to nearest even (#914); the combine folded into the
 *   card sum (#701); the shared expert beside the routed ones (#686);
 *   router logits in fp32 (#763).  "bloomery 0.3.9", From our contributors:
 *   the router's normalisation policy is a named value (#772).
 *
 * Formats (the pages name them; the bit layouts are the OCP Microscaling ones):
 *   - NVFP4 tensor W[N][K]: codes uint8[N][K/2], element 2i in bits 0..3 and
 *     element 2i+1 in bits 4..7; scales uint8[N][K/16], one E4M3 byte per 16
 *     consecutive K values, row-major; one fp32 tensor scale.
 *   - E2M1: sign bit 3, magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
 *   - E4M3 ("FN"): bias 7, max 448, 0x7F/0xFF NaN, no infinities.
 *   - NVFP4 quantiser (weights and W4A4 activations), fp32 arithmetic:
 *       ts = amax / 2688;  s = E4M3_rne_sat((block_amax / 6) / ts);
 *       code = E2M1_rne_sat(x / (E4M3(s) * ts)).
 *
 * Conventions for every entry point:
 *   - Every pointer argument is DEVICE memory unless its comment says host;
 *     the caller owns it.  Pointers must be 16-byte aligned
 *     (MOE_ERR_MISALIGNED otherwise).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  No call below allocates or synchronises
 *     except moe_plan_create / moe_plan_destroy / moe_plan_sync_status.
 *   - Host-side checks return an error at once and launch nothing.  Errors
 *     found on the device (a non-finite activation, a wait that ran out) set
 *     the plan's error word, which moe_plan_sync_status returns; outputs are
 *     unspecified after a device error.
 *   - A plan is used by one stream at a time.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, T > max_tokens ... */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* H or I not a multiple of 256/128, k > E ... */
    MOE_ERR_MISALIGNED = 3,        /* a pointer not 16-byte aligned */
    MOE_ERR_NONFINITE = 4,         /* device: an activation is NaN or infinite */
    MOE_ERR_TIMEOUT = 5,           /* device: a bounded wait ran out */
    MOE_ERR_CUDA = 6,              /* a CUDA runtime call failed */
    MOE_ERR_OOM = 7,               /* moe_plan_create could not allocate */
    MOE_ERR_DEVICE = 8             /* device: an internal check failed */
} moe_status;

typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1 } moe_router_kind;

/* Word type of the router weight: fp32, or the checkpoint's bf16 words read
 * as they are stored ("NVIDIA FP4-Local checkpoints on DGX Spark ... #565",
 * section 4 Round 1: the router kept in its BF16 words, #732).  A bf16 word
 * widens to fp32 exactly, so the logits keep the fixed fp32 order below; the
 * router reads half the bytes. */
typedef enum { MOE_ROUTER_F32 = 0, MOE_ROUTER_BF16 = 1 } moe_router_dtype;

/* Block format of the expert weights.
 *   NVFP4: E2M1 codes, one E4M3 scale a 16-value block, one fp32 tensor scale a
 *          weight (the format described above).
 *   MXFP4: E2M1 codes, one E8M0 scale (2^(byte - 127)) a 32-value block, no
 *          tensor scale; the OCP Microscaling conversion: byte =
 *          clamp(floor(log2(block amax)) - 2 + 127, 0, 254), code =
 *          E2M1_rne_sat(x / 2^(byte - 127)).  The pages name MXFP4 routed
 *          experts and an MXFP4 routed prompt GEMM on block-scaled tensor cores
 *          ("NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 6
 *          Round 3; "bloomery 0.3.13", Also, #1154) and MX blocks of 32 with an
 *          E8M0 scale (#521).  In W4A4 the activations and the SwiGLU output
 *          are then MXFP4 as well (every block on its own scale, no batch
 *          amax).  MXFP4 plans need H, I (and the shared I) multiples of 512;
 *          they run on the CUDA cores, W4A4 also on the tcgen05 block-scaled
 *          MMAs (kind::mxf4, E8M0 scales), and W4A16 also on the warp MMAs
 *          (whose f16 operands hold code x scale exactly only for block scales
 *          from 2^-23 to 2^13: a weight block outside that range is a device
 *          error there). */
typedef enum { MOE_WEIGHTS_NVFP4 = 0, MOE_WEIGHTS_MXFP4 = 1 } moe_weight_format;

/* W4A16: activations stay bf16; the SwiGLU output is rounded to bf16 (RNE)
 *        before the down product.
 * W4A4:  activations are NVFP4-quantised (tensor scale from the batch amax);
 *        the SwiGLU output of all routed rows is rounded to fp32 and
 *        NVFP4-quantised with the tensor scale from its own batch amax (the
 *        shared expert's with its own). */
typedef enum { MOE_W4A16 = 0, MOE_W4A4 = 1 } moe_mode;

typedef struct {
    int32_t hidden;       /* H: multiple of 256, at most 8192 */
    int32_t inter;        /* I: per-expert intermediate, multiple of 128, at most 8192 */
    int32_t num_experts;  /* E: 1..1024 */
    int32_t top_k;        /* k: 1..min(E, 32) */
    int32_t max_tokens;   /* largest T a call may pass (sizes the workspace) */
    int32_t router;       /* moe_router_kind */
    int32_t renormalize;  /* 1: weights renormalised over the top-k; 0: not */
    int32_t mode;         /* moe_mode */
    int32_t has_shared;   /* 1: a shared expert is added to every token */
    int32_t shared_inter; /* shared expert's intermediate (multiple of 128, at most 8192) */
    int32_t router_dtype; /* moe_router_dtype of router_w in moe_route / moe_forward */
    int32_t weight_format; /* moe_weight_format of the expert weights */
} moe_config;

/* One weight stacked over `count` experts: codes [count][N][K/2] and
 *   NVFP4: scales [count][N][K/16] (E4M3), tensor_scale [count] fp32;
 *   MXFP4: scales [count][N][K/32] (E8M0), tensor_scale ignored (may be NULL).
 * All device memory. */
typedef struct {
    const uint8_t *codes;
    const uint8_t *scales;
    const float *tensor_scale;
} moe_nvfp4;

/* gate and up are [I][H]; down is [H][I].  For the routed set count = E; for
 * the shared expert count = 1 and I = shared_inter. */
typedef struct {
    moe_nvfp4 gate, up, down;
} moe_expert_set;

typedef struct moe_plan_s *moe_plan;

/* Validate `cfg` (host memory), then allocate the plan and its device
 * workspace on the current device for cfg->max_tokens tokens.  *out receives
 * the plan (NULL on error).  This and moe_plan_set_profiling are the only
 * calls that allocate. */
moe_status moe_plan_create(const moe_config *cfg, moe_plan *out);

/* Free the plan and its workspace (synchronises the device first). */
moe_status moe_plan_destroy(moe_plan plan);

/* Router + grouping only (the steps "route" and "group by expert").
 *   x_bf16      [T][H] bf16 activations
 *   router_w    [E][H] fp32, or bf16 words when cfg.router_dtype is
 *               MOE_ROUTER_BF16 (16-byte aligned either way)
 *   router_bias [E] fp32 or NULL; added to the logits, so it moves both the
 *               selection and the weights
 * Outputs (device, caller-owned):
 *   topk_ids       [T][k] int32, experts by decreasing logit, ties -> lower id
 *   topk_w         [T][k] fp32 routing weights
 *   expert_offsets [E+1] int32, exclusive prefix of per-expert pair counts
 *   sorted_rows    [T*k] int32, pair indices t*k+j grouped by expert, each
 *                  expert's pairs in increasing t*k+j
 * Logits are fp32 with a fixed order: position h of the H dimension belongs to
 * lane h mod 32, each lane sums fmaf in increasing h from +0, the 32 lane
 * sums are combined by an xor butterfly over offsets 16, 8, 4, 2, 1, and the
 * bias is added last.  Indices and offsets are therefore reproducible bit for
 * bit. */
moe_status moe_route(moe_plan plan, const void *x_bf16, int32_t T, const void *router_w,
                     const float *router_bias, int32_t *topk_ids, float *topk_w,
                     int32_t *expert_offsets, int32_t *sorted_rows, void *stream);

/* The whole MoE FFN: route, group, [W4A4: quantise x], permute, gate/up +
 * SwiGLU, down with the routing weight, combine, [+ shared expert], bf16 out.
 *   routed: E experts' NVFP4 gate/up/down (host struct of device pointers)
 *   shared: NULL, or the shared expert (count 1) when cfg.has_shared
 *   out_bf16 [T][H] bf16, written with one round-to-nearest-even of the fp32
 *            sum.  T = 0 is a no-op. */
moe_status moe_forward(moe_plan plan, const void *x_bf16, int32_t T, const void *router_w,
                       const float *router_bias, const moe_expert_set *routed,
                       const moe_expert_set *shared, void *out_bf16, void *stream);

/* moe_forward with HOST activations and output: copies x (host, ideally
 * pinned) to the plan's device staging buffer, runs moe_forward, and copies
 * the result back to out_bf16_host.  The weights stay device pointers.
 * The copies are ordered on `stream`; the call returns before they finish
 * (synchronise the stream before reading out_bf16_host). */
moe_status moe_forward_host(moe_plan plan, const void *x_bf16_host, int32_t T, const void *router_w,
                            const float *router_bias, const moe_expert_set *routed,
                            const moe_expert_set *shared, void *out_bf16_host, void *stream);

/* W4A4 activation quantisation on its own (the step moe_forward runs first in
 * W4A4): tensor scale from the amax of all of x[T][H], then per 16-block
 * E4M3 scales and E2M1 codes.
 *   codes [T][H/2], scales [T][H/16], tensor_scale [1] fp32 (device).
 * An MXFP4 plan writes MXFP4 instead: scales [T][H/32] E8M0, tensor_scale 1. */
moe_status moe_quantize_act(moe_plan plan, const void *x_bf16, int32_t T, uint8_t *codes,
                            uint8_t *scales, float *tensor_scale, void *stream);

/* NVFP4 quantisation of fp32 weights w[batch][rows][cols] (device), one
 * tensor scale per batch item (amax of that item / 2688).  Writes codes
 * [batch][rows][cols/2], scales [batch][rows][cols/16], tensor_scale [batch].
 * cols must be a multiple of 16.  Needs no plan and no workspace:
 * tensor_scale doubles as the amax accumulator while the call runs. */
moe_status moe_quantize_nvfp4(const float *w, int32_t batch, int32_t rows, int32_t cols,
                              uint8_t *codes, uint8_t *scales, float *tensor_scale, void *stream);

/* Test hook: the device's fp32 -> E4M3 and fp32 -> E2M1 conversions, exactly
 * as the quantisers above apply them (round to nearest even, saturating to the
 * largest finite value; the sign is kept).  For every i < n, dst[i] =
 *   format MOE_FMT_E4M3: the E4M3 byte of src[i];
 *   format MOE_FMT_E2M1: the 4-bit E2M1 code of src[i] in bits 0..3.
 * src [n] fp32 and dst [n] uint8 are device memory (src 16-byte aligned).
 * Needs no plan.  MOE_ERR_INVALID_ARG for an unknown format or n < 0. */
typedef enum { MOE_FMT_E4M3 = 0, MOE_FMT_E2M1 = 1 } moe_format;
moe_status moe_convert_f32(const float *src, int64_t n, int32_t format, uint8_t *dst, void *stream);

/* MXFP4 quantisation (OCP MX, see moe_weight_format) of fp32 weights
 * w[rows][cols] (device; stack experts as rows): codes [rows][cols/2], E8M0
 * scales [rows][cols/32].  cols must be a multiple of 32.  Needs no plan. */
moe_status moe_quantize_mxfp4(const float *w, int64_t rows, int32_t cols, uint8_t *codes, uint8_t *scales,
                              void *stream);

/* Synchronise `stream`, then return and clear the plan's device error word
 * (MOE_OK, MOE_ERR_NONFINITE, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE). */
moe_status moe_plan_sync_status(moe_plan plan, void *stream);

/* Device address and size of a plan workspace buffer, for tests that check a
 * step in isolation.  name: "h_codes", "h_scales", "h_scale_atoms" (W4A4 on
 * the tensor cores: the SwiGLU scales in 512-byte atoms of 128 rows x 4
 * blocks, byte (r % 32) * 16 + (r % 128 / 32) * 4 + b % 4 of atom
 * (r / 128, b / 4)), "h_ts", "x_ts", "acc", "counts" (pairs an expert, where
 * the grouping runs as a launch of its own), "padded_offsets", "offsets",
 * "sorted", "pad_pair", "tiles", "h".
 * Returns MOE_ERR_INVALID_ARG for an unknown name. */
moe_status moe_plan_debug_buffer(moe_plan plan, const char *name, void **ptr, size_t *bytes);

/* W4A4 with MXFP4 weights on the tensor cores quantises the SwiGLU output in
 * the gate/up launch (every 32-value block on its own scale, one pass) and by
 * default writes only its codes and scales.  keep = 1: also store the fp32 h
 * (debug buffer "h"), for stage-by-stage checks.  Every other path stores h
 * anyway.  MOE_ERR_INVALID_ARG for a NULL plan. */
moe_status moe_plan_keep_h(moe_plan plan, int32_t keep);

/* Expert-FFN implementation moe_forward uses.  CUDA_CORE: weight-streaming
 * kernels on the CUDA cores (any shape).  TENSOR_CORE: grouped GEMMs on the
 * 5th-generation tensor cores (tcgen05; W4A4 block-scaled FP4, W4A16 with the
 * weights widened to f16 in tensor memory).  WARP_MMA (W4A16 only): the
 * weights widened in registers straight into warp-level f16 MMAs, for tiles
 * of up to 32 token rows.  AUTO picks WARP_MMA for W4A16 batches with fewer
 * than 2 (token, expert) pairs an expert on average (decode), the tcgen05
 * GEMMs for larger W4A16 batches and for W4A4 batches of 64 or more pairs,
 * and CUDA_CORE otherwise; the tensor paths need H and I multiples of 256.
 * MXFP4 W4A16 plans take no TENSOR_CORE (AUTO: WARP_MMA).  All compute the
 * same function (the tolerance of the parity tests covers their different
 * summation orders). */
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_CUDA_CORE = 1, MOE_PATH_TENSOR_CORE = 2, MOE_PATH_WARP_MMA = 3 } moe_path;

/* Select the expert-FFN implementation for later calls on this plan.
 * MOE_ERR_UNSUPPORTED_SHAPE if MOE_PATH_TENSOR_CORE or MOE_PATH_WARP_MMA is
 * asked for a plan whose mode or shapes it does not cover. */
moe_status moe_plan_set_path(moe_plan plan, int32_t path);

/* Stages of moe_forward, for moe_plan_read_profile. */
typedef enum {
    MOE_STAGE_ROUTE = 0,      /* logits + top-k (one kernel for T <= 16, else two) */
    MOE_STAGE_GROUP = 1,      /* histogram scan, stable placement, work lists */
    MOE_STAGE_QUANT_X = 2,    /* W4A4 activation quantisation */
    MOE_STAGE_PERMUTE = 3,    /* gather of activations into per-expert tiles */
    MOE_STAGE_GATE_UP = 4,    /* gate + up + SwiGLU */
    MOE_STAGE_QUANT_H = 5,    /* W4A4 quantisation of the SwiGLU output */
    MOE_STAGE_DOWN = 6,       /* down + routing weight + scatter-add */
    MOE_STAGE_FINALIZE = 7,   /* bf16 write of the combine */
    MOE_NUM_STAGES = 8
} moe_stage;

/* Turn per-stage timing on (1) or off (0).  While on, moe_forward records a
 * CUDA event pair on its stream around every stage (events come from a pool
 * the plan allocates here) and counts the kernels it launches. */
moe_status moe_plan_set_profiling(moe_plan plan, int32_t enable);

/* Synchronise the device, then add into ms[MOE_NUM_STAGES] the summed event
 * time of every stage recorded since the last read, and into
 * launches[MOE_NUM_STAGES] / calls[MOE_NUM_STAGES] the kernels launched and
 * the stage executions; clears the record.  Host arrays; any may be NULL. */
moe_status moe_plan_read_profile(moe_plan plan, float *ms, int64_t *launches, int64_t *calls);

/* Failure-detection check: launch one block whose waits use the same bounded
 * mbarrier wait as the expert kernels, on a barrier nothing will arrive on,
 * with the bound set to `wait_ns` nanoseconds (at most one second).  The wait
 * runs out, the kernel records MOE_ERR_TIMEOUT in the plan's error word and
 * returns normally; moe_plan_sync_status then reports it and the context stays
 * usable.  Faults nothing and hangs nothing. */
moe_status moe_plan_check_timeout(moe_plan plan, int64_t wait_ns, void *stream);

/* Routing and grouping, as moe_route, for callers that cannot allocate device
 * memory: code running inside another allocator's arena or under a
 * memory-capped runtime, or a host that forbids device allocations after
 * start-up.  The pages have no counterpart of this entry point; it exists for
 * those callers only.
 *
 * It needs no plan and calls no cudaMalloc, cudaFree or other allocating
 * routine.  Its scratch (logits, counts, offsets, placement) is one
 * file-scope device array of about 5.6 MB, held on every GPU that loads the
 * library until the process exits.  Limits: T * num_experts <= 2^20,
 * T * top_k <= 2^16, num_experts <= 1024, hidden a multiple of 256 up to
 * 8192; beyond them it returns MOE_ERR_UNSUPPORTED_SHAPE and launches nothing.
 * The first call on a device looks up the array's device address and sets the
 * grouping kernel's shared-memory size; make that first call before any stream
 * capture.  Every call shares the one array: calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.
 * The counts are cleared at the start of each call.  Outputs and argument
 * layout are moe_route's, with an fp32 router weight; router:
 * moe_router_kind; renormalize: 0 or 1.
 * Device-side findings (a non-finite activation) are not reported here. */
moe_status moe_route_static(const void *x_bf16, int32_t T, int32_t hidden, const float *router_w,
                            const float *router_bias, int32_t num_experts, int32_t top_k, int32_t router,
                            int32_t renormalize, int32_t *topk_ids, float *topk_w, int32_t *expert_offsets,
                            int32_t *sorted_rows, void *stream);

/* Text of a status code (static storage). */
const char *moe_status_string(moe_status s);

/* Library version string (static storage). */
const char *moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
