"""CPU oracle for the routed MoE FFN over NVFP4 weights.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never loads it, and it shares no code with the CUDA path.

Two halves:
  * ``moe_oracle.c`` (compiled here into ``_build/liboracle.so``): the parts whose
    result must be bit-exact -- E2M1/E4M3 codecs, the NVFP4 quantiser in fp32,
    the router logits in a fixed fp32 order, top-k and the stable grouping.
  * this module: ctypes wrappers and the FFN in FP64 with numpy (a matmul is
    the only library step), following the definition

        out[t] = sum_j w[t][j] * FFN_{id[t][j]}(x_t)  (+ FFN_shared(x_t))
        FFN_e(v) = Wd_e ( silu(Wg_e v) * (Wu_e v) ),   silu(z) = z / (1 + e^-z)

    with every weight dequantised as E2M1(code) * E4M3(scale) * tensor_scale.
    The SwiGLU output enters the down product rounded as the mode says: to
    bf16 (W4A16) or NVFP4 with its batch tensor scale (W4A4).

Sources (page title, section): "NVIDIA FP4-Local checkpoints on DGX Spark ...
#565", section 4 Round 1 -- gate, up and SwiGLU of the routed experts (#766),
one FP32 tensor scale per expert weight (#517, #545), activations rounded to
FP4 in the W4A4 GEMM (#687), the SwiGLU output quantised before the down GEMM
(#760), down rows in BF16 rounded to nearest even (#914), the card sum folded
into the combine (#701), the shared expert added beside the routed ones (#686);
"bloomery 0.3.9", New: an f64 oracle with a band for sums whose order is the
hardware's.

Parity status: the codecs (E2M1, E4M3, E8M0), the NVFP4 and MXFP4
quantisers, router, top-k, grouping and the FFN are pinned by the tests in
``tests/test_oracle_*.py`` (tables, library
conversions, brute force, identities, a hand-worked example, a dense-MLP
special case).  Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_lock = threading.Lock()
_lib = None

ROUTER_SOFTMAX = 0
ROUTER_SIGMOID = 1
MODE_W4A16 = 0
MODE_W4A4 = 1
FMT_NVFP4 = 0      # E2M1 codes, E4M3 scale a 16-value block, fp32 tensor scale
FMT_MXFP4 = 1      # E2M1 codes, E8M0 scale a 32-value block (OCP MX), no tensor scale


def build_library(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (no fused multiply-add contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            _SRC, "-o", _SO + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build_library()
            L = ctypes.CDLL(_SO)
            c = ctypes
            P = c.c_void_p
            L.oracle_e2m1_value.argtypes = [c.c_int]
            L.oracle_e2m1_value.restype = c.c_double
            L.oracle_e4m3_value.argtypes = [c.c_int]
            L.oracle_e4m3_value.restype = c.c_double
            L.oracle_e2m1_table.argtypes = [P]
            L.oracle_e4m3_table.argtypes = [P]
            L.oracle_e4m3_from_f32.argtypes = [c.c_float]
            L.oracle_e4m3_from_f32.restype = c.c_uint8
            L.oracle_e2m1_from_f32.argtypes = [c.c_float]
            L.oracle_e2m1_from_f32.restype = c.c_uint8
            L.oracle_e4m3_from_f32_array.argtypes = [P, c.c_int64, P]
            L.oracle_e2m1_from_f32_array.argtypes = [P, c.c_int64, P]
            L.oracle_f64_to_bf16.argtypes = [c.c_double]
            L.oracle_f64_to_bf16.restype = c.c_uint16
            L.oracle_f64_to_bf16_array.argtypes = [P, c.c_int64, P]
            L.oracle_nvfp4_tensor_scale.argtypes = [P, c.c_int64]
            L.oracle_nvfp4_tensor_scale.restype = c.c_float
            L.oracle_nvfp4_quantize.argtypes = [P, c.c_int64, c.c_int64, c.c_float, P, P]
            L.oracle_router_logits.argtypes = [P, c.c_int32, c.c_int32, P, c.c_int32, P, P]
            L.oracle_topk.argtypes = [P, c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32, P, P]
            L.oracle_group.argtypes = [P, c.c_int64, c.c_int32, P, P]
            L.oracle_e8m0_value.argtypes = [c.c_int]
            L.oracle_e8m0_value.restype = c.c_double
            L.oracle_e8m0_table.argtypes = [P]
            L.oracle_mxfp4_quantize.argtypes = [P, c.c_int64, c.c_int64, P, P]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ codecs

def e2m1_table() -> np.ndarray:
    out = np.zeros(16, np.float64)
    lib().oracle_e2m1_table(_p(out))
    return out


def e4m3_table() -> np.ndarray:
    out = np.zeros(256, np.float64)
    lib().oracle_e4m3_table(_p(out))
    return out


def e4m3_from_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.zeros(x.shape, np.uint8)
    lib().oracle_e4m3_from_f32_array(_p(x), x.size, _p(out))
    return out


def e2m1_from_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.zeros(x.shape, np.uint8)
    lib().oracle_e2m1_from_f32_array(_p(x), x.size, _p(out))
    return out


def f64_to_bf16(x) -> np.ndarray:
    """FP64 -> bf16 bit patterns (uint16), one round-to-nearest-even."""
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    out = np.zeros(x.shape, np.uint16)
    lib().oracle_f64_to_bf16_array(_p(x), x.size, _p(out))
    return out


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_to_f32(b) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ NVFP4

def tensor_scale(x) -> float:
    """amax / (6*448) of the whole tensor, in fp32."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    return float(np.float32(lib().oracle_nvfp4_tensor_scale(_p(x), x.size)))


def quantize(x, ts: float | None = None):
    """NVFP4-quantise a [rows][cols] fp32 matrix.  Returns (codes, scales, ts)."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    assert x.ndim == 2 and x.shape[1] % 16 == 0
    if ts is None:
        ts = tensor_scale(x)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    lib().oracle_nvfp4_quantize(_p(x), rows, cols, ctypes.c_float(ts), _p(codes), _p(scales))
    return codes, scales, float(np.float32(ts))


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[.., K/2] bytes -> [.., K] 4-bit codes, element 2i from the low nibble."""
    codes = np.asarray(codes, np.uint8)
    q = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    q[..., 0::2] = codes & 0x0F
    q[..., 1::2] = codes >> 4
    return q


def dequantize(codes, scales, ts) -> np.ndarray:
    """NVFP4 -> FP64: E2M1(code) * E4M3(scale) * tensor_scale."""
    q = unpack_codes(codes)
    s = np.repeat(e4m3_table()[np.asarray(scales, np.uint8)], 16, axis=-1)
    return e2m1_table()[q] * s * float(ts)


# ------------------------------------------------------------------ MXFP4

def e8m0_table() -> np.ndarray:
    out = np.zeros(256, np.float64)
    lib().oracle_e8m0_table(_p(out))
    return out


def quantize_mx(x):
    """MXFP4-quantise a [rows][cols] fp32 matrix (OCP MX: E8M0 scale a
    32-value block, E2M1 codes).  Returns (codes, scales)."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    assert x.ndim == 2 and x.shape[1] % 32 == 0
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 32), np.uint8)
    lib().oracle_mxfp4_quantize(_p(x), rows, cols, _p(codes), _p(scales))
    return codes, scales


def dequantize_mx(codes, scales) -> np.ndarray:
    """MXFP4 -> FP64: E2M1(code) * 2^(scale - 127)."""
    q = unpack_codes(codes)
    s = np.repeat(e8m0_table()[np.asarray(scales, np.uint8)], 32, axis=-1)
    return e2m1_table()[q] * s


def dequant(w, fmt: int = FMT_NVFP4) -> np.ndarray:
    """One packed weight as the expert callback gives it: (codes, scales, ts)
    for NVFP4, (codes, scales[, ignored]) for MXFP4."""
    if fmt == FMT_MXFP4:
        return dequantize_mx(w[0], w[1])
    return dequantize(*w)


# Decisions of the quantiser that lie this close to their rounding boundary
# (relative to the E4M3 argument for a scale, to the block's largest |x/den|
# for a code) are the ones a different fp32 summation order of the quantised
# value can flip: 2^-16 is 16 times the fp32 error of the GEMM sums that feed
# the W4A4 SwiGLU quantiser.
FLIP_MARGIN = 2.0 ** -16
_E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_E2M1_STEP = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0])   # gap between the two codes around each midpoint


def quant_decisions(x, ts: float, margin: float = FLIP_MARGIN):
    """NVFP4-quantise fp32 rows x with tensor scale ts (the c-4 rule) and bound
    what the near-boundary decisions could change.

    Returns (deq, flip, n): deq = the dequantised values (FP64); flip = per
    element, |change| of the dequantised value if every decision within
    `margin` of its boundary went the other way (a block scale: the block
    re-quantised with the neighbouring E4M3 scale; a code: the neighbouring
    E2M1 value); n = the number of such decisions.  This is the band that the
    "f64 oracle with a band for sums whose order is the hardware's" of
    "bloomery 0.3.9" (New) calls for, applied where that order decides an
    integer."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    R, C = x.shape
    codes, scales, ts = quantize(x, ts)
    deq = dequantize(codes, scales, ts)
    flip = np.zeros((R, C), np.float64)
    if R == 0:
        return deq, flip, 0
    ts32 = np.float32(ts)
    xb = x.reshape(R, C // 16, 16)
    bamax = np.abs(xb).max(axis=2)
    q = (bamax / np.float32(6.0)).astype(np.float32) / ts32 if ts32 > 0 else np.zeros_like(bamax)
    pos = np.unique(e4m3_table()[:127])            # finite E4M3 values >= 0, ascending
    mids = (pos[1:] + pos[:-1]) / 2
    qd = q.astype(np.float64)
    j = np.clip(np.searchsorted(mids, qd), 1, len(mids) - 1)
    near = np.where(np.abs(qd - mids[j - 1]) <= np.abs(qd - mids[j]), j - 1, j)   # nearest midpoint
    s_nom = e4m3_table()[scales.astype(np.int64)]
    s_alt = np.where(s_nom == pos[near], pos[near + 1], pos[near])
    den = (s_nom.astype(np.float32) * ts32).astype(np.float32)
    live = den > 0
    scale_flag = live & (np.abs(qd - mids[near]) < margin * qd)
    # codes: |x/den| near an E2M1 midpoint, relative to the block's largest |x/den|
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.abs(xb / np.where(live, den, np.float32(1))[..., None]).astype(np.float64)
    dist = np.abs(v[..., None] - _E2M1_MIDS)
    m = dist.argmin(axis=-1)
    vmax = v.max(axis=2, keepdims=True)
    code_flag = live[..., None] & (dist.min(axis=-1) < margin * vmax)
    fb = flip.reshape(R, C // 16, 16)
    fb += np.where(code_flag, _E2M1_STEP[m] * (s_nom * float(ts))[..., None], 0.0)   # dequantised as dequantize() does
    for r, b in zip(*np.nonzero(scale_flag)):
        d_alt = np.float32(np.float32(s_alt[r, b]) * ts32)         # the quantiser's fp32 divisor
        alt = e2m1_table()[e2m1_from_f32(xb[r, b] / d_alt)] * (s_alt[r, b] * float(ts))
        fb[r, b] += np.abs(alt - deq[r, 16 * b:16 * b + 16])
    return deq, flip, int(code_flag.sum() + scale_flag.sum())


def mx_quant_decisions(x, margin: float = FLIP_MARGIN):
    """MXFP4 counterpart of quant_decisions: quantise fp32 rows x, and bound
    what the decisions within `margin` of their boundary could change.  A
    block scale (E = floor(log2(amax)) - 2) is near its boundary when amax is
    within margin * amax of a power of two: the block is re-quantised with the
    neighbouring exponent.  A code is near its boundary when |x| / 2^E is
    within margin * (the block's largest |x| / 2^E) of an E2M1 midpoint: the
    neighbouring E2M1 value.  Returns (deq, flip, n)."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    R, C = x.shape
    codes, scales = quantize_mx(x)
    deq = dequantize_mx(codes, scales)
    flip = np.zeros((R, C), np.float64)
    if R == 0:
        return deq, flip, 0
    xb = x.reshape(R, C // 32, 32).astype(np.float64)
    X = e8m0_table()[scales.astype(np.int64)]                     # [R][C/32]
    bamax = np.abs(xb).max(axis=2)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(bamax > 0, bamax, 1.0))
    m = np.round(lg)
    near = (bamax > 0) & (np.abs(bamax - np.exp2(m)) < margin * bamax)
    v = np.abs(xb) / X[..., None]
    dist = np.abs(v[..., None] - _E2M1_MIDS)
    mi = dist.argmin(axis=-1)
    vmax = v.max(axis=2, keepdims=True)
    code_flag = dist.min(axis=-1) < margin * vmax
    fb = flip.reshape(R, C // 32, 32)
    fb += np.where(code_flag, _E2M1_STEP[mi] * X[..., None], 0.0)
    for r, b in zip(*np.nonzero(near)):
        s_alt = int(scales[r, b]) + (1 if bamax[r, b] < np.exp2(m[r, b]) else -1)
        s_alt = min(max(s_alt, 0), 254)
        Xa = np.float32(np.ldexp(1.0, s_alt - 127))
        alt = e2m1_table()[e2m1_from_f32(x[r, 32 * b:32 * b + 32] / Xa)] * float(Xa)
        fb[r, b] += np.abs(alt - deq[r, 32 * b:32 * b + 32])
    return deq, flip, int(code_flag.sum() + near.sum())


# ------------------------------------------------------------------ router

def router_logits(x_bf16: np.ndarray, router_w: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """Router logits in the fixed fp32 order (moe_oracle.c).  router_w is fp32
    [E][H], or uint16 bf16 words [E][H] (the router kept in its BF16 words,
    "NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4 Round 1,
    #732): those widen to fp32 exactly, so the same fp32 sums follow."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    if np.asarray(router_w).dtype == np.uint16:
        router_w = bf16_to_f32(router_w)
    w = np.ascontiguousarray(router_w, np.float32)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H and H % 8 == 0
    out = np.zeros((T, E), np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    lib().oracle_router_logits(_p(x), T, H, _p(w), E, None if b is None else _p(b), _p(out))
    return out


def topk(logits: np.ndarray, k: int, kind: int, renormalize: bool = True):
    lg = np.ascontiguousarray(logits, np.float32)
    T, E = lg.shape
    assert 1 <= k <= min(E, 64)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().oracle_topk(_p(lg), T, E, k, kind, int(bool(renormalize)), _p(ids), _p(w))
    return ids, w


def group(ids: np.ndarray, E: int):
    flat = np.ascontiguousarray(ids, np.int32).ravel()
    offsets = np.zeros(E + 1, np.int32)
    rows = np.zeros(flat.size, np.int32)
    lib().oracle_group(_p(flat), flat.size, E, _p(offsets), _p(rows))
    return offsets, rows


# ------------------------------------------------------------------ FFN

def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def route(x_bf16, router_w, router_bias, k, kind, renormalize=True):
    """Router + grouping.  Returns a dict of logits, ids, weights, offsets, rows."""
    E = router_w.shape[0]
    lg = router_logits(x_bf16, router_w, router_bias)
    ids, w = topk(lg, k, kind, renormalize)
    offsets, rows = group(ids, E)
    return dict(logits=lg, ids=ids, weights=w, offsets=offsets, sorted_rows=rows)


def quantize_activations(x_bf16: np.ndarray):
    """W4A4 activation quantisation: tensor scale from the batch amax."""
    xf = bf16_to_f32(x_bf16)
    return quantize(xf)


def swiglu_tensor_scale(h_list) -> float:
    """W4A4 tensor scale of a set of SwiGLU output matrices: the amax over all
    of them (each rounded to fp32 first), divided by 6 * 448 in fp32.  The
    routed rows of a batch form one set, the shared expert's rows another."""
    amax = np.float32(0.0)
    for h in h_list:
        if np.asarray(h).size:
            amax = max(amax, np.float32(np.max(np.abs(np.asarray(h, np.float32)))))
    return float(np.float32(np.float32(amax) / np.float32(2688.0)))


def swiglu_quantize(h_list):
    """W4A4: NVFP4 quantisation of one set of SwiGLU output matrices with their
    shared tensor scale.  Returns ([(codes, scales)], ts)."""
    ts = swiglu_tensor_scale(h_list)
    out = []
    for h in h_list:
        c, sc, _ = quantize(np.asarray(h, np.float32), ts)
        out.append((c, sc))
    return out, ts


def forward(x_bf16, router_w, router_bias, expert, *, k, router_kind, renormalize=True,
            mode=MODE_W4A16, shared=None, keep=False, h_in=None, fmt=FMT_NVFP4):
    """The whole MoE FFN in FP64.

    expert(e) -> ((gc, gs, gts), (uc, us, uts), (dc, ds, dts)): expert e's packed
    NVFP4 gate [I][H], up [I][H] and down [H][I] (the oracle's own quantisation).
    shared: None or the same triple for the shared expert (weight 1, every token).
    h_in: None, or given SwiGLU outputs to run the rest of the path on (a
    stage-isolated check): {e: [rows of expert e in grouped order][I]} for every
    routed expert the batch touches, plus "shared": [T][Is] when a shared expert
    is given.  The oracle then skips the gate/up products and rounds or
    quantises these h values by the mode's rule, then runs down and combine.
    fmt: FMT_NVFP4, or FMT_MXFP4 (MXFP4 weights; expert(e) gives (codes,
    scales, ignored) triples).  In W4A4 the activations and the SwiGLU output
    are then quantised to the same format: MXFP4 blocks of 32 with their own
    E8M0 scales, with no tensor scale ("MXFP4 routed prompt GEMM on the
    block-scaled tensor cores", "NVIDIA FP4-Local checkpoints on DGX Spark
    ... #565", section 6 Round 3; E8M0 blocks of 32 as in the pages' MXFP8
    weights, #521).
    Returns a dict with the route, the FP64 output and its bf16 bit patterns.
    """
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    T, H = x_bf16.shape
    E = router_w.shape[0]
    r = route(x_bf16, router_w, router_bias, k, router_kind, renormalize)
    res = dict(r)
    if mode == MODE_W4A4 and fmt == FMT_MXFP4:
        xc, xs = quantize_mx(bf16_to_f32(x_bf16))
        xin = dequantize_mx(xc, xs)
        res.update(x_codes=xc, x_scales=xs, x_ts=1.0)
    elif mode == MODE_W4A4:
        xc, xs, xts = quantize_activations(x_bf16)
        xin = dequantize(xc, xs, xts)
        res.update(x_codes=xc, x_scales=xs, x_ts=xts)
    else:
        xin = bf16_to_f64(x_bf16)

    offsets, rows = r["offsets"], r["sorted_rows"]
    wflat = r["weights"].ravel()
    out = np.zeros((T, H), np.float64)

    def up_part(weights, X):
        g = X @ dequant(weights[0], fmt).T
        u = X @ dequant(weights[1], fmt).T
        return silu(g) * u

    def down_part(weights, h):
        return h @ dequant(weights[2], fmt).T

    def round_h_bf16(h):
        """W4A16: the SwiGLU output is rounded to bf16 (nearest even) before the
        down product ("down rows in BF16, the product rounding each to nearest
        even", page 3 section 4, #914)."""
        return bf16_to_f64(f64_to_bf16(h))

    def quant_h(h_all):
        """W4A4: SwiGLU output rounded to fp32, quantised with its batch amax
        (MXFP4: block by block, no tensor scale).  Also returns, per matrix,
        the flip band of its near-boundary decisions."""
        h32 = [h.astype(np.float32) for h in h_all]
        if fmt == FMT_MXFP4:
            qs = [mx_quant_decisions(h) for h in h32]
            return [q[0] for q in qs], 1.0, [q[1] for q in qs], sum(q[2] for q in qs)
        ts = swiglu_tensor_scale(h32)
        qs = [quant_decisions(h, ts) for h in h32]
        return [q[0] for q in qs], ts, [q[1] for q in qs], sum(q[2] for q in qs)

    active = [e for e in range(E) if offsets[e + 1] > offsets[e]]
    hs = {}
    for e in active:
        pr = rows[offsets[e]:offsets[e + 1]]
        if h_in is not None:
            hs[e] = np.asarray(h_in[e], np.float64 if mode == MODE_W4A16 else np.float32)
            assert hs[e].shape[0] == pr.size
        else:
            hs[e] = up_part(expert(e), xin[pr // k])
    band = np.zeros((T, H), np.float64)    # W4A4: what near-boundary h decisions could move
    flips = {}
    n_flip = 0
    if mode == MODE_W4A4:
        qh, ts_h, fl, n_flip = quant_h([hs[e] for e in active])
        hs = dict(zip(active, qh))
        flips = dict(zip(active, fl))
        res["h_ts"] = ts_h
    else:
        hs = {e: round_h_bf16(h) for e, h in hs.items()}
    if keep:
        res["h"] = hs
    for e in active:
        pr = rows[offsets[e]:offsets[e + 1]]
        y = down_part(expert(e), hs[e])
        np.add.at(out, pr // k, wflat[pr][:, None] * y)
        if e in flips and flips[e].any():
            np.add.at(band, pr // k, np.abs(wflat[pr])[:, None] * (flips[e] @ np.abs(dequant(expert(e)[2], fmt)).T))

    if shared is not None:
        hsh = np.asarray(h_in["shared"]) if h_in is not None else up_part(shared, xin)
        if mode == MODE_W4A4:
            (hsh,), ts_s, (fs,), ns = quant_h([hsh])
            n_flip += ns
            res["shared_h_ts"] = ts_s
            if fs.any():
                band += fs @ np.abs(dequant(shared[2], fmt)).T
        else:
            hsh = round_h_bf16(hsh)
        out += down_part(shared, hsh)

    res["out"] = out
    res["band"] = band
    res["h_flips"] = n_flip
    res["out_bf16"] = f64_to_bf16(out)
    return res


def bf16_half_ulp(ref) -> np.ndarray:
    """Half a bf16 ulp at each |ref|: the most an exactly rounded bf16 output
    can differ from the FP64 value it rounds (bf16 has 8 significant bits)."""
    a = np.abs(np.asarray(ref, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -126.0) - 8.0), 2.0 ** -134)


def compare_output(got_bf16: np.ndarray, ref_f64: np.ndarray, band: np.ndarray | None = None):
    """Output tolerance.  Element-wise |d| <= 2e-2 * RMS(ref) + half a bf16 ulp
    of ref (+ band), and ||d||_2 / ||ref||_2 <= 5e-3.

    The output is bf16, rounded once from the exact sum: half an ulp of the
    result is the format's own rounding, which an exact implementation also
    makes, so the 2e-2 * RMS bound applies to the computation error on top of
    it.  (With outputs reaching 5 RMS, as the 4096-token prompt's do, the
    exactly rounded output alone can differ from the FP64 value by 2e-2 * RMS.)
    `band` (W4A4) is forward()'s bound on what the SwiGLU quantiser's
    near-boundary decisions can move; it is zero where no such decision
    touches an output."""
    got = bf16_to_f64(got_bf16)
    d = np.abs(got - ref_f64)
    rms = float(np.sqrt(np.mean(ref_f64 ** 2)))
    max_abs = float(np.max(d)) if d.size else 0.0
    rel_l2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref_f64), 1e-300))
    base = 2e-2 * rms + bf16_half_ulp(ref_f64)
    lim = base + (0.0 if band is None else band)
    beyond = d > lim
    ok = (not bool(beyond.any())) and (rel_l2 <= 5e-3) and bool(np.all(np.isfinite(got)))
    excess = d - base
    return ok, dict(max_abs=max_abs, rms=rms, max_abs_over_rms=max_abs / max(rms, 1e-300), rel_l2=rel_l2,
                    max_excess_over_rounding=float(np.max(excess)) / max(rms, 1e-300) if d.size else 0.0,
                    inside_band_only=int(((excess > 0) & ~beyond).sum()), beyond=int(beyond.sum()))
