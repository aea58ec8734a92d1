"""Plain CPU oracle for the QSPEC hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links
or executes anything here, and this package never imports the product.

The arithmetic lives in ``qspec_oracle.c`` (plain C, compiled with
``-ffp-contract=off`` and without fast-math so that every fp32 step is one
IEEE operation).  This module only marshals numpy arrays into it.  Each
function cites the passage of the pages it follows; the readings taken where
the pages are silent are listed at the top of ``qspec_oracle.c``.

Pages cited:
  QSPEC summary   -- "QSPEC: Speculative Decoding with Complementary
                     Quantization Schemes", summary page (molayo1419.me);
                     sections: background terms, QSPEC structure.
  SpecKV blog     -- "SpecKV: compression-aware gamma selection";
                     architecture section (the controller's draft features).

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, brute force or special cases.  The W4A16 reference is
the definition itself in fp64 (pinned by integer special cases); no function
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qspec_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

GROUP = 128
OK, ERR_RANGE, ERR_ZERO_POINT, ERR_NONFINITE = 0, 6, 7, 8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8, u16, u32, i32, f32, f64, u64 = (ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint32,
                                            ctypes.c_int32, ctypes.c_float, ctypes.c_double,
                                            ctypes.c_uint64)
        I = ctypes.c_int
        lib.orc_pack_weights.argtypes = [_P(u8), _P(u16), _P(u16), I, I, _P(u8), _P(u32)]
        lib.orc_pack_weights.restype = I
        lib.orc_quant_act_int4.argtypes = [_P(u16), I, I, I, _P(u8), _P(f32), _P(i32)]
        lib.orc_quant_act_int4.restype = I
        lib.orc_linear_w4a4.argtypes = [_P(u8), _P(f32), _P(u8), _P(u32), I, I, I,
                                        _P(u16), I, _P(i32), _P(f32)]
        lib.orc_linear_w4a4.restype = None
        lib.orc_linear_w4a4_points.argtypes = [_P(u8), _P(f32), _P(u8), _P(u32), I, I, I,
                                               _P(i32), _P(i32), _P(u16)]
        lib.orc_linear_w4a4_points.restype = None
        lib.orc_linear_w4a16.argtypes = [_P(u16), I, _P(u8), _P(u32), I, I, I, _P(f64)]
        lib.orc_linear_w4a16.restype = None
        lib.orc_linear_w4a16_points.argtypes = [_P(u16), I, _P(u8), _P(u32), I, I, I,
                                                _P(i32), _P(i32), _P(f64)]
        lib.orc_linear_w4a16_points.restype = None
        lib.orc_philox4x32_10.argtypes = [_P(u32), _P(u32), _P(u32)]
        lib.orc_philox4x32_10.restype = None
        lib.orc_uniform24.argtypes = [u64, u64, u32, u32]
        lib.orc_uniform24.restype = u32
        lib.orc_qexp.argtypes = [f32]
        lib.orc_qexp.restype = f32
        lib.orc_fixed_softmax_row.argtypes = [_P(u16), I, _P(u64), _P(u64), _P(f32)]
        lib.orc_fixed_softmax_row.restype = I
        lib.orc_verify_greedy.argtypes = [_P(u16), _P(i32), I, I, I, _P(i32), _P(i32)]
        lib.orc_verify_greedy.restype = I
        lib.orc_verify_sample.argtypes = [_P(u16), _P(u16), _P(i32), I, I, I, u64, u64,
                                          _P(i32), _P(i32)]
        lib.orc_verify_sample.restype = I
        lib.orc_draft_sample.argtypes = [_P(u16), I, I, u64, u64, I, _P(i32), _P(f32), _P(f64)]
        lib.orc_draft_sample.restype = I
        lib.orc_kv_overwrite.argtypes = [_P(u16), _P(u16), _P(u16), _P(u16), _P(i32), _P(i32),
                                         I, I, I, I, I, I]
        lib.orc_kv_overwrite.restype = I
        lib.orc_num_threads.argtypes = []
        lib.orc_num_threads.restype = I
        lib.orc_set_num_threads.argtypes = [I]
        lib.orc_set_num_threads.restype = None
        lib.orc_e4m3_value.argtypes = [u8]
        lib.orc_e4m3_value.restype = f64
        lib.orc_e4m3_from_float.argtypes = [f32]
        lib.orc_e4m3_from_float.restype = u8
        lib.orc_e4m3_from_float_array.argtypes = [_P(f32), I, _P(u8)]
        lib.orc_e4m3_from_float_array.restype = None
        lib.orc_quant_weights_fp8.argtypes = [_P(u16), I, I, _P(u8), _P(f32)]
        lib.orc_quant_weights_fp8.restype = I
        lib.orc_quant_act_fp8.argtypes = [_P(u16), I, I, _P(u8), _P(f32)]
        lib.orc_quant_act_fp8.restype = I
        lib.orc_linear_fp8.argtypes = [_P(u8), _P(f32), _P(u8), _P(f32), I, I, I, _P(f64)]
        lib.orc_linear_fp8.restype = None
        _lib = lib
        return lib


def set_num_threads(n: int) -> None:
    """Threads for the oracle's later OpenMP loops."""
    _load().orc_set_num_threads(int(n))


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (its CPU-baseline core count)."""
    return int(_load().orc_num_threads())


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# a1 weight pack -- QSPEC summary, background: 4-bit weights stored with a
# scale s and zero z (W^ = s(W_INT4 - z)); QSPEC structure: one 4-bit weight
# set serves both W4A4 and W4A16.
# ---------------------------------------------------------------------------
def pack_weights(codes, s_bits, z_bits):
    """codes uint8 [N][K] (0..15), s/z fp16 bit patterns uint16 [N][K/128].

    Returns (status, packed uint8 [N][K/2], sz uint32 [N][K/128])."""
    codes, s_bits, z_bits = _c(codes, np.uint8), _c(s_bits, np.uint16), _c(z_bits, np.uint16)
    N, K = codes.shape
    packed = np.zeros((N, K // 2), np.uint8)
    sz = np.zeros((N, K // GROUP), np.uint32)
    st = _load().orc_pack_weights(_ptr(codes, ctypes.c_uint8), _ptr(s_bits, ctypes.c_uint16),
                                  _ptr(z_bits, ctypes.c_uint16), N, K,
                                  _ptr(packed, ctypes.c_uint8), _ptr(sz, ctypes.c_uint32))
    return st, packed, sz


# ---------------------------------------------------------------------------
# a2 activation quantiser -- QSPEC summary, background: W4A4 quantises the
# activations to 4 bits before the low-precision matmul.
# ---------------------------------------------------------------------------
def quant_act_int4(x_bits):
    """x bf16 bit patterns uint16 [M][K].  Returns (status, xq, sx, qs)."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    G = K // GROUP
    xq = np.zeros((M, K // 2), np.uint8)
    sx = np.zeros((M, G), np.float32)
    qs = np.zeros((M, G), np.int32)
    st = _load().orc_quant_act_int4(_ptr(x_bits, ctypes.c_uint16), M, K, K,
                                    _ptr(xq, ctypes.c_uint8), _ptr(sx, ctypes.c_float),
                                    _ptr(qs, ctypes.c_int32))
    return st, xq, sx, qs


# ---------------------------------------------------------------------------
# a3 W4A4 linear -- QSPEC summary, background: 4-bit x 4-bit products,
# accumulation in INT32, then the scale is applied to give a 16-bit result.
# ---------------------------------------------------------------------------
def linear_w4a4(xq, sx, packed, sz, want_I=False, want_acc=False):
    """Returns y (bf16 bits uint16 [M][N]); with want_I also I int32 [M][N][G];
    with want_acc also the fp32 accumulators before the bf16 rounding."""
    xq, sx = _c(xq, np.uint8), _c(sx, np.float32)
    packed, sz = _c(packed, np.uint8), _c(sz, np.uint32)
    M, N, K = xq.shape[0], packed.shape[0], packed.shape[1] * 2
    y = np.zeros((M, N), np.uint16)
    I = np.zeros((M, N, K // GROUP), np.int32) if want_I else None
    acc = np.zeros((M, N), np.float32) if want_acc else None
    _load().orc_linear_w4a4(_ptr(xq, ctypes.c_uint8), _ptr(sx, ctypes.c_float),
                            _ptr(packed, ctypes.c_uint8), _ptr(sz, ctypes.c_uint32), M, N, K,
                            _ptr(y, ctypes.c_uint16), N,
                            _ptr(I, ctypes.c_int32) if want_I else None,
                            _ptr(acc, ctypes.c_float) if want_acc else None)
    res = (y,) + ((I,) if want_I else ()) + ((acc,) if want_acc else ())
    return res if len(res) > 1 else y


def linear_w4a4_points(xq, sx, packed, sz, ms, ns):
    xq, sx = _c(xq, np.uint8), _c(sx, np.float32)
    packed, sz = _c(packed, np.uint8), _c(sz, np.uint32)
    ms, ns = _c(ms, np.int32), _c(ns, np.int32)
    N, K = packed.shape[0], packed.shape[1] * 2
    y = np.zeros(len(ms), np.uint16)
    _load().orc_linear_w4a4_points(_ptr(xq, ctypes.c_uint8), _ptr(sx, ctypes.c_float),
                                   _ptr(packed, ctypes.c_uint8), _ptr(sz, ctypes.c_uint32),
                                   N, K, len(ms), _ptr(ms, ctypes.c_int32),
                                   _ptr(ns, ctypes.c_int32), _ptr(y, ctypes.c_uint16))
    return y


# ---------------------------------------------------------------------------
# a4 W4A16 linear -- QSPEC summary, background: Y = X W^ with
# W^ = s (W_INT4 - z), activations in 16 bits.  fp64 reference.
# ---------------------------------------------------------------------------
def linear_w4a16(x_bits, packed, sz):
    x_bits, packed, sz = _c(x_bits, np.uint16), _c(packed, np.uint8), _c(sz, np.uint32)
    M, K = x_bits.shape
    N = packed.shape[0]
    ref = np.zeros((M, N), np.float64)
    _load().orc_linear_w4a16(_ptr(x_bits, ctypes.c_uint16), K, _ptr(packed, ctypes.c_uint8),
                             _ptr(sz, ctypes.c_uint32), M, N, K, _ptr(ref, ctypes.c_double))
    return ref


def linear_w4a16_points(x_bits, packed, sz, ms, ns):
    x_bits, packed, sz = _c(x_bits, np.uint16), _c(packed, np.uint8), _c(sz, np.uint32)
    ms, ns = _c(ms, np.int32), _c(ns, np.int32)
    K = x_bits.shape[1]
    ref = np.zeros(len(ms), np.float64)
    _load().orc_linear_w4a16_points(_ptr(x_bits, ctypes.c_uint16), K,
                                    _ptr(packed, ctypes.c_uint8), _ptr(sz, ctypes.c_uint32),
                                    packed.shape[0], K, len(ms), _ptr(ms, ctypes.c_int32),
                                    _ptr(ns, ctypes.c_int32), _ptr(ref, ctypes.c_double))
    return ref


# ---------------------------------------------------------------------------
# randomness and fixed-point softmax used by the sampled verification
# ---------------------------------------------------------------------------
def philox4x32_10(counter, key):
    c = np.array(counter, np.uint32)
    k = np.array(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().orc_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32),
                              _ptr(out, ctypes.c_uint32))
    return [int(v) for v in out]


def uniform24(seed, rnd, slot, b):
    return int(_load().orc_uniform24(seed, rnd, slot, b))


def qexp(x: float) -> float:
    return float(_load().orc_qexp(ctypes.c_float(x)))


def fixed_softmax_row(logit_bits):
    """Returns (status, E uint64 [V], S, row max) for one row of bf16 logits."""
    row = _c(logit_bits, np.uint16)
    E = np.zeros(row.shape[0], np.uint64)
    S = ctypes.c_uint64(0)
    m = ctypes.c_float(0)
    st = _load().orc_fixed_softmax_row(_ptr(row, ctypes.c_uint16), row.shape[0],
                                       _ptr(E, ctypes.c_uint64), ctypes.byref(S),
                                       ctypes.byref(m))
    return st, E, int(S.value), float(m.value)


# ---------------------------------------------------------------------------
# a5 greedy verification -- QSPEC summary, background: under greedy decoding
# a draft is accepted when it equals the target's top-1 token; nothing after
# the first rejection is kept; one more token comes from the target.
# ---------------------------------------------------------------------------
def verify_greedy(p_bits, draft):
    p_bits, draft = _c(p_bits, np.uint16), _c(draft, np.int32)
    B, g1, V = p_bits.shape
    gamma = g1 - 1
    assert 1 <= gamma <= 63
    n_acc = np.zeros(B, np.int32)
    out = np.zeros((B, gamma + 1), np.int32)
    st = _load().orc_verify_greedy(_ptr(p_bits, ctypes.c_uint16), _ptr(draft, ctypes.c_int32),
                                   B, gamma, V, _ptr(n_acc, ctypes.c_int32),
                                   _ptr(out, ctypes.c_int32))
    return st, n_acc, out


# ---------------------------------------------------------------------------
# a6 sampled verification -- QSPEC summary, background: accept x with
# probability min(1, p(x|h)/q(x|h)); stop at the first rejection; draw the
# correction token (from the residual max(0, p - q), normalised), or a bonus
# token from the last target distribution when every draft is accepted.
# ---------------------------------------------------------------------------
def verify_sample(p_bits, q_bits, draft, seed, rnd):
    p_bits, q_bits, draft = _c(p_bits, np.uint16), _c(q_bits, np.uint16), _c(draft, np.int32)
    B, g1, V = p_bits.shape
    gamma = g1 - 1
    assert q_bits.shape == (B, gamma, V) and draft.shape == (B, gamma)
    n_acc = np.zeros(B, np.int32)
    out = np.zeros((B, gamma + 1), np.int32)
    st = _load().orc_verify_sample(_ptr(p_bits, ctypes.c_uint16), _ptr(q_bits, ctypes.c_uint16),
                                   _ptr(draft, ctypes.c_int32), B, gamma, V,
                                   ctypes.c_uint64(seed), ctypes.c_uint64(rnd),
                                   _ptr(n_acc, ctypes.c_int32), _ptr(out, ctypes.c_int32))
    return st, n_acc, out


# ---------------------------------------------------------------------------
# draft-side sampling -- QSPEC summary, background: the draft model proposes
# x ~ q(x|h); SpecKV blog, architecture (feature extraction): the gamma
# controller reads the draft softmax's confidence (largest probability) and
# entropy -sum p log(p + 1e-9).
# ---------------------------------------------------------------------------
def draft_sample(q_bits, seed, rnd, step):
    """q_bits: uint16 bf16 logits [B][V]; step: draft position 1..16.
    Returns (status, token int32 [B], confidence float32 [B], entropy float64 [B])."""
    q_bits = _c(q_bits, np.uint16)
    B, V = q_bits.shape
    assert 1 <= step <= 16
    token = np.zeros(B, np.int32)
    conf = np.zeros(B, np.float32)
    ent = np.zeros(B, np.float64)
    st = _load().orc_draft_sample(_ptr(q_bits, ctypes.c_uint16), B, V, ctypes.c_uint64(seed),
                                  ctypes.c_uint64(rnd), step, _ptr(token, ctypes.c_int32),
                                  _ptr(conf, ctypes.c_float), _ptr(ent, ctypes.c_double))
    return st, token, conf, ent


# ---------------------------------------------------------------------------
# a7 KV overwrite -- QSPEC summary, QSPEC structure: for accepted tokens the
# W4A4 KV-cache entries are replaced by the W4A16 ones.
# ---------------------------------------------------------------------------
def kv_overwrite(k_cache, v_cache, k_new, v_new, base_pos, n_acc, gamma):
    """In place on k_cache / v_cache (uint16 [L][B][H][T][D])."""
    L, B, H, T, D = k_cache.shape
    assert k_new.shape == (L, B, gamma + 1, H, D)
    base_pos, n_acc = _c(base_pos, np.int32), _c(n_acc, np.int32)
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    return _load().orc_kv_overwrite(_ptr(k_cache, ctypes.c_uint16), _ptr(v_cache, ctypes.c_uint16),
                                    _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16),
                                    _ptr(base_pos, ctypes.c_int32), _ptr(n_acc, ctypes.c_int32),
                                    L, B, H, T, D, gamma)


# ---------------------------------------------------------------------------
# next-3 SpecQuant Q8 -- SpecQuant summary page, contributions and approach:
# Q4 / Q8 (FP8) / Q16 variants derived post-training from one FP16 parent
# with shared base weights.  E4M3 per output channel for the weights, per
# token for the activations; the FP8 linear of the Q8 model.
# ---------------------------------------------------------------------------
def e4m3_value(b: int) -> float:
    """Value of one E4M3 byte (NaN for S.1111.111)."""
    return float(_load().orc_e4m3_value(int(b) & 0xFF))


def e4m3_from_float(f) -> np.ndarray:
    """fp32 values -> E4M3 bytes (round to nearest even, saturate at 448)."""
    f = _c(np.atleast_1d(np.asarray(f, np.float32)), np.float32)
    out = np.zeros(f.shape, np.uint8)
    _load().orc_e4m3_from_float_array(_ptr(f, ctypes.c_float), f.size, _ptr(out, ctypes.c_uint8))
    return out


def quant_weights_fp8(w16_bits):
    """w16_bits: fp16 bit patterns uint16 [N][K] (the parent weights).
    Returns (status, w8 uint8 [N][K], s8 float32 [N])."""
    w16_bits = _c(w16_bits, np.uint16)
    N, K = w16_bits.shape
    w8 = np.zeros((N, K), np.uint8)
    s8 = np.zeros(N, np.float32)
    st = _load().orc_quant_weights_fp8(_ptr(w16_bits, ctypes.c_uint16), N, K, _ptr(w8, ctypes.c_uint8),
                                       _ptr(s8, ctypes.c_float))
    return st, w8, s8


def quant_act_fp8(x_bits):
    """x_bits: bf16 bit patterns uint16 [M][K].  Returns (status, xq uint8 [M][K], sa float32 [M])."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    xq = np.zeros((M, K), np.uint8)
    sa = np.zeros(M, np.float32)
    st = _load().orc_quant_act_fp8(_ptr(x_bits, ctypes.c_uint16), M, K, _ptr(xq, ctypes.c_uint8),
                                   _ptr(sa, ctypes.c_float))
    return st, xq, sa


def linear_fp8(xq, sa, w8, s8):
    """fp64 reference of the FP8 linear: ref [M][N] = sa[m] s8[n] sum_k xq w8."""
    xq, w8 = _c(xq, np.uint8), _c(w8, np.uint8)
    sa, s8 = _c(sa, np.float32), _c(s8, np.float32)
    M, K = xq.shape
    N = w8.shape[0]
    ref = np.zeros((M, N), np.float64)
    _load().orc_linear_fp8(_ptr(xq, ctypes.c_uint8), _ptr(sa, ctypes.c_float), _ptr(w8, ctypes.c_uint8),
                           _ptr(s8, ctypes.c_float), M, N, K, _ptr(ref, ctypes.c_double))
    return ref
