"""Thin Python binding of libqspec.so (the C ABI in include/qspec.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  The functions
named ``qspec_*`` mirror the C calls one to one (caller-provided outputs);
the short names (``pack_weights`` ...) allocate the outputs with torch and
call the same entry points.

There is no fallback: if libqspec.so is missing or the device is not an
sm_103 part, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libqspec.so")

GROUP = 128
MAX_GAMMA = 16
STATUS = {0: "QSPEC_OK", 1: "QSPEC_ERR_NULL", 2: "QSPEC_ERR_SHAPE", 3: "QSPEC_ERR_ALIGN",
          4: "QSPEC_ERR_LAUNCH", 5: "QSPEC_ERR_WORKSPACE", 6: "QSPEC_ERR_RANGE",
          7: "QSPEC_ERR_ZERO_POINT", 8: "QSPEC_ERR_NONFINITE", 9: "QSPEC_ERR_TIMEOUT",
          10: "QSPEC_ERR_UNSUPPORTED"}
OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAUNCH, ERR_WORKSPACE = 0, 1, 2, 3, 4, 5
ERR_RANGE, ERR_ZERO_POINT, ERR_NONFINITE, ERR_TIMEOUT, ERR_UNSUPPORTED = 6, 7, 8, 9, 10

EXPORTED = ["qspec_version", "qspec_status_string", "qspec_last_cuda_error", "qspec_kernel_launches",
            "qspec_pack_weights",
            "qspec_quant_act_int4", "qspec_linear_w4a4", "qspec_linear_w4a4_bf16", "qspec_linear_w4a16",
            "qspec_verify_workspace_bytes", "qspec_verify_greedy", "qspec_verify_sample",
            "qspec_kv_overwrite", "qspec_verify_sample_noalloc", "qspec_draft_workspace_bytes",
            "qspec_draft_sample", "qspec_debug_linear_bounded", "qspec_quant_weights_fp8",
            "qspec_quant_act_fp8", "qspec_linear_fp8", "qspec_linear_w4a16_kv"]
KERNEL_W4A16_TC, KERNEL_W4A4_GEMV_TC, KERNEL_W4A4_TC = 0, 1, 2
NOALLOC_SCRATCH_BYTES = 1 << 20


class QspecError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = "%s failed: %s" % (where, STATUS.get(status, str(status)))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libqspec.so and declare its prototypes.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libqspec.so is not built (%s); run "
                               "quantized_speculative_decoding_shared_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        vp, i32, sz_t, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
        proto = {
            "qspec_version": ([], i32),
            "qspec_kernel_launches": ([], ctypes.c_ulonglong),
            "qspec_status_string": ([i32], ctypes.c_char_p),
            "qspec_last_cuda_error": ([], ctypes.c_char_p),
            "qspec_pack_weights": ([vp, vp, vp, i32, i32, vp, vp, vp, vp], i32),
            "qspec_quant_act_int4": ([vp, i32, i32, i32, vp, vp, vp, vp, vp], i32),
            "qspec_linear_w4a4": ([vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, vp, vp, vp], i32),
            "qspec_linear_w4a4_bf16": ([vp, i32, vp, vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp],
                                       i32),
            "qspec_linear_w4a16": ([vp, i32, vp, vp, i32, i32, i32, vp, i32, vp, vp], i32),
            "qspec_verify_workspace_bytes": ([i32, i32, i32], sz_t),
            "qspec_verify_greedy": ([vp, vp, i32, i32, i32, vp, vp, vp, sz_t, vp, vp], i32),
            "qspec_verify_sample": ([vp, vp, vp, i32, i32, i32, u64, u64, vp, vp, vp, sz_t, vp, vp],
                                    i32),
            "qspec_kv_overwrite": ([vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp],
                                   i32),
            "qspec_verify_sample_noalloc": ([vp, vp, vp, i32, i32, i32, u64, u64, vp, vp, vp, vp],
                                            i32),
            "qspec_draft_workspace_bytes": ([i32, i32], sz_t),
            "qspec_draft_sample": ([vp, i32, i32, u64, u64, i32, vp, vp, vp, vp, sz_t, vp, vp], i32),
            "qspec_debug_linear_bounded": ([i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, i32,
                                            ctypes.c_uint32, i32, vp, vp], i32),
            "qspec_quant_weights_fp8": ([vp, i32, i32, vp, vp, vp, vp], i32),
            "qspec_quant_act_fp8": ([vp, i32, i32, i32, vp, vp, vp, vp], i32),
            "qspec_linear_fp8": ([vp, vp, vp, vp, i32, i32, i32, vp, i32, vp, vp], i32),
            "qspec_linear_w4a16_kv": ([vp, i32, vp, vp, i32, i32, i32, vp, i32, i32, i32, i32, i32, i32,
                                       vp, vp, vp, vp, vp, vp], i32),
        }
        for name, (args, res) in proto.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        if path is None:
            _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str):
    if rc != OK:
        detail = ""
        if rc == ERR_LAUNCH:
            detail = load_library().qspec_last_cuda_error().decode()
        raise QspecError(rc, where, detail)


def _need(t, dtype, name):
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


# ---------------------------------------------------------------------------
# one-to-one wrappers of the C calls (outputs provided by the caller)
# ---------------------------------------------------------------------------
def qspec_pack_weights(codes, s, z, N, K, packed, sz, dev_status=None, stream=None):
    return load_library().qspec_pack_weights(_ptr(codes), _ptr(s), _ptr(z), N, K, _ptr(packed),
                                             _ptr(sz), _ptr(dev_status), _stream(stream))


def qspec_quant_act_int4(x, M, K, ldx, xq, sx, qs, dev_status=None, stream=None):
    return load_library().qspec_quant_act_int4(_ptr(x), M, K, ldx, _ptr(xq), _ptr(sx), _ptr(qs),
                                               _ptr(dev_status), _stream(stream))


def qspec_linear_w4a4(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I=None, dev_status=None,
                      stream=None):
    return load_library().qspec_linear_w4a4(_ptr(xq), _ptr(sx), _ptr(qs), _ptr(packed), _ptr(sz),
                                            M, N, K, _ptr(y), ldy, _ptr(dbg_I), _ptr(dev_status),
                                            _stream(stream))


def qspec_linear_w4a4_bf16(x, ldx, packed, sz, M, N, K, y, ldy, xq, sx, qs, dbg_I=None,
                           dev_status=None, stream=None):
    return load_library().qspec_linear_w4a4_bf16(_ptr(x), ldx, _ptr(packed), _ptr(sz), M, N, K,
                                                 _ptr(y), ldy, _ptr(xq), _ptr(sx), _ptr(qs),
                                                 _ptr(dbg_I), _ptr(dev_status), _stream(stream))


def qspec_linear_w4a16(x, ldx, packed, sz, M, N, K, y, ldy, dev_status=None, stream=None):
    return load_library().qspec_linear_w4a16(_ptr(x), ldx, _ptr(packed), _ptr(sz), M, N, K,
                                             _ptr(y), ldy, _ptr(dev_status), _stream(stream))


def qspec_linear_w4a16_kv(x, ldx, packed, sz, M, N, K, y, ldy, kv_col0, H, D, T, gamma, k_cache, v_cache,
                          base_pos, n_acc, dev_status=None, stream=None):
    return load_library().qspec_linear_w4a16_kv(_ptr(x), ldx, _ptr(packed), _ptr(sz), M, N, K, _ptr(y), ldy,
                                                kv_col0, H, D, T, gamma, _ptr(k_cache), _ptr(v_cache),
                                                _ptr(base_pos), _ptr(n_acc), _ptr(dev_status), _stream(stream))


def qspec_verify_workspace_bytes(B, gamma, V):
    return int(load_library().qspec_verify_workspace_bytes(B, gamma, V))


def qspec_verify_greedy(p, draft, B, gamma, V, n_acc, out, workspace, ws_bytes, dev_status=None,
                        stream=None):
    return load_library().qspec_verify_greedy(_ptr(p), _ptr(draft), B, gamma, V, _ptr(n_acc),
                                              _ptr(out), _ptr(workspace), ws_bytes,
                                              _ptr(dev_status), _stream(stream))


def qspec_verify_sample(p, q, draft, B, gamma, V, seed, rnd, n_acc, out, workspace, ws_bytes,
                        dev_status=None, stream=None):
    return load_library().qspec_verify_sample(_ptr(p), _ptr(q), _ptr(draft), B, gamma, V,
                                              ctypes.c_uint64(seed), ctypes.c_uint64(rnd),
                                              _ptr(n_acc), _ptr(out), _ptr(workspace), ws_bytes,
                                              _ptr(dev_status), _stream(stream))


def qspec_verify_sample_noalloc(p, q, draft, B, gamma, V, seed, rnd, n_acc, out, dev_status=None,
                                stream=None):
    """Sampled verification with the library's built-in scratch array: for
    callers that cannot allocate device memory (see include/qspec.h)."""
    return load_library().qspec_verify_sample_noalloc(_ptr(p), _ptr(q), _ptr(draft), B, gamma, V,
                                                      ctypes.c_uint64(seed), ctypes.c_uint64(rnd),
                                                      _ptr(n_acc), _ptr(out), _ptr(dev_status),
                                                      _stream(stream))


def qspec_draft_workspace_bytes(B, V):
    return int(load_library().qspec_draft_workspace_bytes(B, V))


def qspec_draft_sample(q, B, V, seed, rnd, step, token, confidence, entropy, workspace, ws_bytes,
                       dev_status=None, stream=None):
    return load_library().qspec_draft_sample(_ptr(q), B, V, ctypes.c_uint64(seed), ctypes.c_uint64(rnd),
                                             step, _ptr(token), _ptr(confidence), _ptr(entropy),
                                             _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))


def qspec_kv_overwrite(k_cache, v_cache, k_new, v_new, base_pos, n_acc, L, B, H, T, D, gamma,
                       dev_status=None, stream=None):
    return load_library().qspec_kv_overwrite(_ptr(k_cache), _ptr(v_cache), _ptr(k_new),
                                             _ptr(v_new), _ptr(base_pos), _ptr(n_acc), L, B, H, T,
                                             D, gamma, _ptr(dev_status), _stream(stream))


def qspec_kernel_launches():
    """Kernel launches this library has issued (graph captures count once)."""
    return int(load_library().qspec_kernel_launches())


def qspec_debug_linear_bounded(kernel, x, xq, sx, qs, packed, sz, M, N, K, y, ldy, wait_limit,
                               stall, dev_status=None, stream=None):
    """Test diagnostic: one tensor-core linear kernel with a chosen bound on
    its barrier waits (and, with stall, a wait made to run out)."""
    return load_library().qspec_debug_linear_bounded(kernel, _ptr(x), _ptr(xq), _ptr(sx), _ptr(qs),
                                                     _ptr(packed), _ptr(sz), M, N, K, _ptr(y), ldy,
                                                     ctypes.c_uint32(wait_limit), stall,
                                                     _ptr(dev_status), _stream(stream))


def qspec_quant_weights_fp8(w16, N, K, w8, s8, dev_status=None, stream=None):
    return load_library().qspec_quant_weights_fp8(_ptr(w16), N, K, _ptr(w8), _ptr(s8), _ptr(dev_status),
                                                  _stream(stream))


def qspec_quant_act_fp8(x, M, K, ldx, xq, sa, dev_status=None, stream=None):
    return load_library().qspec_quant_act_fp8(_ptr(x), M, K, ldx, _ptr(xq), _ptr(sa), _ptr(dev_status),
                                              _stream(stream))


def qspec_linear_fp8(xq, sa, w8, s8, M, N, K, y, ldy, dev_status=None, stream=None):
    return load_library().qspec_linear_fp8(_ptr(xq), _ptr(sa), _ptr(w8), _ptr(s8), M, N, K, _ptr(y), ldy,
                                           _ptr(dev_status), _stream(stream))


# ---------------------------------------------------------------------------
# allocating conveniences (torch tensors in, torch tensors out)
# ---------------------------------------------------------------------------
def pack_weights(codes, s, z, dev_status=None, stream=None):
    """codes uint8 [N][K], s / z fp16 [N][K/128] -> (packed uint8 [N][K/2], sz int32 [N][K/128])."""
    _need(codes, torch.uint8, "codes")
    _need(s, torch.float16, "s")
    _need(z, torch.float16, "z")
    N, K = codes.shape
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=codes.device)
    sz = torch.empty((N, K // GROUP), dtype=torch.int32, device=codes.device)
    _check(qspec_pack_weights(codes, s, z, N, K, packed, sz, dev_status, stream),
           "qspec_pack_weights")
    return packed, sz


def quant_act_int4(x, dev_status=None, stream=None):
    """x bf16 [M][K] -> (xq uint8 [M][K/2], sx fp32 [M][G], qs int32 [M][G])."""
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=x.device)
    qs = torch.empty((M, K // GROUP), dtype=torch.int32, device=x.device)
    _check(qspec_quant_act_int4(x, M, K, K, xq, sx, qs, dev_status, stream), "qspec_quant_act_int4")
    return xq, sx, qs


def linear_w4a4(xq, sx, qs, packed, sz, want_I=False, out=None, dev_status=None, stream=None):
    M, N, K = xq.shape[0], packed.shape[0], packed.shape[1] * 2
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    I = (torch.empty((M, N, K // GROUP), dtype=torch.int32, device=xq.device) if want_I else None)
    _check(qspec_linear_w4a4(xq, sx, qs, packed, sz, M, N, K, y, y.stride(0), I, dev_status,
                             stream), "qspec_linear_w4a4")
    return (y, I) if want_I else y


def linear_w4a4_bf16(x, packed, sz, want_I=False, out=None, dev_status=None, stream=None):
    """Quantise bf16 activations and run the W4A4 linear in one call:
    returns (y, xq, sx, qs) (and I when want_I), equal to quant_act_int4
    followed by linear_w4a4."""
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    dev = x.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=dev)
    qs = torch.empty((M, K // GROUP), dtype=torch.int32, device=dev)
    I = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=dev) if want_I else None
    _check(qspec_linear_w4a4_bf16(x, x.stride(0), packed, sz, M, N, K, y, y.stride(0), xq, sx, qs, I,
                                  dev_status, stream), "qspec_linear_w4a4_bf16")
    return (y, xq, sx, qs, I) if want_I else (y, xq, sx, qs)


def linear_w4a16(x, packed, sz, out=None, dev_status=None, stream=None):
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(qspec_linear_w4a16(x, x.stride(0), packed, sz, M, N, K, y, y.stride(0), dev_status,
                              stream), "qspec_linear_w4a16")
    return y


def verify_workspace(B, gamma, V, device="cuda"):
    n = qspec_verify_workspace_bytes(B, gamma, V)
    if n == 0:
        raise QspecError(ERR_SHAPE, "qspec_verify_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def verify_greedy(p, draft, workspace=None, dev_status=None, stream=None):
    B, g1, V = p.shape
    gamma = g1 - 1
    ws = workspace if workspace is not None else verify_workspace(B, gamma, V, p.device)
    n_acc = torch.empty(B, dtype=torch.int32, device=p.device)
    out = torch.empty((B, gamma + 1), dtype=torch.int32, device=p.device)
    _check(qspec_verify_greedy(p, draft, B, gamma, V, n_acc, out, ws, ws.numel(), dev_status,
                               stream), "qspec_verify_greedy")
    return n_acc, out


def verify_sample(p, q, draft, seed, rnd, workspace=None, dev_status=None, stream=None):
    B, g1, V = p.shape
    gamma = g1 - 1
    ws = workspace if workspace is not None else verify_workspace(B, gamma, V, p.device)
    n_acc = torch.empty(B, dtype=torch.int32, device=p.device)
    out = torch.empty((B, gamma + 1), dtype=torch.int32, device=p.device)
    _check(qspec_verify_sample(p, q, draft, B, gamma, V, seed, rnd, n_acc, out, ws, ws.numel(),
                               dev_status, stream), "qspec_verify_sample")
    return n_acc, out


def draft_workspace(B, V, device="cuda"):
    n = qspec_draft_workspace_bytes(B, V)
    if n == 0:
        raise QspecError(ERR_SHAPE, "qspec_draft_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def draft_sample(q, seed, rnd, step, workspace=None, dev_status=None, stream=None):
    """q bf16 [B][V] draft logits of draft position step (1..16) ->
    (token int32 [B], confidence fp32 [B], entropy fp32 [B])."""
    _need(q, torch.bfloat16, "q")
    B, V = q.shape
    ws = workspace if workspace is not None else draft_workspace(B, V, q.device)
    token = torch.empty(B, dtype=torch.int32, device=q.device)
    conf = torch.empty(B, dtype=torch.float32, device=q.device)
    ent = torch.empty(B, dtype=torch.float32, device=q.device)
    _check(qspec_draft_sample(q, B, V, seed, rnd, step, token, conf, ent, ws, ws.numel(), dev_status,
                              stream), "qspec_draft_sample")
    return token, conf, ent


def kv_overwrite(k_cache, v_cache, k_new, v_new, base_pos, n_acc, dev_status=None, stream=None):
    L, B, H, T, D = k_cache.shape
    gamma = k_new.shape[2] - 1
    _check(qspec_kv_overwrite(k_cache, v_cache, k_new, v_new, base_pos, n_acc, L, B, H, T, D,
                              gamma, dev_status, stream), "qspec_kv_overwrite")


def quant_weights_fp8(w16, dev_status=None, stream=None):
    """Parent weights fp16 [N][K] -> (w8 uint8 [N][K] E4M3, s8 fp32 [N])."""
    _need(w16, torch.float16, "w16")
    N, K = w16.shape
    w8 = torch.empty((N, K), dtype=torch.uint8, device=w16.device)
    s8 = torch.empty(N, dtype=torch.float32, device=w16.device)
    _check(qspec_quant_weights_fp8(w16, N, K, w8, s8, dev_status, stream), "qspec_quant_weights_fp8")
    return w8, s8


def quant_act_fp8(x, dev_status=None, stream=None):
    """bf16 [M][K] -> (xq uint8 [M][K] E4M3, sa fp32 [M])."""
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sa = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(qspec_quant_act_fp8(x, M, K, x.stride(0), xq, sa, dev_status, stream), "qspec_quant_act_fp8")
    return xq, sa


def linear_fp8(xq, sa, w8, s8, out=None, dev_status=None, stream=None):
    M, K = xq.shape
    N = w8.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _check(qspec_linear_fp8(xq, sa, w8, s8, M, N, K, y, y.stride(0), dev_status, stream), "qspec_linear_fp8")
    return y
