"""Thin Python binding of the C ABI in ``include/vq.h``.

Argument marshalling only: every function takes torch CUDA tensors, checks
that they are contiguous, passes their device pointers, sizes and the current
CUDA stream to the function of the same name in ``libvq.so``, and raises
``VQError`` on a non-zero status. No step of the computation happens here,
and there is no fallback: if the library has not been built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvq.so")
# The same kernels built with -DVQ_CHECK_BOUNDS: every global store (and the
# gathers that have no hardware bounds) is tested against its buffer's extent,
# a miss is skipped and sets bit 1 of the device status word (vq_device_error).
CHECKED_LIB_PATH = os.path.join(_HERE, "libvq_checked.so")

VQ_BF16, VQ_F16, VQ_F32 = 0, 1, 2
_ACT = {torch.bfloat16: VQ_BF16, torch.float16: VQ_F16, torch.float32: VQ_F32}

# Every symbol include/vq.h declares, with its ctypes signature.
_P, _I, _S, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
SIGNATURES = {
    "vq_linear_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "vq_linear": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _P, _S, _P]),
    "vq_linear_host": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _S, _P]),
    "vq_vocab_argmax_workspace_bytes": (_S, [_I]),
    "vq_vocab_argmax": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _S, _P]),
    "vq_vocab_argmax_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P]),
    "vq_vocab_argmax_top2_workspace_bytes": (_S, [_I]),
    "vq_vocab_argmax_top2": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P]),
    "verify_accept_walk": (_I, [_P, _P, _I, _I, _P, _P]),
    "kv_compact_per_row": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P]),
    "verify_round_workspace_bytes": (_S, [_I, _I]),
    "verify_round": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                          _I, _P, _P, _P, _P, _P, _S, _P]),
    "verify_round_multi": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P, _P,
                                _S, _P]),
    "verify_attention_workspace_bytes": (_S, [_I, _I, _I, _I, _I, _I]),
    "verify_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _D, _D,
                              _I, _P, _P, _S, _P]),
    "vq_plan": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "vq_strerror": (ctypes.c_char_p, [_I]),
    "vq_device_error": (_I, [_P, _I, _P]),
    "vq_wait_selftest": (_I, [_P, _P, _P]),
}

_lib = None
_lock = threading.Lock()


class VQError(RuntimeError):
    pass


def open_library(path: str) -> ctypes.CDLL:
    """Loads a build of the library at `path` and declares every signature."""
    if not os.path.exists(path):
        raise VQError("CUDA library %s is missing: build it with "
                      "speculative_block_draft_02_gb300.build.build()" % path)
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = open_library(LIB_PATH)
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise VQError("%s failed: %s (%d)" % (what, lib().vq_strerror(rc).decode(), rc))


def _ptr(t):
    """The device address of a contiguous CUDA tensor as an int (ctypes passes
    it as the void* of the signature), None for None."""
    if t is None:
        return None
    if not t.is_cuda:
        raise VQError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise VQError("expected a contiguous tensor")
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    """The cudaStream_t to enqueue on: `stream`, else the current stream of the
    current device (read without building a Stream object, which costs a few
    microseconds per call)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def vq_linear_workspace_bytes(M: int, K: int, N: int, act=torch.bfloat16) -> int:
    return int(lib().vq_linear_workspace_bytes(M, K, N, _ACT[act]))


def vq_vocab_argmax_workspace_bytes(M: int) -> int:
    return int(lib().vq_vocab_argmax_workspace_bytes(M))


def vq_linear(x, qw, scales, biases, y=None, workspace=None, stream=None):
    """y[M][N] = x[M][K] @ dequant(qw, scales, biases)^T, in x's dtype."""
    M, K = x.shape
    N = qw.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.nbytes
    rc = lib().vq_linear(_ptr(x), M, K, N, _ptr(qw), _ptr(scales), _ptr(biases), _ptr(y),
                         _ACT[x.dtype], _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vq_linear")
    return y


def vq_linear_host(x_host, qw, scales, biases, y_host, x_dev, y_dev, workspace=None, stream=None):
    """vq_linear with x and y in page-locked host memory: enqueues the copy of
    x_host into x_dev, the projection into y_dev and the copy into y_host on
    the stream (synchronize it before reading y_host)."""
    M, K = x_host.shape
    N = qw.shape[0]
    for t in (x_host, y_host):
        if t.is_cuda or not t.is_contiguous():
            raise VQError("expected a contiguous host tensor")
    if x_dev.shape != x_host.shape or y_dev.shape != y_host.shape or x_dev.dtype != x_host.dtype \
            or y_dev.dtype != y_host.dtype:
        raise VQError("device buffers must match the host tensors' shapes and dtypes")
    ws_bytes = 0 if workspace is None else workspace.nbytes
    rc = lib().vq_linear_host(x_host.data_ptr(), M, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                              y_host.data_ptr(), _ACT[x_host.dtype], _ptr(x_dev), _ptr(y_dev),
                              _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vq_linear_host")
    return y_host


def vq_vocab_argmax(x, qw, scales, biases, workspace, argmax=None, maxval=None, stream=None):
    """(argmax int32[M], maxval float32[M]) of x @ dequant(W)^T, logits never stored."""
    M, K = x.shape
    N = qw.shape[0]
    if argmax is None:
        argmax = torch.empty(M, dtype=torch.int32, device=x.device)
    rc = lib().vq_vocab_argmax(_ptr(x), M, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                               _ACT[x.dtype], _ptr(argmax), _ptr(maxval), _ptr(workspace),
                               workspace.nbytes, _stream(stream))
    _check(rc, "vq_vocab_argmax")
    return argmax, maxval


def vq_vocab_argmax_top2_workspace_bytes(M: int) -> int:
    return int(lib().vq_vocab_argmax_top2_workspace_bytes(M))


def vq_vocab_argmax_top2(x, qw, scales, biases, workspace, argmax=None, maxval=None, second=None,
                         stream=None):
    """(argmax int32[M], maxval float32[M], second float32[M]): the arg max and the
    runner-up logit of x @ dequant(W)^T, logits never stored."""
    M, K = x.shape
    N = qw.shape[0]
    if argmax is None:
        argmax = torch.empty(M, dtype=torch.int32, device=x.device)
    if maxval is None:
        maxval = torch.empty(M, dtype=torch.float32, device=x.device)
    if second is None:
        second = torch.empty(M, dtype=torch.float32, device=x.device)
    rc = lib().vq_vocab_argmax_top2(_ptr(x), M, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                                    _ACT[x.dtype], _ptr(argmax), _ptr(maxval), _ptr(second),
                                    _ptr(workspace), workspace.nbytes,
                                    _stream(stream))
    _check(rc, "vq_vocab_argmax_top2")
    return argmax, maxval, second


def vq_vocab_argmax_noalloc(x, qw, scales, biases, argmax=None, maxval=None, stream=None):
    """vq_vocab_argmax with the library's own fixed scratch instead of a workspace."""
    M, K = x.shape
    N = qw.shape[0]
    if argmax is None:
        argmax = torch.empty(M, dtype=torch.int32, device=x.device)
    rc = lib().vq_vocab_argmax_noalloc(_ptr(x), M, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                                       _ACT[x.dtype], _ptr(argmax), _ptr(maxval), _stream(stream))
    _check(rc, "vq_vocab_argmax_noalloc")
    return argmax, maxval


def verify_accept_walk(draft, target, accept=None, stream=None):
    B, L = draft.shape
    if accept is None:
        accept = torch.empty(B, dtype=torch.int32, device=draft.device)
    rc = lib().verify_accept_walk(_ptr(draft), _ptr(target), B, L, _ptr(accept), _stream(stream))
    _check(rc, "verify_accept_walk")
    return accept


def kv_compact_per_row(tensors, prefix_len, src_off, keep, max_keep: int, new_len=None,
                       status=None, stream=None):
    t0 = tensors[0]
    B, H, S_cap, D = t0.shape
    arr = (ctypes.c_void_p * len(tensors))(*[_ptr(t) for t in tensors])
    if new_len is None:
        new_len = torch.empty(B, dtype=torch.int32, device=t0.device)
    rc = lib().kv_compact_per_row(ctypes.cast(arr, ctypes.c_void_p), len(tensors), B, H, S_cap, D,
                                  t0.element_size(), _ptr(prefix_len), _ptr(src_off), _ptr(keep),
                                  max_keep, _ptr(new_len), _ptr(status), _stream(stream))
    _check(rc, "kv_compact_per_row")
    return new_len


def verify_round_workspace_bytes(B: int, L: int) -> int:
    return int(lib().verify_round_workspace_bytes(B, L))


def verify_round(h, qw, scales, biases, tokens, workspace, kv=None, prefix_len=None, src_off=None,
                 new_len=None, status=None, target=None, accept=None, bonus=None, stream=None):
    """One fold-layout verify round: (target int32[B][L], accept int32[B], bonus int32[B],
    new_len int32[B] or None). tokens is int32 [B][L] (row 0 of each block = the committed
    token); kv, if given, is the list of [B][H][S_cap][D] cache tensors to commit."""
    B, L = tokens.shape
    M, K = h.shape
    N = qw.shape[0]
    dev = h.device
    if target is None:
        target = torch.empty((B, L), dtype=torch.int32, device=dev)
    if accept is None:
        accept = torch.empty(B, dtype=torch.int32, device=dev)
    if bonus is None:
        bonus = torch.empty(B, dtype=torch.int32, device=dev)
    if kv:
        t0 = kv[0]
        _, H, S_cap, D = t0.shape
        arr = (ctypes.c_void_p * len(kv))(*[_ptr(t) for t in kv])
        if new_len is None:
            new_len = torch.empty(B, dtype=torch.int32, device=dev)
        kv_args = (ctypes.cast(arr, ctypes.c_void_p), len(kv), H, S_cap, D, t0.element_size(),
                   _ptr(prefix_len), _ptr(src_off), _ptr(new_len), _ptr(status))
    else:
        kv_args = (None, 0, 0, 0, 0, 0, None, None, None, None)
    rc = lib().verify_round(_ptr(h), B, L, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                            _ACT[h.dtype], _ptr(tokens), _ptr(target), _ptr(accept), _ptr(bonus),
                            *kv_args, _ptr(workspace), workspace.nbytes,
                            _stream(stream))
    _check(rc, "verify_round")
    return target, accept, bonus, (new_len if kv else None)


class KvSet(ctypes.Structure):
    """vq_kv_set: one set of caches committed by verify_round_multi."""
    _fields_ = [("tensors", ctypes.c_void_p), ("n_tensors", ctypes.c_int32),
                ("H", ctypes.c_int32), ("S_cap", ctypes.c_int32), ("D", ctypes.c_int32),
                ("elem_bytes", ctypes.c_int32), ("prefix_len", ctypes.c_void_p),
                ("src_off", ctypes.c_void_p), ("new_len", ctypes.c_void_p)]


def verify_round_multi(h, qw, scales, biases, tokens, workspace, sets=(), status=None,
                       target=None, accept=None, bonus=None, stream=None):
    """One fold-layout verify round committing several cache sets: (target
    int32[B][L], accept int32[B], bonus int32[B], [new_len int32[B] per set]).
    Each set is (kv, prefix_len, src_off): a list of [B][H][S_cap][D] cache
    tensors of one shape and that set's int32[B] prefix lengths and block
    offsets (e.g. the target's attention cache and the drafter's context)."""
    B, L = tokens.shape
    M, K = h.shape
    N = qw.shape[0]
    dev = h.device
    if target is None:
        target = torch.empty((B, L), dtype=torch.int32, device=dev)
    if accept is None:
        accept = torch.empty(B, dtype=torch.int32, device=dev)
    if bonus is None:
        bonus = torch.empty(B, dtype=torch.int32, device=dev)
    descs = (KvSet * max(1, len(sets)))()
    keep_alive, new_lens = [], []
    for i, (kv, prefix_len, src_off) in enumerate(sets):
        t0 = kv[0]
        _, H, S_cap, D = t0.shape
        arr = (ctypes.c_void_p * len(kv))(*[_ptr(t) for t in kv])
        keep_alive.append(arr)
        nl = torch.empty(B, dtype=torch.int32, device=dev)
        new_lens.append(nl)
        descs[i] = KvSet(ctypes.cast(arr, ctypes.c_void_p), len(kv), H, S_cap, D,
                         t0.element_size(), _ptr(prefix_len), _ptr(src_off), _ptr(nl))
    rc = lib().verify_round_multi(_ptr(h), B, L, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                                  _ACT[h.dtype], _ptr(tokens), _ptr(target), _ptr(accept),
                                  _ptr(bonus), ctypes.cast(descs, ctypes.c_void_p), len(sets),
                                  _ptr(status), _ptr(workspace),
                                  workspace.nbytes, _stream(stream))
    _check(rc, "verify_round_multi")
    return target, accept, bonus, new_lens


class _Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kernel", "rows_padded", "stages", "prefetch",
                                               "k_splits", "units", "grid", "launches")] + \
               [("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


def verify_attention_workspace_bytes(B: int, L: int, Hq: int, Hkv: int, D: int,
                                     S_cap: int) -> int:
    return int(lib().verify_attention_workspace_bytes(B, L, Hq, Hkv, D, S_cap))


def verify_attention(q, k_new, v_new, k_cache, v_cache, prefix_len, src_off, workspace,
                     rotary_dim: int, theta: float, scale: float, out=None, status=None,
                     stream=None):
    """Attention of the verify block q [B][L][Hq][D] over the per-row caches
    [B][Hkv][S_cap][D] (updated in place with the block's rotated keys and its
    values at slots src_off + j); returns out [B][L][Hq][D]."""
    B, L, Hq, D = q.shape
    Hkv, S_cap = k_cache.shape[1], k_cache.shape[2]
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise VQError("verify_attention takes bf16 or f16 tensors")
    for t in (k_new, v_new, k_cache, v_cache):
        if t.dtype != q.dtype:
            raise VQError("verify_attention: every tensor must have q's dtype")
    if tuple(k_new.shape) != (B, L, Hkv, D) or tuple(v_new.shape) != (B, L, Hkv, D) or \
            tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != D:
        raise VQError("verify_attention: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    rc = lib().verify_attention(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(prefix_len), _ptr(src_off), _ptr(out), B, L, Hq, Hkv, D,
                                S_cap, rotary_dim, float(theta), float(scale), _ACT[q.dtype],
                                _ptr(status), _ptr(workspace),
                                workspace.nbytes,
                                _stream(stream))
    _check(rc, "verify_attention")
    return out


def vq_wait_selftest(status, report, stream=None):
    """Runs the bounded-wait self-test (about two seconds) into status int32[2]
    and report int64[8] on the device."""
    _check(lib().vq_wait_selftest(_ptr(status), _ptr(report), _stream(stream)),
           "vq_wait_selftest")


def vq_plan(M: int, K: int, N: int, act=torch.bfloat16, argmax: bool = False,
            sm_count: int = 152) -> dict:
    """The launch plan of a projection (or arg max) call, computed on the host."""
    p = _Plan()
    _check(lib().vq_plan(M, K, N, _ACT[act], int(argmax), sm_count,
                         ctypes.cast(ctypes.byref(p), ctypes.c_void_p)), "vq_plan")
    return {n: getattr(p, n) for n, _ in _Plan._fields_}


def vq_device_error(clear: bool = False, stream=None) -> int:
    out = ctypes.c_int32(0)
    rc = lib().vq_device_error(ctypes.cast(ctypes.byref(out), ctypes.c_void_p), int(clear),
                               _stream(stream))
    _check(rc, "vq_device_error")
    return int(out.value)
