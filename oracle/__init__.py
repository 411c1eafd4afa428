"""Plain CPU oracle for the block-verification hot path.

TEST INFRASTRUCTURE ONLY: the parity reference for the CUDA library. Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may build, import or call it; the product package never does, and it shares
no code with the CUDA sources.

The arithmetic lives in ``vq_oracle.c`` (scalar C, fp64); this module builds
it with gcc and marshals numpy arrays into it. What each function computes,
and which passage of the pages it follows, is stated in the C file:

* ``vq_linear``   -- the W4 group-64 affine verification projection
  (dflash-mlx #7, PR description: VerifyQuantizedLinear).
* ``argmax``      -- greedy target tokens, lowest index on ties, decided on
  fp32-rounded logits (ds4 #778, commit 1 message: greedy at temperature 0).
* ``accept_walk`` -- longest matching draft prefix per row
  (mlxcel #2865, Summary).
* ``kv_compact``  -- per-row KV commit to a contiguous valid prefix
  (mlxcel #2865, Summary).
* ``verify_attention`` -- the verify block's attention, rotated at every row's
  own logical positions, no query seeing the stale gap (mlxcel #2865, Summary and commit
  message), with ``round_bits`` its rounding to the 16-bit storage formats.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vq_oracle.c")
_SO = os.path.join(_HERE, "_vq_oracle.so")
_lock = threading.Lock()
_lib = None

BF16, F16, F32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available). Returns the .so path."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_vq_linear.argtypes = [p, i, i, i, i, p, p, p, p, i, p, i]
            lib.oracle_vq_linear.restype = i
            lib.oracle_argmax.argtypes = [p, i, i, p, p, p]
            lib.oracle_argmax.restype = None
            lib.oracle_accept_walk.argtypes = [p, p, i, i, p]
            lib.oracle_accept_walk.restype = None
            lib.oracle_kv_compact.argtypes = [p, i, i, i, i, i, i, p, p, p, i, p, p]
            lib.oracle_kv_compact.restype = None
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_double.restype = ctypes.c_double
            lib.oracle_round_bits.argtypes = [ctypes.c_double, i]
            lib.oracle_round_bits.restype = ctypes.c_uint16
            lib.oracle_verify_attention.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i,
                                                    ctypes.c_double, ctypes.c_double, i, p, p,
                                                    p, i]
            lib.oracle_verify_attention.restype = i
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """Threads the oracle's OpenMP loops would use (1 without OpenMP)."""
    return _load().oracle_num_threads()


def _act_dtype(x: np.ndarray, act_dtype: int | None) -> int:
    if act_dtype is not None:
        return act_dtype
    if x.dtype == np.float32:
        return F32
    raise ValueError("16-bit activations are passed as uint16 bits with an explicit act_dtype")


def vq_linear(x: np.ndarray, qw: np.ndarray, scales: np.ndarray, biases: np.ndarray,
              act_dtype: int | None = None, cols=None, threads: int | None = None) -> np.ndarray:
    """fp64 y[M][N] (or y[M][len(cols)]) of the W4 projection.

    x: [M][K] as uint16 bits (bf16/f16, act_dtype required) or float32.
    qw: uint32 [N][K/8]; scales, biases: uint16 bf16 bits [N][K/64].
    """
    lib = _load()
    dt = _act_dtype(x, act_dtype)
    x = np.ascontiguousarray(x)
    qw = np.ascontiguousarray(qw, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    biases = np.ascontiguousarray(biases, dtype=np.uint16)
    M, K = x.shape
    N = qw.shape[0]
    assert qw.shape == (N, K // 8) and scales.shape == (N, K // 64) == biases.shape
    if cols is None:
        c_ptr, n_cols = None, N
    else:
        cols = np.ascontiguousarray(cols, dtype=np.int32)
        c_ptr, n_cols = _ptr(cols), len(cols)
    y = np.empty((M, n_cols), dtype=np.float64)
    rc = lib.oracle_vq_linear(_ptr(x), dt, M, K, N, _ptr(qw), _ptr(scales), _ptr(biases),
                              c_ptr, n_cols, _ptr(y), threads or num_threads())
    if rc != 0:
        raise ValueError("oracle_vq_linear rejected its arguments")
    return y


def argmax(logits: np.ndarray):
    """(idx int32[M], maxval float32[M], second float32[M]) per the fp32 decision."""
    lib = _load()
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    M, N = logits.shape
    idx = np.empty(M, dtype=np.int32)
    mx = np.empty(M, dtype=np.float32)
    sec = np.empty(M, dtype=np.float32)
    lib.oracle_argmax(_ptr(logits), M, N, _ptr(idx), _ptr(mx), _ptr(sec))
    return idx, mx, sec


def fold_accept(tokens: np.ndarray, target: np.ndarray):
    """Fold layout (ds4 #778, PR description: the committed token verified as
    row 0 of its block): tokens[b][0] is the committed token, tokens[b][1..]
    the drafts, target[b][j] the greedy token after position j. Draft j+1 is
    accepted while it equals target[b][j], i.e. the accept walk of the drafts
    against the targets of the rows before them. Returns (accept, bonus,
    keep) with bonus = target[b][accept[b]] and keep = accept + 1."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    target = np.ascontiguousarray(target, dtype=np.int32)
    B, L = tokens.shape
    assert target.shape == (B, L) and L >= 1
    if L == 1:
        acc = np.zeros(B, dtype=np.int32)
    else:
        acc = accept_walk(tokens[:, 1:], target[:, :-1])
    bonus = target[np.arange(B), acc].astype(np.int32)
    return acc, bonus, (acc + 1).astype(np.int32)


def accept_walk(draft: np.ndarray, target: np.ndarray) -> np.ndarray:
    lib = _load()
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    target = np.ascontiguousarray(target, dtype=np.int32)
    B, L = draft.shape
    assert target.shape == (B, L)
    acc = np.empty(B, dtype=np.int32)
    lib.oracle_accept_walk(_ptr(draft), _ptr(target), B, L, _ptr(acc))
    return acc


def kv_compact(tensors, prefix_len, src_off, keep, max_keep: int):
    """In-place on a list of numpy arrays [B][H][S_cap][D]; returns (new_len, status)."""
    lib = _load()
    t0 = tensors[0]
    B, H, S_cap, D = t0.shape
    for t in tensors:
        assert t.shape == t0.shape and t.dtype == t0.dtype and t.flags["C_CONTIGUOUS"]
    arr = (ctypes.c_void_p * len(tensors))(*[t.ctypes.data for t in tensors])
    pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
    so = np.ascontiguousarray(src_off, dtype=np.int32)
    kp = np.ascontiguousarray(keep, dtype=np.int32)
    new_len = np.empty(B, dtype=np.int32)
    status = np.zeros(1, dtype=np.int32)
    lib.oracle_kv_compact(ctypes.cast(arr, ctypes.c_void_p), len(tensors), B, H, S_cap, D,
                          t0.dtype.itemsize, _ptr(pl), _ptr(so), _ptr(kp), max_keep,
                          _ptr(new_len), _ptr(status))
    return new_len, int(status[0])


def bf16_to_double(h: int) -> float:
    return _load().oracle_bf16_to_double(h)


def f16_to_double(h: int) -> float:
    return _load().oracle_f16_to_double(h)


def round_bits(v: float, dtype: int) -> int:
    """Bits of v rounded to bf16 (dtype 0) or f16 (dtype 1), nearest even."""
    return int(_load().oracle_round_bits(float(v), dtype))


def verify_attention(q, k_new, v_new, k_cache, v_cache, prefix_len, src_off, dtype: int,
                     rotary_dim: int, theta: float, scale: float, threads: int | None = None):
    """Verify-block attention; k_cache / v_cache are updated in place.

    q [B][L][Hq][D], k_new / v_new [B][L][Hkv][D], caches [B][Hkv][S_cap][D]: uint16
    bits of dtype (0 bf16, 1 f16). Returns (out fp64 [B][L][Hq][D], k_rot fp64
    [B][L][Hkv][D] before rounding, status).
    """
    lib = _load()
    B, L, Hq, D = q.shape
    Hkv = k_new.shape[2]
    S_cap = k_cache.shape[2]
    arrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k_new, v_new)]
    assert arrs[1].shape == arrs[2].shape == (B, L, Hkv, D)
    for c in (k_cache, v_cache):
        assert c.dtype == np.uint16 and c.flags["C_CONTIGUOUS"] and c.shape == (B, Hkv, S_cap, D)
    pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
    so = np.ascontiguousarray(src_off, dtype=np.int32)
    out = np.empty((B, L, Hq, D), dtype=np.float64)
    k_rot = np.empty((B, L, Hkv, D), dtype=np.float64)
    status = np.zeros(1, dtype=np.int32)
    rc = lib.oracle_verify_attention(_ptr(arrs[0]), _ptr(arrs[1]), _ptr(arrs[2]), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(pl), _ptr(so), B, L, Hq, Hkv, D, S_cap,
                                     rotary_dim, float(theta), float(scale), dtype, _ptr(out),
                                     _ptr(k_rot), _ptr(status), threads or num_threads())
    if rc != 0:
        raise ValueError("oracle_verify_attention rejected its arguments")
    return out, k_rot, int(status[0])
