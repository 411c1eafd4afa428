"""Seeded synthetic inputs for the verification hot path.

This module only draws random inputs and stores them in the library's formats.
It holds none of the method's arithmetic (no dequantization, projection, arg
max, accept walk or compaction), so both the CUDA path and the CPU oracle can
consume exactly the same bytes from it.

Formats:
  * activations: [M][K] bf16 or f16 as uint16 bit patterns (rounded to nearest
    even from a float32 draw), or float32;
  * weights: qw uint32 [N][K/8]. Eight independent codes uniform on 0..15
    packed into a word are exactly a uniformly random 32-bit word, so the
    words are drawn directly; scales / biases are bf16 bit patterns [N][K/64];
  * draft tokens int32 [B][L]; KV tensors fp16 [B][H][S_cap][D].

Every tensor has its own generator, keyed by (seed, tensor name), so adding or
reshaping one tensor does not change the others.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np
import torch

GROUP = 64
ACT_DTYPES = ("bf16", "f16", "f32")


def rng_for(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([seed, zlib.crc32(name.encode())])


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def act_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return to_bf16_bits(a)
    if dtype == "f16":
        return to_f16_bits(a)
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    raise ValueError(dtype)


def activations(seed: int, M: int, K: int, dtype: str = "bf16", scale: float = 1.0,
                name: str = "x") -> np.ndarray:
    """x[M][K] ~ scale * N(0, 1), stored in `dtype`."""
    r = rng_for(seed, name)
    a = (r.standard_normal((M, K), dtype=np.float32) * np.float32(scale)).astype(np.float32)
    return act_bits(a, dtype)


@dataclass
class W4Weights:
    qw: np.ndarray       # uint32 [N][K/8]
    scales: np.ndarray   # uint16 bf16 bits [N][K/64]
    biases: np.ndarray   # uint16 bf16 bits [N][K/64]

    @property
    def N(self) -> int:
        return self.qw.shape[0]

    @property
    def K(self) -> int:
        return self.qw.shape[1] * 8

    @property
    def nbytes(self) -> int:
        return self.qw.nbytes + self.scales.nbytes + self.biases.nbytes


def w4_weights(seed: int, N: int, K: int, name: str = "w") -> W4Weights:
    """Codes uniform 0..15, scale ~ U(0.005, 0.02), bias ~ U(-0.1, 0.1), as bf16."""
    assert K % GROUP == 0
    qw = rng_for(seed, name + ".qw").integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint32)
    s = rng_for(seed, name + ".scales").uniform(0.005, 0.02, size=(N, K // GROUP))
    b = rng_for(seed, name + ".biases").uniform(-0.1, 0.1, size=(N, K // GROUP))
    return W4Weights(qw, to_bf16_bits(s.astype(np.float32)), to_bf16_bits(b.astype(np.float32)))


def drafts_from_target(seed: int, target: np.ndarray, vocab: int, p: float = 0.7,
                       name: str = "draft") -> np.ndarray:
    """Draft tokens against a target block [B][L].

    Per position, while no miss has occurred, the draft equals the target with
    probability p; otherwise it is a token guaranteed to differ. After the
    first miss the remaining positions are uniform random tokens.
    """
    r = rng_for(seed, name)
    B, L = target.shape
    out = np.empty((B, L), dtype=np.int32)
    for b in range(B):
        missed = False
        for j in range(L):
            t = int(target[b, j])
            if missed:
                out[b, j] = int(r.integers(0, vocab))
            elif r.random() < p:
                out[b, j] = t
            else:
                out[b, j] = (t + 1 + int(r.integers(0, vocab - 1))) % vocab
                missed = True
    return out


@dataclass
class CommitCase:
    tensors: list            # n_tensors arrays fp16 [B][H][S_cap][D]
    prefix_len: np.ndarray   # int32 [B]
    src_off: np.ndarray      # int32 [B]
    keep: np.ndarray         # int32 [B]
    block: int


def commit_case(seed: int, layers: int = 8, B: int = 4, H: int = 8, S_cap: int = 2048,
                D: int = 128, block: int = 16, prefix_lo: int = 200, prefix_hi: int = 1800,
                keep=None, src_off=None, name: str = "kv") -> CommitCase:
    """Rectangular KV cache with per-row valid prefixes and a shared verify block.

    K and V of each layer are separate tensors (2 * layers of them), filled with
    fp16 ~ N(0, 1). prefix_len ~ U{prefix_lo..prefix_hi}; the verify block sits at
    the shared offset S = max prefix_len (the rectangular cache), unless src_off is
    given; keep ~ U{0..block} unless given.
    """
    r = rng_for(seed, name + ".lens")
    prefix = r.integers(prefix_lo, prefix_hi + 1, size=B).astype(np.int32)
    if src_off is None:
        src_off = np.full(B, int(prefix.max()), dtype=np.int32)
    if keep is None:
        keep = rng_for(seed, name + ".keep").integers(0, block + 1, size=B).astype(np.int32)
    vals = rng_for(seed, name + ".vals")
    tensors = [vals.standard_normal((B, H, S_cap, D), dtype=np.float32).astype(np.float16)
               for _ in range(2 * layers)]
    return CommitCase(tensors, prefix, np.asarray(src_off, dtype=np.int32),
                      np.asarray(keep, dtype=np.int32), block)


@dataclass
class AttentionCase:
    q: np.ndarray            # uint16 bits [B][L][Hq][D]
    k_new: np.ndarray        # uint16 bits [B][L][Hkv][D]
    v_new: np.ndarray        # uint16 bits [B][L][Hkv][D]
    k_cache: np.ndarray      # uint16 bits [B][Hkv][S_cap][D]
    v_cache: np.ndarray      # uint16 bits [B][Hkv][S_cap][D]
    prefix_len: np.ndarray   # int32 [B]
    src_off: np.ndarray      # int32 [B]
    dtype: str


def attention_case(seed: int, B: int = 4, L: int = 16, Hq: int = 32, Hkv: int = 8,
                   D: int = 128, S_cap: int = 2048, prefix_lo: int = 200,
                   prefix_hi: int = 1800, dtype: str = "f16", src_off=None, prefix_len=None,
                   name: str = "attn") -> AttentionCase:
    """The verify block's attention inputs over a rectangular cache.

    q, k_new, v_new and every cache slot (the valid prefix, the stale gap and the
    unused tail alike) ~ N(0, 1) in `dtype`. prefix_len ~ U{prefix_lo..prefix_hi}
    unless given; the verify block sits at the shared offset max prefix_len (the
    rectangular cache) unless src_off is given.
    """
    if prefix_len is None:
        prefix_len = rng_for(seed, name + ".lens").integers(prefix_lo, prefix_hi + 1, size=B)
    prefix_len = np.asarray(prefix_len, dtype=np.int32)
    if src_off is None:
        src_off = np.full(B, int(prefix_len.max()), dtype=np.int32)

    def draw(tag, shape):
        a = rng_for(seed, name + "." + tag).standard_normal(shape, dtype=np.float32)
        return act_bits(a, dtype)

    return AttentionCase(draw("q", (B, L, Hq, D)), draw("k_new", (B, L, Hkv, D)),
                         draw("v_new", (B, L, Hkv, D)), draw("k_cache", (B, Hkv, S_cap, D)),
                         draw("v_cache", (B, Hkv, S_cap, D)), prefix_len,
                         np.asarray(src_off, dtype=np.int32), dtype)


# The seeded workloads, by what they are. Seed 0 throughout.
WORKLOADS = {
    "tiny_w4_verify_m8_k512_n1024": dict(M=8, K=512, N=1024, dtype="bf16", x_scale=1.0,
                                          B=1, L=8),
    "verify_w4_m8_k5120_n17408": dict(M=8, K=5120, N=17408, dtype="bf16", x_scale=1.0),
    "verify_w4_m8_k5120_n1024": dict(M=8, K=5120, N=1024, dtype="bf16", x_scale=1.0),
    "sweep_w4_k5120_n17408": dict(Ms=(1, 4, 8, 16), K=5120, N=17408,
                                  dtypes=("bf16", "f16", "f32"), x_scale=0.5),
    "vocab_argmax_b4_l16_k2560_n151936": dict(M=64, K=2560, N=151936, dtype="bf16",
                                              x_scale=1.0, B=4, L=16, p=0.7),
    "commit_b4_l16_then_verify_m64": dict(layers=8, B=4, H=8, S_cap=2048, D=128, block=16,
                                          M=64, K=5120, N=17408, dtype="bf16"),
    # the verify block's attention over the same cache shape (fp16, 8 KV heads x 128,
    # prefixes ~U(200, 1800)), with 32 query heads (4 per KV head) and rotary
    # embedding over all 128 dimensions at base 1e6
    "verify_attention_b4_l16_hq32_hkv8_d128": dict(B=4, L=16, Hq=32, Hkv=8, D=128, S_cap=2048,
                                                   prefix_lo=200, prefix_hi=1800, dtype="f16",
                                                   rotary_dim=128, theta=1.0e6),
}
