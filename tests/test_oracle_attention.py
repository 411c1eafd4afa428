"""Pins for the oracle's verify-block attention, checked against things other
than itself.

The rounding to the 16-bit storage formats is pinned to numpy's and torch's
conversions; the rotary embedding to hand-worked values of its closed form and
to its defining property (a dot product of two rotated vectors depends only on
their position difference); the attention to closed forms (equal keys give the
mean of the visible values, a single visible key gives its value), to torch's
scaled-dot-product attention on explicitly gathered masks, and to the
invariances of the mask (stale gap and unused slots never matter, the block is
causal). A wrong pairing or rotation sign, a position off by the prefix, a
wrong query-to-KV-head map or a mask that lets the stale gap in fails one of
them.
"""
import math

import numpy as np
import pytest
import torch

from speculative_block_draft_02_gb300 import synth

BF16, F16 = 0, 1
DT = {"bf16": BF16, "f16": F16}


def run(oracle_mod, case, rotary_dim, theta, scale=None):
    D = case.q.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    out, k_rot, st = oracle_mod.verify_attention(case.q, case.k_new, case.v_new, kc, vc,
                                                 case.prefix_len, case.src_off, DT[case.dtype],
                                                 rotary_dim, theta, scale)
    return out, k_rot, st, kc, vc


def decode(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- rounding


def test_round_bits_f16_matches_numpy(oracle_mod):
    r = np.random.default_rng(1)
    vals = list(r.standard_normal(3000) * np.exp(r.uniform(-20, 12, 3000)))
    # exact ties between neighbours (normal and subnormal), the overflow edge
    for a in (1, 2, 3, 1023, 1024, 2047):
        vals += [(a + 0.5) * 2.0 ** -10, (a + 0.5) * 2.0 ** -24, -(a + 0.5) * 2.0 ** 3]
    vals += [65504.0, 65519.99, 65520.0, -65520.0, 1e-9, -1e-9, 0.0, -0.0, 2.0 ** -25,
             3 * 2.0 ** -26]
    ref = np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.round_bits(v, F16) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_round_bits_bf16_matches_torch(oracle_mod):
    r = np.random.default_rng(2)
    u = r.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    u[:500] = (u[:500] & 0xFFFF0000) | 0x8000          # exact ties
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.round_bits(float(v), BF16) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- rotary embedding


def test_rope_hand_case(oracle_mod):
    # D = 8, rotary_dim 4 (pairs (0, 2) and (1, 3)), base 10000; prefix 3, block at 5
    D, S_cap = 8, 8
    c = synth.attention_case(0, B=1, L=2, Hq=1, Hkv=1, D=D, S_cap=S_cap, prefix_len=[3],
                             src_off=[5], dtype="f16")
    k = np.zeros((1, 2, 1, D), dtype=np.float32)
    k[0, 0, 0, 0] = 1.0                       # e0 at position 3
    k[0, 1, 0, 1] = 1.0                       # e1 + 2 e6 at position 4
    k[0, 1, 0, 6] = 2.0
    c.k_new = synth.to_f16_bits(k)
    out, k_rot, st, kc, vc = run(oracle_mod, c, 4, 10000.0)
    assert st == 0
    e0 = np.zeros(D)
    e0[0], e0[2] = math.cos(3.0), math.sin(3.0)            # angle 3 * 10000^0
    e1 = np.zeros(D)
    e1[1], e1[3] = math.cos(0.04), math.sin(0.04)          # angle 4 * 10000^(-1/2)
    e1[6] = 2.0                                            # beyond rotary_dim: unchanged
    np.testing.assert_allclose(k_rot[0, 0, 0], e0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(k_rot[0, 1, 0], e1, rtol=0, atol=1e-15)
    # the block's slots hold the rounded rotated keys and the values as given
    for j in range(2):
        want = [oracle_mod.round_bits(v, F16) for v in k_rot[0, j, 0]]
        assert list(kc[0, 0, 5 + j]) == want
        assert np.array_equal(vc[0, 0, 5 + j], c.v_new[0, j, 0])


def test_rope_depends_only_on_position_differences(oracle_mod):
    B, L, D = 2, 6, 64
    c = synth.attention_case(3, B=B, L=L, Hq=1, Hkv=1, D=D, S_cap=1024, prefix_len=[7, 700],
                             src_off=[900, 900], dtype="bf16")
    c.k_new[1] = c.k_new[0]                  # the same vectors, shifted by 693 positions
    _, k_rot, st, _, _ = run(oracle_mod, c, D, 10000.0)
    assert st == 0
    g0 = k_rot[0, :, 0] @ k_rot[0, :, 0].T
    g1 = k_rot[1, :, 0] @ k_rot[1, :, 0].T
    np.testing.assert_allclose(g1, g0, rtol=0, atol=1e-9)
    # and it is a rotation: norms are kept
    x = decode(c.k_new[0, :, 0], "bf16")
    np.testing.assert_allclose(np.linalg.norm(k_rot[0, :, 0], axis=1), np.linalg.norm(x, axis=1),
                               rtol=1e-12)
    # but not the identity: the positions do turn the vectors
    assert np.abs(k_rot[0, :, 0] - x).max() > 0.1


# ---------------------------------------------------------------- attention


def visible_slots(P, S, j):
    return list(range(P)) + [S + i for i in range(j + 1)]


def test_equal_keys_give_the_mean_of_the_visible_values(oracle_mod):
    B, L, Hq, Hkv, D, S_cap = 3, 5, 4, 2, 16, 96
    c = synth.attention_case(4, B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, S_cap=S_cap,
                             prefix_len=[0, 17, 40], src_off=[3, 60, 40], dtype="f16")
    one = c.k_new[0, 0, 0].copy()
    c.k_cache[:] = one
    c.k_new[:] = one
    # values in the stale gap and the unused tail are huge: any leak shows
    vals = decode(c.v_cache, "f16")
    for b in range(B):
        P, S = int(c.prefix_len[b]), int(c.src_off[b])
        vals[b, :, P:S] = 1000.0
        vals[b, :, S + L:] = -1000.0
    c.v_cache = synth.to_f16_bits(vals.astype(np.float32))
    out, _, st, kc, vc = run(oracle_mod, c, 0, 10000.0)
    assert st == 0
    V = decode(vc, "f16")
    for b in range(B):
        P, S = int(c.prefix_len[b]), int(c.src_off[b])
        for j in range(L):
            for hq in range(Hq):
                want = V[b, hq // (Hq // Hkv), visible_slots(P, S, j)].mean(axis=0)
                np.testing.assert_allclose(out[b, j, hq], want, rtol=1e-12, atol=1e-12)


def test_single_visible_key_returns_its_value(oracle_mod):
    c = synth.attention_case(5, B=2, L=3, Hq=2, Hkv=1, D=32, S_cap=40, prefix_len=[0, 0],
                             src_off=[0, 30], dtype="bf16")
    out, _, st, _, _ = run(oracle_mod, c, 32, 1e6)
    assert st == 0
    for b in range(2):
        for hq in range(2):
            assert np.array_equal(out[b, 0, hq], decode(c.v_new[b, 0, 0], "bf16"))


def sdpa_reference(q_rot, kc, vc, prefix_len, src_off, L, scale):
    """torch's scaled-dot-product attention over all S_cap slots with the mask
    written out slot by slot; query heads map to KV heads in blocks of G."""
    B, _, Hq, D = q_rot.shape
    Hkv, S_cap = kc.shape[1], kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, L, Hq, D))
    for b in range(B):
        P, S = int(prefix_len[b]), int(src_off[b])
        mask = np.zeros((L, S_cap), dtype=bool)
        for j in range(L):
            mask[j, visible_slots(P, S, j)] = True
        q = torch.from_numpy(q_rot[b].transpose(1, 0, 2).copy())            # [Hq][L][D]
        k = torch.from_numpy(kc[b]).repeat_interleave(G, dim=0)             # [Hq][S_cap][D]
        v = torch.from_numpy(vc[b]).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=torch.from_numpy(mask), scale=scale)
        out[b] = o.numpy().transpose(1, 0, 2)
    return out


@pytest.mark.parametrize("dtype,rotary_dim", [("f16", 0), ("bf16", 0), ("f16", 32),
                                              ("bf16", 24)])
def test_matches_torch_sdpa(oracle_mod, dtype, rotary_dim):
    B, L, Hq, Hkv, D, S_cap = 3, 7, 6, 2, 32, 160
    c = synth.attention_case(6, B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, S_cap=S_cap,
                             prefix_len=[0, 45, 120], src_off=[9, 130, 120], dtype=dtype)
    scale = 0.3
    out, _, st, kc, vc = run(oracle_mod, c, rotary_dim, 1e4, scale)
    assert st == 0
    # the queries rotated as the oracle rotates keys at the same positions: pass q as
    # the block's keys of a call with one KV head per query head, and read the rounded
    # rotated vectors back from the slots that call writes
    qc = synth.attention_case(0, B=B, L=L, Hq=Hq, Hkv=Hq, D=D, S_cap=S_cap,
                              prefix_len=c.prefix_len, src_off=c.src_off, dtype=dtype)
    qc.k_new = c.q.copy()
    _, _, st2, qkc, _ = run(oracle_mod, qc, rotary_dim, 1e4, scale)
    assert st2 == 0
    q_rot = np.stack([qkc[b, :, int(c.src_off[b]):int(c.src_off[b]) + L].transpose(1, 0, 2)
                      for b in range(B)])
    ref = sdpa_reference(decode(q_rot, dtype), decode(kc, dtype), decode(vc, dtype),
                         c.prefix_len, c.src_off, L, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_stale_gap_and_unused_slots_never_matter(oracle_mod):
    B, L, S_cap = 3, 8, 300
    c = synth.attention_case(7, B=B, L=L, Hq=4, Hkv=2, D=64, S_cap=S_cap,
                             prefix_len=[10, 150, 200], src_off=[250, 250, 200], dtype="bf16")
    out, _, _, kc, vc = run(oracle_mod, c, 64, 1e6)
    r = np.random.default_rng(8)
    for b in range(B):
        P, S = int(c.prefix_len[b]), int(c.src_off[b])
        for t in list(range(P, S)) + list(range(S, S_cap)):   # gap, block slots, tail
            c.k_cache[b, :, t] = r.integers(0, 2 ** 16, size=c.k_cache[b, :, t].shape)
            c.v_cache[b, :, t] = r.integers(0, 2 ** 16, size=c.v_cache[b, :, t].shape)
    out2, _, _, kc2, vc2 = run(oracle_mod, c, 64, 1e6)
    assert np.array_equal(out, out2)
    for b in range(B):
        S = int(c.src_off[b])
        assert np.array_equal(kc[b, :, S:S + L], kc2[b, :, S:S + L])
        assert np.array_equal(vc[b, :, S:S + L], vc2[b, :, S:S + L])


def test_block_is_causal(oracle_mod):
    L, j0 = 9, 3
    c = synth.attention_case(9, B=2, L=L, Hq=4, Hkv=4, D=32, S_cap=128, prefix_len=[20, 64],
                             dtype="f16")
    out, _, _, _, _ = run(oracle_mod, c, 32, 1e4)
    r = np.random.default_rng(10)
    for a in (c.q, c.k_new, c.v_new):
        a[:, j0 + 1:] = synth.to_f16_bits(r.standard_normal(a[:, j0 + 1:].shape)
                                          .astype(np.float32))
    out2, _, _, _, _ = run(oracle_mod, c, 32, 1e4)
    assert np.array_equal(out[:, :j0 + 1], out2[:, :j0 + 1])
    assert not np.array_equal(out[:, j0 + 1:], out2[:, j0 + 1:])


def test_cache_writes_and_rows_out_of_range(oracle_mod):
    B, L, S_cap = 5, 4, 64
    # rows 1, 2 and 3 are out of range: block before the prefix, block past the
    # end, negative prefix
    c = synth.attention_case(11, B=B, L=L, Hq=2, Hkv=1, D=16, S_cap=S_cap,
                             prefix_len=[10, 30, 5, -1, 60], src_off=[30, 20, 61, 0, 60],
                             dtype="bf16")
    out, k_rot, st, kc, vc = run(oracle_mod, c, 16, 1e4)
    assert st == 1
    for b in (1, 2, 3):
        assert np.array_equal(kc[b], c.k_cache[b]) and np.array_equal(vc[b], c.v_cache[b])
        assert not out[b].any()
    for b in (0, 4):
        S = int(c.src_off[b])
        keep = np.ones(S_cap, dtype=bool)
        keep[S:S + L] = False
        assert np.array_equal(kc[b][:, keep], c.k_cache[b][:, keep])
        assert np.array_equal(vc[b][:, keep], c.v_cache[b][:, keep])
        assert np.array_equal(vc[b, 0, S:S + L], c.v_new[b, :, 0])
        want = np.array([[oracle_mod.round_bits(v, BF16) for v in row] for row in k_rot[b, :, 0]],
                        dtype=np.uint16)
        assert np.array_equal(kc[b, 0, S:S + L], want)
        assert np.isfinite(out[b]).all() and np.abs(out[b]).max() > 0
