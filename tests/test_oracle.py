"""Pins for the CPU oracle, checked against things other than itself.

Each test fixes one part of the oracle with something the pages or the
mathematics determine independently: a hand-worked example, closed forms,
library routines for the number formats, invariants of a linear map, and
hand-built accept / arg max / compaction cases. A plausible mistake (nibble
order, group index, dropped bias term, sign, transposed operand, off-by-one in
the walk, overlap in the compaction) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    return synth.to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ---------------------------------------------------------------- number formats


def test_bf16_decoder_matches_torch_on_every_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_to_double(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_decoder_matches_numpy_on_every_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_double(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- projection


def _hand_case():
    with open(os.path.join(GOLDEN, "w4_hand_case.json")) as f:
        g = json.load(f)
    K, N, M = g["K"], g["N"], g["M"]
    qw = np.array([[int(h, 16) for h in row] for row in g["qw_hex"]], dtype=np.uint32)
    x = np.zeros((M, K), dtype=np.float32)
    for m, spec in g["x_rows"].items():
        m = int(m)
        if "ones" in spec:
            a, b = spec["ones"]
            x[m, a:b] = 1.0
        for k, v in spec.get("points", []):
            x[m, k] = v
    return g, qw, bf16(g["scales"]), bf16(g["biases"]), x


def test_hand_worked_example(oracle_mod):
    g, qw, s, b, x = _hand_case()
    y = oracle_mod.vq_linear(synth.to_bf16_bits(x), qw, s, b, act_dtype=oracle_mod.BF16)
    assert np.array_equal(y, np.array(g["expected_y"]))


def test_nibble_order_one_hot(oracle_mod):
    # word 0x76543210 holds codes 0..7 in k order, 0xfedcba98 codes 8..15
    K, N = 64, 1
    qw = np.zeros((N, K // 8), dtype=np.uint32)
    qw[0, 0], qw[0, 1] = 0x76543210, 0xFEDCBA98
    s, b = bf16([[0.5]]), bf16([[0.25]])
    x = np.eye(K, dtype=np.float32)             # x = e_k for row m = k
    y = oracle_mod.vq_linear(x, qw, s, b)
    expect = [0.5 * c + 0.25 for c in range(16)] + [0.25] * (K - 16)
    assert np.array_equal(y[:, 0], np.array(expect))


def test_group_index_at_boundaries(oracle_mod):
    K, N = 192, 2
    qw = np.full((N, K // 8), 0x55555555, dtype=np.uint32)      # every code 5
    s = bf16([[1.0, 2.0, 4.0], [0.5, 0.25, 0.125]])
    b = bf16([[0.5, -1.0, 8.0], [0.0, 1.0, -2.0]])
    ks = [0, 63, 64, 127, 128, 191]
    x = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = oracle_mod.vq_linear(x, qw, s, b)
    row0 = {0: 5.5, 1: 9.0, 2: 28.0}
    row1 = {0: 2.5, 1: 2.25, 2: -1.375}
    for i, k in enumerate(ks):
        assert y[i, 0] == row0[k // 64]
        assert y[i, 1] == row1[k // 64]


def test_zero_codes_closed_form(oracle_mod):
    # all codes 0: y[m][n] = sum_g bias[n][g] * (sum of x[m][k] over group g)
    M, K, N = 5, 320, 24
    w = synth.w4_weights(3, N, K)
    x = synth.activations(3, M, K, "f32")
    qw = np.zeros_like(w.qw)
    y = oracle_mod.vq_linear(x, qw, w.scales, w.biases)
    bias = torch.from_numpy(w.biases.view(np.int16)).view(torch.bfloat16).double().numpy()
    xs = x.astype(np.float64).reshape(M, K // 64, 64).sum(-1)
    expect = xs @ bias.T
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_constant_code_closed_form(oracle_mod):
    K, N = 5120, 4
    for c in (0, 7, 15):
        qw = np.full((N, K // 8), int("%x" % c * 8, 16), dtype=np.uint32)
        s = bf16(np.full((N, K // 64), 0.0078125))
        b = bf16(np.full((N, K // 64), -0.046875))
        x = np.ones((2, K), dtype=np.float32)
        y = oracle_mod.vq_linear(x, qw, s, b)
        assert np.all(y == K * (0.0078125 * c - 0.046875))


def _codes_by_hex(qw):
    """Codes read from each word's hex digits, least significant digit first."""
    N, W = qw.shape
    out = np.zeros((N, W * 8), dtype=np.float64)
    for n in range(N):
        for j in range(W):
            digits = format(int(qw[n, j]), "08x")[::-1]
            for i, d in enumerate(digits):
                out[n, 8 * j + i] = int(d, 16)
    return out


def test_unit_scale_zero_bias_is_a_plain_matmul(oracle_mod):
    M, K, N = 3, 128, 17
    w = synth.w4_weights(5, N, K)
    s = bf16(np.ones((N, K // 64)))
    b = bf16(np.zeros((N, K // 64)))
    x = synth.activations(5, M, K, "f32")
    y = oracle_mod.vq_linear(x, w.qw, s, b)
    expect = x.astype(np.float64) @ _codes_by_hex(w.qw).T
    assert np.allclose(y, expect, rtol=1e-13, atol=1e-12)


def test_scale_and_bias_terms_superpose(oracle_mod):
    # y(codes, s, b) = y(codes, s, 0) + y(0, *, b): the bias term is additive
    M, K, N = 4, 256, 9
    w = synth.w4_weights(6, N, K)
    x = synth.activations(6, M, K, "f32")
    zeros = bf16(np.zeros((N, K // 64)))
    full = oracle_mod.vq_linear(x, w.qw, w.scales, w.biases)
    scale_part = oracle_mod.vq_linear(x, w.qw, w.scales, zeros)
    bias_part = oracle_mod.vq_linear(x, np.zeros_like(w.qw), w.scales, w.biases)
    assert np.allclose(full, scale_part + bias_part, rtol=1e-12, atol=1e-11)
    # and doubling every scale doubles the scale part exactly
    s2 = bf16(2.0 * torch.from_numpy(w.scales.view(np.int16)).view(torch.bfloat16).float().numpy())
    assert np.array_equal(oracle_mod.vq_linear(x, w.qw, s2, zeros), 2.0 * scale_part)


def test_rows_are_independent_and_permute(oracle_mod):
    M, K, N = 8, 512, 40
    w = synth.w4_weights(7, N, K)
    x = synth.activations(7, M, K, "bf16")
    y = oracle_mod.vq_linear(x, w.qw, w.scales, w.biases, act_dtype=oracle_mod.BF16)
    for m in range(M):
        y1 = oracle_mod.vq_linear(x[m:m + 1], w.qw, w.scales, w.biases, act_dtype=oracle_mod.BF16)
        assert np.array_equal(y1[0], y[m])
    perm = np.random.default_rng(0).permutation(M)
    yp = oracle_mod.vq_linear(x[perm], w.qw, w.scales, w.biases, act_dtype=oracle_mod.BF16)
    assert np.array_equal(yp, y[perm])


def test_column_subset_matches_full(oracle_mod):
    M, K, N = 4, 256, 50
    w = synth.w4_weights(8, N, K)
    x = synth.activations(8, M, K, "bf16")
    full = oracle_mod.vq_linear(x, w.qw, w.scales, w.biases, act_dtype=oracle_mod.BF16)
    cols = np.array([49, 0, 17, 17, 3], dtype=np.int32)
    sub = oracle_mod.vq_linear(x, w.qw, w.scales, w.biases, act_dtype=oracle_mod.BF16, cols=cols)
    assert np.array_equal(sub, full[:, cols])


def test_activation_dtypes_agree_on_common_values(oracle_mod):
    # values exactly representable in bf16, f16 and f32 give identical y
    M, K, N = 2, 128, 6
    w = synth.w4_weights(9, N, K)
    r = np.random.default_rng(9)
    x = (r.integers(-64, 64, size=(M, K)) / 16.0).astype(np.float32)
    y32 = oracle_mod.vq_linear(x, w.qw, w.scales, w.biases)
    yb = oracle_mod.vq_linear(synth.to_bf16_bits(x), w.qw, w.scales, w.biases,
                              act_dtype=oracle_mod.BF16)
    yh = oracle_mod.vq_linear(synth.to_f16_bits(x), w.qw, w.scales, w.biases,
                              act_dtype=oracle_mod.F16)
    assert np.array_equal(y32, yb) and np.array_equal(y32, yh)


def test_linear_in_x(oracle_mod):
    M, K, N = 3, 192, 11
    w = synth.w4_weights(10, N, K)
    a = (np.random.default_rng(1).integers(-8, 8, size=(M, K)) / 4.0).astype(np.float32)
    c = (np.random.default_rng(2).integers(-8, 8, size=(M, K)) / 4.0).astype(np.float32)
    ya = oracle_mod.vq_linear(a, w.qw, w.scales, w.biases)
    yc = oracle_mod.vq_linear(c, w.qw, w.scales, w.biases)
    yac = oracle_mod.vq_linear(a + c, w.qw, w.scales, w.biases)
    assert np.allclose(yac, ya + yc, rtol=1e-12, atol=1e-10)


def test_rejects_bad_shapes(oracle_mod):
    w = synth.w4_weights(0, 4, 64)
    with pytest.raises(ValueError):
        oracle_mod.vq_linear(np.ones((1, 64), np.float32), w.qw, w.scales, w.biases,
                             cols=np.array([4], dtype=np.int32))


# ---------------------------------------------------------------- arg max


def test_argmax_hand_cases(oracle_mod):
    inf, nan = math.inf, math.nan
    rows = [
        [2.0, 2.0, 2.0, 2.0],              # all equal -> 0
        [1.0, 5.0, 3.0, 5.0],              # duplicated max -> lower index 1
        [0.0, -1.0, 2.0, 9.5],             # max at the last index
        [-inf, -inf, -3.0, -inf],          # -inf entries
        [-inf, -inf, -inf, -inf],          # all -inf -> 0
        [nan, 1.0, nan, 0.5],              # NaN never wins
        [nan, nan, nan, nan],              # all NaN -> 0
        [1.0, 0.0, 1.0 + 1e-12, 0.0],      # equal once rounded to fp32 -> 0
        [1.0, 0.0, 1.0 + 2 ** -23, 0.0],   # one fp32 ulp apart -> 2
    ]
    idx, mx, sec = oracle_mod.argmax(np.array(rows))
    assert idx.tolist() == [0, 1, 3, 2, 0, 1, 0, 0, 2]
    assert mx[1] == 5.0 and mx[3] == -3.0 and np.isnan(mx[6])
    # runner-up: the largest value at any other index, NaN skipped, -inf if none;
    # a tie for the maximum makes it equal to the maximum
    assert sec.tolist() == [2.0, 5.0, 2.0, -inf, -inf, 0.5, -inf, 1.0, 1.0]
    _, _, one = oracle_mod.argmax(np.array([[3.0], [nan]]))
    assert one.tolist() == [-inf, -inf]


def test_argmax_runner_up_matches_sorting(oracle_mod):
    # against numpy: the runner-up is the second entry of the descending sort
    # of the row's non-NaN fp32 values (duplicates kept)
    r = np.random.default_rng(5)
    rows = r.integers(-4, 5, size=(200, 7)).astype(np.float64) * 0.5
    rows[r.random(rows.shape) < 0.1] = np.nan
    idx, mx, sec = oracle_mod.argmax(rows)
    for m in range(rows.shape[0]):
        v = rows[m][~np.isnan(rows[m])].astype(np.float32)
        if v.size == 0:
            assert idx[m] == 0 and np.isnan(mx[m]) and sec[m] == -np.inf
            continue
        s = np.sort(v)[::-1]
        assert mx[m] == s[0] and rows[m][idx[m]] == s[0]
        assert sec[m] == (s[1] if s.size > 1 else -np.inf)


# ---------------------------------------------------------------- accept walk


def test_fold_accept_hand_cases(oracle_mod):
    # rows: [committed, d1, d2, d3] against target [t0, t1, t2, t3] (t_j follows position j)
    tokens = np.array([[7, 10, 11, 99],      # d1 = t0, d2 = t1, d3 != t2 -> accept 2, bonus t2
                       [7, 10, 11, 12],      # every draft accepted -> accept 3, bonus t3
                       [7, 55, 11, 12],      # first draft misses -> accept 0, bonus t0
                       [7, 10, 11, 12]])     # same drafts, other targets (below)
    target = np.array([[10, 11, 12, 13],
                       [10, 11, 12, 13],
                       [10, 11, 12, 13],
                       [10, 77, 12, 13]])    # t1 differs -> accept 1, bonus 77
    acc, bonus, keep = oracle_mod.fold_accept(tokens, target)
    assert acc.tolist() == [2, 3, 0, 1]
    assert bonus.tolist() == [12, 13, 10, 77]
    assert keep.tolist() == [3, 4, 1, 2]
    # a block of one token: nothing to accept, the bonus is the target of row 0
    acc, bonus, keep = oracle_mod.fold_accept(np.array([[5]]), np.array([[9]]))
    assert acc.tolist() == [0] and bonus.tolist() == [9] and keep.tolist() == [1]



def test_accept_walk_hand_cases(oracle_mod):
    big = 2 ** 31 - 1
    tgt = np.array([
        [5, 6, 7, 8, 9, 10, 11, 12],       # full accept -> 8
        [5, 6, 7, 8, 9, 10, 11, 12],       # first-token miss -> 0
        [5, 6, 7, 8, 9, 10, 11, 12],       # partial 3, later positions match again
        [big, -1, 0, 0, 0, 0, 0, 0],       # large and negative ids -> 2
    ], dtype=np.int32)
    dft = tgt.copy()
    dft[1, 0] = 4
    dft[2, 3] = 0
    dft[3, 2] = 1
    assert oracle_mod.accept_walk(dft, tgt).tolist() == [8, 0, 3, 2]
    one = np.array([[3], [4]], dtype=np.int32)
    assert oracle_mod.accept_walk(one, np.array([[3], [5]], dtype=np.int32)).tolist() == [1, 0]


# ---------------------------------------------------------------- KV compaction


def _encoded_cache(n_tensors, B, H, S, D):
    """fp16 slots whose bits name (tensor, b, h, slot, d): checkable in closed form."""
    t, b, h, s, d = np.meshgrid(np.arange(n_tensors), np.arange(B), np.arange(H),
                                np.arange(S), np.arange(D), indexing="ij")
    code = ((t * 7 + b * 5 + h * 3) * 4099 + s * 13 + d) % 65536
    return [code[i].astype(np.uint16).view(np.float16).copy() for i in range(n_tensors)]


def _expected_after(before, prefix, src, keep):
    out = [a.copy() for a in before]
    for a, b0 in zip(out, before):
        for b in range(a.shape[0]):
            p, s, c = prefix[b], src[b], keep[b]
            a[b, :, p:p + c, :] = b0[b, :, s:s + c, :]
    return out


def test_kv_compact_closed_form(oracle_mod):
    n_t, B, H, S, D = 4, 6, 3, 64, 8
    prefix = np.array([10, 40, 30, 0, 20, 50], dtype=np.int32)
    src = np.array([44, 44, 34, 44, 20, 50], dtype=np.int32)
    keep = np.array([16, 3, 16, 0, 16, 9], dtype=np.int32)
    # rows: far move, short move, overlapping (S - p = 4 < keep = 16), keep 0,
    # no-op (prefix == src), and a move at the very end of the cache
    before = _encoded_cache(n_t, B, H, S, D)
    cache = [a.copy() for a in before]
    new_len, status = oracle_mod.kv_compact(cache, prefix, src, keep, max_keep=16)
    assert status == 0
    assert new_len.tolist() == (prefix + keep).tolist()
    for got, exp in zip(cache, _expected_after(before, prefix, src, keep)):
        assert np.array_equal(got.view(np.uint16), exp.view(np.uint16))


def test_kv_compact_out_of_range_rows_are_skipped(oracle_mod):
    n_t, B, H, S, D = 2, 4, 2, 32, 4
    before = _encoded_cache(n_t, B, H, S, D)
    cache = [a.copy() for a in before]
    prefix = np.array([4, 30, 2, 1], dtype=np.int32)
    src = np.array([20, 20, 28, 5], dtype=np.int32)
    keep = np.array([4, 4, 8, 17], dtype=np.int32)     # row 1: p+keep > S; row 2: src+keep > S; row 3: keep > max
    new_len, status = oracle_mod.kv_compact(cache, prefix, src, keep, max_keep=16)
    assert status & 1
    assert new_len.tolist() == [8, -1, -1, -1]
    exp = _expected_after(before, prefix[:1].tolist() + [0] * 3, src[:1].tolist() + [0] * 3,
                          keep[:1].tolist() + [0] * 3)
    for got, e in zip(cache, exp):
        assert np.array_equal(got.view(np.uint16), e.view(np.uint16))
