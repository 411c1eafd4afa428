"""GPU parity: the CUDA library, called through its C ABI, against the oracle.

Projections must meet the tolerance in parity.py; arg max indices, accept
lengths and compacted KV must match bit for bit. Every projection, the
full-size workloads included, is compared with the oracle element by element
over its whole output (the oracle takes well under a second for the largest
of them); small shapes span several 128-row units, several 512-wide stages and
ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import (Guarded, ORACLE_DT, TOL, assert_proj_close, out_to_f64, proj_error, to_dev_act,
                    to_dev_weights)
from speculative_block_draft_02_gb300 import binding as vq
from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_block_draft_02_gb300 import build

    build.build()
    vq.lib()
    oracle.build()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0


def _workspace(M, K, N, dtype):
    nb = vq.vq_linear_workspace_bytes(M, K, N, parity_torch(dtype))
    return torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None


def parity_torch(dtype):
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]


def run_linear(x_bits, w, dtype, ws=None):
    x = to_dev_act(x_bits, dtype)
    qw, s, b = to_dev_weights(w)
    M, K = x.shape
    if ws is None:
        ws = _workspace(M, K, w.N, dtype)
    y = Guarded((M, w.N), x.dtype, fill=float("nan"))
    vq.vq_linear(x, qw, s, b, y=y.t, workspace=ws)
    y.check()
    return out_to_f64(y.t)


def oracle_linear(x_bits, w, dtype, cols=None):
    return oracle.vq_linear(x_bits, w.qw, w.scales, w.biases, act_dtype=ORACLE_DT[dtype],
                            cols=cols)


# ------------------------------------------------------------------ projection


def test_linear_tiny_workload():
    # M=8 bf16 ~N(0,1), K=512, N=1024, seed 0
    w = synth.w4_weights(0, 1024, 512)
    x = synth.activations(0, 8, 512, "bf16")
    assert_proj_close(run_linear(x, w, "bf16"), oracle_linear(x, w, "bf16"), "bf16")


RAGGED = [
    (1, 512, 1, "bf16"), (3, 512, 129, "bf16"), (8, 1024, 1000, "bf16"), (5, 512, 257, "f16"),
    (12, 1024, 300, "bf16"), (16, 512, 384, "f16"), (24, 512, 200, "bf16"),
    (33, 1024, 130, "bf16"), (64, 512, 1024, "bf16"), (64, 1536, 260, "f16"),
    (1, 512, 77, "f32"), (7, 1024, 500, "f32"), (16, 512, 256, "f32"), (32, 512, 129, "f32"),
    (8, 2048, 4100, "bf16"), (2, 512, 128 * 160 + 3, "bf16"),
]


@pytest.mark.parametrize("M,K,N,dtype", RAGGED)
def test_linear_ragged_shapes(M, K, N, dtype):
    seed = M * 131 + N
    w = synth.w4_weights(seed, N, K)
    x = synth.activations(seed, M, K, dtype)
    assert_proj_close(run_linear(x, w, dtype), oracle_linear(x, w, dtype), dtype)


# wide N with M <= 8: several row blocks per block, so x is converted once
# into a per-block fp16 table (the x-table variant)
@pytest.mark.parametrize("M,K,N,dtype", [(8, 1024, 60000, "bf16"), (5, 512, 70001, "f16"),
                                         (1, 2048, 58500, "bf16")])
def test_linear_wide_n_x_table(M, K, N, dtype):
    w = synth.w4_weights(M + K, N, K)
    x = synth.activations(M + K, M, K, dtype)
    assert_proj_close(run_linear(x, w, dtype), oracle_linear(x, w, dtype), dtype)


# 16-bit x with M > 16 and an N wide enough that K is not split: the
# tensor-core (tcgen05) kernel, M padded to 32 / 64 rows
TC_SHAPES = [(17, 512, 12345, "bf16"), (24, 1024, 10000, "f16"), (32, 1024, 9800, "f16"),
             (33, 512, 9729, "bf16"), (40, 512, 9999, "bf16"), (64, 1024, 10001, "bf16"),
             (64, 512, 9730, "f16")]


@pytest.mark.parametrize("M,K,N,dtype", TC_SHAPES)
def test_linear_tensor_core_path(M, K, N, dtype):
    seed = 7 * M + K + N
    w = synth.w4_weights(seed, N, K)
    x = synth.activations(seed, M, K, dtype)
    assert_proj_close(run_linear(x, w, dtype), oracle_linear(x, w, dtype), dtype)


# long K on the tcgen05 kernel: the group row sums are taken per stage from
# the x tile (a table for all of K would not fit beside two stages)
@pytest.mark.parametrize("M,K,N,dtype", [(64, 8192, 9800, "bf16"), (40, 17408, 9728, "f16")])
def test_linear_tensor_core_long_k(M, K, N, dtype):
    seed = 11 * M + K
    w = synth.w4_weights(seed, N, K)
    x = synth.activations(seed, M, K, dtype)
    assert_proj_close(run_linear(x, w, dtype), oracle_linear(x, w, dtype), dtype)


def test_vocab_argmax_tensor_core_long_k():
    M, K, N = 64, 8192, 12000
    w = synth.w4_weights(77, N, K)
    x = synth.activations(77, M, K, "bf16")
    idx, mx, ws = run_vocab(x, w)
    check_argmax(idx, mx, oracle_linear(x, w, "bf16"))
    assert not ws.any()


@pytest.mark.parametrize("M,K,N,dtype", [(17, 512, 3000, "bf16"), (20, 1024, 9000, "f16"),
                                         (64, 1024, 40000, "f16")])
def test_vocab_argmax_tensor_core_path(M, K, N, dtype):
    w = synth.w4_weights(M * 3 + N, N, K)
    x = synth.activations(M * 3 + N, M, K, dtype)
    idx, mx, ws = run_vocab(x, w, dtype)
    check_argmax(idx, mx, oracle_linear(x, w, dtype))
    assert not ws.any(), "workspace must be left zeroed"


def test_linear_x_table_handles_large_and_tiny_rows():
    # the per-row fp16 scaling keeps rows of very different magnitude exact
    M, K, N = 4, 1024, 60000
    w = synth.w4_weights(44, N, K)
    base = np.random.default_rng(44).standard_normal((M, K)).astype(np.float32)
    base[0] *= 3.0e4      # beyond fp16 range once multiplied by codes
    base[1] *= 1.0e-6     # deep below fp16's normal range
    base[2, ::7] = 0.0
    x = synth.to_bf16_bits(base)
    y = run_linear(x, w, "bf16")
    r = oracle_linear(x, w, "bf16")
    for m in range(M):
        assert_proj_close(y[m:m + 1], r[m:m + 1], "bf16")


@pytest.mark.parametrize("M,K,N", [(8, 5120, 1024), (4, 4096, 256), (16, 2560, 640)])
def test_linear_split_k_is_exact_and_repeatable(M, K, N):
    w = synth.w4_weights(11, N, K)
    x = synth.activations(11, M, K, "bf16")
    ws = _workspace(M, K, N, "bf16")
    assert ws is not None, "narrow N is expected to split K"
    y1 = run_linear(x, w, "bf16", ws)
    y2 = run_linear(x, w, "bf16", ws)        # the workspace must come back zeroed
    assert np.array_equal(y1, y2)
    assert_proj_close(y1, oracle_linear(x, w, "bf16"), "bf16")


@pytest.mark.parametrize("N", [17408, 1024])
def test_linear_paper_shape_full(N):
    # M=8, K=5120, N=17408 and N=1024, bf16 ~N(0,1): the headline verify
    # projection and its narrow-output case, every output element
    w = synth.w4_weights(0, N, 5120)
    x = synth.activations(0, 8, 5120, "bf16")
    assert_proj_close(run_linear(x, w, "bf16"), oracle_linear(x, w, "bf16"), "bf16")


@pytest.fixture(scope="module")
def sweep_weights():
    return synth.w4_weights(0, 17408, 5120)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_linear_block_size_and_dtype_sweep(sweep_weights, M, dtype):
    x = synth.activations(0, M, 5120, dtype, scale=0.5)
    y = run_linear(x, sweep_weights, dtype)
    assert_proj_close(y, oracle_linear(x, sweep_weights, dtype), dtype)


def test_rows_are_independent_and_permute():
    # a row's result does not depend on the other rows of the block: M=1 and
    # the M=8 block agree bit for bit (same code path), the M=16 block agrees
    # within the tolerance (its rows take the general path), and permuting the
    # rows permutes the output
    w = synth.w4_weights(21, 700, 1024)
    x16 = synth.activations(21, 16, 1024, "bf16")
    y16 = run_linear(x16, w, "bf16")
    y8 = run_linear(x16[:8].copy(), w, "bf16")
    y1 = run_linear(x16[5:6].copy(), w, "bf16")
    assert np.array_equal(y8[5], y1[0])
    r8 = oracle_linear(x16[:8].copy(), w, "bf16")
    assert_proj_close(y8, r8, "bf16")
    assert_proj_close(y16[:8], r8, "bf16")
    for M, xs, ys in ((16, x16, y16), (8, x16[:8].copy(), y8)):
        perm = np.random.default_rng(M).permutation(M)
        yp = run_linear(xs[perm].copy(), w, "bf16")
        assert np.array_equal(yp, ys[perm])


def test_linear_paper_shape_is_deterministic():
    w = synth.w4_weights(0, 17408, 5120)
    x = synth.activations(0, 8, 5120, "bf16")
    ys = [run_linear(x, w, "bf16") for _ in range(3)]
    assert all(np.array_equal(ys[0], y) for y in ys[1:])


# ------------------------------------------------------------------ arg max


def run_vocab(x_bits, w, dtype="bf16"):
    x = to_dev_act(x_bits, dtype)
    qw, s, b = to_dev_weights(w)
    M = x.shape[0]
    ws = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    gi, gm = Guarded((M,), torch.int32, fill=-1), Guarded((M,), torch.float32, fill=float("nan"))
    idx, mx = vq.vq_vocab_argmax(x, qw, s, b, ws, argmax=gi.t, maxval=gm.t)
    gi.check()
    gm.check()
    return idx.cpu().numpy(), mx.cpu().numpy(), ws


def check_argmax(idx, mx, logits):
    """Bit-exact indices, except rows whose fp32 top two are within the
    accumulation error of each other: there either index is correct, and
    the GPU's pick must be one of the near-tied maxima."""
    r_idx, r_max, r_sec = oracle.argmax(logits)
    near = 0
    for m in range(len(idx)):
        margin = 1e-4 * max(1.0, abs(float(r_max[m])))
        if float(r_max[m]) - float(r_sec[m]) < margin:
            near += 1
            assert float(logits[m, idx[m]]) >= float(r_max[m]) - margin
        else:
            assert idx[m] == r_idx[m], (m, idx[m], r_idx[m])
        assert abs(float(mx[m]) - float(logits[m, idx[m]])) <= 1e-5 * max(1.0, abs(float(mx[m])))
    return near


def test_vocab_argmax_tiny_workload():
    w = synth.w4_weights(0, 1024, 512)
    x = synth.activations(0, 8, 512, "bf16")
    idx, mx, ws = run_vocab(x, w)
    assert check_argmax(idx, mx, oracle_linear(x, w, "bf16")) == 0
    assert not ws.any(), "workspace must be left zeroed"


def test_vocab_argmax_exact_tie_takes_lowest_index():
    N, K, M = 3000, 1024, 8
    w = synth.w4_weights(31, N, K)
    x = synth.activations(31, M, K, "bf16")
    r_idx, _, _ = oracle.argmax(oracle_linear(x, w, "bf16"))
    # copy the winning row of output row 0 to an earlier index: an exact tie
    a = int(r_idx[0])
    lo = 3 if a > 3 else N - 1
    for arr in (w.qw, w.scales, w.biases):
        arr[lo] = arr[a]
    idx, _, _ = run_vocab(x, w)
    assert idx[0] == min(lo, a)


@pytest.mark.parametrize("M,K,N", [(3, 512, 1000), (16, 1024, 5000), (64, 512, 2049),
                                   (33, 1536, 777), (8, 512, 60000), (2, 1024, 77777)])
def test_vocab_argmax_ragged(M, K, N):
    w = synth.w4_weights(M + N, N, K)
    x = synth.activations(M + N, M, K, "bf16")
    idx, mx, _ = run_vocab(x, w)
    check_argmax(idx, mx, oracle_linear(x, w, "bf16"))


def run_vocab_top2(x_bits, w, dtype="bf16"):
    x = to_dev_act(x_bits, dtype)
    qw, s, b = to_dev_weights(w)
    M = x.shape[0]
    ws = torch.zeros(vq.vq_vocab_argmax_top2_workspace_bytes(M), dtype=torch.uint8,
                     device="cuda")
    gi, gm = Guarded((M,), torch.int32, fill=-1), Guarded((M,), torch.float32, fill=float("nan"))
    gs = Guarded((M,), torch.float32, fill=float("nan"))
    idx, mx, sec = vq.vq_vocab_argmax_top2(x, qw, s, b, ws, argmax=gi.t, maxval=gm.t, second=gs.t)
    for g in (gi, gm, gs):
        g.check()
    return idx.cpu().numpy(), mx.cpu().numpy(), sec.cpu().numpy(), ws, M


def check_runner_up(idx, sec, logits):
    """The runner-up must be the largest fp32 logit at any index other than
    the one the kernel picked, within the fp32 accumulation error."""
    f = logits.astype(np.float32)
    for m in range(len(idx)):
        row = np.delete(f[m], idx[m])
        row = row[~np.isnan(row)]
        want = row.max() if row.size else -np.inf
        if np.isinf(want):
            assert sec[m] == want
        else:
            assert abs(float(sec[m]) - float(want)) <= 1e-5 * max(1.0, abs(float(want))), (m, sec[m], want)


# every arg max kernel: x table (M <= 8, wide N), per-stage x (M <= 16, fp32 x),
# tcgen05 (16-bit x, M > 16)
@pytest.mark.parametrize("M,K,N,dtype", [(8, 512, 60000, "bf16"), (3, 1024, 5000, "f16"),
                                         (12, 512, 3001, "bf16"), (7, 512, 2000, "f32"),
                                         (24, 1024, 9000, "bf16"), (64, 512, 20000, "f16")])
def test_vocab_argmax_top2(M, K, N, dtype):
    w = synth.w4_weights(M * 5 + N, N, K)
    x = synth.activations(M * 5 + N, M, K, dtype)
    idx, mx, sec, ws, _ = run_vocab_top2(x, w, dtype)
    logits = oracle_linear(x, w, dtype)
    check_argmax(idx, mx, logits)
    check_runner_up(idx, sec, logits)
    assert np.all(sec <= mx)
    assert not ws[: vq.vq_vocab_argmax_workspace_bytes(M)].any(), "keys must be left zeroed"
    # the same arg max as the call without the runner-up
    idx2, mx2, _ = run_vocab(x, w, dtype)
    assert np.array_equal(idx, idx2) and np.array_equal(mx, mx2)


def test_vocab_argmax_top2_exact_tie_and_single_column():
    N, K, M = 3000, 512, 20
    w = synth.w4_weights(37, N, K)
    x = synth.activations(37, M, K, "bf16")
    r_idx, _, _ = oracle.argmax(oracle_linear(x, w, "bf16"))
    a = int(r_idx[0])
    lo = 5 if a > 5 else N - 1
    for arr in (w.qw, w.scales, w.biases):
        arr[lo] = arr[a]
    idx, mx, sec, _, _ = run_vocab_top2(x, w)
    assert idx[0] == min(lo, a) and sec[0] == mx[0], "a tie for the maximum: margin 0"
    w1 = synth.w4_weights(38, 1, K)
    idx, mx, sec, _, _ = run_vocab_top2(synth.activations(38, 4, K, "bf16"), w1)
    assert np.all(idx == 0) and np.all(sec == -np.inf)


def test_vocab_argmax_full_workload_and_accept():
    # M=64 (B=4 x block 16), K=2560, N=151936 vocab; drafts match the target
    # with p=0.7 per position until the first miss
    cfg = synth.WORKLOADS["vocab_argmax_b4_l16_k2560_n151936"]
    w = synth.w4_weights(0, cfg["N"], cfg["K"])
    x = synth.activations(0, cfg["M"], cfg["K"], "bf16")
    idx, mx, _ = run_vocab(x, w)
    logits = oracle_linear(x, w, "bf16")
    # no row of this workload has its top two logits within the near-tie
    # margin (the smallest relative top-1/top-2 gap is 8.3e-4), so every index
    # must match bit for bit
    assert check_argmax(idx, mx, logits) == 0
    r_idx, _, _ = oracle.argmax(logits)
    target = r_idx.reshape(cfg["B"], cfg["L"])
    draft = synth.drafts_from_target(0, target, cfg["N"], cfg["p"])
    acc = vq.verify_accept_walk(torch.from_numpy(draft).cuda(),
                                torch.from_numpy(idx.reshape(cfg["B"], cfg["L"])).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), oracle.accept_walk(draft, target))


# ------------------------------------------------------------------ accept walk


@pytest.mark.parametrize("B,L", [(1, 8), (4, 16), (1, 1), (7, 40), (1000, 16), (3, 100)])
def test_accept_walk(B, L):
    r = np.random.default_rng(B * 1000 + L)
    target = r.integers(-5, 2 ** 31 - 1, size=(B, L), dtype=np.int64).astype(np.int32)
    draft = target.copy()
    for b in range(B):
        j = int(r.integers(0, L + 1))
        if j < L:
            draft[b, j] ^= 1 + int(r.integers(0, 1000))
            # positions after the miss may match again
            if j + 1 < L and r.random() < 0.5:
                draft[b, j + 1:] = target[b, j + 1:]
    acc = vq.verify_accept_walk(torch.from_numpy(draft).cuda(), torch.from_numpy(target).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), oracle.accept_walk(draft, target))


# ------------------------------------------------------------------ KV commit


def _kv_to_dev(tensors):
    return [torch.from_numpy(t.view(np.int16).copy()).cuda() for t in tensors]


def _run_compact(case, max_keep=16):
    src = _kv_to_dev(case.tensors)
    guarded = [Guarded(t.shape, t.dtype, fill=t) for t in src]
    dev = [g.t for g in guarded]
    del src
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    new_len = vq.kv_compact_per_row(dev, i32(case.prefix_len), i32(case.src_off), i32(case.keep),
                                    max_keep, status=status)
    for g in guarded:
        g.check()
    return dev, new_len.cpu().numpy(), int(status.item())


def test_kv_compact_full_workload():
    # 8 layers x {K,V} x [4][8][2048][128] fp16, prefix ~U{200..1800},
    # verify block at the shared offset max(prefix), keep ~U{0..16}
    case = synth.commit_case(0)
    dev, new_len, status = _run_compact(case)
    ref = [t.copy() for t in case.tensors]
    r_len, r_status = oracle.kv_compact(ref, case.prefix_len, case.src_off, case.keep, 16)
    assert status == r_status == 0
    assert np.array_equal(new_len, r_len)
    for d, r in zip(dev, ref):
        assert np.array_equal(d.cpu().numpy(), r.view(np.int16))


def test_kv_compact_edge_cases():
    # overlapping ranges, keep 0, no-op, move to the cache end, keep = max,
    # and rows whose ranges leave the cache (skipped, flagged)
    case = synth.commit_case(5, layers=2, B=8, H=3, S_cap=64, D=64, block=16, prefix_lo=0,
                             prefix_hi=40,
                             keep=[16, 0, 16, 5, 16, 3, 17, 16],
                             src_off=[44, 44, 20, 59, 48, 2, 40, 50])
    case.prefix_len[:] = [30, 10, 20, 10, 5, 62, 1, 0]
    dev, new_len, status = _run_compact(case)
    ref = [t.copy() for t in case.tensors]
    r_len, r_status = oracle.kv_compact(ref, case.prefix_len, case.src_off, case.keep, 16)
    assert status == r_status == 1
    assert np.array_equal(new_len, r_len)
    assert r_len.tolist() == [46, 10, 36, 15, 21, -1, -1, -1]
    for d, r in zip(dev, ref):
        assert np.array_equal(d.cpu().numpy(), r.view(np.int16))


def test_commit_then_next_block_verify():
    # the per-row commit followed by the next block's M=64 verify projection
    cfg = synth.WORKLOADS["commit_b4_l16_then_verify_m64"]
    case = synth.commit_case(0)
    dev, new_len, _ = _run_compact(case)
    assert np.array_equal(new_len, case.prefix_len + case.keep)
    w = synth.w4_weights(0, cfg["N"], cfg["K"])
    x = synth.activations(0, cfg["M"], cfg["K"], "bf16", name="x_next")
    assert_proj_close(run_linear(x, w, "bf16"), oracle_linear(x, w, "bf16"), "bf16")


# ------------------------------------------------------------ one verify round


@pytest.mark.parametrize("B,L,K,N,layers", [(4, 16, 512, 20000, 2), (1, 8, 512, 3000, 1),
                                            (8, 8, 1024, 12000, 0), (2, 1, 512, 5000, 1)])
def test_verify_round_fold_layout(B, L, K, N, layers):
    """vocab arg max -> fold accept -> KV commit in one call, against the
    oracle composed the same way: target = arg max of the oracle logits,
    (accept, bonus, keep) = fold accept, then the per-row commit with keep."""
    M = B * L
    w = synth.w4_weights(B * 100 + L, N, K)
    hx = synth.activations(B * 100 + L, M, K, "bf16", name="hidden")
    logits = oracle_linear(hx, w, "bf16")
    r_target, _, _ = oracle.argmax(logits)
    r_target = r_target.reshape(B, L)
    # committed token in column 0, then drafts against the targets of the rows before
    r = np.random.default_rng(B + L)
    tokens = np.empty((B, L), dtype=np.int32)
    tokens[:, 0] = r.integers(0, N, size=B)
    if L > 1:
        tokens[:, 1:] = synth.drafts_from_target(B + L, r_target[:, :-1], N)
    r_acc, r_bonus, r_keep = oracle.fold_accept(tokens, r_target)

    h = to_dev_act(hx, "bf16")
    qw, sc, bi = to_dev_weights(w)
    ws = torch.zeros(vq.verify_round_workspace_bytes(B, L), dtype=torch.uint8, device="cuda")
    tok = torch.from_numpy(tokens).cuda()
    if layers:
        case = synth.commit_case(B + L, layers=layers, B=B, H=2, S_cap=512, D=64, block=L,
                                 prefix_lo=20, prefix_hi=400, keep=r_keep)
        kv = _kv_to_dev(case.tensors)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        target, acc, bonus, new_len = vq.verify_round(
            h, qw, sc, bi, tok, ws, kv=kv, prefix_len=i32(case.prefix_len),
            src_off=i32(case.src_off), status=status)
    else:
        target, acc, bonus, new_len = vq.verify_round(h, qw, sc, bi, tok, ws)
    torch.cuda.synchronize()
    target = target.cpu().numpy()
    assert check_argmax(target.reshape(-1), np.zeros(M, np.float32) + logits.max(axis=1),
                        logits) == 0
    assert np.array_equal(target, r_target)
    assert np.array_equal(acc.cpu().numpy(), r_acc)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)
    assert not ws[: vq.vq_vocab_argmax_workspace_bytes(M)].any()
    if layers:
        ref = [t.copy() for t in case.tensors]
        r_len, r_status = oracle.kv_compact(ref, case.prefix_len, case.src_off, r_keep, L)
        assert int(status.item()) == r_status == 0
        assert np.array_equal(new_len.cpu().numpy(), r_len)
        for d, rr in zip(kv, ref):
            assert np.array_equal(d.cpu().numpy(), rr.view(np.int16))


def test_verify_round_commits_the_drafter_context_too():
    """Per-row drafter context: one round commits the target's attention cache
    and the drafter's context cache, each with its own layers, heads, head
    size, capacity, prefix lengths and block offset, both with keep = accept
    + 1 -- against the oracle composed the same way (fold accept, then the
    per-row commit of each set)."""
    B, L, K, N = 4, 16, 512, 20000
    M = B * L
    w = synth.w4_weights(404, N, K)
    hx = synth.activations(404, M, K, "bf16", name="hidden")
    logits = oracle_linear(hx, w, "bf16")
    r_target = oracle.argmax(logits)[0].reshape(B, L)
    r = np.random.default_rng(404)
    tokens = np.empty((B, L), dtype=np.int32)
    tokens[:, 0] = r.integers(0, N, size=B)
    tokens[:, 1:] = synth.drafts_from_target(404, r_target[:, :-1], N)
    r_acc, r_bonus, r_keep = oracle.fold_accept(tokens, r_target)
    # the target's cache: 2 layers x {K, V} of [4][2][512][64] fp16, verify
    # block at the shared offset max(prefix); the drafter's: 1 layer x {K, V}
    # of [4][4][1024][128], its own (shorter) prefixes, block right after the
    # longest of them, and one row whose block sits right after its prefix
    tgt = synth.commit_case(405, layers=2, B=B, H=2, S_cap=512, D=64, block=L, prefix_lo=20,
                            prefix_hi=400, keep=r_keep, name="target_kv")
    dft = synth.commit_case(406, layers=1, B=B, H=4, S_cap=1024, D=128, block=L, prefix_lo=5,
                            prefix_hi=300, keep=r_keep, name="drafter_kv")
    dft.src_off[2] = dft.prefix_len[2]
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    sets, devs = [], []
    for case in (tgt, dft):
        kv = _kv_to_dev(case.tensors)
        devs.append(kv)
        sets.append((kv, i32(case.prefix_len), i32(case.src_off)))
    ws = torch.zeros(vq.verify_round_workspace_bytes(B, L), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    target, acc, bonus, new_lens = vq.verify_round_multi(
        to_dev_act(hx, "bf16"), *to_dev_weights(w), torch.from_numpy(tokens).cuda(), ws,
        sets=sets, status=status)
    torch.cuda.synchronize()
    assert np.array_equal(target.cpu().numpy(), r_target)
    assert np.array_equal(acc.cpu().numpy(), r_acc)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)
    assert int(status.item()) == 0
    for case, kv, nl in zip((tgt, dft), devs, new_lens):
        ref = [t.copy() for t in case.tensors]
        r_len, r_status = oracle.kv_compact(ref, case.prefix_len, case.src_off, r_keep, L)
        assert r_status == 0
        assert np.array_equal(nl.cpu().numpy(), r_len)
        for d, rr in zip(kv, ref):
            assert np.array_equal(d.cpu().numpy(), rr.view(np.int16))


# K a multiple of 64 but not of 512: a last stage of 1..7 groups (zero-filled
# past K), scales and biases loaded without a tensor map; the mma.sync kernel
# (M <= 16, fp32 x, K splits) and the tcgen05 kernel (16-bit x, M > 16)
GENERAL_K = [(8, 576, 17408, "bf16"), (16, 576, 3000, "f16"), (64, 576, 17408, "bf16"),
             (8, 2880, 5000, "bf16"), (16, 2880, 17408, "bf16"), (64, 2880, 12000, "f16"),
             (8, 5184, 17408, "bf16"), (16, 5184, 9000, "f16"), (64, 5184, 17408, "bf16"),
             (7, 2880, 1000, "f32"), (8, 5184, 1024, "bf16"), (33, 576, 10001, "bf16"),
             (3, 64, 300, "bf16")]


@pytest.mark.parametrize("M,K,N,dtype", GENERAL_K)
def test_linear_k_multiple_of_64(M, K, N, dtype):
    seed = 3 * M + K + N
    w = synth.w4_weights(seed, N, K)
    x = synth.activations(seed, M, K, dtype)
    assert_proj_close(run_linear(x, w, dtype), oracle_linear(x, w, dtype), dtype)


@pytest.mark.parametrize("M,K,N", [(8, 576, 20000), (64, 2880, 30000), (64, 5184, 12000),
                                   (16, 5184, 4000)])
def test_vocab_argmax_k_multiple_of_64(M, K, N):
    w = synth.w4_weights(M + K, N, K)
    x = synth.activations(M + K, M, K, "bf16")
    idx, mx, ws = run_vocab(x, w)
    assert check_argmax(idx, mx, oracle_linear(x, w, "bf16")) == 0
    assert not ws.any(), "workspace must be left zeroed"
