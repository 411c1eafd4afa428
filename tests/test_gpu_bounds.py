"""The bounds-checked build (libvq_checked.so, compiled with VQ_CHECK_BOUNDS).

In that build every global store of every kernel (and the row gathers whose
addresses the kernel computes itself) is tested against the extent of the
buffer it writes or reads; an access outside it is skipped and sets bit 1 of
the library's device status word. Here each entry point runs on the parity
shapes (the full-size workloads, ragged tails, both projection layouts, split
K, the tensor-core kernels, the arg max variants, the KV commit, one verify
round and the attention) through the normal and the checked build, on the
same inputs: the results must be identical bit for bit and the checked
build's status word must stay 0. Together with the guard bands that the
parity tests put around every output, this stands in for a memory checker.
"""
import numpy as np
import pytest
import torch

from parity import to_dev_act, to_dev_weights
from speculative_block_draft_02_gb300 import binding as vq
from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.gpu

_TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def checked():
    from speculative_block_draft_02_gb300 import build

    build.build()
    vq.lib()
    handle = vq.open_library(build.build(checked=True))
    torch.cuda.init()
    return handle


def both(checked, run):
    """run() through the normal build, then through the checked one; returns
    both results as lists of host byte strings and the checked build's status."""
    normal = [bytes(t.cpu().contiguous().view(torch.uint8).numpy()) for t in run()]
    saved = vq._lib
    vq._lib = checked
    try:
        vq.vq_device_error(clear=True)
        chk = [bytes(t.cpu().contiguous().view(torch.uint8).numpy()) for t in run()]
        torch.cuda.synchronize()
        err = vq.vq_device_error()
    finally:
        vq._lib = saved
    return normal, chk, err


def assert_same(checked, run):
    normal, chk, err = both(checked, run)
    assert err == 0, "the checked build flagged an access out of bounds (status %#x)" % err
    assert len(normal) == len(chk)
    for i, (a, b) in enumerate(zip(normal, chk)):
        assert a == b, "result %d differs between the normal and the checked build" % i


def _proj_inputs(M, K, N, dtype, seed):
    w = synth.w4_weights(seed, N, K)
    x = to_dev_act(synth.activations(seed, M, K, dtype), dtype)
    return (x, *to_dev_weights(w))


# (M, K, N, dtype): the headline shape and its narrow (split-K) case, M=16 and
# M=64 at full size, fp32 activations, ragged tails, the tcgen05 kernel with
# long K
LINEAR = [(8, 5120, 17408, "bf16"), (8, 5120, 1024, "bf16"), (16, 5120, 17408, "bf16"),
          (64, 5120, 17408, "bf16"), (4, 5120, 17408, "f32"), (7, 1024, 500, "f32"),
          (3, 512, 129, "bf16"), (12, 1024, 300, "f16"), (33, 1024, 130, "bf16"),
          (2, 512, 128 * 160 + 3, "bf16"), (40, 17408, 9728, "f16"), (17, 512, 12345, "bf16")]


@pytest.mark.parametrize("M,K,N,dtype", LINEAR)
def test_linear_checked_build(checked, M, K, N, dtype):
    x, qw, s, b = _proj_inputs(M, K, N, dtype, M + K + N)

    def run():
        nb = vq.vq_linear_workspace_bytes(M, K, N, _TD[dtype])
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
        y = vq.vq_linear(x, qw, s, b, workspace=ws)
        return [y] + ([ws] if ws is not None else [])

    assert_same(checked, run)


@pytest.mark.parametrize("M,K,N,dtype", [(64, 2560, 151936, "bf16"), (8, 1024, 40000, "bf16"),
                                         (17, 512, 3000, "bf16"), (5, 1024, 9000, "f32"),
                                         (64, 1024, 40000, "f16")])
def test_vocab_argmax_checked_build(checked, M, K, N, dtype):
    x, qw, s, b = _proj_inputs(M, K, N, dtype, 3 * M + N)

    def run():
        ws = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        mx = torch.empty(M, dtype=torch.float32, device="cuda")
        idx, mx = vq.vq_vocab_argmax(x, qw, s, b, ws, maxval=mx)
        ws2 = torch.zeros(vq.vq_vocab_argmax_top2_workspace_bytes(M), dtype=torch.uint8,
                          device="cuda")
        i2, m2, sec = vq.vq_vocab_argmax_top2(x, qw, s, b, ws2)
        return [idx, mx, ws, i2, m2, sec, ws2]

    assert_same(checked, run)


def test_accept_walk_and_kv_commit_checked_build(checked):
    case = synth.commit_case(0)
    edge = synth.commit_case(5, layers=2, B=8, H=3, S_cap=64, D=64, block=16, prefix_lo=0,
                             prefix_hi=40, keep=[16, 0, 16, 5, 16, 3, 17, 16],
                             src_off=[44, 44, 20, 59, 48, 2, 40, 50])
    edge.prefix_len[:] = [30, 10, 20, 10, 5, 62, 1, 0]
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    r = np.random.default_rng(9)
    draft = i32(r.integers(0, 4, size=(33, 16)))
    target = i32(r.integers(0, 4, size=(33, 16)))

    def run():
        out = [vq.verify_accept_walk(draft, target)]
        for c in (case, edge):
            kv = [torch.from_numpy(t.view(np.int16).copy()).cuda() for t in c.tensors]
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            out.append(vq.kv_compact_per_row(kv, i32(c.prefix_len), i32(c.src_off), i32(c.keep),
                                             16, status=status))
            out += [status] + kv
        return out

    assert_same(checked, run)


def test_verify_round_checked_build(checked):
    B, L, K, N = 4, 16, 512, 20000
    M = B * L
    x, qw, s, b = _proj_inputs(M, K, N, "bf16", 404)
    r = np.random.default_rng(404)
    tok = torch.from_numpy(r.integers(0, N, size=(B, L)).astype(np.int32)).cuda()
    case = synth.commit_case(20, layers=2, B=B, H=2, S_cap=512, D=64, block=L, prefix_lo=20,
                             prefix_hi=400, keep=[1, 16, 3, 8])
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()

    def run():
        ws = torch.zeros(vq.verify_round_workspace_bytes(B, L), dtype=torch.uint8, device="cuda")
        kv = [torch.from_numpy(t.view(np.int16).copy()).cuda() for t in case.tensors]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        target, acc, bonus, new_len = vq.verify_round(x, qw, s, b, tok, ws, kv=kv,
                                                      prefix_len=i32(case.prefix_len),
                                                      src_off=i32(case.src_off), status=status)
        return [target, acc, bonus, new_len, status] + kv

    assert_same(checked, run)


# (B, L, Hq, Hkv, D, S_cap, prefix_len, src_off, dtype, rotary_dim): the
# full-size workload, two row groups, the block at the cache end (a key box
# past the tensor's end), D=64 bf16, rows out of range (flagged, skipped), and
# a rotary width that is not a multiple of 16 (one pair per rotation step)
ATTN = [
    (4, 16, 32, 8, 128, 2048, None, None, "f16", 128),
    (2, 10, 16, 2, 64, 400, [5, 250], [260, 250], "f16", 64),
    (1, 8, 4, 2, 64, 100, [90], [92], "f16", 64),
    (2, 8, 4, 4, 64, 300, [129, 255], [200, 292], "bf16", 32),
    (4, 8, 8, 2, 128, 256, [40, 100, 10, 200], [60, 90, 248, 250], "f16", 64),
    (2, 8, 4, 2, 64, 300, [100, 37], [120, 37], "f16", 40),
]


@pytest.mark.parametrize("B,L,Hq,Hkv,D,S_cap,prefix,src,dtype,rd", ATTN)
def test_verify_attention_checked_build(checked, B, L, Hq, Hkv, D, S_cap, prefix, src, dtype, rd):
    kw = dict(prefix_len=prefix, src_off=src) if prefix is not None else dict(prefix_lo=200,
                                                                               prefix_hi=1800)
    case = synth.attention_case(B * 31 + L, B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, S_cap=S_cap,
                                dtype=dtype, **kw)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).cuda().view(
        _TD[dtype])
    q, kn, vn = dev(case.q), dev(case.k_new), dev(case.v_new)
    pl = torch.from_numpy(case.prefix_len).cuda()
    so = torch.from_numpy(case.src_off).cuda()

    def run():
        kc, vc = dev(case.k_cache), dev(case.v_cache)
        ws = torch.zeros(vq.verify_attention_workspace_bytes(B, L, Hq, Hkv, D, S_cap),
                         dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.zeros_like(q)
        vq.verify_attention(q, kn, vn, kc, vc, pl, so, ws, rd, 1e6, D ** -0.5, out=out,
                            status=status)
        return [out, kc, vc, status]

    assert_same(checked, run)
