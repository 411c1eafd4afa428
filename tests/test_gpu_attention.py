"""GPU parity of verify_attention, called through the C ABI, against the oracle.

The output must meet the tolerance in parity.py; the cache slots the call
appends (the block's rotated keys) too, against the oracle's rotated keys
before rounding; the appended values and every other cache slot must match bit
for bit. Small shapes cover several key chunks with ragged tails, rows without
a prefix, without a stale gap and with the block at the end of the cache,
grouped query heads over one and two row groups, both storage types, both head
sizes and full, partial and no rotation; the full-size workload is checked in
full.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, Guarded, proj_error
from speculative_block_draft_02_gb300 import binding as vq
from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "f16": torch.float16}
ODT = {"bf16": 0, "f16": 1}


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


def dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(TDT[dtype]).cuda()


def bits_of(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def f64_of(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_both(case, rotary_dim, theta, scale=None, ws_fill=0xFF):
    """Runs the GPU call and the oracle on the same case; returns both results."""
    B, L, Hq, D = case.q.shape
    Hkv, S_cap = case.k_cache.shape[1], case.k_cache.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dt = case.dtype
    q, kn, vn = dev(case.q, dt), dev(case.k_new, dt), dev(case.v_new, dt)
    gk = Guarded(case.k_cache.shape, TDT[dt], fill=dev(case.k_cache, dt))
    gv = Guarded(case.v_cache.shape, TDT[dt], fill=dev(case.v_cache, dt))
    kc, vc = gk.t, gv.t
    pl = torch.from_numpy(case.prefix_len).cuda()
    so = torch.from_numpy(case.src_off).cuda()
    nb = vq.verify_attention_workspace_bytes(B, L, Hq, Hkv, D, S_cap)
    # the workspace needs no initial contents: start it as NaN bytes
    ws = torch.full((nb,), ws_fill, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    go = Guarded(q.shape, q.dtype, fill=float("nan"))
    out = go.t
    vq.verify_attention(q, kn, vn, kc, vc, pl, so, ws, rotary_dim, theta, scale, out=out,
                        status=status)
    for g in (gk, gv, go):
        g.check()
    kco, vco = case.k_cache.copy(), case.v_cache.copy()
    r_out, r_krot, r_st = oracle.verify_attention(case.q, case.k_new, case.v_new, kco, vco,
                                                  case.prefix_len, case.src_off, ODT[dt],
                                                  rotary_dim, theta, scale)
    return dict(out=out, kc=kc, vc=vc, status=int(status.item()), r_out=r_out, r_krot=r_krot,
                r_st=r_st, kco=kco, vco=vco)


def check(case, res):
    dt = case.dtype
    B, L = case.q.shape[:2]
    S_cap = case.k_cache.shape[2]
    assert res["status"] == res["r_st"]
    err = proj_error(f64_of(res["out"]), res["r_out"], dt)
    assert err <= TOL[dt], "output error %.3e" % err
    kc, vc = bits_of(res["kc"]), bits_of(res["vc"])
    for b in range(B):
        P, S = int(case.prefix_len[b]), int(case.src_off[b])
        if not (P >= 0 and S >= P and S + L <= S_cap):
            assert np.array_equal(kc[b], case.k_cache[b]) and np.array_equal(vc[b], case.v_cache[b])
            assert not res["out"][b].any()
            continue
        other = np.ones(S_cap, dtype=bool)
        other[S:S + L] = False
        assert np.array_equal(kc[b][:, other], case.k_cache[b][:, other])
        assert np.array_equal(vc[b][:, other], case.v_cache[b][:, other])
        assert np.array_equal(vc[b][:, S:S + L], case.v_new[b].transpose(1, 0, 2))
        got = f64_of(res["kc"][b, :, S:S + L])
        want = res["r_krot"][b].transpose(1, 0, 2)
        kerr = proj_error(got, want, dt)
        assert kerr <= TOL[dt], "appended key error %.3e (row %d)" % (kerr, b)
    return err


# (B, L, Hq, Hkv, D, S_cap, prefix_len, src_off, dtype, rotary_dim, theta)
CASES = [
    # three rows: no prefix, a gap, none; several 64-key chunks with ragged tails
    (3, 16, 8, 2, 128, 520, [0, 137, 300], None, "f16", 128, 1e6),
    # block ends at the cache end; src_off per row; partial rotation; bf16; D 64
    (2, 8, 4, 4, 64, 300, [129, 255], [200, 292], "bf16", 32, 1e4),
    # 8 query heads per KV head: L*G = 80 rows -> two row groups
    (2, 10, 16, 2, 64, 400, [5, 250], [260, 250], "f16", 64, 1e4),
    # one key per query: no prefix, L = 1, no rotation
    (1, 1, 2, 1, 128, 64, [0], [0], "bf16", 0, 1e4),
    # the largest block, one query head per KV head
    (4, 64, 8, 8, 128, 1024, [900, 3, 500, 128], None, "bf16", 128, 1e6),
    # prefix lengths on chunk edges (127, 128, 129) with the block after them
    (3, 16, 4, 2, 128, 400, [127, 128, 129], [127, 150, 300], "f16", 96, 5e5),
    # a chunk that reaches the block near the cache end: its 64-row box of the
    # last KV head runs past the end of the cache tensor (zero-filled rows)
    (1, 8, 4, 2, 64, 100, [90], [92], "f16", 64, 1e4),
    # rotary widths that are not multiples of 16 (one pair per rotation step,
    # for the queries and for the prefetched block keys)
    (2, 8, 4, 2, 64, 300, [100, 37], [120, 37], "f16", 40, 1e4),
    (1, 16, 8, 2, 128, 200, [70], None, "bf16", 6, 1e4),
]


@pytest.mark.parametrize("B,L,Hq,Hkv,D,S_cap,prefix,src,dtype,rd,theta", CASES)
def test_verify_attention_matches_oracle(B, L, Hq, Hkv, D, S_cap, prefix, src, dtype, rd, theta):
    case = synth.attention_case(B * 1000 + L, B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, S_cap=S_cap,
                                prefix_len=prefix, src_off=src, dtype=dtype)
    check(case, run_both(case, rd, theta))


def test_verify_attention_rows_out_of_range_are_flagged():
    # rows 1 and 3 are out of range (block before the prefix, block past the end)
    case = synth.attention_case(17, B=4, L=8, Hq=4, Hkv=2, D=64, S_cap=256,
                                prefix_len=[40, 100, 10, 200], src_off=[60, 90, 248, 250],
                                dtype="f16")
    res = run_both(case, 64, 1e4)
    assert res["status"] == 1
    check(case, res)


def test_verify_attention_full_workload():
    cfg = synth.WORKLOADS["verify_attention_b4_l16_hq32_hkv8_d128"]
    case = synth.attention_case(0, B=cfg["B"], L=cfg["L"], Hq=cfg["Hq"], Hkv=cfg["Hkv"],
                                D=cfg["D"], S_cap=cfg["S_cap"], prefix_lo=cfg["prefix_lo"],
                                prefix_hi=cfg["prefix_hi"], dtype=cfg["dtype"])
    res = run_both(case, cfg["rotary_dim"], cfg["theta"])
    assert res["status"] == 0
    check(case, res)


def test_verify_attention_is_deterministic_and_ignores_workspace_contents():
    case = synth.attention_case(23, B=2, L=16, Hq=8, Hkv=2, D=128, S_cap=700,
                                prefix_len=[333, 600], dtype="bf16")
    a = run_both(case, 128, 1e6, ws_fill=0xFF)
    b = run_both(case, 128, 1e6, ws_fill=0x00)
    assert torch.equal(a["out"], b["out"])
    assert torch.equal(a["kc"], b["kc"]) and torch.equal(a["vc"], b["vc"])


def test_stuck_waits_give_up_and_flag_their_status():
    """The kernels' bounded waits, made to run out on purpose on a barrier that
    nothing arrives at: each gives up after its limit with the status flagged,
    and the GPU stays usable afterwards."""
    limit = 2 ** 31
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    report = torch.zeros(8, dtype=torch.int64, device="cuda")
    vq.vq_wait_selftest(status, report)
    torch.cuda.synchronize()
    r = report.cpu().tolist()
    assert r[0] == 1 and r[1] < limit // 64          # a completed barrier passes at once
    assert r[2] == 0 and limit <= r[3] < 2 * limit   # a stuck one gives up at the limit
    assert r[4] == 1                                 # and raises the block's abort flag
    assert r[5] == 0 and r[6] < limit                # which ends the next wait before its own limit
    assert limit <= r[7] < 2 * limit                 # the teardown wait is bounded too
    assert status.cpu().tolist() == [1, 1]
    assert vq.vq_device_error() == 0                 # the library's own word is untouched
    # the context still works: a small attention call right after matches the oracle
    case = synth.attention_case(29, B=1, L=4, Hq=2, Hkv=1, D=64, S_cap=200, prefix_len=[150],
                                dtype="f16")
    check(case, run_both(case, 64, 1e4))
