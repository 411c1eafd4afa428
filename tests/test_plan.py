"""The launch planner, on the host (vq_plan touches no device): which kernel a
call runs, its stage ring, K split, grid and memory, for a 152-SM GB300."""
import pytest
import torch

SMS = 152
LIMIT = 232448          # opt-in shared memory per block
SLICE = 8992            # prepared x slice per 512-wide stage (M <= 8)


@pytest.fixture(scope="module")
def vq():
    from speculative_block_draft_02_gb300 import binding, build

    build.build()
    binding.lib()
    return binding


def plan(vq, M, K, N, act=torch.bfloat16, argmax=False, sms=SMS):
    return vq.vq_plan(M, K, N, act, argmax, sms)


def test_headline_projection(vq):
    p = plan(vq, 8, 5120, 17408)
    assert p["kernel"] == 2 and p["launches"] == 2          # prepared slices + projection
    assert p["k_splits"] == 1 and p["units"] == p["grid"] == 136
    assert p["prefetch"] == 3 and p["stages"] >= 4
    assert p["workspace_bytes"] == -(-10 * SLICE // 256) * 256
    assert p["smem_bytes"] <= LIMIT


def test_next_block_verify_runs_on_tcgen05(vq):
    p = plan(vq, 64, 5120, 17408)
    assert p["kernel"] == 3 and p["rows_padded"] == 64 and p["launches"] == 2
    assert p["stages"] == 2 and p["workspace_bytes"] == 80 * 64 * 4   # group row sums
    p = plan(vq, 24, 5120, 17408, torch.float16)
    assert p["kernel"] == 3 and p["rows_padded"] == 32


def test_small_m_and_fp32_stay_on_mma_sync(vq):
    # 16-bit x with M <= 16: prepared slices, one per n8 tile (two at M = 16)
    p = plan(vq, 16, 5120, 17408)
    assert p["kernel"] == 2 and p["launches"] == 2 and p["stages"] == 4
    assert p["workspace_bytes"] == -(-10 * 2 * SLICE // 256) * 256
    assert plan(vq, 16, 5120, 17408, argmax=True)["kernel"] == 0
    assert plan(vq, 8, 5120, 17408, torch.float32)["kernel"] == 0
    assert plan(vq, 32, 512, 17408, torch.float32)["kernel"] == 0


def test_long_k_sums_the_x_groups_per_stage(vq):
    # a table of group row sums for all of K would leave the tcgen05 kernel one
    # stage: the groups are summed per stage instead, with no extra kernel
    p = plan(vq, 64, 5120, 17408)
    assert p["kernel"] == 3 and p["launches"] == 2 and p["workspace_bytes"] == 80 * 64 * 4
    for K in (8192, 17408, 65536):
        p = plan(vq, 64, K, 17408)
        assert p["kernel"] == 3 and p["stages"] == 2 and p["launches"] == 1
        assert p["workspace_bytes"] == 0
        p = plan(vq, 64, K, 151936, argmax=True)
        assert p["kernel"] == 3 and p["launches"] == 1
    # the documented limits of the other kernels
    with pytest.raises(Exception):
        plan(vq, 64, 6656, 1024)              # K split at M > 32
    with pytest.raises(Exception):
        plan(vq, 16, 33280, 151936, argmax=True)
    assert plan(vq, 16, 33280, 17408)["kernel"] == 2     # prepared slices: any K
    with pytest.raises(Exception):
        plan(vq, 32, 13312, 17408, torch.float32)


def test_narrow_n_splits_k_to_fill_the_gpu(vq):
    p = plan(vq, 8, 5120, 1024)            # 8 row blocks of 128
    assert p["k_splits"] == 10 and p["units"] == 80 and p["grid"] == 80
    # slices, then split counters (one per row block, 16-byte rounded), then
    # fp32 partials [S][M][N]
    assert p["workspace_bytes"] == -(-10 * SLICE // 256) * 256 + 32 + 10 * 8 * 1024 * 4
    p = plan(vq, 64, 512, 1024)
    assert p["k_splits"] == 1 and p["units"] == 8         # one stage of K: nothing to split
    # half the SMs or more busy: no split
    assert plan(vq, 8, 5120, 128 * 76)["k_splits"] == 1
    assert plan(vq, 8, 5120, 128 * 75)["k_splits"] > 1


def test_vocab_argmax(vq):
    p = plan(vq, 64, 2560, 151936, argmax=True)
    assert p["kernel"] == 3 and p["launches"] == 1
    assert p["units"] == 1187 and p["grid"] == SMS
    assert p["workspace_bytes"] == 528
    p = plan(vq, 8, 1024, 60000, argmax=True)             # several row blocks per block
    assert p["kernel"] == 1 and p["units"] == 469
    assert plan(vq, 8, 1024, 3000, argmax=True)["kernel"] == 0   # too few to pay for the table


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("argmax", [False, True])
def test_plan_invariants(vq, act, argmax):
    for M in (1, 3, 8, 9, 16, 17, 32, 33, 64):
        if act == torch.float32 and M > 32:
            continue
        for K in (512, 2560, 5120):
            for N in (1, 300, 5000, 17408, 151936):
                p = plan(vq, M, K, N, act, argmax)
                assert 2 <= p["stages"] <= 8 and 1 <= p["prefetch"] <= p["stages"]
                assert p["smem_bytes"] <= LIMIT
                assert p["rows_padded"] >= M and p["rows_padded"] in (8, 16, 32, 64)
                assert 1 <= p["grid"] <= min(SMS, p["units"])
                assert p["units"] == -(-N // 128) * p["k_splits"]
                assert p["k_splits"] <= K // 512
                if argmax:
                    assert p["k_splits"] == 1 and p["workspace_bytes"] == -(-(M * 8 + 4) // 16) * 16
                if p["kernel"] == 3:
                    assert act != torch.float32 and M > 16 and p["k_splits"] == 1


@pytest.mark.parametrize("K", [64, 576, 2880, 5184])
def test_k_multiple_of_64_runs_on_the_per_stage_x_kernels(vq, K):
    # a last stage of 1..7 groups; scales and biases by plain loads, so such
    # shapes run on the per-stage x kernels (mma.sync, or tcgen05 for 16-bit
    # x with M > 16 and no K split), with or without a K split
    for M, act, argmax, N in ((8, torch.bfloat16, False, 17408), (16, torch.float16, False, 4096),
                              (64, torch.bfloat16, False, 17408), (8, torch.bfloat16, True, 151936),
                              (64, torch.bfloat16, True, 151936), (7, torch.float32, False, 1000),
                              (8, torch.bfloat16, False, 1024), (24, torch.float16, False, 12000)):
        p = plan(vq, M, K, N, act, argmax)
        if M > 16 and act != torch.float32 and p["k_splits"] == 1:
            assert p["kernel"] == 3
        else:
            assert p["kernel"] == 0 and p["launches"] == 1
        assert p["k_splits"] <= -(-K // 512)
        assert p["units"] == -(-N // 128) * p["k_splits"]
        assert p["smem_bytes"] <= LIMIT and p["stages"] >= 2


def test_plan_rejects_bad_shapes(vq):
    from speculative_block_draft_02_gb300.binding import VQError

    for args in ((0, 512, 16), (65, 512, 16), (8, 100, 16), (8, 512, 0), (8, 544, 16)):
        with pytest.raises(VQError):
            plan(vq, *args)
    with pytest.raises(VQError):
        plan(vq, 33, 512, 16, torch.float32)
    with pytest.raises(VQError):
        plan(vq, 8, 512, 16, sms=0)
