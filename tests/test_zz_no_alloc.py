"""vq_vocab_argmax_noalloc: the arg max entry point that allocates nothing.

Some callers cannot allocate device memory: serving runtimes that forbid
cudaMalloc once they are running, and plug-ins inside a host application that
owns all device memory. For them the library keeps the arg max scratch in a
fixed array of its own.
This test calls that entry point through the C ABI, twice in a row (the
array keeps the previous call's contents), and checks each call against the
CPU oracle's arg max of the same logits (indices bit for bit, max values
within the tolerance the other arg max tests use) and against vq_vocab_argmax
with a caller-provided workspace (identical indices and max values). It lives
in a file that pytest collects last, and needs no state from the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_block_draft_02_gb300 import binding as vq
from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(w, x):
    qw = torch.from_numpy(w.qw.view(np.int32).copy()).cuda()
    s = torch.from_numpy(w.scales.view(np.int16).copy()).cuda()
    b = torch.from_numpy(w.biases.view(np.int16).copy()).cuda()
    xd = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return xd, qw, s, b


@pytest.mark.parametrize("M,K,N", [(8, 512, 1024), (64, 2560, 20000), (3, 1024, 5000)])
def test_noalloc_argmax_matches_workspace_entry_point(M, K, N):
    from speculative_block_draft_02_gb300 import build

    build.build()
    oracle.build()
    w = synth.w4_weights(M * 7 + 1, N, K)
    x = synth.activations(M * 7 + 1, M, K, "bf16")
    # the oracle's greedy tokens, decided on its fp64 logits rounded to fp32;
    # no row of these shapes has a near tie (top two within 1e-4 relative)
    logits = oracle.vq_linear(x, w.qw, w.scales, w.biases, act_dtype=oracle.BF16)
    o_idx, o_max, o_sec = oracle.argmax(logits)
    margin = 1e-4 * np.maximum(1.0, np.abs(o_max.astype(np.float64)))
    assert np.all(o_max.astype(np.float64) - o_sec > margin)
    xd, qw, s, b = _dev(w, x)
    ws = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    ref_i, ref_v = vq.vq_vocab_argmax(xd, qw, s, b, ws,
                                      maxval=torch.empty(M, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    ref_i, ref_v = ref_i.cpu().numpy(), ref_v.cpu().numpy()
    for _ in range(2):
        idx, mx = vq.vq_vocab_argmax_noalloc(
            xd, qw, s, b, maxval=torch.empty(M, dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        idx, mx = idx.cpu().numpy(), mx.cpu().numpy()
        assert np.array_equal(idx, o_idx)
        assert np.all(np.abs(mx - o_max) <= 1e-5 * np.maximum(1.0, np.abs(o_max)))
        assert np.array_equal(idx, ref_i) and np.array_equal(mx, ref_v)
    assert vq.vq_device_error() == 0


def test_noalloc_argmax_rejects_m_beyond_its_array():
    from speculative_block_draft_02_gb300 import build

    build.build()
    w = synth.w4_weights(5, 256, 512)
    x = synth.activations(5, 65, 512, "bf16")
    xd, qw, s, b = _dev(w, x)
    with pytest.raises(vq.VQError):
        vq.vq_vocab_argmax_noalloc(xd, qw, s, b)
