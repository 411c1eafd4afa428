"""Back-to-back calls on one stream.

The projection kernels are launched with programmatic stream serialization:
a call may start while the kernel before it is finishing, requests its first
weight stages at once, and reads x (and writes its outputs and workspace)
only after that kernel has completed. These tests chain calls whose x is the
previous call's output, sharing one workspace, with no synchronization in
between, and compare with the same call made after a full synchronization on
a separate copy of that x (same kernels, so bit for bit). The buffer the first
call writes starts out as NaN, so a read that came too early would show.
"""
import numpy as np
import pytest
import torch

from speculative_block_draft_02_gb300 import binding as vq
from speculative_block_draft_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev_weights(seed, N, K):
    w = synth.w4_weights(seed, N, K)
    return tuple(torch.from_numpy(a.view(np.int32 if a.dtype == np.uint32 else np.int16).copy())
                 .cuda() for a in (w.qw, w.scales, w.biases))


def _dev_x(seed, M, K, dtype):
    xb = synth.activations(seed, M, K, dtype)
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(xb.view(np.int16).copy()).view(t).cuda()


def _ws(M, K, N, t):
    return torch.zeros(max(vq.vq_linear_workspace_bytes(M, K, N, t), 16), dtype=torch.uint8,
                       device="cuda")


# (M, K1, N1 = K2, N2), chosen so that the second call (the one that reads the
# first's output) covers each kernel: M <= 8 the prepared-slice kernel, M > 16
# with a wide N the tcgen05 kernel, M = 16 with a narrow N the split-K mma.sync
# kernel
CHAINS = [(8, 512, 4096, 2048, "bf16"), (5, 1024, 2048, 17408, "f16"),
          (64, 512, 5120, 17408, "bf16"), (33, 512, 2048, 12000, "f16"),
          (16, 512, 4096, 1024, "bf16")]


@pytest.mark.parametrize("M,K1,N1,N2,dtype", CHAINS)
def test_chained_projections_read_the_previous_output(M, K1, N1, N2, dtype):
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    x = _dev_x(M + K1, M, K1, dtype)
    w1 = _dev_weights(1, N1, K1)
    w2 = _dev_weights(2, N2, N1)
    ws = torch.zeros(max(_ws(M, K1, N1, t).numel(), _ws(M, N1, N2, t).numel()),
                     dtype=torch.uint8, device="cuda")
    y1 = torch.full((M, N1), float("nan"), dtype=t, device="cuda")
    y2 = torch.empty((M, N2), dtype=t, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):   # repeated chains on the same buffers and workspace
        vq.vq_linear(x, *w1, y=y1, workspace=ws)
        vq.vq_linear(y1, *w2, y=y2, workspace=ws)
    torch.cuda.synchronize()
    assert not torch.isnan(y1).any()
    y1c = y1.clone()
    ref = vq.vq_linear(y1c, *w2, workspace=_ws(M, N1, N2, t))
    torch.cuda.synchronize()
    assert torch.equal(y2, ref)
    assert vq.vq_device_error() == 0


@pytest.mark.parametrize("M,K1,N1,N2", [(8, 512, 2048, 60000), (64, 512, 2560, 20000)])
def test_argmax_after_projection_reads_its_output(M, K1, N1, N2):
    x = _dev_x(M + N2, M, K1, "bf16")
    w1 = _dev_weights(3, N1, K1)
    w2 = _dev_weights(4, N2, N1)
    wsl = _ws(M, K1, N1, torch.bfloat16)
    wsa = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    h = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(M, dtype=torch.int32, device="cuda")
    mx = torch.empty(M, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    vq.vq_linear(x, *w1, y=h, workspace=wsl)
    vq.vq_vocab_argmax(h, *w2, wsa, argmax=idx, maxval=mx)
    torch.cuda.synchronize()
    hc = h.clone()
    wsb = torch.zeros_like(wsa)
    ridx, rmx = vq.vq_vocab_argmax(hc, *w2, wsb, maxval=torch.empty_like(mx))
    torch.cuda.synchronize()
    assert torch.equal(idx, ridx)
    assert torch.equal(mx, rmx)
    assert not wsa.any()



@pytest.mark.parametrize("M,K,N,dtype", [(8, 5120, 17408, "bf16"), (3, 512, 1000, "f16"),
                                         (7, 1024, 500, "f32"), (64, 1024, 9800, "bf16"),
                                         (8, 5120, 1024, "bf16")])
def test_linear_host_buffers_match_device_call(M, K, N, dtype):
    """vq_linear_host (x in and y out through page-locked host memory, enqueued
    with the projection) gives what vq_linear gives on the same inputs, bit for
    bit, twice in a row on the same buffers and workspace (narrow N splits K,
    so the workspace must come back zeroed)."""
    from parity import to_dev_act

    qw, s, b = _dev_weights(M + K + N, N, K)
    x = to_dev_act(synth.activations(M + K + N, M, K, dtype), dtype)
    nb = vq.vq_linear_workspace_bytes(M, K, N, x.dtype)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
    y_ref = vq.vq_linear(x, qw, s, b, workspace=ws).cpu()
    x_host = x.cpu().pin_memory()
    y_host = torch.empty((M, N), dtype=x.dtype).pin_memory()
    x_dev = torch.empty_like(x)
    y_dev = torch.empty((M, N), dtype=x.dtype, device="cuda")
    for _ in range(2):
        y_host.fill_(float("nan"))
        vq.vq_linear_host(x_host, qw, s, b, y_host, x_dev, y_dev, workspace=ws)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(y_host.view(torch.uint8), y_ref.view(torch.uint8))


def test_linear_host_pageable_and_mixed_buffers():
    """Host buffers the device cannot address directly (ordinary pageable memory)
    go through the copies: same bits as vq_linear, with pageable x and pinned y
    and the other way round."""
    from parity import to_dev_act

    M, K, N = 8, 5120, 17408
    qw, s, b = _dev_weights(91, N, K)
    x = to_dev_act(synth.activations(91, M, K, "bf16"), "bf16")
    nb = vq.vq_linear_workspace_bytes(M, K, N, x.dtype)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
    y_ref = vq.vq_linear(x, qw, s, b, workspace=ws).cpu()
    x_dev = torch.empty_like(x)
    y_dev = torch.empty((M, N), dtype=x.dtype, device="cuda")
    for x_pin, y_pin in ((False, False), (False, True), (True, False)):
        x_host = x.cpu().pin_memory() if x_pin else x.cpu().clone()
        y_host = torch.full((M, N), float("nan"), dtype=x.dtype)
        if y_pin:
            y_host = y_host.pin_memory()
        vq.vq_linear_host(x_host, qw, s, b, y_host, x_dev, y_dev, workspace=ws)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(y_host.view(torch.uint8), y_ref.view(torch.uint8)), (x_pin, y_pin)
