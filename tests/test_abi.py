"""The C-ABI library builds for sm_103a, loads, and exports what vq.h declares.

No compute calls here (no GPU needed): only symbol checks and the host-side
argument validation, which rejects bad calls before any CUDA work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vq.h")


@pytest.fixture(scope="module")
def vqlib():
    from speculative_block_draft_02_gb300 import binding, build

    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_functions()
    for n in ("vq_linear", "vq_vocab_argmax", "verify_accept_walk", "kv_compact_per_row"):
        assert n in names


def test_library_exports_every_declared_symbol(vqlib):
    from speculative_block_draft_02_gb300 import binding

    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(vqlib, n), n
    assert set(names) == set(binding.SIGNATURES)


def test_library_is_built_for_sm_103a():
    from speculative_block_draft_02_gb300 import build

    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_strerror(vqlib):
    for code in (0, -1, -2, -3, -4, -5):
        assert vqlib.vq_strerror(code)
    assert vqlib.vq_strerror(-99) == b"unknown status"


def test_vocab_workspace_size(vqlib):
    assert vqlib.vq_vocab_argmax_workspace_bytes(64) == 528
    assert vqlib.vq_vocab_argmax_workspace_bytes(1) == 16
    assert vqlib.vq_vocab_argmax_workspace_bytes(0) == 0
    assert vqlib.vq_vocab_argmax_workspace_bytes(65) == 0
    # keys and counter, then one 16-byte candidate per (block, row), 256 blocks
    assert vqlib.vq_vocab_argmax_top2_workspace_bytes(64) == 528 + 256 * 64 * 16
    assert vqlib.vq_vocab_argmax_top2_workspace_bytes(1) == 16 + 256 * 16
    assert vqlib.vq_vocab_argmax_top2_workspace_bytes(0) == 0
    assert vqlib.vq_vocab_argmax_top2_workspace_bytes(65) == 0


def test_host_validation_rejects_before_any_launch(vqlib):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    # M out of range, K not a multiple of 64, bad dtype
    assert vqlib.vq_linear(fake, 0, 512, 16, fake, fake, fake, fake, 0, None, 0, None) == -1
    assert vqlib.vq_linear(fake, 65, 512, 16, fake, fake, fake, fake, 0, None, 0, None) == -1
    assert vqlib.vq_linear(fake, 8, 100, 16, fake, fake, fake, fake, 0, None, 0, None) == -1
    assert vqlib.vq_linear(fake, 8, 544, 16, fake, fake, fake, fake, 0, None, 0, None) == -1
    assert vqlib.vq_linear(fake, 8, 512, 16, fake, fake, fake, fake, 7, None, 0, None) == -1
    assert vqlib.vq_linear(fake, 33, 512, 16, fake, fake, fake, fake, 2, None, 0, None) == -4
    # null and misaligned pointers
    assert vqlib.vq_linear(None, 8, 512, 16, fake, fake, fake, fake, 0, None, 0, None) == -1
    assert vqlib.vq_linear(P(0x1002), 8, 512, 16, fake, fake, fake, fake, 0, None, 0, None) == -2
    assert vqlib.vq_vocab_argmax(fake, 8, 512, 16, fake, fake, fake, 0, None, None, fake, 64,
                                 None) == -1
    # verify_round: B*L <= 64, outputs required, workspace checked before any launch
    assert vqlib.verify_round_workspace_bytes(4, 16) == 528 + 16
    assert vqlib.verify_round_workspace_bytes(8, 9) == 0
    rnd = lambda B, L, tok, ws, nb: vqlib.verify_round(
        fake, B, L, 512, 100, fake, fake, fake, 0, tok, fake, fake, fake, None, 0, 0, 0, 0, 0,
        None, None, None, None, ws, nb, None)
    assert rnd(8, 9, fake, fake, 4096) == -1
    assert rnd(4, 16, None, fake, 4096) == -1
    assert rnd(4, 16, fake, None, 0) == -5
    assert rnd(4, 16, fake, fake, 16) == -5
    # the top-2 call needs its runner-up output, 4-byte aligned
    assert vqlib.vq_vocab_argmax_top2(fake, 8, 512, 16, fake, fake, fake, 0, fake, None, None,
                                      fake, 1 << 20, None) == -1
    assert vqlib.vq_vocab_argmax_top2(fake, 8, 512, 16, fake, fake, fake, 0, fake, None,
                                      P(0x1001), fake, 1 << 20, None) == -2
    assert vqlib.verify_accept_walk(fake, fake, 0, 8, fake, None) == -1
    assert vqlib.verify_accept_walk(fake, fake, 4, 0, fake, None) == -1
    assert vqlib.verify_accept_walk(P(0x1001), fake, 4, 8, fake, None) == -2
    arr = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    tp = ctypes.cast(arr, P)
    assert vqlib.kv_compact_per_row(tp, 0, 4, 8, 2048, 128, 2, fake, fake, fake, 16, fake, None,
                                    None) == -1
    assert vqlib.kv_compact_per_row(tp, 65, 4, 8, 2048, 128, 2, fake, fake, fake, 16, fake, None,
                                    None) == -1
    assert vqlib.kv_compact_per_row(tp, 2, 4, 8, 2048, 3, 2, fake, fake, fake, 16, fake, None,
                                    None) == -2
    assert vqlib.kv_compact_per_row(tp, 2, 4, 8, 2048, 128, 2, fake, fake, fake, 1000, fake,
                                    None, None) == -4
    bad = (ctypes.c_void_p * 2)(0x1000, 0x2008)
    assert vqlib.kv_compact_per_row(ctypes.cast(bad, P), 2, 4, 8, 2048, 128, 2, fake, fake, fake,
                                    16, fake, None, None) == -2


def test_verify_attention_workspace_and_host_validation(vqlib):
    P = ctypes.c_void_p
    # the partial results stay in the clusters' shared memory: no workspace
    assert vqlib.verify_attention_workspace_bytes(4, 16, 32, 8, 128, 2048) == 0
    assert vqlib.verify_attention_workspace_bytes(2, 10, 16, 2, 64, 100) == 0

    fake = P(0x1000)

    def call(q=fake, out=fake, B=4, L=16, Hq=32, Hkv=8, D=128, S_cap=2048, rd=128, theta=1e6,
             scale=0.088, dtype=1):
        # every call below fails validation before any CUDA work
        return vqlib.verify_attention(q, fake, fake, fake, fake, fake, fake, out, B, L, Hq, Hkv, D,
                                      S_cap, rd, theta, scale, dtype, None, None, 0, None)

    assert call(B=0) == -1
    assert call(Hq=30) == -1                       # not a multiple of Hkv
    assert call(S_cap=8) == -1                     # shorter than the block
    assert call(rd=7) == -1 and call(rd=130) == -1
    assert call(theta=0.0) == -1 and call(theta=float("nan")) == -1
    assert call(scale=float("inf")) == -1
    assert call(dtype=2) == -1                     # fp32 tensors are not taken
    assert call(q=None) == -1
    assert call(D=96, rd=96) == -4
    assert call(L=65, S_cap=4096) == -4
    assert call(q=P(0x1008)) == -2                 # 16-byte alignment
    assert call(out=P(0x1001)) == -2


def test_wait_selftest_host_validation(vqlib):
    P = ctypes.c_void_p
    assert vqlib.vq_wait_selftest(None, P(0x1000), None) == -1
    assert vqlib.vq_wait_selftest(P(0x1000), None, None) == -1
    assert vqlib.vq_wait_selftest(P(0x1002), P(0x1000), None) == -2
    assert vqlib.vq_wait_selftest(P(0x1000), P(0x1004), None) == -2


def test_linear_host_validation(vqlib):
    P = ctypes.c_void_p
    fake = P(0x1000)

    def call(xh=fake, yh=fake, xd=fake, yd=fake, M=8, K=512, N=128, act=0):
        # every call below fails validation before any CUDA work
        return vqlib.vq_linear_host(xh, M, K, N, fake, fake, fake, yh, act, xd, yd, None, 0, None)

    assert call(xh=None) == -1
    assert call(yh=None) == -1
    assert call(xd=None) == -1 and call(yd=None) == -1
    assert call(M=0) == -1 and call(K=0) == -1 and call(N=0) == -1
    assert call(act=7) == -1
