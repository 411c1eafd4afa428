"""Host logic of bench.py that the reported numbers depend on (no GPU).

The digest that ties a committed ncu summary to the code must follow the code
and nothing else, and the algorithmic byte and FLOP counts of the attention
must follow their closed forms.
"""
import os

import numpy as np

import bench
from speculative_block_draft_02_gb300 import synth


def test_code_only_strips_comments_but_not_strings():
    src = ('int a = 1; // gone\n/* gone\n too */ const char* s = "keep // and /* this */";\n'
           "char q = '\"'; asm(\"ld.global.v4.u32 {%0}, [%1];\"); // gone\n  x  =  y;\n")
    out = bench.code_only(src)
    assert "gone" not in out and "too" not in out
    assert '"keep // and /* this */"' in out
    assert "'\"'" in out and '"ld.global.v4.u32 {%0}, [%1];"' in out
    assert out.endswith("x = y;")


def test_code_only_digit_separators_are_not_character_literals():
    a = "int n = 1'000; // count\nint m = 2;\n"
    b = "int n = 1'000; /* other */ int m = 2;"
    out = bench.code_only(a)
    assert "count" not in out and out == bench.code_only(b)
    assert out == "int n = 1'000; int m = 2;"


def test_code_only_ignores_layout_and_comments_only():
    a = "template <int D>\n__global__ void k(float* p) {\n  p[0] = D;  // store\n}\n"
    b = "template <int D> __global__ void k(float* p) { /* note */ p[0] = D; }"
    c = "template <int D> __global__ void k(float* p) { p[1] = D; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)


def test_every_committed_profile_matches_its_sources():
    pdir = os.path.join(bench.ROOT, "profiles")
    names = [n for n in os.listdir(pdir) if n.endswith(".md")]
    assert names
    for n in names:
        units = bench.ATTENTION_UNITS if n.startswith("verify_attention") else None
        tag = n[:-3]
        assert bench.profiled_traffic(tag, units) is not None, n


def test_attention_bytes_and_flops_closed_form():
    case = synth.attention_case(0, B=2, L=4, Hq=6, Hkv=2, D=64, S_cap=64, prefix_len=[10, 3],
                                dtype="f16")
    prefix_kv = (10 + 3) * 2 * 64 * 2 * 2            # slots x heads x D x bytes x (K, V)
    block_in = (2 * 4 * 6 * 64 + 2 * 2 * 4 * 2 * 64) * 2
    appended = 2 * 2 * 4 * 2 * 64 * 2                # (K, V) x B x L x heads x D x bytes
    out = 2 * 4 * 6 * 64 * 2
    assert bench.attention_bytes(case) == prefix_kv + block_in + appended + out
    # visible (query, key) pairs: every query sees the prefix and the block up to itself
    pairs = sum(p * 4 + (1 + 2 + 3 + 4) for p in (10, 3))
    assert bench.attention_flops(case) == 2 * 2 * pairs * 6 * 64
    assert isinstance(bench.attention_bytes(case), (int, np.integer))
