"""Shared helpers of the GPU parity tests: device copies and the tolerance.

Tolerance (the stated bar for projections): 2e-3 for bf16 / f16 outputs and
1e-5 for fp32 outputs, as a max relative error against the fp64 oracle r:

    err = max_i  max(0, |y_i - r_i| - h_i) / max(|r_i|, rms(r))

where h_i is half a unit in the last place of the output format at r_i. The
output cast itself is allowed its half ulp: bf16 carries 8 significant bits,
so rounding alone can move a value by up to 2^-8 (3.9e-3) relative, which no
2e-3 bound can contain; the bar applies to everything else (the fp32
accumulation, the dequantization, the group folding). Relative error is taken
against max(|r_i|, rms(r)) so that outputs near zero, where any relative
measure is undefined, are judged against the typical output magnitude.
"""
from __future__ import annotations

import numpy as np
import torch

from speculative_block_draft_02_gb300 import synth

TOL = {"bf16": 2e-3, "f16": 2e-3, "f32": 1e-5}
_FRAC_BITS = {"bf16": 7, "f16": 10, "f32": 23}
TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
ORACLE_DT = {"bf16": 0, "f16": 1, "f32": 2}


def half_ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    _, e = np.frexp(np.abs(v))                  # |v| = f * 2^e, f in [0.5, 1)
    h = np.ldexp(1.0, e - 2 - _FRAC_BITS[dtype])
    if dtype == "f16":
        h = np.maximum(h, 2.0 ** -25)          # subnormal spacing
    return h


def proj_error(y: np.ndarray, r: np.ndarray, dtype: str) -> float:
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 1.0
    scale = np.maximum(np.abs(r), rms if rms > 0 else 1.0)
    h = half_ulp(np.maximum(np.abs(r), np.abs(y)), dtype)
    excess = np.maximum(np.abs(y - r) - h, 0.0) / scale
    return float(excess.max()) if excess.size else 0.0


def assert_proj_close(y, r, dtype: str):
    err = proj_error(y, r, dtype)
    assert err <= TOL[dtype], "max relative error %.3e exceeds %.1e (%s)" % (err, TOL[dtype], dtype)
    return err


def to_dev_act(x_bits: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x_bits, dtype=np.float32)).cuda()
    t = torch.from_numpy(x_bits.view(np.int16).copy())
    return t.view(TORCH_DT[dtype]).cuda()


def to_dev_weights(w: synth.W4Weights):
    qw = torch.from_numpy(w.qw.view(np.int32).copy()).cuda()
    s = torch.from_numpy(w.scales.view(np.int16).copy()).cuda()
    b = torch.from_numpy(w.biases.view(np.int16).copy()).cuda()
    return qw, s, b


def out_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


# Canary guard regions (a stand-in for a memory checker): an output handed to a
# kernel is a view into a larger device buffer whose bytes on both sides hold a
# known pattern; check() fails if any of them changed, i.e. if the kernel wrote
# outside the tensor it was given.
GUARD_BYTES = 4096      # on each side; keeps the tensor 256-byte aligned
_CANARY = 0xA5


class Guarded:
    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((n + 2 * GUARD_BYTES,), _CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
        if fill is not None:
            if isinstance(fill, torch.Tensor):
                self.t.copy_(fill)
            else:
                self.t.fill_(fill)

    def check(self):
        torch.cuda.synchronize()
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.n:]
        assert bool((head == _CANARY).all()) and bool((tail == _CANARY).all()), \
            "a kernel wrote outside the %d-byte tensor it was given" % self.n
