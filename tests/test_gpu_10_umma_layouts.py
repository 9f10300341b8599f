"""The decode kernel's two tcgen05 contractions, one tile each, against a plain
float64 matrix product (operand layouts, descriptors and TMEM lane mapping).

Score form: S[96 x 64] = Q[96 x 576] . T^T with Q staged by one 3-D TMA box and
copied into TMEM (24 heads per 32-lane quarter) and the 64-token page T staged by
one 3-D TMA box.  PV form:
O[512 x 96] = T[:, :512]^T . P^T with the page (one 3-D box of chunks 0..7) as an
MN-major operand and P^T written by threads in the 128-byte-swizzled K-major
layout.  Products of bf16 values are exact, so the only
difference from float64 is f32 accumulation."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.gpu_common import dump

pytestmark = pytest.mark.gpu


def _check(d, ref, absref, name):
    d = d.double().cpu().numpy()
    ref = ref.cpu().numpy()
    bound = 64 * 2.0**-24 * absref.cpu().numpy() + 1e-30
    ok = np.all(np.abs(d - ref) <= bound)
    if not ok:
        dump(name, d=d, ref=ref)
    assert ok, f"{name}: max |diff| / bound = {np.max(np.abs(d - ref) / bound):.3g}"


def test_score_contraction_tile(gpu_lib):
    g = torch.Generator(device="cuda").manual_seed(1)
    a = torch.randn(96, 576, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(64, 576, generator=g, device="cuda").to(torch.bfloat16)
    d = torch.full((128, 64), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.diag_umma(0, a, b, d)
    torch.cuda.synchronize()
    t = b.double()
    ref = a.double() @ t.T
    absref = a.double().abs() @ t.abs().T
    _check(d[:96], ref, absref, "diag_score")


def test_pv_contraction_tile(gpu_lib):
    g = torch.Generator(device="cuda").manual_seed(2)
    p = torch.rand(96, 64, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(64, 576, generator=g, device="cuda").to(torch.bfloat16)
    d = torch.full((512, 96), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.diag_umma(1, p, b, d)
    torch.cuda.synchronize()
    t = b[:, :512].double()
    ref = t.T @ p.double().T
    absref = t.abs().T @ p.double().abs().T
    _check(d, ref, absref, "diag_pv")
