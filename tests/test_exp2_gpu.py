"""GPU pins of the software exp2 (FMA-pipe polynomial) against fp64 2^x, at
the accuracy M4.6 "FlashAttention-3/4 Hardware Pipelines" 0x09 states for a
degree-3 range-reduced exp2: maximum relative fp32 error near 9e-5 on [0, 1),
and, once rounded to bf16 as the kernels consume it, at most one bf16 code
from the correctly rounded value (the pages' mean post-bf16 error 1.41e-3 is
that of ideal bf16 rounding)."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_gb300 import gbattn_exp2_paths

pytestmark = pytest.mark.gpu


def _grid():
    frac = np.linspace(0.0, 1.0, 1 << 16, endpoint=False)
    wide = np.linspace(-126.0, 20.0, 1 << 18)
    x = np.concatenate([frac, wide, -frac * 40]).astype(np.float32)
    return x[: len(x) // 2 * 2]


def test_software_exp2_relative_error():
    x = _grid()
    y_poly, y_hw = gbattn_exp2_paths(torch.from_numpy(x).cuda())
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y_poly.cpu().numpy().astype(np.float64) / ref - 1.0)
    assert rel.max() <= 1.0e-4, rel.max()
    on01 = (x >= 0) & (x < 1)
    assert 3e-5 <= rel[on01].max() <= 1.0e-4       # a degree-3 fit: not exact, not worse
    rel_hw = np.abs(y_hw.cpu().numpy().astype(np.float64) / ref - 1.0)
    assert rel_hw.max() <= 1e-6


def test_software_exp2_after_bf16_rounding():
    x = _grid()
    y_poly, _ = gbattn_exp2_paths(torch.from_numpy(x).cuda())
    ref = torch.from_numpy(np.exp2(x.astype(np.float64))).to(torch.bfloat16)  # correctly rounded
    got = y_poly.cpu().to(torch.bfloat16)
    codes = lambda t: t.view(torch.int16).numpy().astype(np.int64)  # noqa: E731 (positive values)
    assert np.abs(codes(got) - codes(ref)).max() <= 1
    rel = np.abs(got.double().numpy() / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.mean() <= 2.0e-3


def test_software_exp2_clamp():
    x = torch.tensor([-1000.0, -127.0, -126.0, 127.0, 0.0, 1.0], device="cuda")
    y, _ = gbattn_exp2_paths(x)
    y = y.cpu().numpy()
    assert y[0] == y[1] == y[2] == np.float32(2.0 ** -126)
    assert abs(y[3] / 2.0 ** 127 - 1) <= 1e-4 and y[4] == 1.0 and y[5] == 2.0
