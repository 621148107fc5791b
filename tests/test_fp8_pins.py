"""CPU pins of the E4M3 codebook the FP8 tests decode through (torch's
float8_e4m3fn), against the format facts M4.6 "FlashAttention-3/4 Hardware
Pipelines" 0x06 states: largest finite magnitude 448, smallest positive
subnormal 2^-9, three fraction bits."""
import numpy as np
import torch


def test_e4m3_range_and_spacing():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = codes.float().numpy()
    finite = vals[np.isfinite(vals)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = np.sort(finite[finite > 0])
    assert pos[0] == 2.0 ** -9
    # three fraction bits: 8 codes per binade above the subnormals
    assert np.all(np.isin([1.0, 1.125, 1.25, 1.875, 2.0, 2.25], pos))
    assert 1.0625 not in pos
    # the only non-finite codes are the two NaNs (no infinities in E4M3FN)
    assert np.isnan(vals).sum() == 2 and not np.isinf(vals).any()


def test_e4m3_round_to_nearest_even():
    x = torch.tensor([1.0625, 1.1875, 448.0, 2.0 ** -10, 3 * 2.0 ** -10])
    y = x.to(torch.float8_e4m3fn).float().tolist()
    assert y == [1.0, 1.25, 448.0, 0.0, 2.0 ** -8]
