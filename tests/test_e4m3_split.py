"""The two-term e4m3 form of a bf16 query row that the FP8-key decode feeds its e4m3 MMAs.

The kernel scales a query row by a power of two that puts its largest magnitude in [128, 256) and
writes each element x as hi + lo, hi = e4m3(x), lo = e4m3(x - hi) (round to nearest even).  The
claim it rests on: a bf16 value has eight significant bits and an e4m3 term holds four, so hi + lo
equals x exactly whenever x is at least 2^-10 of the row's largest magnitude (the remainder then
stays above e4m3's smallest subnormal, 2^-9), and smaller elements are off by at most 2^-10 in
those scaled units (2^-18 of the largest).  Checked here on every positive bf16 value from 2^-40 to
the largest that rounds into [128, 256), with PyTorch's e4m3 conversion as the rounding.
"""

import torch


def _e4m3(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).to(torch.float64)


def _all_bf16(lo_exp: int, hi_exp: int) -> torch.Tensor:
    """Every positive bf16 value in [2^lo_exp, 2^hi_exp), as float64."""
    bits = torch.arange(0, 1 << 15, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16).to(torch.float64)
    return vals[(vals >= 2.0 ** lo_exp) & (vals < 2.0 ** hi_exp)]


def test_two_e4m3_terms_hold_a_bf16_value_exactly_down_to_2_pow_minus_10_of_the_row_maximum():
    x = _all_bf16(-2, 8)  # the scaled row: largest magnitude in [128, 256), elements >= 2^-10 of it
    hi = _e4m3(x)
    lo = _e4m3(x - hi)
    assert torch.equal(hi + lo, x)
    assert torch.equal(-(_e4m3(-x) + _e4m3(-x - _e4m3(-x))), x)  # and with the sign


def test_smaller_elements_err_by_at_most_2_pow_minus_10_in_scaled_units():
    x = _all_bf16(-40, -2)
    hi = _e4m3(x)
    lo = _e4m3(x - hi)
    err = (hi + lo - x).abs()
    assert float(err.max()) <= 2.0 ** -10


def test_the_row_scale_puts_the_largest_magnitude_in_128_256():
    # 2^(134 - biased exponent of amax): amax in [2^(e - 127), 2^(e - 126)) lands in [128, 256).
    amax = _all_bf16(-100, 100)
    e = (amax.to(torch.float32).view(torch.int32) >> 23) & 0xFF
    scaled = amax * torch.pow(2.0, (134 - e).to(torch.float64))
    assert bool(((scaled >= 128) & (scaled < 256)).all())
    # the largest bf16 value below 256 still has an exact two-term form (hi may round up to 256)
    top = scaled.max().reshape(1)
    assert torch.equal(_e4m3(top) + _e4m3(top - _e4m3(top)), top)
