"""The FP8 decode's reading of q as two e4m3 parts ("Qwen2大模型架构解析与
vLLM优化实践" section 6.3 names fp8_e4m3fn; the split is this library's way
to keep the bf16 query exact against e4m3 codes): with 2^e putting the
head's largest |q| in [128, 256), hi = e4m3(q 2^e) and lo = e4m3(q 2^e - hi)
sum to q 2^e exactly for every scaled |q| >= 2^-2 -- every bf16 q within a
factor 2^9 of that maximum -- and within 2^-10 (half e4m3's subnormal step,
2^-17 of the maximum) below it.  (At 2^-3 the residue's last bit, 2^-10,
falls below the step: the split is not exact there.)  Checked here over every positive bf16 value of the range, with
torch's own round-to-nearest-even e4m3 conversion (independent of the
kernels)."""
import torch


def e4m3(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).to(torch.float32)


def all_bf16_between(lo: float, hi: float) -> torch.Tensor:
    bits = torch.arange(0, 1 << 15, dtype=torch.int32)  # every non-negative bf16
    v = (bits << 16).view(torch.float32)
    return v[(v >= lo) & (v < hi)]


def test_two_part_split_is_exact_near_the_maximum():
    # scaled values: the maximum in [128, 256), everything from 2^-2 up
    q = all_bf16_between(2.0 ** -2, 256.0)
    hi = e4m3(q)
    lo = e4m3(q - hi)
    assert torch.equal(hi + lo, q)
    assert torch.equal(-(e4m3(-q) + e4m3(-q - e4m3(-q))), q)  # and for negative values


def test_two_part_split_error_below_2_pow_minus_10_under_it():
    q = all_bf16_between(2.0 ** -30, 2.0 ** -2)
    hi = e4m3(q)
    lo = e4m3(q - hi)
    err = (hi + lo - q).abs()
    assert float(err.max()) <= 2.0 ** -10
    # the bound is reached: the parts cannot hold what lies below e4m3's step
    assert float(err.max()) == 2.0 ** -10


def test_power_of_two_scale_is_exact():
    # q * 2^e and back is exact for bf16 q (the kernel scales by 2^e, the
    # softmax by 2^-e) whatever e in [-126, 126] the head's maximum picks
    q = all_bf16_between(2.0 ** -20, 2.0 ** 20)
    for e in (-100, -7, 0, 7, 100):
        f = 2.0 ** e
        assert torch.equal((q * f) * (1.0 / f), q)
