"""The output tolerance rule of the parity tests, checked on the CPU.

The attention output must be within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the
oracle wherever a T value can be that close, i.e. wherever half an ulp of T at
the reference value fits in the tolerance.  Only above that (bf16 |o| >= 4,
fp16 |o| >= 8) is a faithfully rounded output (less than one ulp away)
accepted instead."""
import numpy as np
import pytest
import torch

from gqa_cases import TOL, ulp, within_tolerance


def test_tolerance_applies_below_the_floor_range():
    # bf16 |o| in [2, 4): half an ulp is 2^-7 = 0.0078 < 0.01, so 0.01 holds
    ok, n = within_tolerance(np.array([0.0099, 0.0101, 0.0101]), np.array([3.0, 3.0, -2.5]), "bf16")
    assert ok.tolist() == [True, False, False] and n == 0
    # fp16 |o| in [4, 8): half an ulp is 2^-9 = 0.00195 < 0.002
    ok, n = within_tolerance(np.array([0.0019, 0.0025]), np.array([5.0, -7.9]), "fp16")
    assert ok.tolist() == [True, False] and n == 0


def test_faithful_rounding_above_it():
    # bf16 at 4.72: ulp 2^-5 = 0.03125; the correctly rounded value 4.71875 is
    # 0.00125 away, and anything closer than one ulp passes
    assert float(torch.tensor(4.72, dtype=torch.float64).to(torch.bfloat16)) == 4.71875
    ok, n = within_tolerance(np.array([0.00125, 0.02, 0.0313]), np.array([4.72, 4.72, 4.72]), "bf16")
    assert ok.tolist() == [True, True, False] and n == 3
    # fp16 at 9.0: ulp 2^-7 = 0.0078
    ok, n = within_tolerance(np.array([0.005, 0.008]), np.array([9.0, -9.0]), "fp16")
    assert ok.tolist() == [True, False] and n == 2


def test_ulp_of_both_types():
    assert ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert ulp(np.array([3.9]), "bf16")[0] == 2.0 ** -6
    assert ulp(np.array([1.0]), "fp16")[0] == 2.0 ** -10
    assert ulp(np.array([-8.5]), "fp16")[0] == 2.0 ** -7
    # the floor starts exactly where half an ulp exceeds the tolerance
    for dtype, start in (("bf16", 4.0), ("fp16", 8.0)):
        below = np.nextafter(start, 0.0)
        assert 0.5 * ulp(np.array([below]), dtype)[0] <= TOL[dtype] < 0.5 * ulp(np.array([start]), dtype)[0]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_correctly_rounded_outputs_always_pass(dtype):
    """The rule never rejects a T output that is the reference rounded to
    nearest (the best any kernel can do)."""
    gen = torch.Generator().manual_seed(5)
    ref = torch.randn(200000, generator=gen, dtype=torch.float64) * 6.0
    t = {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]
    got = ref.to(torch.float32).to(t).to(torch.float64)
    ok, _ = within_tolerance(np.abs(got - ref).numpy(), ref.numpy(), dtype)
    assert ok.all()
