"""The error metrics the GPU parity tests use, checked on the CPU."""
import numpy as np

import parity_util as pu
from exact_io_aware_29_gb300 import synth


def test_bf16_half_ulp_is_half_the_spacing():
    # bf16 keeps 8 significant bits: the spacing at 1 is 2^-7, at 4.5 it is 2^-5
    assert pu.bf16_half_ulp(1.0) == 2.0 ** -8
    assert pu.bf16_half_ulp(-1.99) == 2.0 ** -8
    assert pu.bf16_half_ulp(4.5) == 2.0 ** -6
    assert pu.bf16_half_ulp(0.0) == 2.0 ** -134     # subnormal spacing 2^-133
    # every value rounds to bf16 within half an ulp (the input rounding routine)
    x = np.random.default_rng(1).standard_normal(10000) * 10.0 ** np.random.default_rng(2).uniform(-20, 20, 10000)
    r = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(x.astype(np.float32)))
    assert np.all(np.abs(r - x.astype(np.float32)) <= pu.bf16_half_ulp(x) * (1 + 2.0 ** -7))


def test_o_err_discounts_only_the_output_rounding():
    ref = np.array([4.51, 0.3, -2.0])
    exact_rounded = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(ref.astype(np.float32)))
    assert pu.o_err(exact_rounded, ref) <= 0.0           # rounding alone costs nothing
    off = exact_rounded + np.array([0.0, 0.011 + pu.bf16_half_ulp(0.3), 0.0])
    assert pu.o_err(off, ref) > 0.01                      # anything beyond it counts
    assert pu.o_err(np.array([np.inf]), np.array([np.inf])) <= 0.0
