"""Pins for the oracle's value helpers against library routines: bf16 decode
and bf16 rounding against torch's bfloat16 conversions (round to nearest,
ties to even, from fp32 values), the activation-rounding choice per dtype,
and the capacity formula's use of the fp32 capacity factor."""
import numpy as np
import torch

from oracle import moe_oracle as O


def test_decode_bf16_bits_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF            # skip inf / NaN patterns
    bits = bits[finite]
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.decode(bits), ref)


def test_round_bf16_matches_torch_rne():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(200_000) * 10.0 ** rng.integers(-30, 30, 200_000),
        # exact halfway cases: 8 significant bits plus a trailing 1 bit
        (rng.integers(128, 256, 10_000) * 2 + 1) * 2.0 ** rng.integers(-100, 100, 10_000),
    ]).astype(np.float32)
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_bf16(v.astype(np.float64)), ref)
    # ties go to the even neighbour
    assert O.round_bf16(np.float64(1.0 + 2.0 ** -8)) == 1.0
    assert O.round_bf16(np.float64(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6


def test_activation_rounding_per_dtype():
    v = np.array([1.0 + 2.0 ** -12, np.pi])
    assert np.array_equal(O.act_rounder("bf16", True)(v), O.round_bf16(v))
    assert np.array_equal(O.act_rounder("f32", True)(v), v.astype(np.float32).astype(np.float64))
    assert np.array_equal(O.act_rounder("bf16", False)(v), v)
    assert np.array_equal(O.f32_rounder(True)(v), v.astype(np.float32).astype(np.float64))


def test_capacity_takes_the_fp32_capacity_factor():
    # the layer receives CF as fp32: 0.1f = 0.100000001490116..., so
    # CF * 1000 * 1 / 1 is just above 100 and the capacity is 101
    assert O.capacity(0.1, 1000, 1, 1) == 101
    assert float(np.float32(0.1)) * 1000 > 100
