"""The oracle's IEEE round-to-nearest-even into fp16 / bf16, pinned against
torch's and numpy's own conversions and against the definition (nearest
member, ties to even) checked by brute force."""
import numpy as np
import pytest
import torch

from oracle import rounding as R


def _stratified_f32(low_bits: int, extra_lows, seed: int) -> np.ndarray:
    """Every pattern of the high (32 - low_bits) bits, combined with the low
    patterns that decide rounding: zero, one, just below / at / just above
    the tie, all ones, plus random ones."""
    hi = np.arange(1 << (32 - low_bits), dtype=np.uint64) << np.uint64(low_bits)
    half = 1 << (low_bits - 1)
    rng = np.random.default_rng(seed)
    lows = [0, 1, half - 1, half, half + 1, (1 << low_bits) - 1, *extra_lows]
    lows += list(rng.integers(0, 1 << low_bits, size=4))
    bits = (hi[:, None] | np.array(lows, dtype=np.uint64)[None, :]).reshape(-1).astype(np.uint32)
    return bits.view(np.float32)


def _torch_bits(x: np.ndarray, dt) -> np.ndarray:
    return torch.from_numpy(x).to(dt).view(torch.int16).numpy().view(np.uint16)


def _same_or_both_nan(a_bits, b_bits, decode):
    a, b = decode(a_bits), decode(b_bits)
    nan = np.isnan(a)
    assert np.array_equal(nan, np.isnan(b))
    assert np.array_equal(a_bits[~nan], b_bits[~nan])


def test_f32_to_bf16_matches_torch_on_every_high_half():
    x = _stratified_f32(16, [0x7FFF, 0x8000], seed=1)
    _same_or_both_nan(R.f32_to_bf16_bits(x), _torch_bits(x, torch.bfloat16), R.bf16_bits_to_f64)


def test_f32_to_f16_matches_torch_on_every_high_pattern():
    # 13 low bits decide rounding of normal fp16 results; subnormal results
    # drop more, which the random low patterns and the full high sweep cover.
    x = _stratified_f32(13, [0x0FFF, 0x1000], seed=2)
    _same_or_both_nan(R.f32_to_f16_bits(x), _torch_bits(x, torch.float16), R.f16_bits_to_f64)


def test_f32_to_f16_subnormal_range_exhaustive_band():
    # every float with exponent field 100..113 (results in fp16's subnormal
    # and lowest normal binades) and a dense sample of mantissas
    rng = np.random.default_rng(3)
    exps = np.arange(100, 114, dtype=np.uint32)
    mants = np.concatenate([np.arange(0, 1 << 23, 977, dtype=np.uint32),
                            rng.integers(0, 1 << 23, 20000).astype(np.uint32)])
    bits = ((exps[:, None] << np.uint32(23)) | mants[None, :]).reshape(-1)
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    x = bits.view(np.float32)
    assert np.array_equal(R.f32_to_f16_bits(x), _torch_bits(x, torch.float16))


def test_f64_to_f16_one_rounding_matches_numpy():
    rng = np.random.default_rng(4)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        np.ldexp(rng.integers(1, 1 << 12, 100000).astype(np.float64) + 0.5, rng.integers(-36, 5, 100000)),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 + 2.0 ** -60],
    ])
    ours = R.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)  # numpy rounds double to half directly
    assert np.array_equal(ours, ref)


def _bf16_neighbours_ok(x: np.ndarray, bits: np.ndarray):
    """Definition check: the result is a nearest bf16 member; on a tie its
    last significand bit is 0."""
    val = R.bf16_bits_to_f64(bits)
    fin = np.isfinite(val)
    b = bits[fin].astype(np.int64)
    v = val[fin]
    xx = x[fin]
    # neighbours one step away in the bit encoding (same sign side)
    up = R.bf16_bits_to_f64(np.clip(b + 1, 0, 0xFFFF).astype(np.uint16))
    dn = R.bf16_bits_to_f64(np.clip(b - 1, 0, 0xFFFF).astype(np.uint16))
    err = np.abs(xx - v)
    for nb in (up, dn):
        ok = ~np.isfinite(nb) | (np.sign(nb) != np.sign(v)) & (v != 0) | (np.abs(xx - nb) >= err)
        assert ok.all()
        tie = np.isfinite(nb) & (np.abs(xx - nb) == err) & (nb != v)
        assert ((b[tie] & 1) == 0).all()


def test_f64_to_bf16_is_nearest_ties_even():
    rng = np.random.default_rng(5)
    mant = rng.integers(1 << 52, 1 << 53, 300000, dtype=np.int64).astype(np.float64)
    x = np.ldexp(mant, rng.integers(-190, 70, 300000)) * np.where(rng.random(300000) < 0.5, -1, 1)
    # exact ties: 9 significant bits ending in 1
    ties = np.ldexp(rng.integers(256, 512, 20000).astype(np.float64) * 2 + 1, rng.integers(-140, 60, 20000))
    x = np.concatenate([x, ties, -ties])
    _bf16_neighbours_ok(x, R.f64_to_bf16_bits(x))


def test_f64_to_bf16_differs_from_double_rounding_through_f32():
    # a double just above a bf16 tie whose float32 rounding lands exactly on
    # the tie: rounding twice goes to even (down), once goes up.
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40])
    once = R.f64_to_bf16_bits(x)[0]
    twice = R.f32_to_bf16_bits(x.astype(np.float32))[0]
    assert R.bf16_bits_to_f64(np.array([once]))[0] == 1.0 + 2.0 ** -7
    assert R.bf16_bits_to_f64(np.array([twice]))[0] == 1.0


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_widening_is_exact_inverse(dt):
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    val = R.storage_to_f64(allbits, dt)
    fin = np.isfinite(val)
    tdt = torch.float16 if dt == "f16" else torch.bfloat16
    ref = torch.from_numpy(allbits.view(np.int16)).view(tdt).to(torch.float64).numpy()
    assert np.array_equal(val[fin], ref[fin])
    assert np.array_equal(np.isnan(val), np.isnan(ref))
    back = R.round_f64(val[fin], dt)
    assert np.array_equal(back, allbits[fin])
