"""Pins for the oracle's number formats: RNE encoding and exact decoding of binary16 and
bfloat16, checked against numpy's float16 cast and torch's bfloat16 cast (library routines),
on random values plus ties, subnormals, overflow edges, infinities and NaN."""
import numpy as np
import torch

import oracle


def _specials():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e-8, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), 6.1e-5, 1e30, -1e30,
            3.3895313892515355e38, 1.1754943508222875e-38, 9.2e-41, float("inf"), float("-inf")]
    # exact ties between neighbouring f16 / bf16 values
    for e in (-3, 0, 5):
        base = 2.0 ** e
        vals += [base * (1 + 2.0 ** -11), base * (1 + 3 * 2.0 ** -11), base * (1 + 2.0 ** -8),
                 base * (1 + 3 * 2.0 ** -8)]
    return np.array(vals, dtype=np.float32)


def _random(n=20000, seed=7):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(n).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 6, n).astype(np.float32)
    bits = rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    bits = bits[np.isfinite(bits)]
    return np.concatenate([a, bits, _specials()]).astype(np.float32)


def test_encode_f16_matches_numpy():
    x = _random()
    got = oracle.encode(x, "f16")
    want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_encode_bf16_matches_torch():
    x = _random(seed=11)
    got = oracle.encode(x, "bf16")
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_encode_nan_is_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    for dt in ("f16", "bf16"):
        back = oracle.decode(oracle.encode(x, dt), dt)
        assert np.all(np.isnan(back))


def test_decode_exact():
    allbits = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    d16 = oracle.decode(allbits, "f16")
    ref16 = allbits.view(np.float16).astype(np.float64)
    same = (d16 == ref16) | (np.isnan(d16) & np.isnan(ref16))
    assert same.all()
    dbf = oracle.decode(allbits, "bf16")
    refbf = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (dbf == refbf) | (np.isnan(dbf) & np.isnan(refbf))
    assert same.all()
