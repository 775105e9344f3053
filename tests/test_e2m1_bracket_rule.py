"""The NVFP4 quantiser's rounding rule, checked in float32 arithmetic on the host.

The kernel converts two brackets of the exact quotient v = x / s with the hardware's RNE
E2M1 conversion: y_up = x * RN(RN(1/s) (1 + 2^-20)) and y_dn = x * RN(RN(1/s) (1 - 2^-20)).
Equal codes are taken as the code of v (RNE rounding is monotonic). Unequal codes send fp32
inputs to an exact path. For bf16 inputs the tie goes to the neighbour with a clear last bit.
Here numpy float32 stands in for the kernel's fp32 arithmetic, and an exact float64 RNE stands
in for the conversion. On values at, next to and away from every midpoint under every nonzero
UE4M3 scale, the rule must reproduce the exact rounding of v.
"""
import numpy as np

from oracle import formats

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _rne_index(v):
    """Exact RNE magnitude index of |v| on the E2M1 grid (satfinite): ties to the even index."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    idx = np.zeros(a.shape, dtype=np.int64)
    for i, m in enumerate(formats.E2M1_MIDS):
        idx += (a > m) | ((a == m) & (i % 2 == 1))
    return idx


def _to_bf16(x):
    """Round float32 values to bf16 (RNE), returned as float32."""
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return b.view(np.float32)


def _inputs(rng, s, n):
    pts = np.concatenate([formats.E2M1_MIDS, GRID])
    ties = (rng.choice(pts, n) * s).astype(np.float32)
    ulps = rng.integers(1, 64, n) * rng.choice([-1, 1], n)
    near = (ties.astype(np.float64) * (1 + ulps * 2.0 ** -24)).astype(np.float32)
    wide = (rng.standard_normal(n) * 2.0 * s).astype(np.float32)
    return [ties, near, wide]


def test_bracket_rule_reproduces_exact_rounding():
    rng = np.random.default_rng(3)
    scales = formats.decode_ue4m3(np.arange(1, 127, dtype=np.uint8)).astype(np.float32)
    for s in scales:
        inv = np.float32(1.0) / s                      # RN(1/s)
        inv_up = np.float32(inv * np.float32(1.0 + 2.0 ** -20))
        inv_dn = np.float32(inv * np.float32(1.0 - 2.0 ** -20))
        for x in _inputs(rng, float(s), 1500):
            for kind in ("fp32", "bf16"):
                xs = _to_bf16(x) if kind == "bf16" else x
                exact = _rne_index(xs.astype(np.float64) / float(s))
                up = _rne_index(xs * inv_up)
                dn = _rne_index(xs * inv_dn)
                same = up == dn
                assert np.array_equal(up[same], exact[same])  # equal brackets: the exact code
                assert np.all(np.abs(up - dn) <= 1)           # at most one midpoint between them
                if kind == "bf16":
                    even = np.where(up % 2 == 0, up, dn)       # the tie goes to the even neighbour
                    assert np.array_equal(even[~same], exact[~same])
