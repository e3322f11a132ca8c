"""The transpose's slot -> (query, chunk start) division: below 2^24 the library
takes q = trunc(float32(n) * float32(1/d)) and corrects it once by the sign and
size of n - q d.  This checks that arithmetic (float32 round-to-nearest product,
as the device computes it) against exact integer division: the estimate is
within one of the quotient and the corrected value is exact, on random values,
every multiple of d +-1 and the ends of the range."""
import numpy as np
import pytest

LIMIT = 1 << 24


def _quot(n: np.ndarray, d: int) -> np.ndarray:
    inv = np.float32(1.0) / np.float32(d)
    q = np.trunc(n.astype(np.float32) * inv).astype(np.int64)
    assert np.all(np.abs(q - n // d) <= 1)
    r = n - q * d
    return np.where(r < 0, q - 1, np.where(r >= d, q + 1, q))


@pytest.mark.parametrize("d", [1, 2, 3, 7, 31, 32, 33, 47, 48, 64, 100, 128, 255, 256,
                               1000, 1024, 4096, 65535, 65536, (1 << 20) + 7])
def test_float_reciprocal_division_is_exact(d):
    rng = np.random.default_rng(d)
    n = rng.integers(0, LIMIT, size=1 << 20, dtype=np.int64)
    m = np.arange(0, LIMIT, d, dtype=np.int64)[: 1 << 18]
    edges = np.concatenate([m, m[1:] - 1, np.minimum(m + 1, LIMIT - 1),
                            np.arange(LIMIT - 4096, LIMIT, dtype=np.int64),
                            np.arange(0, 4096, dtype=np.int64)])
    for x in (n, edges):
        assert np.array_equal(_quot(x, d), x // d)
