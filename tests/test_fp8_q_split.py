"""The fp8 decode kernel multiplies the raw E4M3 K codes with Q split into two
E4M3 terms: q * 2^e = hi + lo, with 2^e chosen per query head so that
max|q| * 2^e lies in (224, 448], hi the nearest E4M3 value to q * 2^e and lo
the nearest E4M3 value to what is left. This pins the property the kernel
relies on, with torch's own E4M3 type (no GPU): for bf16 q the split is exact
wherever the scaled value is at least 2^-2, and off by at most 2^-10 (scaled)
below that, where lo falls under the E4M3 subnormal step 2^-9."""
import math

import pytest
import torch

E4M3 = getattr(torch, "float8_e4m3fn", None)
pytestmark = pytest.mark.skipif(E4M3 is None, reason="torch without float8_e4m3fn")


def split(q):
    amax = q.abs().max().item()
    e = math.floor(math.log2(448.0 / amax))
    if amax * 2.0 ** e > 448.0:
        e -= 1
    x = q * 2.0 ** e
    hi = x.to(E4M3).float()
    lo = (x - hi).to(E4M3).float()
    return x, hi, lo, e


@pytest.mark.parametrize("seed", range(4))
def test_hi_plus_lo_is_the_scaled_bf16_row(seed):
    g = torch.Generator().manual_seed(seed)
    for trial in range(300):
        scale = 10.0 ** (torch.rand(1, generator=g).item() * 12 - 6)
        q = torch.randn(128, generator=g) * scale
        if trial % 5 == 0:
            q[torch.randint(0, 128, (12,), generator=g)] *= 1e-3   # a few tiny entries
        q = q.to(torch.bfloat16).float()
        x, hi, lo, e = split(q)
        assert 224.0 < x.abs().max().item() <= 448.0
        err = (hi + lo - x).abs()
        big = x.abs() >= 0.25
        assert torch.equal(hi[big] + lo[big], x[big])
        assert err.max().item() <= 2.0 ** -10


def test_scaled_row_never_saturates_and_zero_rows_stay_zero():
    q = torch.tensor([448.0, -448.0, 1.0, 0.0]).to(torch.bfloat16).float()
    x, hi, lo, e = split(q)
    assert e == 0 and torch.equal(hi + lo, x)
    z = torch.zeros(128)
    assert torch.equal(z.to(E4M3).float(), z)
