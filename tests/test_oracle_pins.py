"""The fp64 oracle against the facts that pin it (pages' values, closed forms,
invariants).  CPU only."""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_matches_torch_fp64_on_tiny_shapes(orc):
    """Extra cross-check (not a pin by itself): torch's own fp64 softmax and
    matmul on tiny shapes, causal and non-causal."""
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(7)
    for (B, H, N, d) in [(1, 1, 1, 1), (1, 2, 5, 3), (2, 1, 16, 8), (1, 1, 33, 64)]:
        q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
        k = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
        v = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
        scale = d ** -0.5
        for causal in (False, True):
            s = (q @ k.transpose(-1, -2)) * scale
            if causal:
                s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
            o_t = torch.softmax(s, dim=-1) @ v
            lse_t = torch.logsumexp(s, dim=-1)
            o, lse = orc.attention_fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal=causal,
                                       threads=2)
            np.testing.assert_allclose(o, o_t.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lse_t.numpy(), rtol=0, atol=1e-12)


def test_rejects_bad_arguments(orc):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(oracle.OracleError):
        orc.attention_rows(q, q, q, [(0, 4)], 1.0)  # row index out of range
    with pytest.raises(oracle.OracleError):
        orc.attention_rows(q, q, q, [(1, 0)], 1.0)  # head index out of range
    with pytest.raises(oracle.OracleError):
        orc.online_row([1.0, 2.0], [1.0, 1.0], [(0, 1)])  # blocks miss a score
    with pytest.raises(oracle.OracleError):
        orc.online_row([1.0, 2.0], [1.0, 1.0], [(0, 2), (1, 1)])  # overlap
