"""The log-sum-exp combine entry point on the GPU against the oracle's merge, and
the tree law on the device: any permutation of the partials merges to the same result."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import check_lse, check_out
from long_context_decode_04_b300 import ta

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _partials(R, N, D, seed, empty_frac=0.1):
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.normal(0, 3, (R, N))
    l = rng.uniform(0.5, 50, (R, N))
    o = rng.normal(0, 1, (R, N, D)) * l[..., None]
    empty = rng.random((R, N)) < empty_frac
    m[empty] = -np.inf
    l[empty] = 0
    o[empty] = 0
    return m.astype(np.float32), l.astype(np.float32), o.astype(np.float32)


@pytest.mark.parametrize("N", [1, 2, 37, 64, 65, 4096, 5000])
@pytest.mark.parametrize("D", [64, 128])
def test_combine_matches_oracle(N, D):
    R = 9
    m, l, o = _partials(R, N, D, seed=N * 7 + D)
    ro, rl = oracle.combine(m.astype(np.float64), l.astype(np.float64), o.astype(np.float64))
    out, lse = ta.combine(*(torch.from_numpy(a).to(DEV) for a in (m, l, o)))
    torch.cuda.synchronize()
    check_out(out.cpu().numpy(), ro, bf16=False)
    check_lse(lse.cpu().numpy(), rl)
    out_b, _ = ta.combine(*(torch.from_numpy(a).to(DEV) for a in (m, l, o)), out_dtype=torch.bfloat16)
    check_out(out_b.float().cpu().numpy(), ro, bf16=True)


@pytest.mark.parametrize("N", [5, 64, 300])
def test_combine_permutation_invariance(N):
    R, D = 4, 128
    m, l, o = _partials(R, N, D, seed=100 + N)
    out, lse = ta.combine(*(torch.from_numpy(a).to(DEV) for a in (m, l, o)))
    rng = np.random.Generator(np.random.PCG64(N))
    for _ in range(3):
        perm = rng.permutation(N)
        out2, lse2 = ta.combine(*(torch.from_numpy(np.ascontiguousarray(a[:, perm])).to(DEV) for a in (m, l, o)))
        assert torch.max(torch.abs(out - out2)).item() < 1e-5
        assert torch.max(torch.abs(lse - lse2)).item() < 1e-5


def test_combine_all_empty_row():
    R, N, D = 3, 70, 64
    m, l, o = _partials(R, N, D, seed=5)
    m[1] = -np.inf
    l[1] = 0
    o[1] = 0
    out, lse = ta.combine(*(torch.from_numpy(a).to(DEV) for a in (m, l, o)))
    assert torch.all(out[1] == 0) and torch.isneginf(lse[1])
    assert torch.isfinite(lse[0]) and torch.isfinite(lse[2])


def test_combine_of_oracle_chunk_partials_equals_single_pass():
    """Partials of real chunks (from the oracle) merged on the device give the attention result."""
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, S, D = 1, 4, 2, 900, 128
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    bounds = [0, 1, 100, 100, 450, 899, 900]
    parts = [oracle.decode_partials(q, k, v, 0.09, 0, h, bounds) for h in range(Hq)]
    m = np.stack([p[0] for p in parts]).astype(np.float32)
    l = np.stack([p[1] for p in parts]).astype(np.float32)
    o = np.stack([p[2] for p in parts]).astype(np.float32)
    out, lse = ta.combine(*(torch.from_numpy(a).to(DEV) for a in (m, l, o)))
    ro, rl = oracle.decode(q, k, v, 0.09)
    check_out(out.cpu().numpy(), ro, bf16=False)
    check_lse(lse.cpu().numpy(), rl)
