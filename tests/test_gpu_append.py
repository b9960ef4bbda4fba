"""lcsw_append_token on the GPU: each sequence's newest row of k_idx, K and V
written from the packed staging rows, bit for bit, and nothing else (the
plain definition is the numpy assignment below)."""
import numpy as np
import pytest
import torch

import long_context_sparse_weighted_b300 as lcsw
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _bits(shape, rng):
    return rng.integers(0, 1 << 16, shape, dtype=np.uint16)


@pytest.mark.parametrize("d_idx,d_qk,d_v", [(64, 128, 128), (64, 192, 128), (64, 576, 0)])
def test_append_token_writes_the_newest_rows(d_idx, d_qk, d_v):
    rng = np.random.default_rng(700 + d_qk)
    B, L = 5, 300
    seq = np.array([300, 1, 0, 157, 64], np.int32)
    k_idx, K = _bits((B, L, d_idx), rng), _bits((B, L, d_qk), rng)
    V = _bits((B, L, d_v), rng) if d_v else None
    rows = _bits((B, d_idx + d_qk + d_v), rng)
    t16 = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    gk, gK = t16(k_idx), t16(K)
    gV = t16(V) if d_v else None
    lcsw.append_token(t16(rows), dev(seq), gk, gK, gV)
    torch.cuda.synchronize()
    for b in range(B):
        if seq[b] > 0:
            t = seq[b] - 1
            k_idx[b, t] = rows[b, :d_idx]
            K[b, t] = rows[b, d_idx:d_idx + d_qk]
            if d_v:
                V[b, t] = rows[b, d_idx + d_qk:]
    back = lambda g: g.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(back(gk), k_idx)
    assert np.array_equal(back(gK), K)
    if d_v:
        assert np.array_equal(back(gV), V)
