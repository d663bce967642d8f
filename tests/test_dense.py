"""Dense causal gated attention (the full-attention control branch of the
break-even measurement) on the GPU against the fp64 oracle with every
position kept, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import check_outputs, to_host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


@pytest.mark.parametrize("L,Hq,d", [(700, 16, 128), (333, 20, 64), (9, 3, 128)])
def test_dense_matches_oracle(sa, L, Hq, d):
    g = torch.Generator().manual_seed(L)
    q = (torch.randn((L, Hq, d), generator=g) / math.sqrt(d) * 2).to(torch.bfloat16)
    k = (torch.randn((L, d), generator=g) / math.sqrt(d) * 2).to(torch.bfloat16)
    v = (torch.randn((L, d), generator=g) / math.sqrt(d)).to(torch.bfloat16)
    gate = torch.randn((L, Hq), generator=g)
    scale = 1 / math.sqrt(d)
    out = sa.attention_dense_causal(q.to(DEV), k.to(DEV), v.to(DEV), gate.to(DEV), scale)
    torch.cuda.synchronize()
    idx = np.full((L, L), -1, dtype=np.int32)
    for t in range(L):
        idx[t, :t + 1] = np.arange(t + 1)
    ref = oracle.attend(q, k, v, d, d, d, gate, np.arange(L), np.zeros(L), idx, scale)
    check_outputs(to_host(out).double().numpy(), ref, torch.bfloat16, "dense out")


def _dense_case(sa, L, Hq, d, rows, q_gain=2.0, k_ramp=0.0, seed=None):
    g = torch.Generator().manual_seed(L if seed is None else seed)
    q = (torch.randn((L, Hq, d), generator=g) / math.sqrt(d) * q_gain).to(torch.bfloat16)
    ramp = 1.0 + k_ramp * torch.arange(L, dtype=torch.float32)[:, None] / L
    k = (torch.randn((L, d), generator=g) / math.sqrt(d) * 2 * ramp).to(torch.bfloat16)
    v = (torch.randn((L, d), generator=g) / math.sqrt(d)).to(torch.bfloat16)
    gate = torch.randn((L, Hq), generator=g)
    scale = 1 / math.sqrt(d)
    out = sa.attention_dense_causal(q.to(DEV), k.to(DEV), v.to(DEV), gate.to(DEV), scale)
    torch.cuda.synchronize()
    assert sa.device_errors(reset=True) == 0
    rows = np.asarray(rows)
    idx = np.full((len(rows), L), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        idx[i, :t + 1] = np.arange(t + 1)
    ref = oracle.attend(q, k, v, d, d, d, gate, rows, np.zeros(len(rows)), idx, scale)
    check_outputs(to_host(out)[rows].double().numpy(), ref, torch.bfloat16, "dense out")


def test_dense_tensor_core_single_cta(sa):
    # 9 queries: one CTA of two 8-query tiles, the second mostly past the end
    _dense_case(sa, 9, 16, 128, np.arange(9))


def test_dense_tensor_core_many_tiles(sa):
    # 4100 rows: 65 key tiles for the last CTA, a ragged last CTA and tile
    rows = np.concatenate([np.arange(0, 70), np.arange(2040, 2060), np.arange(4030, 4100)])
    _dense_case(sa, 4100, 16, 128, rows)


def test_dense_tensor_core_rising_scores(sa):
    # large logits (standard deviation up to about 6) whose key norms grow
    # with the position: a row's maximum rises tile after tile, so O is
    # rescaled in TMEM part way through; the values keep their small scale
    rows = np.concatenate([np.arange(1000, 1010), np.arange(2980, 3000)])
    _dense_case(sa, 3000, 16, 128, rows, q_gain=96.0, k_ramp=3.0, seed=77)
