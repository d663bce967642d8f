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
