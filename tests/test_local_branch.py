"""Branch fusion with a sliding-window local branch (out = g * sparse +
(1 - g) * local) on the GPU against the fp64 oracle, through the C ABI. The
sparse branch's index set is checked against the oracle's scores with the
token path's rule, and the fused output is compared over that set."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import certain_zero_scores, check_kept_set, check_outputs, to_host
from workloads import get_config, make_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


@pytest.mark.parametrize("L,K,W", [(700, 128, 64), (300, 64, 1), (260, 32, 512)])
def test_local_fusion_matches_oracle(sa, L, K, W):
    cfg = get_config("prefill_8k", L=L, K=K)
    inp = make_prefill(cfg, seed=L + W)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((L, K), dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(cfg.dqk)
    out = sa.sparse_attn_prefill_local(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"], K, scale, W,
                                       idx_out=idx)
    torch.cuda.synchronize()
    rows = np.arange(L)
    idx_h = to_host(idx).numpy()
    args = (inp["q_idx"], inp["w"], inp["k_idx"], rows, np.zeros_like(rows), rows + 1, inp["q_scale"],
            inp["k_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for t in rows:
        check_kept_set(idx_h[t], ref_scores[t], K, f"row {t}", cz[t])
    widx = np.full((L, W), -1, dtype=np.int32)
    for t in rows:
        pos = np.arange(max(0, t - W + 1), t + 1)
        widx[t, :len(pos)] = pos
    _, sp = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"], rows,
                          np.zeros_like(rows), idx_h, scale, want_pre=True)
    _, lo = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"], rows,
                          np.zeros_like(rows), widx, scale, want_pre=True)
    g = 1.0 / (1.0 + np.exp(-inp["gate"].double().numpy()))[:, :, None]
    check_outputs(to_host(out).double().numpy(), g * sp + (1 - g) * lo, cfg.attn_dtype, "fused out")
