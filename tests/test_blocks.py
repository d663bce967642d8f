"""Block-granular selection (block-level routing: mean-pooled keys per block,
blocks scored and selected, exact attention inside the kept blocks) on the
GPU against the fp64 oracle, through the C ABI. The kept blocks follow the
token path's acceptance rule applied to block scores; the outputs are checked
over the GPU's own kept positions."""
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


@pytest.mark.parametrize("L,K,B", [(1500, 256, 64), (777, 96, 16), (300, 64, 1), (2100, 512, 128)])
def test_blocks_match_oracle(sa, L, K, B):
    cfg = get_config("prefill_8k", L=L, K=K)
    inp = make_prefill(cfg, seed=L + B)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((L, K), dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(cfg.dqk)
    out = sa.sparse_attn_prefill_blocks(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"], K, scale,
                                        B, idx_out=idx)
    torch.cuda.synchronize()
    idx_h = to_host(idx).numpy()
    out_h = to_host(out).double().numpy()
    rows = np.arange(L)
    pooled = oracle.pool_keys_bf16(inp["k_idx"], B)
    scores = oracle.indexer(inp["q_idx"], inp["w"], pooled, rows, np.zeros_like(rows), rows // B + 1)
    cz = certain_zero_scores(inp["q_idx"], inp["w"], pooled, rows, np.zeros_like(rows), rows // B + 1)
    for t in rows:
        valid = idx_h[t][idx_h[t] >= 0]
        n_valid = len(valid)
        assert (idx_h[t][n_valid:] == -1).all() and (np.diff(valid) > 0).all() and (valid <= t).all()
        blocks = np.unique(valid // B)
        # every visible position of a kept block is kept
        expect = [p for b in blocks for p in range(b * B, min((b + 1) * B, t + 1))]
        assert valid.tolist() == expect, f"row {t}"
        padded = np.full(K // B, -1, dtype=np.int64)
        padded[:len(blocks)] = blocks
        check_kept_set(padded, scores[t], K // B, f"row {t} blocks", cz[t])
    ref = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"], rows,
                        np.zeros_like(rows), idx_h, scale)
    check_outputs(out_h, ref, cfg.attn_dtype, "blocks out")
