"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (one sparse_attn_prefill / sparse_attn_decode call over the
whole workload), checked against the fp64 oracle on sampled query rows: the
oracle evaluates each sampled row from scratch, so sampling loses nothing for
those rows. The inputs are the seeded synthetic workloads of `workloads`."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import certain_zero_scores, check_kept_set, check_outputs, to_host
from workloads import get_config, make_decode, make_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


def _sample_rows(L, K, n_random, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, K - 2, K - 1, K, K + 1, L // 2, L - 2, L - 1]
    rnd = rng.choice(L, size=n_random, replace=False)
    return np.unique(np.clip(np.concatenate([fixed, rnd]), 0, L - 1))


@pytest.mark.parametrize("name,n_random", [("tiny", 40), ("prefill_8k", 24), ("prefill_128k", 12)])
def test_prefill_full_size(sa, name, n_random):
    cfg = get_config(name)
    inp = make_prefill(cfg, seed=0)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(cfg.dqk)
    out = sa.sparse_attn_prefill(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"],
                                 cfg.K, scale, q_scale=d["q_scale"], k_scale=d["k_scale"], idx_out=idx)
    torch.cuda.synchronize()
    del d
    rows = _sample_rows(cfg.L, cfg.K, n_random, seed=5)
    idx_h = to_host(idx[torch.as_tensor(rows, device=DEV)]).numpy()
    out_h = to_host(out[torch.as_tensor(rows, device=DEV)]).double().numpy()
    args = (inp["q_idx"], inp["w"], inp["k_idx"], rows, np.zeros_like(rows), rows + 1, inp["q_scale"],
            inp["k_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for i, t in enumerate(rows):
        check_kept_set(idx_h[i], ref_scores[i], cfg.K, f"{name} row {t}", cz[i])
    ref = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"], rows,
                        np.zeros_like(rows), idx_h, scale)
    check_outputs(out_h, ref, cfg.attn_dtype, f"{name} out")


@pytest.mark.parametrize("name,n_seq,over", [("decode_mla", 6, {}), ("decode_ragged", 6, {}), ("decode_128k", 4, {}),
                                             ("decode_128k", 4, dict(idx_dtype=torch.float8_e4m3fn))])
def test_decode_full_size(sa, name, n_seq, over):
    cfg = get_config(name, **over)
    inp = make_decode(cfg, seed=0)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if inp["v_cache"] is inp["k_cache"]:
        d["v_cache"] = d["k_cache"]
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(cfg.dqk)
    out = sa.sparse_attn_decode(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"],
                                d["k_idx_cache"], d["seq_start"], d["ctx_len"], max(inp["lens"]), cfg.K,
                                scale, dv=cfg.dv, q_scale=d["q_scale"], k_idx_scale=d["k_idx_scale"],
                                ld_k=inp["ld_k"], ld_v=inp["ld_v"], idx_out=idx)
    torch.cuda.synchronize()
    del d
    lens = np.asarray(inp["lens"])
    rng = np.random.default_rng(6)
    seqs = np.unique(np.concatenate([[int(np.argmax(lens)), int(np.argmin(lens))],
                                     rng.choice(cfg.B, size=n_seq, replace=False)]))
    idx_h = to_host(idx).numpy()
    out_h = to_host(out).double().numpy()
    starts = inp["seq_start"].numpy()
    args = (inp["q_idx"], inp["w"], inp["k_idx_cache"], seqs, starts[seqs], lens[seqs], inp["q_scale"],
            inp["k_idx_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for i, b in enumerate(seqs):
        check_kept_set(idx_h[b], ref_scores[i], cfg.K, f"{name} seq {b}", cz[i])
    ref = oracle.attend(inp["q"], inp["k_cache"], inp["v_cache"], inp["ld_k"], inp["ld_v"], cfg.dv,
                        inp["gate"], seqs, starts[seqs], idx_h[seqs], scale)
    check_outputs(out_h[seqs], ref, cfg.attn_dtype, f"{name} out")
