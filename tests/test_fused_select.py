"""The fused indexer + Top-K path of the prefill (rows whose history is long
enough: a sampled threshold, a filtering tensor-core pass that stores only the
pairs at or above it, and an exact selection among those pairs) against the
fp64 oracle, through the C ABI. Rows below the fused region take the
materialised path in the same call, so both sides of the switch are checked."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import certain_zero_scores, check_kept_set, check_outputs, to_host
from workloads import get_config, make_prefill, quantize_rows_e4m3

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


def fmix32(h):
    """MurmurHash3's 32-bit finaliser (its published definition)."""
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h


def sampled_positions(L, lg=4, seed=0x9E3779B9):
    """The library's stratified key sample: one position per stratum of 2^lg,
    at offset fmix32(i ^ seed) mod 2^lg inside stratum i."""
    pos = [(i << lg) + (fmix32(i ^ seed) & ((1 << lg) - 1)) for i in range((L >> lg) + 1)]
    return np.array([p for p in pos if p < L], dtype=np.int64)


def _run(sa, cfg, inp):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_prefill(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"],
                                 cfg.K, 1 / math.sqrt(cfg.dqk), q_scale=d["q_scale"],
                                 k_scale=d["k_scale"], idx_out=idx)
    torch.cuda.synchronize()
    return to_host(out), to_host(idx).numpy()


def _check_rows(cfg, inp, out, idx, rows):
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    args = (inp["q_idx"], inp["w"], inp["k_idx"], rows, np.zeros_like(rows), rows + 1, inp["q_scale"],
            inp["k_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for i, t in enumerate(rows):
        check_kept_set(idx[t], ref_scores[i], cfg.K, f"row {t}", cz[i])
    ref = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"],
                        rows, np.zeros_like(rows), idx[rows], 1 / math.sqrt(cfg.dqk))
    check_outputs(out[rows].double().numpy(), ref, cfg.attn_dtype, "prefill out")


def _rows(lo, hi, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    return np.concatenate([rng.choice(np.arange(lo, hi), size=n, replace=False), np.asarray(extra, dtype=np.int64)])


def test_fused_fp8_rows(sa):
    # FP8 indexer, 8 heads x 64: rows from 16384 on are fused (four passes of 2048)
    cfg = get_config("prefill_128k", L=24576)
    inp = make_prefill(cfg, seed=21)
    out, idx = _run(sa, cfg, inp)
    _check_rows(cfg, inp, out, idx, _rows(16384, cfg.L, 40, 1, extra=(16382, 16383, 16384, 16385, 18431, 18432,
                                                                     20479, 20480, 24574, 24575, 5000)))


def test_fused_bf16_rows_with_boosted_keys(sa):
    # bf16 indexer, 4 heads x 64, every 256th key boosted: fused from row 49152
    cfg = get_config("prefill_8k", L=65536)
    inp = make_prefill(cfg, seed=22)
    out, idx = _run(sa, cfg, inp)
    _check_rows(cfg, inp, out, idx, _rows(49152, cfg.L, 16, 2, extra=(49151, 49152, 51199, 51200, 65535, 30000)))


def test_fused_fp8_rows_signed_w(sa):
    # head weights of either sign through the sampled threshold and the filter pass
    cfg = get_config("prefill_128k", L=20480)
    inp = make_prefill(cfg, seed=24)
    inp["w"] = torch.randn(inp["w"].shape, generator=torch.Generator().manual_seed(6))
    out, idx = _run(sa, cfg, inp)
    _check_rows(cfg, inp, out, idx, _rows(16384, cfg.L, 24, 4, extra=(16383, 16384, 18432, 20479, 3000)))


def test_fused_rows_whose_sample_misleads_fall_back(sa):
    # every sampled key is made near-identical and far above the others, so
    # the sampled threshold keeps ~n/16 pairs (< K) in every fused row: each
    # of those rows is rescored and selected by the fallback
    cfg = get_config("prefill_128k", L=20480)
    inp = make_prefill(cfg, seed=23)
    g = torch.Generator().manual_seed(5)
    ki = inp["k_idx"].float() * inp["k_scale"][:, None]
    pos = torch.as_tensor(sampled_positions(cfg.L))
    ki[pos] = 4.0 + 0.1 * torch.randn((len(pos), cfg.di), generator=g)
    inp["k_idx"], inp["k_scale"] = quantize_rows_e4m3(ki)
    out, idx = _run(sa, cfg, inp)
    _check_rows(cfg, inp, out, idx, _rows(16384, cfg.L, 24, 3, extra=(16384, 18432, 20479)))

