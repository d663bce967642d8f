"""Gradients of the gated attention over a fixed index set (the training path)
on the GPU against the fp64 oracle, through the C ABI.

Tolerance, from the arithmetic: inputs are decoded exactly, every product and
sum runs in fp32, so each gradient element carries the rounding of fp32 sums of
at most K * max(d, Hq) terms (relative 2^-24 per addition); the key and value
rows additionally sum over every query that selected them, in an order that
varies between runs. 1e-3 relative plus 2e-4 of the tensor's largest
magnitude covers that with a wide margin while a wrong term, sign or index
(errors of order one relative) cannot pass."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import to_host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    tol = 1e-3 * np.abs(ref) + 2e-4 * np.abs(ref).max()
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements off, worst {np.abs(got - ref).max():.3g}"


def _causal_selection(L, K, seed, full=False):
    rng = np.random.default_rng(seed)
    idx = np.full((L, K), -1, dtype=np.int32)
    for t in range(L):
        m = min(K, t + 1)
        idx[t, :m] = np.arange(m) if full else np.sort(rng.choice(t + 1, size=m, replace=False))
    return idx


def _case(sa, L, Hq, d, K, dtype, seed, full=False):
    g = torch.Generator().manual_seed(seed)
    std = 1 / math.sqrt(d)
    q = (torch.randn((L, Hq, d), generator=g) * std * 3).to(dtype)
    k = (torch.randn((L, d), generator=g) * std * 3).to(dtype)
    v = (torch.randn((L, d), generator=g) * std).to(dtype)
    gate = torch.randn((L, Hq), generator=g)
    dout = torch.randn((L, Hq, d), generator=g).to(dtype)
    idx = _causal_selection(L, K, seed, full)
    scale = 1 / math.sqrt(d)
    dq, dk, dv, dg = sa.sparse_attn_backward(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(idx).to(DEV),
                                             gate.to(DEV), dout.to(DEV), scale)
    torch.cuda.synchronize()
    ref = oracle.attend_backward(q, k, v, d, d, d, gate, np.arange(L), np.zeros(L), idx, scale, dout, n_keys=L)
    for name, got, r in zip(("dq", "dk", "dv", "dgate"), (dq, dk, dv, dg), ref):
        _close(to_host(got).double().numpy(), r, name)


@pytest.mark.parametrize("L,Hq,d,K,dtype", [
    (300, 16, 128, 64, torch.bfloat16),       # several chunks, ragged tail, short rows padded
    (257, 5, 64, 40, torch.bfloat16),
    (130, 3, 64, 200, torch.float32),          # K > n everywhere: every row keeps its whole history
])
def test_backward_matches_oracle(sa, L, Hq, d, K, dtype):
    _case(sa, L, Hq, d, K, dtype, seed=L + K)


def test_backward_on_forward_selection(sa):
    # the index set the prefill returns, at a size that spans many chunks
    from workloads import get_config, make_prefill
    cfg = get_config("prefill_8k", L=1024, K=256)
    inp = make_prefill(cfg, seed=31)
    d_ = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(cfg.dqk)
    sa.sparse_attn_prefill(d_["q"], d_["k"], d_["v"], d_["q_idx"], d_["k_idx"], d_["w"], d_["gate"], cfg.K, scale,
                           idx_out=idx)
    g = torch.Generator().manual_seed(7)
    dout = torch.randn((cfg.L, cfg.Hq, cfg.dv), generator=g).to(torch.bfloat16)
    dq, dk, dv, dg = sa.sparse_attn_backward(d_["q"], d_["k"], d_["v"], idx, d_["gate"], dout.to(DEV), scale)
    torch.cuda.synchronize()
    idx_h = to_host(idx).numpy()
    ref = oracle.attend_backward(inp["q"], inp["k"], inp["v"], cfg.dqk, cfg.dv, cfg.dv, inp["gate"],
                                 np.arange(cfg.L), np.zeros(cfg.L), idx_h, scale, dout, n_keys=cfg.L)
    for name, got, r in zip(("dq", "dk", "dv", "dgate"), (dq, dk, dv, dg), ref):
        _close(to_host(got).double().numpy(), r, name)
