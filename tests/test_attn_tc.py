"""The prefill rows' gathered attention on the tensor core (kernel choice
SA_ATTN_TCGEN05: tiles of 128 kept key/value rows in swizzled shared memory,
S^T and O^T accumulated in TMEM by tcgen05.mma), against the oracle: rows with
many 128-key tiles, ragged last tiles, more than one group of 16 heads, and
scores that rise along a row so that the running maxima are raised in the
middle of a row; the same prefill cases as the default kernel's tests."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import certain_zero_scores, check_kept_set, check_outputs, to_host
from workloads import get_config, make_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import indexer_top_sparse_03_b300 as m
    m.load_library()
    prev = m.set_prefill_attention_kernel(m.ATTN_TCGEN05)
    yield m
    m.set_prefill_attention_kernel(prev)


def _run(sa, cfg, inp):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_prefill(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"],
                                 cfg.K, 1 / math.sqrt(cfg.dqk), q_scale=d["q_scale"],
                                 k_scale=d["k_scale"], idx_out=idx)
    torch.cuda.synchronize()
    assert sa.device_errors(reset=True) == 0
    return to_host(out), to_host(idx).numpy()


def _check(cfg, inp, out, idx, rows):
    rows = np.asarray(rows)
    args = (inp["q_idx"], inp["w"], inp["k_idx"], rows, np.zeros_like(rows), rows + 1, inp["q_scale"],
            inp["k_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for i, t in enumerate(rows):
        check_kept_set(idx[t], ref_scores[i], cfg.K, f"row {t}", cz[i])
    ref = oracle.attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], cfg.dv, inp["gate"],
                        rows, np.zeros_like(rows), idx[rows], 1 / math.sqrt(cfg.dqk))
    check_outputs(out[rows].double().numpy(), ref, cfg.attn_dtype, "prefill out")


def test_rows_of_sixteen_tiles(sa):
    # rows from 4K on are gathered (below, the dense kernel): K = 2048 kept
    # rows = 16 tiles of 128 keys
    cfg = get_config("prefill_8k", L=8600)
    inp = make_prefill(cfg, seed=31)
    out, idx = _run(sa, cfg, inp)
    _check(cfg, inp, out, idx, np.concatenate([np.arange(8192, 8600), np.arange(8186, 8192), [0, 2047, 4100]]))


def test_two_head_groups(sa):
    cfg = get_config("prefill_8k", L=1500, K=256, Hq=32)
    inp = make_prefill(cfg, seed=32)
    out, idx = _run(sa, cfg, inp)
    _check(cfg, inp, out, idx, np.arange(cfg.L))


@pytest.mark.parametrize("K", [512, 300])
def test_scores_rising_along_the_row(sa, K):
    # large logits whose key norms grow with the position: the kept rows come
    # in ascending position, so a row's later tiles hold larger scores and
    # the running maxima are raised (O^T rescaled in TMEM) part way through.
    # The values keep the workload's scale: the bf16 softmax weights carry a
    # rounding error of 2^-8 relative each, i.e. up to 2^-8 * sum(w |v|) on
    # an output, which the output tolerance covers for values of that scale.
    cfg = get_config("prefill_8k", L=2600, K=K, qkv_std=2.45)
    inp = make_prefill(cfg, seed=33)
    ramp = 1.0 + 3.0 * torch.arange(cfg.L, dtype=torch.float32) / cfg.L
    inp["k"] = (inp["k"].float() * ramp[:, None]).to(inp["k"].dtype)
    inp["v"] = (inp["v"].float() / (2.45 * math.sqrt(128))).to(inp["v"].dtype)
    out, idx = _run(sa, cfg, inp)
    _check(cfg, inp, out, idx, np.arange(2 * K, cfg.L, 3))


@pytest.mark.parametrize("name,over", [
    ("prefill_8k", dict(L=1500, K=256)),
    ("prefill_128k", dict(L=1300, K=200)),          # ragged last tiles (72 of 128 rows)
    ("prefill_8k", dict(L=1100, K=257)),            # last tile holds one kept row
])
def test_prefill_cases(sa, name, over):
    cfg = get_config(name, **over)
    inp = make_prefill(cfg, seed=11)
    out, idx = _run(sa, cfg, inp)
    _check(cfg, inp, out, idx, np.arange(cfg.L))


def test_selector_rejects_unknown_values(sa):
    from indexer_top_sparse_03_b300 import SparseAttnError
    with pytest.raises(SparseAttnError):
        sa.set_prefill_attention_kernel(7)
    assert sa.set_prefill_attention_kernel(sa.ATTN_TCGEN05) == sa.ATTN_TCGEN05
