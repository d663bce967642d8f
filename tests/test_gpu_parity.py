"""CUDA library vs the fp64 oracle, through the C ABI, at sizes the oracle
finishes in seconds (several tiles, ragged tails), plus edge cases."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import (RTOL_SCORE, certain_zero_scores, check_kept_set, check_outputs, check_scores,
                    score_denominators, to_host)
from workloads import get_config, make_decode, make_prefill, quantize_rows_e4m3

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sa(cuda_ok):
    import indexer_top_sparse_03_b300 as pkg
    from indexer_top_sparse_03_b300.build import build
    build()
    pkg.load_library()
    return pkg


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _indexer_inputs(T, N, Hi, di, dtype, seed, signed_w=False):
    g = _gen(seed)
    qf = torch.randn((T, Hi, di), generator=g)
    kf = torch.randn((N, di), generator=g)
    w = torch.randn((T, Hi), generator=g)
    w = w if signed_w else torch.softmax(w, -1)
    if dtype == torch.float8_e4m3fn:
        q, qs = quantize_rows_e4m3(qf)
        k, ks = quantize_rows_e4m3(kf)
        return q, qs, w, k, ks
    return qf.to(dtype), None, w, kf.to(dtype), None


# ---------------------------------------------------------------------------
# indexer_score
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float8_e4m3fn])
@pytest.mark.parametrize("Hi,di", [(1, 16), (4, 32), (4, 64), (8, 64), (32, 128), (3, 48)])
def test_indexer_score(sa, dtype, Hi, di):
    T, N = 203, 389
    q, qs, w, k, ks = _indexer_inputs(T, N, Hi, di, dtype, seed=Hi * 1000 + di)
    dq = lambda x: None if x is None else x.to(DEV)
    for off in (0, 186, -7, N):
        got = sa.indexer_score(dq(q), dq(w), dq(k), dq(qs), dq(ks), causal_offset=off)
        got = to_host(got).double().numpy()
        rows = np.arange(T)
        n = np.clip(rows + 1 + off, 0, N)
        ref = oracle.indexer(q, w, k, rows, np.zeros(T), n, qs, ks)
        den = score_denominators(q, w, k, rows, np.zeros(T), n, qs, ks)
        for t in range(T):
            check_scores(got[t, :n[t]], ref[t], den[t], RTOL_SCORE[dtype], f"off={off} t={t}")
            assert np.isnan(got[t, n[t]:]).all(), "positions beyond n_t must stay unwritten"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float8_e4m3fn])
@pytest.mark.parametrize("Hi,di", [(4, 64), (8, 64), (3, 48)])
def test_indexer_score_signed_w(sa, dtype, Hi, di):
    # head weights of either sign (the header allows any real w): scores can be
    # negative, and a head's ReLU term can cancel another's
    T, N = 150, 333
    q, qs, w, k, ks = _indexer_inputs(T, N, Hi, di, dtype, seed=7 + Hi * 100 + di, signed_w=True)
    assert (w < 0).any() and (w > 0).any()
    dq = lambda x: None if x is None else x.to(DEV)
    for off in (0, 120):
        got = to_host(sa.indexer_score(dq(q), dq(w), dq(k), dq(qs), dq(ks), causal_offset=off)).double().numpy()
        rows = np.arange(T)
        n = np.clip(rows + 1 + off, 0, N)
        ref = oracle.indexer(q, w, k, rows, np.zeros(T), n, qs, ks)
        den = score_denominators(q, w, k, rows, np.zeros(T), n, qs, ks)
        for t in range(T):
            check_scores(got[t, :n[t]], ref[t], den[t], RTOL_SCORE[dtype], f"signed w off={off} t={t}")


def test_indexer_all_negative_dots_give_exact_zero(sa):
    T, N, Hi, di = 40, 70, 4, 64
    g = _gen(1)
    k = torch.randn((N, di), generator=g).abs().to(torch.bfloat16)
    q = (-torch.rand((T, Hi, di), generator=g)).to(torch.bfloat16)
    w = torch.softmax(torch.randn((T, Hi), generator=g), -1)
    got = to_host(sa.indexer_score(q.to(DEV), w.to(DEV), k.to(DEV), causal_offset=N))
    assert (got == 0).all()


# ---------------------------------------------------------------------------
# topk_select: bit-exact against the oracle's sort on the same fp32 values
# ---------------------------------------------------------------------------

def _topk_case(sa, rows, K, ld=None):
    n = [len(r) for r in rows]
    ld = ld or max(max(n), 1)
    buf = torch.full((len(rows), ld), float("nan"), dtype=torch.float32)
    for i, r in enumerate(rows):
        buf[i, :len(r)] = torch.as_tensor(r, dtype=torch.float32)
    lens = torch.tensor(n, dtype=torch.int32)
    got = to_host(sa.topk_select(buf.to(DEV), lens.to(DEV), K)).numpy()
    ref = oracle.topk([buf[i, :n[i]].double().numpy() for i in range(len(rows))], K)
    for i in range(len(rows)):
        m = min(K, n[i])
        assert np.array_equal(got[i, :m], np.sort(ref[i, :m])), f"row {i} (n={n[i]})"
        assert (got[i, m:] == -1).all()


@pytest.mark.parametrize("K", [1, 7, 64, 2048])
def test_topk_random_rows(sa, K):
    rng = np.random.default_rng(K)
    lens = [0, 1, K - 1 if K > 1 else 0, K, K + 1, 3 * K + 5, 12000, 12289, 40000]
    rows = [rng.standard_normal(n).astype(np.float32) for n in lens]
    _topk_case(sa, rows, K)


def test_topk_heavy_ties_signed_zeros_and_negatives(sa):
    rng = np.random.default_rng(5)
    K = 100
    rows = [rng.integers(-2, 3, size=5000).astype(np.float32),       # few distinct values
            np.zeros(300, np.float32),                                # all equal
            np.where(rng.random(700) < 0.5, -0.0, 0.0).astype(np.float32),
            -np.abs(rng.standard_normal(900)).astype(np.float32),     # all negative
            np.repeat(rng.standard_normal(10), 50).astype(np.float32),
            np.concatenate([np.full(20000, 1.5), np.full(20000, 2.5)]).astype(np.float32)]
    _topk_case(sa, rows, K)


# calls whose rows all fit the shared-memory stage (row stride <= 16384) take
# the small-CTA kernel; the cases above include a longer row and so do not
@pytest.mark.parametrize("K", [1, 7, 64, 2048])
def test_topk_short_rows(sa, K):
    rng = np.random.default_rng(100 + K)
    lens = [0, 1, K - 1 if K > 1 else 0, K, K + 1, 2 * K + 3, 5001, 12289, 16384]
    rows = [rng.standard_normal(n).astype(np.float32) for n in lens]
    _topk_case(sa, rows, K)


def test_topk_short_rows_ties_and_unaligned_stride(sa):
    rng = np.random.default_rng(6)
    K = 100
    rows = [rng.integers(-2, 3, size=5000).astype(np.float32),
            np.zeros(300, np.float32),
            np.where(rng.random(700) < 0.5, -0.0, 0.0).astype(np.float32),
            -np.abs(rng.standard_normal(900)).astype(np.float32),
            np.repeat(rng.standard_normal(10), 50).astype(np.float32),
            np.concatenate([np.full(2000, 1.5), np.full(3001, 2.5)]).astype(np.float32)]
    _topk_case(sa, rows, K, ld=5001)              # odd stride: rows 1.. start off 16-byte boundaries
    _topk_case(sa, rows, K, ld=16384)


def test_topk_long_rows_from_global_memory(sa):
    rng = np.random.default_rng(9)
    rows = [rng.standard_normal(n).astype(np.float32) * 3 for n in (131072, 200001)]
    _topk_case(sa, rows, 2048)


def test_topk_row_len_clamped_to_stride(sa):
    buf = torch.arange(10, dtype=torch.float32).reshape(1, 10).to(DEV)
    lens = torch.tensor([50], dtype=torch.int32, device=DEV)      # clamped to ld_s = 10
    got = to_host(sa.topk_select(buf, lens, 3)).numpy()
    assert got.tolist() == [[7, 8, 9]]


# ---------------------------------------------------------------------------
# prefill: all rows at small sizes
# ---------------------------------------------------------------------------

def _run_prefill(sa, cfg, inp):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_prefill(d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["w"], d["gate"],
                                 cfg.K, 1 / math.sqrt(cfg.dqk), q_scale=d["q_scale"],
                                 k_scale=d["k_scale"], idx_out=idx)
    torch.cuda.synchronize()
    return to_host(out), to_host(idx).numpy()


def _check_prefill_rows(cfg, inp, out, idx, rows):
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


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("prefill_8k", dict(L=1500, K=256)),
    ("prefill_128k", dict(L=1300, K=200)),
    ("prefill_8k", dict(L=700, K=1024)),          # K >= n for every row: full causal attention
    # dense rows below 4K (2K on the mma.sync dense kernel) with K not a
    # multiple of the 8-row CTA: CTAs straddle the start of the masked rows
    # (K) and the end of the dense rows
    ("prefill_8k", dict(L=333, K=200)),           # every row on the dense kernel, rows >= 200 masked
    ("prefill_8k", dict(L=1100, K=257)),          # dense rows 0..1027, gathered rows 1028..1099
])
def test_prefill_parity(sa, name, over):
    cfg = get_config(name, **over)
    inp = make_prefill(cfg, seed=11)
    out, idx = _run_prefill(sa, cfg, inp)
    _check_prefill_rows(cfg, inp, out, idx, np.arange(cfg.L))


@pytest.mark.parametrize("name,over", [
    ("prefill_8k", dict(L=1500, K=256)),
    ("prefill_128k", dict(L=1300, K=200)),
])
def test_prefill_parity_signed_w(sa, name, over):
    # head weights of either sign: many scores are negative, and the K-th best
    # can be negative or zero
    cfg = get_config(name, **over)
    inp = make_prefill(cfg, seed=17)
    inp["w"] = torch.randn(inp["w"].shape, generator=_gen(18))
    out, idx = _run_prefill(sa, cfg, inp)
    _check_prefill_rows(cfg, inp, out, idx, np.arange(cfg.L))


def test_prefill_latent_row(sa):
    # one 576-wide row per token, values are its first 512 columns
    cfg = get_config("prefill_8k", L=300, K=64, dqk=576, dv=512, qkv_std=1 / 24)
    inp = make_prefill(cfg, seed=12)
    kv = inp["k"]
    inp = dict(inp, v=kv, ld_v=576)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_prefill(d["q"], d["k"], d["k"], d["q_idx"], d["k_idx"], d["w"], d["gate"],
                                 cfg.K, 1 / math.sqrt(576), dv=512, idx_out=idx)
    torch.cuda.synchronize()
    _check_prefill_rows(cfg, inp, to_host(out), to_host(idx).numpy(), np.arange(cfg.L))


def test_prefill_zero_indexer_keeps_lowest_positions(sa):
    cfg = get_config("prefill_8k", L=400, K=32)
    inp = make_prefill(cfg, seed=13)
    inp["q_idx"] = torch.zeros_like(inp["q_idx"])          # every score is exactly 0
    out, idx = _run_prefill(sa, cfg, inp)
    for t in range(cfg.L):
        m = min(cfg.K, t + 1)
        assert idx[t, :m].tolist() == list(range(m))
    _check_prefill_rows(cfg, inp, out, idx, np.arange(0, cfg.L, 7))


# ---------------------------------------------------------------------------
# decode: all sequences at small sizes
# ---------------------------------------------------------------------------

def _run_decode(sa, cfg, inp):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if inp["v_cache"] is inp["k_cache"]:
        d["v_cache"] = d["k_cache"]                        # keep the latent row aliased
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_decode(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"],
                                d["k_idx_cache"], d["seq_start"], d["ctx_len"], max(inp["lens"]),
                                cfg.K, 1 / math.sqrt(cfg.dqk), dv=cfg.dv, q_scale=d["q_scale"],
                                k_idx_scale=d["k_idx_scale"], ld_k=inp["ld_k"], ld_v=inp["ld_v"],
                                idx_out=idx)
    torch.cuda.synchronize()
    return to_host(out), to_host(idx).numpy()


def _check_decode(cfg, inp, out, idx, seqs=None):
    seqs = np.arange(cfg.B) if seqs is None else np.asarray(seqs)
    lens = np.asarray(inp["lens"])
    starts = inp["seq_start"].numpy()
    args = (inp["q_idx"], inp["w"], inp["k_idx_cache"], seqs, starts[seqs], lens[seqs], inp["q_scale"],
            inp["k_idx_scale"])
    ref_scores = oracle.indexer(*args)
    cz = certain_zero_scores(*args)
    for i, b in enumerate(seqs):
        check_kept_set(idx[b], ref_scores[i], cfg.K, f"seq {b}", cz[i])
    ref = oracle.attend(inp["q"], inp["k_cache"], inp["v_cache"], inp["ld_k"], inp["ld_v"], cfg.dv,
                        inp["gate"], seqs, starts[seqs], idx[seqs], 1 / math.sqrt(cfg.dqk))
    check_outputs(out[seqs].double().numpy(), ref, cfg.attn_dtype, "decode out")


@pytest.mark.parametrize("name,over", [
    ("decode_ragged", dict(B=8, ctx_range=(), ctx_list=(1, 100, 2047, 2048, 2049, 4097, 9000, 0))),
    ("decode_mla", dict(B=5, ctx=6000)),
    ("decode_128k", dict(B=3, ctx=20000, K=512)),
    # FP8-e4m3 indexer keys with one fp32 scale per cached row
    ("decode_ragged", dict(B=8, ctx_range=(), ctx_list=(1, 100, 2047, 2048, 2049, 4097, 9000, 0),
                           idx_dtype=torch.float8_e4m3fn)),
    ("decode_128k", dict(B=3, ctx=20000, K=512, idx_dtype=torch.float8_e4m3fn, Hi=8)),
    ("decode_128k", dict(B=2, ctx=5000, K=300, idx_dtype=torch.float8_e4m3fn, di=128, Hi=16)),
])
def test_decode_parity(sa, name, over):
    cfg = get_config(name, **over)
    inp = make_decode(cfg, seed=21)
    out, idx = _run_decode(sa, cfg, inp)
    _check_decode(cfg, inp, out, idx)


def test_decode_prepared_step_matches_the_call(sa):
    # DecodeStep builds the argument structure once; each call must give what
    # sparse_attn_decode gives on the buffers' current contents
    cfg = get_config("decode_ragged", B=6, ctx_range=(), ctx_list=(1, 2047, 2049, 5000, 9000, 0))
    inp = make_decode(cfg, seed=23)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=DEV)
    step = sa.DecodeStep(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"], d["k_idx_cache"],
                         d["seq_start"], d["ctx_len"], max(inp["lens"]), cfg.K, 1 / math.sqrt(cfg.dqk),
                         q_scale=d["q_scale"], k_idx_scale=d["k_idx_scale"], idx_out=idx)
    for seed in (0, 1):
        if seed:                                  # new contents in the same buffers
            d["q"].copy_(torch.randn(d["q"].shape, generator=_gen(24)).to(d["q"].dtype))
            d["q_idx"].copy_(torch.randn(d["q_idx"].shape, generator=_gen(25)).to(d["q_idx"].dtype))
        got = step().clone()
        got_idx = idx.clone()
        ref = sa.sparse_attn_decode(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"],
                                    d["k_idx_cache"], d["seq_start"], d["ctx_len"], max(inp["lens"]), cfg.K,
                                    1 / math.sqrt(cfg.dqk), q_scale=d["q_scale"], k_idx_scale=d["k_idx_scale"],
                                    idx_out=idx)
        torch.cuda.synchronize()
        assert torch.equal(got_idx, idx)
        assert torch.equal(got, ref)
    inp["q"], inp["q_idx"] = to_host(d["q"]), to_host(d["q_idx"])
    _check_decode(cfg, inp, to_host(got), to_host(got_idx).numpy())


def test_decode_step_with_host_buffers(sa):
    # sparse_attn_decode_host: the packed per-step inputs come from pinned host
    # memory and the output goes back there; it must equal the device call
    cfg = get_config("decode_ragged", B=5, ctx_range=(), ctx_list=(3, 2048, 2049, 7000, 0))
    inp = make_decode(cfg, seed=26)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    names = ("q", "q_idx", "w", "gate")
    sizes = [inp[k].numel() * inp[k].element_size() for k in names]
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    dev_in = torch.empty(sum(sizes), dtype=torch.uint8, device=DEV)
    host_in = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
    view = {}
    for k, o, n in zip(names, offs, sizes):
        view[k] = dev_in[o:o + n].view(inp[k].dtype).view(inp[k].shape)
        host_in[o:o + n].copy_(inp[k].contiguous().view(-1).view(torch.uint8))
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=DEV)
    step = sa.DecodeStep(view["q"], view["q_idx"], view["w"], view["gate"], d["k_cache"], d["v_cache"],
                         d["k_idx_cache"], d["seq_start"], d["ctx_len"], max(inp["lens"]), cfg.K,
                         1 / math.sqrt(cfg.dqk), idx_out=idx)
    host_out = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16).pin_memory()
    step.run_host(host_in, dev_in, host_out)
    torch.cuda.synchronize()
    ref = sa.sparse_attn_decode(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"],
                                d["k_idx_cache"], d["seq_start"], d["ctx_len"], max(inp["lens"]), cfg.K,
                                1 / math.sqrt(cfg.dqk))
    torch.cuda.synchronize()
    assert torch.equal(host_out, to_host(ref))
    _check_decode(cfg, inp, host_out, to_host(idx).numpy())


def test_decode_parity_signed_w(sa):
    cfg = get_config("decode_ragged", B=6, ctx_range=(), ctx_list=(100, 2049, 3000, 4097, 9000, 20000))
    inp = make_decode(cfg, seed=24)
    inp["w"] = torch.randn(inp["w"].shape, generator=_gen(25))
    out, idx = _run_decode(sa, cfg, inp)
    _check_decode(cfg, inp, out, idx)


def test_decode_repeated_calls_reuse_workspace(sa):
    cfg = get_config("decode_ragged", B=4, ctx_range=(), ctx_list=(3000, 5000, 2500, 4100))
    inp = make_decode(cfg, seed=22)
    a_out, a_idx = _run_decode(sa, cfg, inp)
    b_out, b_idx = _run_decode(sa, cfg, inp)
    assert np.array_equal(a_idx, b_idx)
    assert torch.equal(a_out, b_out)


def test_decode_latent_row_given_as_separate_value_copy(sa):
    # the same numbers, but v handed over as its own buffer: the attention kernel
    # then gathers K and V rows separately (single-buffered, 576 + 512 wide rows)
    cfg = get_config("decode_mla", B=3, ctx=3000)
    inp = make_decode(cfg, seed=23)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    v_copy = inp["k_cache"][:, :cfg.dv].contiguous().to(DEV)
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=DEV)
    out = sa.sparse_attn_decode(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], v_copy,
                                d["k_idx_cache"], d["seq_start"], d["ctx_len"], 3000, cfg.K,
                                1 / math.sqrt(cfg.dqk), dv=cfg.dv, idx_out=idx)
    torch.cuda.synchronize()
    _check_decode(cfg, inp, to_host(out), to_host(idx).numpy())


# ---------------------------------------------------------------------------
# tensor-core indexer over many tiles and work items (pipeline wrap-around)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hi,di", [(torch.bfloat16, 4, 64), (torch.float8_e4m3fn, 8, 64),
                                         (torch.bfloat16, 16, 32), (torch.float8_e4m3fn, 4, 128)])
def test_indexer_score_many_tiles(sa, dtype, Hi, di):
    T, N = 1500, 2600
    q, qs, w, k, ks = _indexer_inputs(T, N, Hi, di, dtype, seed=77 + Hi + di)
    dq = lambda x: None if x is None else x.to(DEV)
    off = N - T                                   # the last query sees every key
    got = to_host(sa.indexer_score(dq(q), dq(w), dq(k), dq(qs), dq(ks), causal_offset=off)).double().numpy()
    rows = np.arange(T)
    n = np.clip(rows + 1 + off, 0, N)
    ref = oracle.indexer(q, w, k, rows, np.zeros(T), n, qs, ks)
    den = score_denominators(q, w, k, rows, np.zeros(T), n, qs, ks)
    for t in range(T):
        check_scores(got[t, :n[t]], ref[t], den[t], RTOL_SCORE[dtype], f"t={t}")
        assert np.isnan(got[t, n[t]:]).all()


# ---------------------------------------------------------------------------
# decode Top-K paths: the whole threshold bin kept, and a bin too full for
# the candidate list (exact radix select over the row)
# ---------------------------------------------------------------------------

def _decode_with_indexer(sa, ctx_list, K, k_sign_fn, seed):
    cfg = get_config("decode_ragged", B=len(ctx_list), ctx_range=(), ctx_list=tuple(ctx_list), K=K)
    inp = make_decode(cfg, seed=seed)
    ntot = inp["total_rows"]
    e0 = torch.zeros(cfg.di)
    e0[0] = 1.0
    sign = torch.as_tensor(k_sign_fn(ntot), dtype=torch.float32)
    inp["k_idx_cache"] = (sign[:, None] * e0[None, :]).to(torch.bfloat16)
    inp["q_idx"] = e0.expand(cfg.B, cfg.Hi, cfg.di).contiguous().to(torch.bfloat16)
    out, idx = _run_decode(sa, cfg, inp)
    _check_decode(cfg, inp, out, idx)
    return cfg, inp, idx


def test_decode_topk_exactly_k_in_top_bin(sa):
    # scores are 1 at exactly K positions of each sequence and 0 elsewhere
    rng = np.random.default_rng(3)
    lens = [9000, 20000]
    K = 300
    sign = np.full(sum(lens), -1.0)
    keep = []
    start = 0
    for n in lens:
        pos = np.sort(rng.choice(n, size=K, replace=False))
        sign[start + pos] = 1.0
        keep.append(pos)
        start += n
    _, _, idx = _decode_with_indexer(sa, lens, K, lambda n: sign, seed=41)
    for b in range(len(lens)):
        assert np.array_equal(idx[b], keep[b])


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_topk_boundary_between_adjacent_tied_positions(sa, fp8):
    # the K-th best score is 0 and the boundary falls between two zero-score
    # positions that differ only in their lowest bits (999 | 1000, 1969 | 1970):
    # the lower one must be kept, the higher one dropped
    lens = [5000, 3000, 2050]
    K = 2000
    rng = np.random.default_rng(8)
    sign = np.full(sum(lens), -1.0)
    keep, start = [], 0
    for b, n in enumerate(lens):
        pos = np.arange(n - 1000, n) if b < 2 else np.sort(rng.choice(n, size=30, replace=False))
        sign[start + pos] = 1.0
        zeros = np.setdiff1d(np.arange(n), pos)[:K - len(pos)]
        keep.append(np.sort(np.concatenate([pos, zeros])))
        start += n
    cfg = get_config("decode_ragged", B=len(lens), ctx_range=(), ctx_list=tuple(lens), K=K,
                     idx_dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16)
    inp = make_decode(cfg, seed=43)
    e0 = torch.zeros(cfg.di)
    e0[0] = 1.0
    kf = torch.as_tensor(sign, dtype=torch.float32)[:, None] * e0[None, :]
    qf = e0.expand(cfg.B, cfg.Hi, cfg.di).contiguous()
    if fp8:
        inp["k_idx_cache"], inp["k_idx_scale"] = quantize_rows_e4m3(kf)
        inp["q_idx"], inp["q_scale"] = quantize_rows_e4m3(qf)
    else:
        inp["k_idx_cache"], inp["q_idx"] = kf.to(torch.bfloat16), qf.to(torch.bfloat16)
    out, idx = _run_decode(sa, cfg, inp)
    for b in range(len(lens)):
        assert np.array_equal(idx[b], keep[b]), f"seq {b}"
    _check_decode(cfg, inp, out, idx)


def test_decode_topk_all_scores_tied(sa):
    # every score is exactly 0: the K lowest positions win (too many ties for
    # the candidate list, so the row takes the full radix select)
    lens = [40000, 3000, 2048]
    _, _, idx = _decode_with_indexer(sa, lens, 2048, lambda n: -np.ones(n), seed=42)
    for b, n in enumerate(lens):
        assert np.array_equal(idx[b], np.arange(2048))


def test_topk_long_rows_crowded_boundary_bin(sa):
    # long rows whose boundary bin holds thousands of tied keys (and rows whose
    # candidate count overflows the list): both take the exact fallback path
    rng = np.random.default_rng(17)
    a = rng.random(20000).astype(np.float32) * 0.5
    a[rng.choice(20000, 1500, replace=False)] = 5.0
    rest = np.flatnonzero(a < 1.0)
    a[rng.choice(rest, 3500, replace=False)] = 3.0
    b = np.full(70000, 1.0, np.float32)
    b[::7] = 2.0
    c = rng.standard_normal(90000).astype(np.float32)          # the sampled path proper
    _topk_case(sa, [a, b, c], 2048)
