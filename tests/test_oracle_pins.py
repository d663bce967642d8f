"""Pins for the fp64 oracle: each check ties it to something other than itself
(closed forms, special cases that reduce to a library routine, invariants,
brute force on tiny inputs, and the hand-worked fixture in tests/golden).
CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_layer.json")


# ---------------------------------------------------------------------------
# stored formats
# ---------------------------------------------------------------------------

def test_bf16_decoding_known_patterns():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_f64(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert oracle.bf16_to_f64(0x8000) == 0.0 and math.copysign(1, oracle.bf16_to_f64(0x8000)) < 0


def test_bf16_decoding_matches_torch_for_every_pattern():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.bf16_to_f64(b) for b in range(1 << 16)])
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_decoding_known_patterns():
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0xFE) == -448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert math.isnan(oracle.e4m3_to_f64(0x7F))


def test_e4m3_decoding_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# ---------------------------------------------------------------------------
# indexer
# ---------------------------------------------------------------------------

def _rand(shape, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype)


def test_indexer_basis_keys_pick_coordinates():
    # keys e_0..e_{di-1}, one head, w=1: s_j = max(0, q[j])
    di = 8
    q = _rand((1, 1, di), 1)
    k = torch.eye(di)
    w = torch.ones(1, 1)
    s = oracle.indexer(q, w, k, [0], [0], [di])[0]
    assert np.array_equal(s, np.maximum(q[0, 0].double().numpy(), 0.0))


def test_indexer_head_weights_select_heads():
    # w one-hot on head h, keys e_d: s_d = max(0, q[h, d]) -- catches head mix-ups
    Hi, di = 4, 6
    q = _rand((1, Hi, di), 2)
    k = torch.eye(di)
    for h in range(Hi):
        w = torch.zeros(1, Hi)
        w[0, h] = 1.0
        s = oracle.indexer(q, w, k, [0], [0], [di])[0]
        assert np.array_equal(s, np.maximum(q[0, h].double().numpy(), 0.0)), h


def test_indexer_clips_negative_dots_exactly_to_zero():
    di = 16
    k = _rand((5, di), 3)
    q = -k[2].reshape(1, 1, di).repeat(1, 3, 1)   # every head points away from key 2
    w = torch.tensor([[0.2, 0.3, 0.5]])
    s = oracle.indexer(q, w, k, [0], [0], [5])[0]
    assert s[2] == 0.0


def test_indexer_is_linear_in_weights_and_homogeneous_in_q():
    Hi, di, n = 3, 8, 11
    q = _rand((1, Hi, di), 4)
    k = _rand((n, di), 5)
    wa, wb = _rand((1, Hi), 6).abs(), _rand((1, Hi), 7).abs()
    sa = oracle.indexer(q, wa, k, [0], [0], [n])[0]
    sb = oracle.indexer(q, wb, k, [0], [0], [n])[0]
    sab = oracle.indexer(q, wa + wb, k, [0], [0], [n])[0]
    np.testing.assert_allclose(sab, sa + sb, rtol=1e-6, atol=1e-12)   # fp32 w sum rounding
    s2 = oracle.indexer(q * 2, wa, k, [0], [0], [n])[0]
    assert np.array_equal(s2, 2 * sa)                                 # power-of-2: exact
    assert (sa >= 0).all()                                            # w >= 0 => s >= 0


def test_indexer_matches_numpy_on_tiny_inputs():
    Hi, di, L = 3, 5, 9
    q = _rand((L, Hi, di), 8)
    k = _rand((L, di), 9)
    w = _rand((L, Hi), 10)                          # signed weights too
    rows = np.arange(L)
    got = oracle.indexer(q, w, k, rows, np.zeros(L), rows + 1)
    dots = np.einsum("thd,jd->thj", q.double().numpy(), k.double().numpy())
    ref = np.einsum("th,thj->tj", w.double().numpy(), np.maximum(dots, 0.0))
    for t in range(L):
        np.testing.assert_allclose(got[t], ref[t, :t + 1], rtol=1e-13, atol=1e-13)


def test_indexer_fp8_applies_both_scales():
    Hi, di, n = 2, 16, 7
    qf = _rand((1, Hi, di), 11) * 3
    kf = _rand((n, di), 12) * 5
    w = torch.tensor([[0.25, 0.75]])
    # power-of-two scales: code * scale is exact in fp32, so the fp32 path must agree
    qs = torch.tensor([[2.0 ** -4, 2.0 ** -5]])
    ks = torch.tensor([2.0 ** (-3 - (j % 3)) for j in range(n)])
    q8 = (qf / qs.unsqueeze(-1)).clamp(-448, 448).to(torch.float8_e4m3fn)
    k8 = (kf / ks.unsqueeze(-1)).clamp(-448, 448).to(torch.float8_e4m3fn)
    s8 = oracle.indexer(q8, w, k8, [0], [0], [n], q_scale=qs, k_scale=ks)[0]
    qd = q8.float() * qs.unsqueeze(-1)
    kd = k8.float() * ks.unsqueeze(-1)
    sf = oracle.indexer(qd, w, kd, [0], [0], [n])[0]
    np.testing.assert_allclose(s8, sf, rtol=1e-14, atol=0)
    # general amax/448 scales: agrees with the fp32-rounded dequantised values
    from workloads import quantize_rows_e4m3
    q8, qs = quantize_rows_e4m3(qf)
    k8, ks = quantize_rows_e4m3(kf)
    s8 = oracle.indexer(q8, w, k8, [0], [0], [n], q_scale=qs, k_scale=ks)[0]
    sf = oracle.indexer(q8.float() * qs.unsqueeze(-1), w, k8.float() * ks.unsqueeze(-1),
                        [0], [0], [n])[0]
    np.testing.assert_allclose(s8, sf, rtol=1e-6, atol=1e-6)
    # doubling one key's scale doubles exactly that key's score
    ks2 = ks.clone()
    ks2[3] *= 2
    s8b = oracle.indexer(q8, w, k8, [0], [0], [n], q_scale=qs, k_scale=ks2)[0]
    assert s8b[3] == 2 * s8[3]
    assert np.array_equal(np.delete(s8b, 3), np.delete(s8, 3))


def test_indexer_key_window_and_rows():
    # task r reads keys key_start[r] .. key_start[r]+n[r]-1 and query row qrow[r]
    Hi, di = 2, 4
    q = _rand((3, Hi, di), 13)
    k = _rand((10, di), 14)
    w = torch.ones(3, Hi)
    full = oracle.indexer(q, w, k, [2], [0], [10])[0]
    part = oracle.indexer(q, w, k, [2], [4], [3])[0]
    assert np.array_equal(part, full[4:7])


# ---------------------------------------------------------------------------
# Top-K
# ---------------------------------------------------------------------------

def test_topk_matches_brute_force_sort_with_ties():
    rng = np.random.default_rng(0)
    rows = [rng.integers(-3, 4, size=n).astype(np.float64) for n in (1, 5, 9, 17, 33, 64)]
    K = 6
    got = oracle.topk(rows, K)
    for r, s in enumerate(rows):
        order = np.lexsort((np.arange(len(s)), -s))       # score desc, then position asc
        ref = np.full(K, -1, dtype=np.int32)
        m = min(K, len(s))
        ref[:m] = order[:m]
        assert np.array_equal(got[r], ref), r


def test_topk_short_rows_keep_everything_and_pad():
    s = [np.array([0.5, 2.0, 1.0])]
    got = oracle.topk(s, 5)[0]
    assert sorted(got[:3].tolist()) == [0, 1, 2] and got[3:].tolist() == [-1, -1]


def test_topk_all_equal_scores_take_lowest_positions():
    got = oracle.topk([np.zeros(100)], 10)[0]
    assert got.tolist() == list(range(10))


def test_topk_is_permutation_equivariant():
    rng = np.random.default_rng(1)
    s = rng.standard_normal(200)
    perm = rng.permutation(200)
    a = set(oracle.topk([s], 20)[0].tolist())
    b = set(oracle.topk([s[perm]], 20)[0].tolist())
    assert {int(perm[j]) for j in b} == a


def test_topk_rejects_non_finite():
    with pytest.raises(RuntimeError):
        oracle.topk([np.array([1.0, np.nan])], 1)


# ---------------------------------------------------------------------------
# attention + gate
# ---------------------------------------------------------------------------

def _torch_gated_causal(q, k, v, gate, scale):
    """Gated full causal attention in torch float64 (library routine)."""
    L = q.shape[0]
    logits = torch.einsum("thd,jd->thj", q.double(), k.double()) * scale
    mask = torch.ones(L, L, dtype=torch.bool).tril()
    logits = logits.masked_fill(~mask.unsqueeze(1), float("-inf"))
    p = torch.softmax(logits, dim=-1)
    o = torch.einsum("thj,jd->thd", p, v.double())
    return torch.sigmoid(gate.double()).unsqueeze(-1) * o


def test_attend_with_all_positions_equals_full_causal_attention():
    L, Hq, d = 37, 3, 16
    q, k, v = _rand((L, Hq, d), 20), _rand((L, d), 21), _rand((L, d), 22)
    gate = _rand((L, Hq), 23)
    K = 64                                        # K >= n for every row
    idx = np.full((L, K), -1, dtype=np.int32)
    for t in range(L):
        idx[t, :t + 1] = np.arange(t + 1)[::-1]   # any order
    out = oracle.attend(q, k, v, d, d, d, gate, np.arange(L), np.zeros(L), idx, 0.25)
    ref = _torch_gated_causal(q, k, v, gate, 0.25).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_attend_output_is_convex_combination_of_selected_rows():
    # one-hot values: the pre-gate output equals the softmax weights themselves
    n, d, Hq = 12, 12, 2
    q, k = _rand((1, Hq, d), 24) * 3, _rand((n, d), 25)
    v = torch.eye(n, d)
    sel = np.array([[3, 7, 0, 11, -1, 5]], dtype=np.int32)
    _, pre = oracle.attend(q, k, v, d, d, d, torch.zeros(1, Hq), [0], [0], sel, 1.0,
                           want_pre=True)
    for h in range(Hq):
        p = pre[0, h]
        chosen = [3, 7, 0, 11, 5]
        assert (p >= 0).all() and abs(p.sum() - 1.0) < 1e-12
        assert np.all(np.delete(p, chosen) == 0.0)
        logits = k[chosen].double().numpy() @ q[0, h].double().numpy()
        assert np.array_equal(np.argsort(p[chosen], kind="stable"),
                              np.argsort(logits, kind="stable"))


def test_attend_single_key_and_uniform_weights():
    n, d, Hq = 6, 4, 2
    q, k, v = _rand((1, Hq, d), 26), _rand((n, d), 27), _rand((n, d), 28)
    g0 = torch.zeros(1, Hq)
    one = oracle.attend(q, k, v, d, d, d, g0, [0], [0], np.array([[4, -1, -1]]), 1.0)
    assert np.array_equal(one[0], 0.5 * np.stack([v[4].double().numpy()] * Hq))
    zq = torch.zeros(1, Hq, d)
    uni = oracle.attend(zq, k, v, d, d, d, g0, [0], [0], np.array([[1, 2, 5]]), 1.0)
    mean = v[[1, 2, 5]].double().numpy().mean(axis=0)
    np.testing.assert_allclose(uni[0], 0.5 * np.stack([mean] * Hq), rtol=1e-14)


def test_gate_is_the_logistic_function():
    from scipy.special import expit
    logits = torch.tensor([[-40.0, -3.0, -0.5, 0.0, 0.5, 3.0, 40.0]])
    Hq = logits.shape[1]
    q = torch.zeros(1, Hq, 1)
    k = torch.ones(1, 1)
    v = torch.ones(1, 1)
    out = oracle.attend(q, k, v, 1, 1, 1, logits, [0], [0], np.array([[0]]), 1.0)[0, :, 0]
    np.testing.assert_allclose(out, expit(logits.double().numpy()[0]), rtol=1e-15)
    assert (out >= 0).all() and (out <= 1).all() and out[3] == 0.5


def test_attend_latent_row_values_alias_keys():
    # values are the first dv columns of the key row
    n, dqk, dv, Hq = 5, 8, 6, 2
    kv = _rand((n, dqk), 29)
    q = _rand((1, Hq, dqk), 30)
    g = _rand((1, Hq), 31)
    sel = np.array([[0, 2, 4]], dtype=np.int32)
    a = oracle.attend(q, kv, kv, dqk, dqk, dv, g, [0], [0], sel, 0.5)
    b = oracle.attend(q, kv, kv[:, :dv].contiguous(), dqk, dv, dv, g, [0], [0], sel, 0.5)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# gradients over a fixed index set
# ---------------------------------------------------------------------------

def _bwd_case(seed, L=11, Hq=3, d=8, K=6):
    q, k, v = _rand((L, Hq, d), seed), _rand((L, d), seed + 1), _rand((L, d), seed + 2)
    gate, dout = _rand((L, Hq), seed + 3), _rand((L, Hq, d), seed + 4)
    rng = np.random.default_rng(seed)
    idx = np.full((L, K), -1, dtype=np.int32)
    for t in range(L):                       # a causal selection, some rows short
        m = min(K, t + 1)
        idx[t, :m] = np.sort(rng.choice(t + 1, size=m, replace=False))
    return q, k, v, gate, dout, idx


def test_backward_matches_float64_autograd():
    L, Hq, d, K, scale = 11, 3, 8, 6, 0.3
    q, k, v, gate, dout, idx = _bwd_case(40, L, Hq, d, K)
    dq, dk, dv, dg = oracle.attend_backward(q, k, v, d, d, d, gate, np.arange(L), np.zeros(L), idx, scale,
                                            dout, n_keys=L)
    # the same forward in torch float64; autograd derives the gradients
    qt, kt, vt, gt = (x.double().requires_grad_() for x in (q, k, v, gate))
    outs = []
    for t in range(L):
        sel = torch.as_tensor(idx[t][idx[t] >= 0], dtype=torch.long)
        p = torch.softmax(scale * qt[t] @ kt[sel].T, dim=-1)
        outs.append(torch.sigmoid(gt[t]).unsqueeze(-1) * (p @ vt[sel]))
    (torch.stack(outs) * dout.double()).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_backward_matches_central_differences_of_the_forward():
    L, Hq, d, K, scale = 7, 2, 4, 4, 0.7
    q, k, v, gate, dout, idx = _bwd_case(50, L, Hq, d, K)
    dq, dk, dv, dg = oracle.attend_backward(q, k, v, d, d, d, gate, np.arange(L), np.zeros(L), idx, scale,
                                            dout, n_keys=L)
    dd = dout.double().numpy()

    def loss(qq, kk, vv, gg):
        out = oracle.attend(qq, kk, vv, d, d, d, gg, np.arange(L), np.zeros(L), idx, scale)
        return float((out * dd).sum())

    def secant(t, pos, analytic, which):
        lo, hi = t.clone(), t.clone()
        x = float(t[pos])
        lo[pos], hi[pos] = x - 1e-3, x + 1e-3      # stored fp32: the secant uses the stored values
        args_lo = [q, k, v, gate]
        args_hi = [q, k, v, gate]
        args_lo[which], args_hi[which] = lo, hi
        num = (loss(*args_hi) - loss(*args_lo)) / (float(hi[pos]) - float(lo[pos]))
        assert abs(num - analytic) <= 1e-5 * max(1.0, abs(analytic)), (which, pos, num, analytic)

    for pos in [(3, 1, 2), (6, 0, 0), (0, 1, 3)]:
        secant(q, pos, dq[pos], 0)
    for pos in [(0, 1), (2, 3), (5, 0)]:
        secant(k, pos, dk[pos], 1)
        secant(v, pos, dv[pos], 2)
    for pos in [(4, 1), (6, 0)]:
        secant(gate, pos, dg[pos], 3)


def test_backward_single_key_closed_form():
    # one selected key: p = 1, so the logits get no gradient and dv = g * dout
    d, Hq = 4, 2
    q, k, v = _rand((1, Hq, d), 60), _rand((3, d), 61), _rand((3, d), 62)
    gate, dout = _rand((1, Hq), 63), _rand((1, Hq, d), 64)
    idx = np.array([[2, -1]], dtype=np.int32)
    dq, dk, dv, dg = oracle.attend_backward(q, k, v, d, d, d, gate, [0], [0], idx, 1.0, dout, n_keys=3)
    g = 1 / (1 + np.exp(-gate.double().numpy()[0]))
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15      # zero up to rounding
    np.testing.assert_allclose(dv[2], (g[:, None] * dout.double().numpy()[0]).sum(0), rtol=1e-14)
    assert np.all(dv[:2] == 0)
    np.testing.assert_allclose(dg[0], g * (1 - g) * (dout.double().numpy()[0] * v[2].double().numpy()).sum(-1),
                               rtol=1e-14)


# ---------------------------------------------------------------------------
# the composed layer
# ---------------------------------------------------------------------------

def _golden_num(x):
    if isinstance(x, str):
        return {"ln2": math.log(2), "ln3": math.log(3), "-ln3": -math.log(3)}[x]
    return float(x)


def _golden_tensor(x):
    arr = np.vectorize(_golden_num, otypes=[np.float64])(np.array(x, dtype=object))
    return torch.tensor(arr, dtype=torch.float32)


def test_hand_worked_prefill_example():
    g = json.load(open(GOLDEN))["prefill"]
    T = lambda key: _golden_tensor(g[key])
    inp = dict(q=T("q"), k=T("k"), v=T("v"), ld_k=2, ld_v=2, q_idx=T("q_idx"),
               k_idx=T("k_idx"), w=T("w"), gate=T("gate"))
    res = oracle.prefill_layer(inp, g["K"], 1.0)
    for t in range(3):
        assert np.array_equal(res["scores"][t], np.array(g["scores"][t], dtype=np.float64))
        sel = sorted(int(j) for j in res["idx"][t] if j >= 0)
        assert sel == g["selected"][t]
    np.testing.assert_allclose(res["out"], np.array(g["out"]), rtol=0, atol=2e-7)


def test_hand_worked_decode_example():
    g = json.load(open(GOLDEN))["decode"]
    T = lambda key: _golden_tensor(g[key])
    inp = dict(q=T("q"), k_cache=T("k"), v_cache=T("v"), ld_k=2, ld_v=2,
               q_idx=T("q_idx"), k_idx_cache=T("k_idx"), w=T("w"), gate=T("gate"),
               seq_start=torch.tensor(g["seq_start"]), ctx_len=torch.tensor(g["ctx_len"]))
    for case in g["cases"]:
        res = oracle.decode_layer(inp, case["K"], 2, 1.0)
        for b in range(2):
            assert np.array_equal(res["scores"][b], np.array(case["scores"][b], float))
            assert sorted(int(j) for j in res["idx"][b] if j >= 0) == case["selected"][b]
        np.testing.assert_allclose(res["out"], np.array(case["out"]), rtol=0, atol=2e-7)


def test_prefill_layer_with_large_k_is_gated_full_causal_attention():
    from workloads import get_config, make_prefill
    cfg = get_config("tiny", L=80, K=128)
    inp = make_prefill(cfg, seed=3)
    scale = 1 / math.sqrt(cfg.dqk)
    res = oracle.prefill_layer(inp, cfg.K, scale)
    ref = _torch_gated_causal(inp["q"], inp["k"], inp["v"], inp["gate"], scale).numpy()
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-13)


def test_decode_layer_with_large_k_is_gated_full_attention():
    from workloads import get_config, make_decode
    cfg = get_config("decode_ragged", B=3, ctx_range=(), ctx_list=(5, 17, 9), K=32)
    inp = make_decode(cfg, seed=4)
    scale = 1 / math.sqrt(cfg.dqk)
    res = oracle.decode_layer(inp, cfg.K, cfg.dv, scale)
    for b, (s0, n) in enumerate(zip(inp["seq_start"].tolist(), inp["lens"])):
        q = inp["q"][b].double()
        k = inp["k_cache"][s0:s0 + n].double()
        v = inp["v_cache"][s0:s0 + n].double()
        p = torch.softmax(q @ k.T * scale, dim=-1)
        ref = torch.sigmoid(inp["gate"][b].double()).unsqueeze(-1) * (p @ v)
        np.testing.assert_allclose(res["out"][b], ref.numpy(), rtol=1e-11, atol=1e-13)


def test_prefill_layer_sparse_rows_differ_from_full_and_keep_k():
    from workloads import get_config, make_prefill
    cfg = get_config("tiny", L=200, K=16)
    inp = make_prefill(cfg, seed=5)
    res = oracle.prefill_layer(inp, cfg.K, 1 / math.sqrt(cfg.dqk), rows=[3, 15, 16, 199])
    kept = (res["idx"] >= 0).sum(axis=1).tolist()
    assert kept == [4, 16, 16, 16]
    # the kept set of row 199 is exactly its 16 best scores
    s = res["scores"][3]
    order = np.lexsort((np.arange(len(s)), -s))[:16]
    assert set(order.tolist()) == set(res["idx"][3].tolist())


def test_thread_count_report():
    assert oracle.threads_used(3, 100) == 3
    assert oracle.threads_used(8, 2) == 2
    assert oracle.threads_used(0, 10 ** 6) >= 1


# ---------------------------------------------------------------------------
# block-level routing
# ---------------------------------------------------------------------------

def test_pooled_keys_are_block_means():
    k = torch.tensor([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0], [-2.0, 0.5]]).to(torch.bfloat16)
    p = oracle.pool_keys_bf16(k, 2)
    assert p.dtype == torch.bfloat16
    assert p.float().tolist() == [[2.0, 3.0], [6.0, 7.0], [-2.0, 0.5]]      # last block: its one row
    same = torch.full((8, 4), 0.375).to(torch.bfloat16)
    assert torch.equal(oracle.pool_keys_bf16(same, 4), same[:2])


def test_blocks_of_one_position_are_the_token_path():
    from workloads import get_config, make_prefill
    cfg = get_config("prefill_8k", L=90, K=16, Hq=2)
    inp = make_prefill(cfg, seed=5)
    scale = 1 / math.sqrt(cfg.dqk)
    tok = oracle.prefill_layer(inp, cfg.K, scale)
    blk = oracle.prefill_blocks_layer(inp, cfg.K, 1, scale)
    assert np.array_equal(np.sort(np.where(tok["idx"] < 0, 1 << 30, tok["idx"]), axis=1),
                          np.where(blk["idx"] < 0, 1 << 30, blk["idx"]))
    np.testing.assert_allclose(tok["out"], blk["out"], rtol=1e-13, atol=1e-16)   # summation order differs


def test_blocks_covering_the_history_give_full_causal_attention():
    from workloads import get_config, make_prefill
    cfg = get_config("prefill_8k", L=70, K=128, Hq=2)
    inp = make_prefill(cfg, seed=6)
    scale = 1 / math.sqrt(cfg.dqk)
    res = oracle.prefill_blocks_layer(inp, cfg.K, 16, scale)          # 8 blocks kept >= every row's 5
    ref = _torch_gated_causal(inp["q"], inp["k"], inp["v"], inp["gate"], scale).numpy()
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-13)
    for i, t in enumerate(res["rows"]):
        assert res["idx"][i].tolist() == list(range(t + 1)) + [-1] * (cfg.K - t - 1)


# ---------------------------------------------------------------------------
# branch fusion with a sliding-window local branch
# ---------------------------------------------------------------------------

def test_local_fusion_with_whole_history_is_ungated_causal_attention():
    from workloads import get_config, make_prefill
    cfg = get_config("tiny", L=60, K=64, Hq=2)
    inp = make_prefill(cfg, seed=8)
    scale = 1 / math.sqrt(cfg.dqk)
    res = oracle.prefill_local_layer(inp, cfg.K, 64, scale)          # both branches see every position
    ungated = _torch_gated_causal(inp["q"], inp["k"], inp["v"], torch.full_like(inp["gate"], 60.0), scale).numpy()
    np.testing.assert_allclose(res["out"], ungated, rtol=1e-12, atol=1e-14)


def test_local_fusion_gate_extremes_pick_one_branch():
    from workloads import get_config, make_prefill
    cfg = get_config("tiny", L=50, K=8, Hq=2)
    inp = make_prefill(cfg, seed=9)
    scale = 1 / math.sqrt(cfg.dqk)
    L = cfg.L
    for sign in (1.0, -1.0):
        inp["gate"] = torch.full((L, cfg.Hq), 60.0 * sign)
        res = oracle.prefill_local_layer(inp, cfg.K, 5, scale)
        if sign > 0:                                           # g = 1: the sparse branch, pre-gate
            sp = oracle.prefill_layer(inp, cfg.K, scale)
            _, pre = oracle.attend(inp["q"], inp["k"], inp["v"], cfg.dqk, cfg.dv, cfg.dv, inp["gate"], np.arange(L),
                                   np.zeros(L), sp["idx"], scale, want_pre=True)
        else:                                                  # g = 0: attention over the last 5 positions
            widx = np.array([[p if p >= 0 else -1 for p in range(t - 4, t + 1)] for t in range(L)], dtype=np.int32)
            _, pre = oracle.attend(inp["q"], inp["k"], inp["v"], cfg.dqk, cfg.dv, cfg.dv, inp["gate"], np.arange(L),
                                   np.zeros(L), widx, scale, want_pre=True)
        np.testing.assert_allclose(res["out"], pre, rtol=1e-12, atol=1e-14)
