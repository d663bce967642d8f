"""Comparison rules between the CUDA library and the fp64 oracle.

Acceptance bounds (stated for the layer's bf16 path; the fp32 path is held to
the same ones):
  * indexer scores: |s_gpu - s_ref| <= RTOL_SCORE * denom, where denom is the
    forward-error scale of the score, max(|s_ref|, sum_h |w| sum_d |q k|)
    (a plain |s_ref| would make exactly cancelling scores untestable);
    RTOL_SCORE = 1e-3 (bf16/fp32 inputs) or 5e-2 (FP8 inputs).
  * kept index sets: identical, except positions whose reference score lies
    within 1e-3 relative of the reference K-th best score. Exact ties are not
    near-ties: when the K-th best reference score is exactly 0 and a set of
    positions certainly scores exactly 0 on the GPU too (every head's dot
    product is negative by more than any fp32 evaluation error), the GPU must
    keep the lowest positions of that set, as the tie rule says.
  * gated outputs, computed by the oracle over the GPU's own kept set:
    |o_gpu - o_ref| <= 2e-2 + 1e-2 |o_ref|, and additionally the tighter bound
    TIGHT_ATOL + TIGHT_RTOL |o_ref| derived from the arithmetic: bf16 output
    rounding (2^-9 relative), bf16-rounded softmax weights (2^-9 relative per
    weight, normalised by their own sum) and fp32 accumulation.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

RTOL_SCORE = {torch.float32: 1e-3, torch.bfloat16: 1e-3, torch.float8_e4m3fn: 5e-2}
BOUNDARY_RTOL = 1e-3
OUT_ATOL, OUT_RTOL = 2e-2, 1e-2
TIGHT = {torch.float32: (1e-5, 1e-4), torch.bfloat16: (2e-3, 1.6e-2)}


def abs_codes(t):
    """|x| of a stored tensor without changing its format (e4m3: clear the sign bit)."""
    if t is None:
        return None
    if t.dtype == torch.float8_e4m3fn:
        return (t.view(torch.uint8) & 0x7F).view(torch.float8_e4m3fn)
    return t.abs()


def score_denominators(q_idx, w, k_idx, qrow, key_start, n, q_scale=None, k_scale=None):
    """sum_h |w| sum_d |q k| per position, evaluated by the oracle on |inputs|
    (all terms are non-negative, so its ReLU is inactive)."""
    return oracle.indexer(abs_codes(q_idx), w.abs(), abs_codes(k_idx), qrow, key_start, n,
                          q_scale, k_scale)


def negate_codes(t):
    """-x of a stored tensor without changing its format (e4m3: flip the sign bit)."""
    if t.dtype == torch.float8_e4m3fn:
        return (t.view(torch.uint8) ^ 0x80).view(torch.float8_e4m3fn)
    return -t


TIE_MARGIN = 1e-3


def certain_zero_scores(q_idx, w, k_idx, qrow, key_start, n, q_scale=None, k_scale=None):
    """Per position, True when every indexer head's dot product is negative by
    more than TIE_MARGIN * sum_d |q k|. Any fp32 (or tensor-core) evaluation of
    such a dot is negative, so every head's ReLU gives 0 and the score is
    exactly 0 on the GPU as in the oracle. TIE_MARGIN is far above the
    accumulation error of di products (di * 2^-24 for fp32)."""
    Hi = q_idx.shape[1]
    qn, qa, ka = negate_codes(q_idx), abs_codes(q_idx), abs_codes(k_idx)
    out = None
    for h in range(Hi):
        onehot = torch.zeros_like(w)
        onehot[:, h] = 1.0
        neg = oracle.indexer(qn, onehot, k_idx, qrow, key_start, n, q_scale, k_scale)   # max(0, -dot_h)
        mag = oracle.indexer(qa, onehot, ka, qrow, key_start, n, q_scale, k_scale)      # sum_d |q k|
        ok = [a > TIE_MARGIN * b for a, b in zip(neg, mag)]
        out = ok if out is None else [x & y for x, y in zip(out, ok)]
    return out


def check_scores(got, ref, denom, rtol, what=""):
    got = np.asarray(got, dtype=np.float64)
    scale = np.maximum(np.abs(ref), denom)
    err = np.abs(got - ref)
    bad = err > rtol * scale + 1e-30
    assert not bad.any(), (f"{what}: {bad.sum()} scores off; worst rel "
                           f"{(err / np.maximum(scale, 1e-30)).max():.3e}")


def check_kept_set(got_row, ref_scores, K, what="", certain_zero=None):
    """got_row: int array (ascending, -1 padded) from the GPU. certain_zero:
    the row of certain_zero_scores, which turns on the exact-tie rule when the
    K-th best reference score is 0."""
    n = len(ref_scores)
    m = min(K, n)
    got = np.asarray(got_row)
    sel = got[:m]
    assert (got[m:] == -1).all(), f"{what}: padding"
    assert (sel >= 0).all() and (sel < n).all(), f"{what}: out of range"
    assert (np.diff(sel) > 0).all(), f"{what}: not strictly ascending"
    if n <= K:
        assert np.array_equal(sel, np.arange(n)), f"{what}: short row must keep all"
        return
    order = np.lexsort((np.arange(n), -ref_scores))
    ref_set = set(order[:K].tolist())
    kth = ref_scores[order[K - 1]]
    diff = ref_set.symmetric_difference(set(sel.tolist()))
    for j in diff:
        assert abs(ref_scores[j] - kth) <= BOUNDARY_RTOL * abs(kth), (
            f"{what}: position {j} (score {ref_scores[j]!r}) differs, K-th {kth!r}")
    if kth == 0 and certain_zero is not None:
        tied = np.nonzero((ref_scores == 0) & np.asarray(certain_zero))[0]
        kept = np.isin(tied, sel)
        if kept.any() and not kept.all():
            first_out = int(np.argmin(kept))
            assert not kept[first_out:].any(), (
                f"{what}: exact tie at score 0 broken out of position order: kept "
                f"{tied[first_out:][kept[first_out:]][:3].tolist()} over {tied[first_out]}")


def check_outputs(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    assert (err <= OUT_ATOL + OUT_RTOL * np.abs(ref)).all(), f"{what}: outside 2e-2/1e-2"
    ta, tr = TIGHT[dtype]
    bad = err > ta + tr * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} outputs off, worst abs {err.max():.3e}"


def to_host(t):
    if t is None:
        return None
    return t.detach().cpu()
