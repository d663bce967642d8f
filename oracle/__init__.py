"""fp64 CPU oracle for the gated sparse attention layer — TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. The CUDA library never imports, links or calls it,
and nothing here imports the CUDA library: the two share only the seeded
input generators in ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, one row per task,
pthreads across rows). This wrapper only marshals arguments: it hands the C
code the raw stored bytes (fp32, bf16 bit patterns, e4m3 codes) and the C code
decodes them itself.

Layer steps and where the pages state them:
  indexer  -- score every causal history position with a light, position-free
              score ("Hybrid Attention Architectures...", section 3.1, step 1;
              "From Full Attention to Sparsity", indexer paragraph and the
              positional-encoding paragraph). Formula (the pages give none):
              s[t,j] = sum_h w[t,h] * max(0, q_idx[t,h] . k_idx[j]).
  topk     -- keep the K highest-scoring positions (section 3.1, step 2; the
              pseudocode of section 3.3); an exact tie goes to the lower
              position; a row with n <= K keeps all n.
  attend   -- exact softmax attention over the selected rows only (section
              3.1, step 3; "Hybrid Attention Architecture Evolution...",
              section 3.3: the form of attention is unchanged).
  gate     -- out = sigmoid(gate logit) * attention output, one scalar per
              (token, head) ("Sparse Attention and Hybrid Attention
              Architecture Design", section 4, output gating; section 3.3 of
              the first page returns gate * attn_out).
  attend_backward -- the gradients of the gated attention over a fixed
              index set (the training path), by the chain rule.
  prefill_blocks_layer -- block-level routing: mean-pooled keys per block,
              blocks scored and selected, attention inside the kept blocks.
  prefill_local_layer -- branch fusion with a sliding-window local branch,
              g * sparse + (1 - g) * local.
Parity status: every function here is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, E4M3 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = D
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = D
        lib.oracle_threads_used.argtypes = [I, I64]
        lib.oracle_threads_used.restype = I
        lib.oracle_indexer.argtypes = [P, I, P, P, P, P, I, I, I64, P, P, P, P, P, I]
        lib.oracle_indexer.restype = I
        lib.oracle_topk.argtypes = [P, I64, P, P, I, P, I]
        lib.oracle_topk.restype = I
        lib.oracle_attend.argtypes = [P, I, I, I, I, P, I64, P, I64, I64, P, P, P, I, D, P,
                                      P, P, I]
        lib.oracle_attend.restype = I
        lib.oracle_attend_backward.argtypes = [P, I, I, I, I, P, I64, P, I64, I64, P, P, P, I, D, P, P,
                                               P, P, P, P, I]
        lib.oracle_attend_backward.restype = I
        _lib = lib
    return _lib


def _raw(t):
    """(numpy array of the stored bytes, dtype code) of a CPU tensor or array."""
    if isinstance(t, np.ndarray):
        if t.dtype == np.float32:
            return np.ascontiguousarray(t), F32
        raise TypeError(f"unsupported numpy dtype {t.dtype}")
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.float32:
        return t.numpy(), F32
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), BF16
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy(), E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _f32(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(t, dtype=np.float32)


def _i64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def threads_used(nthreads: int, nrows: int) -> int:
    return _load().oracle_threads_used(nthreads, nrows)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(bits: int) -> float:
    return _load().oracle_e4m3_to_f64(bits)


def indexer(q_idx, w, k_idx, qrow, key_start, n, q_scale=None, k_scale=None,
            nthreads: int = 0):
    """Scores of query rows qrow[r] against keys key_start[r] .. +n[r]-1.

    q_idx [R, Hi, di], w [R, Hi], k_idx [N, di] (fp32/bf16/e4m3 storage; e4m3
    needs q_scale [R, Hi] and k_scale [N]). Returns a list of float64 arrays.
    """
    qa, qd = _raw(q_idx)
    ka, kd = _raw(k_idx)
    if qd != kd:
        raise TypeError("q_idx and k_idx must share a storage type")
    if (qd == E4M3) != (q_scale is not None and k_scale is not None):
        raise ValueError("FP8 indexer inputs need both scales, others none")
    R, Hi, di = q_idx.shape
    qrow, key_start, n = _i64(qrow), _i64(key_start), _i64(n)
    off = np.zeros(len(n), dtype=np.int64)
    if len(n) > 1:
        off[1:] = np.cumsum(n)[:-1]
    out = np.empty(int(n.sum()), dtype=np.float64)
    wa, qs, ks = _f32(w), _f32(q_scale), _f32(k_scale)
    rc = _load().oracle_indexer(_ptr(qa), qd, _ptr(qs), _ptr(wa), _ptr(ka), _ptr(ks),
                                Hi, di, len(n), _ptr(qrow), _ptr(key_start), _ptr(n),
                                _ptr(off), _ptr(out), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_indexer failed ({rc})")
    return [out[o:o + m] for o, m in zip(off, n)]


def topk(rows, K: int, nthreads: int = 0):
    """The K best positions of each score row (score desc, position asc);
    returns int32 [R, K] padded with -1, best first."""
    n = _i64([len(r) for r in rows])
    off = np.zeros(len(n), dtype=np.int64)
    if len(n) > 1:
        off[1:] = np.cumsum(n)[:-1]
    s = np.ascontiguousarray(np.concatenate([np.asarray(r, dtype=np.float64) for r in rows])
                             if len(rows) else np.zeros(0))
    idx = np.empty((len(n), K), dtype=np.int32)
    rc = _load().oracle_topk(_ptr(s), len(n), _ptr(off), _ptr(n), K, _ptr(idx), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_topk failed ({rc})")
    return idx


def attend(q, k_cache, v_cache, ld_k, ld_v, dv, gate, qrow, key_start, idx, scale,
           nthreads: int = 0, want_pre: bool = False):
    """Gated exact attention of query rows qrow[r] over key rows
    key_start[r] + idx[r, i] (idx < 0 skipped). q [R, Hq, dqk]; caches are row
    arrays with row strides ld_k / ld_v (v may alias k). Returns float64
    [len(qrow), Hq, dv] (and the pre-gate output if want_pre)."""
    qa, qd = _raw(q)
    ka, kd = _raw(k_cache)
    va, vd = _raw(v_cache)
    if not (qd == kd == vd):
        raise TypeError("q, k and v must share a storage type")
    _, Hq, dqk = q.shape
    qrow, key_start = _i64(qrow), _i64(key_start)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    R, K = idx.shape
    out = np.empty((R, Hq, dv), dtype=np.float64)
    pre = np.empty_like(out) if want_pre else None
    ga = _f32(gate)
    rc = _load().oracle_attend(_ptr(qa), qd, Hq, dqk, dv, _ptr(ka), ld_k, _ptr(va), ld_v,
                               R, _ptr(qrow), _ptr(key_start), _ptr(idx), K, float(scale),
                               _ptr(ga), _ptr(out), _ptr(pre), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_attend failed ({rc})")
    return (out, pre) if want_pre else out


def attend_backward(q, k, v, ld_k, ld_v, dv, gate, qrow, key_start, idx, scale, dout, n_keys,
                    nthreads: int = 0):
    """Gradients of sum(dout * out) for out = attend(...) over the fixed index
    set idx (the training path: section 3.1 of the first page, the selected set
    is fixed; section 3.3, the gate). dout [R, Hq, dv] in the storage type of
    q. Returns float64 dq [R, Hq, dqk], dk [n_keys, dqk], dv [n_keys, dv] (the
    key and value rows' totals over every task) and dgate [R, Hq] (with
    respect to the gate logits)."""
    qa, qd = _raw(q)
    ka, kd = _raw(k)
    va, vd = _raw(v)
    da, dd = _raw(dout)
    if not (qd == kd == vd == dd):
        raise TypeError("q, k, v and dout must share a storage type")
    _, Hq, dqk = q.shape
    qrow, key_start = _i64(qrow), _i64(key_start)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    R, K = idx.shape
    dq = np.empty((R, Hq, dqk), dtype=np.float64)
    dk = np.zeros((n_keys, dqk), dtype=np.float64)
    dvv = np.zeros((n_keys, dv), dtype=np.float64)
    dgate = np.empty((R, Hq), dtype=np.float64)
    ga = _f32(gate)
    rc = _load().oracle_attend_backward(_ptr(qa), qd, Hq, dqk, dv, _ptr(ka), ld_k, _ptr(va), ld_v, R,
                                        _ptr(qrow), _ptr(key_start), _ptr(idx), K, float(scale), _ptr(ga),
                                        _ptr(da), _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(dgate), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_attend_backward failed ({rc})")
    return dq, dk, dvv, dgate


# ---------------------------------------------------------------------------
# the layer, composed from the three steps above
# ---------------------------------------------------------------------------

def prefill_layer(inp, K: int, scale: float, rows=None, nthreads: int = 0):
    """Causal prefill of one sequence: row t sees positions 0..t.

    Returns dict(scores=[...], idx=int32 [R, K], out=float64 [R, Hq, dv]) for
    the requested rows (all rows by default)."""
    L = inp["q"].shape[0]
    rows = np.arange(L, dtype=np.int64) if rows is None else _i64(rows)
    n = rows + 1
    scores = indexer(inp["q_idx"], inp["w"], inp["k_idx"], rows, np.zeros_like(rows), n,
                     inp.get("q_scale"), inp.get("k_scale"), nthreads)
    idx = topk(scores, K, nthreads)
    dv = inp["v"].shape[1] if inp["v"].dim() == 2 else inp["v"].shape[-1]
    out = attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], dv, inp["gate"],
                 rows, np.zeros_like(rows), idx, scale, nthreads)
    return dict(rows=rows, scores=scores, idx=idx, out=out)


def pool_keys_bf16(k_idx, block: int):
    """Block-level routing's pooled keys ("Sparse Attention and Hybrid
    Attention Architecture Design", block-level routing: keys mean-pooled per
    block): the mean of each block of `block` consecutive rows (a last short
    block averages the rows it has), evaluated in float64 from the stored bf16
    values and stored as bf16 (round to nearest even, through float32)."""
    kf = k_idx.double()
    N = kf.shape[0]
    nb = (N + block - 1) // block
    means = torch.stack([kf[b * block:min(N, (b + 1) * block)].mean(dim=0) for b in range(nb)])
    return means.float().to(torch.bfloat16).contiguous()


def prefill_blocks_layer(inp, K: int, block: int, scale: float, rows=None, nthreads: int = 0):
    """Block-granular causal prefill: query t scores the blocks b with
    b * block <= t through their pooled keys (the indexer formula above),
    keeps the K // block best (ties: lower block), and attends over the
    positions <= t of the kept blocks. Returns the blocks' scores, the kept
    blocks, the kept positions (ascending, -1 padded to K) and the output."""
    L = inp["q"].shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    pooled = pool_keys_bf16(inp["k_idx"], block)
    nblk = rows // block + 1
    scores = indexer(inp["q_idx"], inp["w"], pooled, rows, np.zeros_like(rows), nblk, nthreads=nthreads)
    blk = topk(scores, K // block, nthreads=nthreads)
    idx = np.full((len(rows), K), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        pos = [p for b in sorted(x for x in blk[i] if x >= 0) for p in range(b * block, (b + 1) * block) if p <= t]
        idx[i, :len(pos)] = pos
    out = attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], inp["v"].shape[-1], inp["gate"], rows,
                 np.zeros_like(rows), idx, scale, nthreads=nthreads)
    return dict(rows=rows, scores=scores, blocks=blk, idx=idx, out=out)


def prefill_local_layer(inp, K: int, window: int, scale: float, rows=None, nthreads: int = 0):
    """Branch fusion ("Sparse Attention and Hybrid Attention Architecture
    Design": out = g * sparse + (1 - g) * local): the token-level layer's
    pre-gate output and exact attention over positions max(0, t - window + 1)
    .. t, mixed by g = sigmoid(gate logit)."""
    L = inp["q"].shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    sp = prefill_layer(inp, K, scale, rows=rows, nthreads=nthreads)
    widx = np.full((len(rows), window), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        pos = np.arange(max(0, t - window + 1), t + 1)
        widx[i, :len(pos)] = pos
    dv = inp["v"].shape[-1]
    _, sparse_pre = attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], dv, inp["gate"], rows,
                           np.zeros_like(rows), sp["idx"], scale, nthreads=nthreads, want_pre=True)
    _, local_pre = attend(inp["q"], inp["k"], inp["v"], inp["ld_k"], inp["ld_v"], dv, inp["gate"], rows,
                          np.zeros_like(rows), widx, scale, nthreads=nthreads, want_pre=True)
    g = 1.0 / (1.0 + np.exp(-inp["gate"].double().numpy()[rows]))[:, :, None]
    return dict(rows=rows, idx=sp["idx"], out=g * sparse_pre + (1.0 - g) * local_pre)


def decode_layer(inp, K: int, dv: int, scale: float, seqs=None, nthreads: int = 0):
    """One decode step: sequence b's query sees its ctx_len[b] cached rows
    starting at packed row seq_start[b]."""
    lens = np.asarray(inp["ctx_len"].cpu(), dtype=np.int64)
    starts = np.asarray(inp["seq_start"].cpu(), dtype=np.int64)
    seqs = np.arange(len(lens), dtype=np.int64) if seqs is None else _i64(seqs)
    scores = indexer(inp["q_idx"], inp["w"], inp["k_idx_cache"], seqs, starts[seqs],
                     lens[seqs], inp.get("q_scale"), inp.get("k_idx_scale"), nthreads)
    idx = topk(scores, K, nthreads)
    out = attend(inp["q"], inp["k_cache"], inp["v_cache"], inp["ld_k"], inp["ld_v"], dv,
                 inp["gate"], seqs, starts[seqs], idx, scale, nthreads)
    return dict(seqs=seqs, scores=scores, idx=idx, out=out)
