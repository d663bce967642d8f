"""ctypes binding of libsparse_attn.so, with the names of its C ABI.

Argument marshalling only: torch provides device memory and the current
stream, every step of the layer runs in the library's CUDA kernels. There is
no fallback: if the library is missing or the device is not a CUDA device the
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsparse_attn.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_WORKSPACE, SA_ERR_LAUNCH = 0, -1, -2, -3, -4
SA_F32, SA_BF16, SA_FP8_E4M3 = 0, 1, 2

EXPORTS = ("sa_status_string", "sa_version", "indexer_score", "topk_select",
           "sa_prefill_workspace_size", "sparse_attn_prefill",
           "sa_decode_workspace_size", "sparse_attn_decode", "sparse_attn_decode_noalloc")

_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class PrefillArgs(ctypes.Structure):
    """Mirror of sa_prefill_args."""
    _fields_ = [("L", _I), ("Hq", _I), ("dqk", _I), ("dv", _I), ("Hi", _I), ("di", _I), ("K", _I),
                ("softmax_scale", _F), ("attn_dtype", _I), ("idx_dtype", _I),
                ("q", _P), ("k", _P), ("ld_k", _I64), ("v", _P), ("ld_v", _I64),
                ("q_idx", _P), ("q_scale", _P), ("k_idx", _P), ("k_scale", _P),
                ("w", _P), ("gate", _P), ("out", _P), ("idx_out", _P), ("stage_events", _P)]


class DecodeArgs(ctypes.Structure):
    """Mirror of sa_decode_args."""
    _fields_ = [("B", _I), ("Hq", _I), ("dqk", _I), ("dv", _I), ("Hi", _I), ("di", _I), ("K", _I),
                ("softmax_scale", _F), ("attn_dtype", _I), ("idx_dtype", _I),
                ("q", _P), ("q_idx", _P), ("q_scale", _P), ("w", _P), ("gate", _P),
                ("k_cache", _P), ("ld_k", _I64), ("v_cache", _P), ("ld_v", _I64),
                ("k_idx_cache", _P), ("k_idx_scale", _P), ("seq_start", _P), ("ctx_len", _P),
                ("max_ctx", _I64), ("out", _P), ("idx_out", _P), ("stage_events", _P)]


class BackwardArgs(ctypes.Structure):
    """Mirror of sa_backward_args."""
    _fields_ = [("L", _I), ("Hq", _I), ("dqk", _I), ("dv", _I), ("K", _I), ("dtype", _I),
                ("softmax_scale", _F), ("q", _P), ("k", _P), ("ld_k", _I64), ("v", _P), ("ld_v", _I64),
                ("idx", _P), ("gate", _P), ("dout", _P), ("dq", _P), ("dk", _P), ("dv_out", _P),
                ("dgate", _P)]


class SparseAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def load_library(path: str | None = None):
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m indexer_top_sparse_03_b300.build`")
    lib = ctypes.CDLL(p)
    lib.sa_status_string.argtypes = [_I]
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_version.argtypes = []
    lib.sa_version.restype = _I
    lib.sa_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), _I]
    lib.sa_device_errors.restype = _I
    lib.sa_set_prefill_attention_kernel.argtypes = [_I]
    lib.sa_set_prefill_attention_kernel.restype = _I
    lib.indexer_score.argtypes = [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _P, _I64, _P]
    lib.indexer_score.restype = _I
    lib.topk_select.argtypes = [_P, _I64, _P, _I, _I, _P, _P]
    lib.topk_select.restype = _I
    lib.sa_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
    lib.sa_prefill_workspace_size.restype = _SZ
    lib.sparse_attn_prefill.argtypes = [ctypes.POINTER(PrefillArgs), _P, _SZ, _P]
    lib.sparse_attn_prefill.restype = _I
    lib.sa_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs)]
    lib.sa_decode_workspace_size.restype = _SZ
    lib.sparse_attn_decode.argtypes = [ctypes.POINTER(DecodeArgs), _P, _SZ, _P]
    lib.sparse_attn_decode.restype = _I
    lib.sparse_attn_decode_host.argtypes = [ctypes.POINTER(DecodeArgs), _P, _P, _SZ, _P, _P, _SZ, _P]
    lib.sparse_attn_decode_host.restype = _I
    lib.sparse_attn_decode_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), _P]
    lib.sparse_attn_decode_noalloc.restype = _I
    lib.sa_prefill_blocks_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs), _I]
    lib.sa_prefill_blocks_workspace_size.restype = _SZ
    lib.sparse_attn_prefill_blocks.argtypes = [ctypes.POINTER(PrefillArgs), _I, _P, _SZ, _P]
    lib.sparse_attn_prefill_blocks.restype = _I
    lib.sa_prefill_local_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs), _I]
    lib.sa_prefill_local_workspace_size.restype = _SZ
    lib.sparse_attn_prefill_local.argtypes = [ctypes.POINTER(PrefillArgs), _I, _P, _SZ, _P]
    lib.sparse_attn_prefill_local.restype = _I
    lib.attention_dense_causal.argtypes = [_P, _P, _I64, _P, _I64, _P, _P, _I, _I, _I, _F, _P]
    lib.attention_dense_causal.restype = _I
    lib.sparse_attn_backward.argtypes = [ctypes.POINTER(BackwardArgs), _P]
    lib.sparse_attn_backward.restype = _I
    if path is None:
        _lib = lib
    return lib


def device_errors(reset: bool = False) -> int:
    """The device-side error bits (SA_DEVERR_*) of the current GPU; synchronises."""
    bits = ctypes.c_uint(0)
    _check("sa_device_errors", load_library().sa_device_errors(ctypes.byref(bits), 1 if reset else 0))
    return bits.value


ATTN_AUTO, ATTN_TCGEN05 = 0, 1


def set_prefill_attention_kernel(which: int) -> int:
    """Kernel for the gathered attention of prefill rows (ATTN_AUTO or
    ATTN_TCGEN05), process-wide; returns the previous choice."""
    prev = load_library().sa_set_prefill_attention_kernel(which)
    if prev < 0:
        _check("sa_set_prefill_attention_kernel", prev)
    return prev


def status_string(status: int) -> str:
    return load_library().sa_status_string(status).decode()


def _check(fn: str, status: int):
    if status != SA_OK:
        raise SparseAttnError(fn, status)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SA_F32
    if t == torch.bfloat16:
        return SA_BF16
    if t == torch.float8_e4m3fn:
        return SA_FP8_E4M3
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    return t.data_ptr()


def _stream(device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


_ws_cache: dict = {}


def _events(events):
    """ctypes array of raw cudaEvent_t handles (events must have been created)."""
    if not events:
        return None
    handles = []
    for e in events:
        if e.cuda_event == 0:
            e.record()                      # torch creates the event on first record
        handles.append(e.cuda_event)
    return (ctypes.c_void_p * len(handles))(*handles)


def _workspace(device, nbytes: int, workspace=None):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise SparseAttnError("workspace", SA_ERR_WORKSPACE)
        return workspace
    key = (str(device), )
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


# ---------------------------------------------------------------------------
# the four entry points
# ---------------------------------------------------------------------------

def indexer_score(q_idx, w, k_idx, q_scale=None, k_scale=None, causal_offset: int = 0,
                  scores=None, stream=None):
    """scores[t, j] for j < n_t = clamp(t+1+causal_offset, 0, N); other entries untouched.
    q_idx [T, Hi, di], w [T, Hi], k_idx [N, di]."""
    T, Hi, di = q_idx.shape
    N = k_idx.shape[0]
    if scores is None:
        scores = torch.full((T, N), float("nan"), dtype=torch.float32, device=q_idx.device)
    lib = load_library()
    st = lib.indexer_score(_ptr(q_idx), dtype_code(q_idx.dtype), _ptr(q_scale), _ptr(w), _ptr(k_idx),
                           _ptr(k_scale), T, N, Hi, di, causal_offset, _ptr(scores), scores.stride(0),
                           _stream(q_idx.device, stream))
    _check("indexer_score", st)
    return scores


def topk_select(scores, row_len, K: int, idx_out=None, stream=None):
    """Positions of the K best scores of each row, ascending, -1 padded."""
    T = scores.shape[0]
    if idx_out is None:
        idx_out = torch.empty((T, K), dtype=torch.int32, device=scores.device)
    st = load_library().topk_select(_ptr(scores), scores.stride(0), _ptr(row_len), T, K,
                                    _ptr(idx_out), _stream(scores.device, stream))
    _check("topk_select", st)
    return idx_out


def _prefill_args(q, k, v, q_idx, k_idx, w, gate, K, softmax_scale, q_scale, k_scale, out,
                  idx_out, ld_k, ld_v, dv):
    L, Hq, dqk = q.shape
    a = PrefillArgs()
    a.L, a.Hq, a.dqk, a.dv = L, Hq, dqk, dv
    a.Hi, a.di = q_idx.shape[1], q_idx.shape[2]
    a.K, a.softmax_scale = K, softmax_scale
    a.attn_dtype, a.idx_dtype = dtype_code(q.dtype), dtype_code(q_idx.dtype)
    a.q, a.k, a.ld_k, a.v, a.ld_v = _ptr(q), _ptr(k), ld_k, _ptr(v), ld_v
    a.q_idx, a.q_scale, a.k_idx, a.k_scale = _ptr(q_idx), _ptr(q_scale), _ptr(k_idx), _ptr(k_scale)
    a.w, a.gate, a.out, a.idx_out = _ptr(w), _ptr(gate), _ptr(out), _ptr(idx_out)
    return a


def sparse_attn_prefill(q, k, v, q_idx, k_idx, w, gate, K: int, softmax_scale: float,
                        q_scale=None, k_scale=None, ld_k=None, ld_v=None, dv=None, out=None,
                        idx_out=None, workspace=None, stream=None, stage_events=None):
    """Causal gated sparse attention prefill of one sequence.
    q [L, Hq, dqk]; k rows [L, ld_k]; v rows [L, ld_v] (v may be k); returns out [L, Hq, dv]."""
    L, Hq, dqk = q.shape
    ld_k = k.stride(0) if ld_k is None else ld_k
    ld_v = v.stride(0) if ld_v is None else ld_v
    dv = (v.shape[-1] if v is not k else dqk) if dv is None else dv
    if out is None:
        out = torch.empty((L, Hq, dv), dtype=q.dtype, device=q.device)
    a = _prefill_args(q, k, v, q_idx, k_idx, w, gate, K, softmax_scale, q_scale, k_scale, out,
                      idx_out, ld_k, ld_v, dv)
    ev = _events(stage_events)
    a.stage_events = ctypes.cast(ev, ctypes.c_void_p).value if ev is not None else None
    lib = load_library()
    nbytes = lib.sa_prefill_workspace_size(ctypes.byref(a))
    if nbytes == 0:
        _check("sparse_attn_prefill", lib.sparse_attn_prefill(ctypes.byref(a), None, 0, None))
    ws = _workspace(q.device, nbytes, workspace)
    st = lib.sparse_attn_prefill(ctypes.byref(a), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(q.device, stream))
    _check("sparse_attn_prefill", st)
    return out


def sparse_attn_prefill_blocks(q, k, v, q_idx, k_idx, w, gate, K: int, softmax_scale: float, block_size: int,
                               ld_k=None, ld_v=None, dv=None, out=None, idx_out=None, workspace=None, stream=None,
                               stage_events=None):
    """sparse_attn_prefill with block-granular selection: K / block_size blocks
    of block_size positions kept per query (bf16 indexer inputs)."""
    L, Hq, dqk = q.shape
    ld_k = k.stride(0) if ld_k is None else ld_k
    ld_v = v.stride(0) if ld_v is None else ld_v
    dv = (v.shape[-1] if v is not k else dqk) if dv is None else dv
    if out is None:
        out = torch.empty((L, Hq, dv), dtype=q.dtype, device=q.device)
    a = _prefill_args(q, k, v, q_idx, k_idx, w, gate, K, softmax_scale, None, None, out, idx_out, ld_k, ld_v, dv)
    ev = _events(stage_events)
    a.stage_events = ctypes.cast(ev, ctypes.c_void_p).value if ev is not None else None
    lib = load_library()
    nbytes = lib.sa_prefill_blocks_workspace_size(ctypes.byref(a), block_size)
    if nbytes == 0:
        _check("sparse_attn_prefill_blocks", lib.sparse_attn_prefill_blocks(ctypes.byref(a), block_size, None, 0, None))
    ws = _workspace(q.device, nbytes, workspace)
    st = lib.sparse_attn_prefill_blocks(ctypes.byref(a), block_size, _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(q.device, stream))
    _check("sparse_attn_prefill_blocks", st)
    return out


def sparse_attn_prefill_local(q, k, v, q_idx, k_idx, w, gate, K: int, softmax_scale: float, window: int,
                              q_scale=None, k_scale=None, ld_k=None, ld_v=None, dv=None, out=None, idx_out=None,
                              workspace=None, stream=None):
    """sparse_attn_prefill fused with a sliding-window local branch:
    out = g * sparse + (1 - g) * local, local = attention over the last
    `window` positions (bf16 attention)."""
    L, Hq, dqk = q.shape
    ld_k = k.stride(0) if ld_k is None else ld_k
    ld_v = v.stride(0) if ld_v is None else ld_v
    dv = (v.shape[-1] if v is not k else dqk) if dv is None else dv
    if out is None:
        out = torch.empty((L, Hq, dv), dtype=q.dtype, device=q.device)
    a = _prefill_args(q, k, v, q_idx, k_idx, w, gate, K, softmax_scale, q_scale, k_scale, out, idx_out, ld_k, ld_v,
                      dv)
    lib = load_library()
    nbytes = lib.sa_prefill_local_workspace_size(ctypes.byref(a), window)
    if nbytes == 0:
        _check("sparse_attn_prefill_local", lib.sparse_attn_prefill_local(ctypes.byref(a), window, None, 0, None))
    ws = _workspace(q.device, nbytes, workspace)
    st = lib.sparse_attn_prefill_local(ctypes.byref(a), window, _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(q.device, stream))
    _check("sparse_attn_prefill_local", st)
    return out


def attention_dense_causal(q, k, v, gate, softmax_scale: float, out=None, stream=None):
    """Dense causal gated attention (the full-attention control branch):
    q [L, Hq, d] bf16, k and v rows [L, ld] bf16, gate [L, Hq]; returns out."""
    L, Hq, d = q.shape
    if out is None:
        out = torch.empty((L, Hq, d), dtype=q.dtype, device=q.device)
    st = load_library().attention_dense_causal(_ptr(q), _ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(gate),
                                               _ptr(out), L, Hq, d, softmax_scale, _stream(q.device, stream))
    _check("attention_dense_causal", st)
    return out


def sparse_attn_backward(q, k, v, idx, gate, dout, softmax_scale: float, ld_k=None, ld_v=None,
                         stream=None):
    """Gradients of the gated attention of one causal sequence over the fixed
    index set idx [L, K] (the kept positions of the forward). q [L, Hq, d];
    k, v rows [L, ld]; dout [L, Hq, d] in q's dtype. Returns fp32 dq [L, Hq, d],
    dk [L, d], dv [L, d] and dgate [L, Hq] (with respect to the gate logits)."""
    L, Hq, d = q.shape
    a = BackwardArgs()
    a.L, a.Hq, a.dqk, a.dv, a.K = L, Hq, d, d, idx.shape[1]
    a.dtype, a.softmax_scale = dtype_code(q.dtype), softmax_scale
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.ld_k = k.stride(0) if ld_k is None else ld_k
    a.ld_v = v.stride(0) if ld_v is None else ld_v
    a.idx, a.gate, a.dout = _ptr(idx), _ptr(gate), _ptr(dout)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dv, dg = (torch.empty((L, Hq, d), **f32), torch.empty((L, d), **f32), torch.empty((L, d), **f32),
                      torch.empty((L, Hq), **f32))
    a.dq, a.dk, a.dv_out, a.dgate = _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg)
    _check("sparse_attn_backward", load_library().sparse_attn_backward(ctypes.byref(a), _stream(q.device, stream)))
    return dq, dk, dv, dg


def decode_args(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len, max_ctx: int,
                K: int, softmax_scale: float, dv: int, out, q_scale=None, k_idx_scale=None,
                ld_k=None, ld_v=None, idx_out=None):
    """The sa_decode_args structure for these tensors (for callers of the raw C ABI)."""
    B, Hq, dqk = q.shape
    a = DecodeArgs()
    a.B, a.Hq, a.dqk, a.dv = B, Hq, dqk, dv
    a.Hi, a.di = q_idx.shape[1], q_idx.shape[2]
    a.K, a.softmax_scale = K, softmax_scale
    a.attn_dtype, a.idx_dtype = dtype_code(q.dtype), dtype_code(q_idx.dtype)
    a.q, a.q_idx, a.q_scale, a.w, a.gate = _ptr(q), _ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(gate)
    a.k_cache, a.ld_k = _ptr(k_cache), k_cache.stride(0) if ld_k is None else ld_k
    a.v_cache, a.ld_v = _ptr(v_cache), v_cache.stride(0) if ld_v is None else ld_v
    a.k_idx_cache, a.k_idx_scale = _ptr(k_idx_cache), _ptr(k_idx_scale)
    a.seq_start, a.ctx_len, a.max_ctx = _ptr(seq_start), _ptr(ctx_len), max_ctx
    a.out, a.idx_out = _ptr(out), _ptr(idx_out)
    return a


def decode_workspace_size(args: DecodeArgs) -> int:
    return load_library().sa_decode_workspace_size(ctypes.byref(args))


def sparse_attn_decode(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len,
                       max_ctx: int, K: int, softmax_scale: float, dv=None, q_scale=None,
                       k_idx_scale=None, ld_k=None, ld_v=None, out=None, idx_out=None,
                       workspace=None, stream=None, stage_events=None):
    """One decode step of B sequences over packed caches; returns out [B, Hq, dv]."""
    B, Hq, dqk = q.shape
    dv = (v_cache.shape[-1] if v_cache is not k_cache else dqk) if dv is None else dv
    if out is None:
        out = torch.empty((B, Hq, dv), dtype=q.dtype, device=q.device)
    a = decode_args(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len, max_ctx,
                    K, softmax_scale, dv, out, q_scale, k_idx_scale, ld_k, ld_v, idx_out)
    ev = _events(stage_events)
    a.stage_events = ctypes.cast(ev, ctypes.c_void_p).value if ev is not None else None
    lib = load_library()
    nbytes = lib.sa_decode_workspace_size(ctypes.byref(a))
    if nbytes == 0:
        _check("sparse_attn_decode", lib.sparse_attn_decode(ctypes.byref(a), None, 0, None))
    ws = _workspace(q.device, nbytes, workspace)
    st = lib.sparse_attn_decode(ctypes.byref(a), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(q.device, stream))
    _check("sparse_attn_decode", st)
    return out


class DecodeStep:
    """A decode step prepared once and run many times (a serving loop that
    reuses the same device buffers): the argument structure, the workspace
    and the stream are fixed here, so each call is a single sparse_attn_decode
    call through the C ABI. Arguments as for sparse_attn_decode; the tensors
    must stay allocated, and their contents may change between calls."""

    def __init__(self, q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len,
                 max_ctx: int, K: int, softmax_scale: float, dv=None, q_scale=None, k_idx_scale=None,
                 ld_k=None, ld_v=None, out=None, idx_out=None, workspace=None, stream=None):
        B, Hq, dqk = q.shape
        dv = (v_cache.shape[-1] if v_cache is not k_cache else dqk) if dv is None else dv
        if out is None:
            out = torch.empty((B, Hq, dv), dtype=q.dtype, device=q.device)
        self.out = out
        self._a = decode_args(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len, max_ctx,
                              K, softmax_scale, dv, out, q_scale, k_idx_scale, ld_k, ld_v, idx_out)
        self._a.stage_events = None
        self._lib = load_library()
        nbytes = self._lib.sa_decode_workspace_size(ctypes.byref(self._a))
        if nbytes == 0:
            _check("sparse_attn_decode", self._lib.sparse_attn_decode(ctypes.byref(self._a), None, 0, None))
        self._ws = workspace if workspace is not None else torch.empty(max(nbytes, 256), dtype=torch.uint8,
                                                                          device=q.device)
        self._ws_bytes = self._ws.numel() * self._ws.element_size()
        if self._ws_bytes < nbytes:
            raise SparseAttnError("workspace", SA_ERR_WORKSPACE)
        self._ws_ptr = _ptr(self._ws)
        self._stream = _stream(q.device, stream)
        # the tensors whose addresses the structure holds
        self._keep = (q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len, q_scale,
                      k_idx_scale, idx_out)

    def __call__(self):
        _check("sparse_attn_decode",
               self._lib.sparse_attn_decode(ctypes.byref(self._a), self._ws_ptr, self._ws_bytes, self._stream))
        return self.out

    def run_host(self, host_in, dev_in, host_out):
        """One step with host buffers (sparse_attn_decode_host): host_in's bytes
        go to dev_in (the device buffer this step's q, q_idx, w, gate and
        q_scale live in), the step runs, and the output lands in host_out
        (page-locked CPU tensors for asynchronous copies). Asynchronous on the
        step's stream; returns host_out."""
        if host_in.is_cuda or host_out.is_cuda:
            raise ValueError("host_in and host_out must be CPU tensors")
        nbytes = host_in.numel() * host_in.element_size()
        if host_out.numel() * host_out.element_size() < self.out.numel() * self.out.element_size():
            raise ValueError("host_out is smaller than the output")
        _check("sparse_attn_decode_host",
               self._lib.sparse_attn_decode_host(ctypes.byref(self._a), host_in.data_ptr(), _ptr(dev_in), nbytes,
                                                 host_out.data_ptr(), self._ws_ptr, self._ws_bytes, self._stream))
        return host_out


def sparse_attn_decode_noalloc(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len,
                               max_ctx: int, K: int, softmax_scale: float, dv=None, q_scale=None,
                               k_idx_scale=None, ld_k=None, ld_v=None, out=None, idx_out=None,
                               stream=None):
    """sparse_attn_decode without a workspace, for callers that cannot allocate: the
    library's own fixed scratch array is used (see include/sparse_attn.h). Only
    `out`/`idx_out` are allocated here, and only when not given."""
    B, Hq, dqk = q.shape
    dv = (v_cache.shape[-1] if v_cache is not k_cache else dqk) if dv is None else dv
    if out is None:
        out = torch.empty((B, Hq, dv), dtype=q.dtype, device=q.device)
    a = decode_args(q, q_idx, w, gate, k_cache, v_cache, k_idx_cache, seq_start, ctx_len, max_ctx,
                    K, softmax_scale, dv, out, q_scale, k_idx_scale, ld_k, ld_v, idx_out)
    st = load_library().sparse_attn_decode_noalloc(ctypes.byref(a), _stream(q.device, stream))
    _check("sparse_attn_decode_noalloc", st)
    return out
