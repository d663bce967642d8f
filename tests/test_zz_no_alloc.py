"""sparse_attn_decode_noalloc: the decode step for callers that cannot allocate
device memory (a host that owns every allocation, or code that must not
allocate once serving runs). It uses the library's fixed scratch array instead
of a caller workspace; its results must equal the workspace entry point's.

Collected last on purpose, so a stop-at-first-failure run has already run
every other test when it gets here. Works alone in a fresh process and after
the other tests."""
import ctypes
import math

import numpy as np
import pytest
import torch

from workloads import get_config, make_decode

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _args_and_out(binding, inp, cfg, max_ctx):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if inp["v_cache"] is inp["k_cache"]:
        d["v_cache"] = d["k_cache"]
    out = torch.full((cfg.B, cfg.Hq, cfg.dv), float("nan"), dtype=torch.bfloat16, device=DEV)
    idx = torch.full((cfg.B, cfg.K), -7, dtype=torch.int32, device=DEV)
    a = binding.decode_args(d["q"], d["q_idx"], d["w"], d["gate"], d["k_cache"], d["v_cache"],
                            d["k_idx_cache"], d["seq_start"], d["ctx_len"], max_ctx, cfg.K,
                            1 / math.sqrt(cfg.dqk), cfg.dv, out, ld_k=inp["ld_k"],
                            ld_v=inp["ld_v"], idx_out=idx)
    return a, out, idx, d


@pytest.mark.parametrize("name,over", [
    ("decode_ragged", dict(B=6, ctx_range=(), ctx_list=(1, 2047, 2049, 9000, 30000, 0))),
    ("decode_mla", dict(B=4, ctx=7000)),
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_ok, name, over):
    from indexer_top_sparse_03_b300 import binding
    from indexer_top_sparse_03_b300.build import build
    from parity import OUT_ATOL, OUT_RTOL, TIGHT
    build()
    lib = binding.load_library()
    cfg = get_config(name, **over)
    inp = make_decode(cfg, seed=31)
    max_ctx = max(inp["lens"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    # the existing entry point, with a caller workspace
    a_ref, out_ref, idx_ref, _ = _args_and_out(binding, inp, cfg, max_ctx)
    need = lib.sa_decode_workspace_size(ctypes.byref(a_ref))
    assert 0 < need <= (32 << 20)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    assert lib.sparse_attn_decode(ctypes.byref(a_ref), ws.data_ptr(), need, stream) == 0
    torch.cuda.synchronize()

    ta, tr = TIGHT[torch.bfloat16]
    for call in range(2):
        a, out, idx, _ = _args_and_out(binding, inp, cfg, max_ctx)
        assert lib.sparse_attn_decode_noalloc(ctypes.byref(a), stream) == 0, call
        torch.cuda.synchronize()
        assert torch.equal(idx.cpu(), idx_ref.cpu()), call
        got = out.cpu().double().numpy()
        ref = out_ref.cpu().double().numpy()
        err = np.abs(got - ref)
        assert (err <= OUT_ATOL + OUT_RTOL * np.abs(ref)).all(), call
        assert (err <= ta + tr * np.abs(ref)).all(), call


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_ok):
    from indexer_top_sparse_03_b300 import binding
    lib = binding.load_library()
    cfg = get_config("decode_128k", B=2, ctx=16)
    inp = make_decode(cfg, seed=32)
    a, out, idx, _ = _args_and_out(binding, inp, cfg, 16)
    a.max_ctx = 1 << 24                       # scores alone would need 128 MiB
    assert lib.sa_decode_workspace_size(ctypes.byref(a)) > (32 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.sparse_attn_decode_noalloc(ctypes.byref(a), stream) == binding.SA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and (idx.cpu() == -7).all()    # nothing was enqueued


def test_no_device_error_bits_after_the_gpu_tests(cuda_ok):
    # every bounded wait of the tensor-core indexer completed in the runs above
    import indexer_top_sparse_03_b300 as pkg
    pkg.load_library()
    assert pkg.device_errors() == 0
