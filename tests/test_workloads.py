"""The seeded input generators: shapes, storage types, determinism and the
structure each workload plants. CPU only."""
import math

import torch

from workloads import get_config, make_decode, make_prefill, decode_lengths, quantize_rows_e4m3


def test_prefill_shapes_dtypes_and_determinism():
    cfg = get_config("prefill_8k", L=600)
    a = make_prefill(cfg, seed=1)
    b = make_prefill(cfg, seed=1)
    assert a["q"].shape == (600, 16, 128) and a["q"].dtype == torch.bfloat16
    assert a["k_idx"].shape == (600, 64) and a["q_idx"].shape == (600, 4, 64)
    assert a["w"].shape == (600, 4) and torch.allclose(a["w"].sum(-1), torch.ones(600))
    assert a["gate"].shape == (600, 16) and a["gate"].dtype == torch.float32
    for key in ("q", "k", "v", "q_idx", "k_idx", "w", "gate"):
        assert torch.equal(a[key], b[key]), key
    c = make_prefill(cfg, seed=2)
    assert not torch.equal(a["q"], c["q"])


def test_prefill_boosted_keys():
    cfg = get_config("prefill_8k", L=2048)
    x = make_prefill(cfg, seed=0)["k_idx"].float()
    boosted = x[::256].mean().item()
    rest = torch.cat([x[j * 256 + 1:(j + 1) * 256] for j in range(8)]).mean().item()
    assert boosted > 1.5 and abs(rest) < 0.05


def test_fp8_quantisation_round_trip():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(50, 64, generator=g) * 3
    codes, scale = quantize_rows_e4m3(x)
    assert codes.dtype == torch.float8_e4m3fn and scale.shape == (50,)
    deq = codes.float() * scale.unsqueeze(-1)
    assert (codes.float().abs().amax(-1) == 448).all()
    # e4m3 keeps 3 fraction bits: relative error <= 2^-4 for normal codes
    big = x.abs() > scale.unsqueeze(-1) * 2 ** -6 * 8
    assert ((deq - x).abs()[big] <= x.abs()[big] * 2 ** -4 + 1e-7).all()


def test_planted_direction_rows():
    cfg = get_config("prefill_128k", L=20000)
    inp = make_prefill(cfg, seed=0)
    frac = inp["planted"].float().mean().item()
    assert 0.005 < frac < 0.015
    assert inp["k_idx"].dtype == torch.float8_e4m3fn and inp["k_scale"].shape == (20000,)


def test_decode_lengths_and_packing():
    cfg = get_config("decode_ragged")
    lens = decode_lengths(cfg, seed=0)
    assert len(lens) == 32 and min(lens) >= 4096 and max(lens) <= 524288
    assert lens == decode_lengths(cfg, seed=0)
    small = get_config("decode_ragged", B=3, ctx_range=(), ctx_list=(5, 1, 9))
    inp = make_decode(small, seed=0)
    assert inp["seq_start"].tolist() == [0, 5, 6] and inp["total_rows"] == 15
    assert inp["k_cache"].shape == (15, 128) and inp["k_idx_cache"].shape == (15, 64)


def test_latent_decode_aliases_value_rows():
    cfg = get_config("decode_mla", B=2, ctx=100)
    inp = make_decode(cfg, seed=0)
    assert inp["k_cache"] is inp["v_cache"] and inp["ld_v"] == 576
    assert math.isclose(inp["k_cache"].float().std().item(), 1 / math.sqrt(576), rel_tol=0.05)
