"""Seeded synthetic inputs for the gated sparse attention layer.

This module is the one piece both the fp64 oracle and the CUDA library are fed
from. It only draws random numbers and stores them in the formats the layer
consumes (fp32, bf16, or FP8-e4m3 codes with one fp32 scale per row); it holds
none of the layer's arithmetic (no scoring, no selection, no attention, no
gate).

Workloads (the pages print no input data; shapes follow the model the pages
describe, "Evolution of Hybrid Attention in Open-Source LLMs", section 3 and
its configuration table: an indexer of a few heads, Top-K of 2048, MQA and a
latent KV row as in "Sparse Attention and Hybrid Attention Architecture
Design", section 2):

  tiny          causal prefill, L=512, 8 query heads x 64, 1 KV head, indexer
                4 x 32, K=64, all fp32
  prefill_8k    causal prefill, L=8192, 16 x 128 MQA, indexer 4 x 64, K=2048,
                bf16; every 256th indexer key gets +2 on every element
  decode_mla    decode, 64 sequences x 32768 cached rows, one latent row of
                576 per token (keys use all 576 columns, values the first 512),
                16 query heads, indexer 4 x 64 bf16, K=2048
  prefill_128k  causal prefill, L=131072, 16 x 128 MQA bf16, indexer 8 x 64 in
                FP8-e4m3 with one fp32 scale per row, K=2048; 1% of the indexer
                keys carry a shared planted direction of norm 8
  decode_ragged decode, 32 sequences, context lengths log-uniform in
                [4096, 524288], 16 x 128 MQA bf16, indexer 4 x 64 bf16, K=2048
  decode_128k   decode_ragged's shapes with every context 131072 (the decode
                throughput point at 128K context)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

__all__ = [
    "PrefillConfig", "DecodeConfig", "CONFIGS", "get_config",
    "make_prefill", "make_decode", "quantize_rows_e4m3",
]

E4M3_MAX = 448.0


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    L: int
    Hq: int
    dqk: int
    dv: int
    Hi: int
    di: int
    K: int
    attn_dtype: torch.dtype
    idx_dtype: torch.dtype          # float32, bfloat16 or float8_e4m3fn
    qkv_std: float                  # std of q, k, v
    idx_std: float                  # std of q_idx, k_idx before quantisation
    boost_every: int = 0            # k_idx[j] += boost for j % boost_every == 0
    boost: float = 0.0
    planted_frac: float = 0.0       # Bernoulli rate of rows that get + planted
    planted_norm: float = 0.0
    kind: str = field(default="prefill")


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    dqk: int
    dv: int
    Hi: int
    di: int
    K: int
    attn_dtype: torch.dtype
    idx_dtype: torch.dtype
    qkv_std: float
    idx_std: float
    ctx: int = 0                    # every sequence has this many rows ...
    ctx_range: tuple = ()           # ... or log-uniform in [lo, hi]
    ctx_list: tuple = ()            # ... or exactly these lengths
    latent: bool = False            # one row per token: K = row, V = row[:dv]
    kind: str = field(default="decode")


CONFIGS = {
    "tiny": PrefillConfig("tiny", L=512, Hq=8, dqk=64, dv=64, Hi=4, di=32, K=64,
                          attn_dtype=torch.float32, idx_dtype=torch.float32,
                          qkv_std=1 / math.sqrt(64), idx_std=1 / math.sqrt(32)),
    "prefill_8k": PrefillConfig("prefill_8k", L=8192, Hq=16, dqk=128, dv=128, Hi=4, di=64,
                                K=2048, attn_dtype=torch.bfloat16, idx_dtype=torch.bfloat16,
                                qkv_std=1 / math.sqrt(128), idx_std=1.0,
                                boost_every=256, boost=2.0),
    "decode_mla": DecodeConfig("decode_mla", B=64, Hq=16, dqk=576, dv=512, Hi=4, di=64,
                               K=2048, attn_dtype=torch.bfloat16, idx_dtype=torch.bfloat16,
                               qkv_std=1 / math.sqrt(576), idx_std=1.0, ctx=32768,
                               latent=True),
    "prefill_128k": PrefillConfig("prefill_128k", L=131072, Hq=16, dqk=128, dv=128, Hi=8,
                                  di=64, K=2048, attn_dtype=torch.bfloat16,
                                  idx_dtype=torch.float8_e4m3fn,
                                  qkv_std=1 / math.sqrt(128), idx_std=1.0,
                                  planted_frac=0.01, planted_norm=8.0),
    "decode_ragged": DecodeConfig("decode_ragged", B=32, Hq=16, dqk=128, dv=128, Hi=4, di=64,
                                  K=2048, attn_dtype=torch.bfloat16,
                                  idx_dtype=torch.bfloat16, qkv_std=1 / math.sqrt(128),
                                  idx_std=1.0, ctx_range=(4096, 524288)),
    "decode_128k": DecodeConfig("decode_128k", B=32, Hq=16, dqk=128, dv=128, Hi=4, di=64,
                                K=2048, attn_dtype=torch.bfloat16, idx_dtype=torch.bfloat16,
                                qkv_std=1 / math.sqrt(128), idx_std=1.0, ctx=131072),
}


def get_config(name: str, **overrides):
    """A named workload, optionally with some fields replaced (smaller cases)."""
    return replace(CONFIGS[name], **overrides)


def quantize_rows_e4m3(x: torch.Tensor):
    """Store x ([..., d]) as FP8-e4m3 codes with one fp32 scale per row.

    scale = amax(|row|) / 448 (1 for an all-zero row); code = RNE(x / scale),
    clamped to the finite range. The stored value of an element is code*scale.
    """
    xf = x.float()
    amax = xf.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (xf / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes.contiguous(), scale.contiguous()


def _normal(gen, shape, std, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def _store(x: torch.Tensor, dtype: torch.dtype):
    return x.to(dtype).contiguous()


def _softmax_heads(gen, rows, heads, device):
    return torch.softmax(torch.randn((rows, heads), generator=gen, device=device), dim=-1)


def make_prefill(cfg: PrefillConfig, seed: int = 0, device="cpu"):
    """One causal prefill sequence of cfg.L tokens; tensors drawn in this order:
    q, k, v, q_idx, k_idx, (planted rows), w, gate."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    L = cfg.L
    q = _store(_normal(g, (L, cfg.Hq, cfg.dqk), cfg.qkv_std, device), cfg.attn_dtype)
    k = _store(_normal(g, (L, cfg.dqk), cfg.qkv_std, device), cfg.attn_dtype)
    v = _store(_normal(g, (L, cfg.dv), cfg.qkv_std, device), cfg.attn_dtype)
    qi = _normal(g, (L, cfg.Hi, cfg.di), cfg.idx_std, device)
    ki = _normal(g, (L, cfg.di), cfg.idx_std, device)
    if cfg.boost_every:
        ki[::cfg.boost_every] += cfg.boost
    if cfg.planted_frac > 0:
        u = torch.randn((cfg.di,), generator=g, device=device)
        u = u * (cfg.planted_norm / u.norm())
        rows = torch.rand((L,), generator=g, device=device) < cfg.planted_frac
        ki[rows] += u
    out = dict(q=q, k=k, v=v, ld_k=cfg.dqk, ld_v=cfg.dv)
    out.update(_store_indexer(qi, ki, cfg.idx_dtype))
    out["w"] = _softmax_heads(g, L, cfg.Hi, device).contiguous()
    out["gate"] = _normal(g, (L, cfg.Hq), 1.0, device).contiguous()
    if cfg.planted_frac > 0:
        out["planted"] = rows
    return out


def _store_indexer(qi, ki, dtype):
    if dtype == torch.float8_e4m3fn:
        q8, qs = quantize_rows_e4m3(qi)
        k8, ks = quantize_rows_e4m3(ki)
        return dict(q_idx=q8, q_scale=qs, k_idx=k8, k_scale=ks)
    return dict(q_idx=_store(qi, dtype), q_scale=None, k_idx=_store(ki, dtype), k_scale=None)


def decode_lengths(cfg: DecodeConfig, seed: int = 0):
    """Context length of each sequence (host list)."""
    if cfg.ctx_list:
        return [int(x) for x in cfg.ctx_list]
    if cfg.ctx:
        return [int(cfg.ctx)] * cfg.B
    lo, hi = cfg.ctx_range
    g = torch.Generator()
    g.manual_seed(seed + 7919)
    u = torch.rand((cfg.B,), generator=g, dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(round(float(x))) for x in lens]


def make_decode(cfg: DecodeConfig, seed: int = 0, device="cpu"):
    """One decode step for cfg.B sequences whose caches are packed back to back;
    tensors drawn in this order: caches, k_idx cache, q, q_idx, w, gate."""
    lens = decode_lengths(cfg, seed)
    starts = [0]
    for n in lens[:-1]:
        starts.append(starts[-1] + n)
    ntot = sum(lens)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = dict(ctx_len=torch.tensor(lens, dtype=torch.int32, device=device),
               seq_start=torch.tensor(starts, dtype=torch.int64, device=device),
               lens=lens, total_rows=ntot)
    if cfg.latent:
        kv = _store(_normal(g, (ntot, cfg.dqk), cfg.qkv_std, device), cfg.attn_dtype)
        out.update(k_cache=kv, v_cache=kv, ld_k=cfg.dqk, ld_v=cfg.dqk)
    else:
        kc = _store(_normal(g, (ntot, cfg.dqk), cfg.qkv_std, device), cfg.attn_dtype)
        vc = _store(_normal(g, (ntot, cfg.dv), cfg.qkv_std, device), cfg.attn_dtype)
        out.update(k_cache=kc, v_cache=vc, ld_k=cfg.dqk, ld_v=cfg.dv)
    ki = _normal(g, (ntot, cfg.di), cfg.idx_std, device)
    q = _store(_normal(g, (cfg.B, cfg.Hq, cfg.dqk), cfg.qkv_std, device), cfg.attn_dtype)
    qi = _normal(g, (cfg.B, cfg.Hi, cfg.di), cfg.idx_std, device)
    ix = _store_indexer(qi, ki, cfg.idx_dtype)
    out.update(q=q, q_idx=ix["q_idx"], q_scale=ix["q_scale"],
               k_idx_cache=ix["k_idx"], k_idx_scale=ix["k_scale"])
    out["w"] = _softmax_heads(g, cfg.B, cfg.Hi, device).contiguous()
    out["gate"] = _normal(g, (cfg.B, cfg.Hq), 1.0, device).contiguous()
    return out
