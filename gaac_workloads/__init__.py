"""Seeded synthetic KV-cache workloads.

Shared by the tests (for both the CUDA path and the oracle), the smoke check
and the benchmark.  This module only draws random numbers and arranges BF16
tensors; it holds none of the codec's or the attention's arithmetic.

Distributions (stand-ins for real model KV, which needs trained weights):
  keys     K[b,t,h,c] = N(0,1) * sK[l,h,c],  sK = exp(N(0,1)) (lognormal,
           sigma 1.0), with 4 distinct outlier channels per (layer, head)
           scaled x20
  values   V[b,t,h,c] = N(0,1) * sV[l,h,c],  sV = exp(0.5 N(0,1))
  queries  q ~ N(0,1)
Values are drawn in fp32 and rounded to BF16 (round to nearest even).  Channel
scales are shared by every sequence of a layer.  Every stream has its own seed
1_000_003*config + 1009*layer + stream so each piece is reproducible alone.

Rotary keys (for the positional-drift study of the GAAC page's Appendix C):
make_kv(..., rope_theta=1e6) rotates the fp32 keys before rounding, channel
pairs (c, c+64) by the angle t * theta^(-2c/128) at position t (the half-split
rotary convention of the Qwen3 family, whose rotary base is 1e6).

Model shapes follow the Qwen3 table of the Transformer-FSQ page (appendix,
models and memory): 0.6B and 1.7B have 28 layers, 16 query / 8 kv heads;
8B has 36 layers, 32 query / 8 kv heads; head width 128 throughout.
"""
from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128
BLOCK = 64

S_KSCALE, S_VSCALE, S_OUTLIER, S_K, S_V, S_Q, S_LEN, S_SLOT, S_ADV_MASK, S_ADV_BITS, S_APPEND = range(11)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config: int
    n_layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    seq_len: int            # fixed length, or the upper bound when lengths vary
    min_len: int = 0        # > 0: lengths uniform in [min_len, seq_len]
    n_calib: int = 512
    appends: int = 0        # decode steps that append one token per sequence
    adversarial: float = 0.0  # share of random-bit tokens after the calibration prefix
    paged: bool = False     # full blocks scattered over a shared slot pool

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)


WORKLOADS = {
    0: Workload("single-layer T=4096, 16q/8kv", 0, 1, 1, 16, 8, 4096),
    1: Workload("Qwen3-8B shape decode, T=65536, 36 layers", 1, 36, 1, 32, 8, 65536),
    2: Workload("paged batch 32, Qwen3-1.7B shape, T in [4096,32768], 28 layers", 2, 28, 32, 16, 8, 32768,
                min_len=4096, paged=True),
    3: Workload("prefill 32768 + 256 appends, Qwen3-0.6B shape, batch 8, 28 layers", 3, 28, 8, 16, 8, 32768,
                appends=256),
    4: Workload("adversarial 10% random-bit tokens, batch 4, T=131072, 32q/8kv", 4, 1, 4, 32, 8, 131072,
                adversarial=0.1),
}


def seed_of(config: int, layer: int, stream: int) -> int:
    return 1_000_003 * config + 1009 * layer + stream


def _gen(device, config, layer, stream) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(config, layer, stream))
    return g


def channel_scales(config: int, layer: int, n_kv_heads: int, device="cpu"):
    """(sK, sV) fp32 [n_kv_heads][128]."""
    sk = torch.exp(torch.randn(n_kv_heads, HEAD_DIM, generator=_gen(device, config, layer, S_KSCALE), device=device))
    g = _gen(device, config, layer, S_OUTLIER)
    for h in range(n_kv_heads):
        idx = torch.randperm(HEAD_DIM, generator=g, device=device)[:4]
        sk[h, idx] *= 20.0
    sv = torch.exp(0.5 * torch.randn(n_kv_heads, HEAD_DIM, generator=_gen(device, config, layer, S_VSCALE),
                                     device=device))
    return sk, sv


def rope(k: torch.Tensor, theta: float, first_pos: int = 0) -> torch.Tensor:
    """Rotary position rotation of fp32 keys [..., n_tok, heads, 128] at positions first_pos + t."""
    n_tok = k.shape[-3]
    pos = torch.arange(n_tok, dtype=torch.float64, device=k.device) + first_pos
    inv = theta ** (-torch.arange(HEAD_DIM // 2, dtype=torch.float64, device=k.device) * 2.0 / HEAD_DIM)
    ang = pos[:, None] * inv[None, :]
    cos, sin = torch.cos(ang).float()[:, None, :], torch.sin(ang).float()[:, None, :]
    x1, x2 = k[..., : HEAD_DIM // 2], k[..., HEAD_DIM // 2:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def make_kv(config: int, layer: int, batch: int, n_tok: int, n_kv_heads: int, device="cpu",
            adversarial: float = 0.0, n_clean: int = 512, token_offset: int = 0, rope_theta: float = 0.0):
    """BF16 (K, V), each [batch][n_tok][n_kv_heads][128].

    token_offset selects a different seed stream so that appended tokens are
    drawn independently of the prefill tokens.  With adversarial > 0, each
    (sequence, token) at position >= n_clean is replaced, with that probability,
    by uniform random 16-bit patterns; exponent 255 (Inf/NaN) is avoided by
    clearing bit 7, which maps it to 254."""
    sk, sv = channel_scales(config, layer, n_kv_heads, device)
    shape = (batch, n_tok, n_kv_heads, HEAD_DIM)
    ks, vs = (S_K, S_V) if token_offset == 0 else (10_000 + 2 * token_offset, 10_001 + 2 * token_offset)
    k = torch.randn(shape, generator=_gen(device, config, layer, ks), device=device) * sk
    if rope_theta > 0.0:
        k = rope(k, rope_theta, token_offset)
    k = k.to(torch.bfloat16)
    v = (torch.randn(shape, generator=_gen(device, config, layer, vs), device=device) * sv).to(torch.bfloat16)
    if adversarial > 0.0:
        g = _gen(device, config, layer, S_ADV_MASK)
        mask = torch.rand(batch, n_tok, generator=g, device=device) < adversarial
        pos = torch.arange(n_tok, device=device) + token_offset
        mask &= (pos >= n_clean)[None, :]
        gb = _gen(device, config, layer, S_ADV_BITS)
        for x in (k, v):
            bits = torch.randint(0, 1 << 16, shape, generator=gb, device=device, dtype=torch.int32)
            exp255 = ((bits >> 7) & 0xFF) == 0xFF
            bits = torch.where(exp255, bits & ~0x80, bits)
            rnd = bits.to(torch.int16).view(torch.bfloat16)
            x.copy_(torch.where(mask[:, :, None, None], rnd, x))
    return k, v


def make_q(config: int, layer: int, batch: int, n_q_heads: int, device="cpu", step: int = 0):
    g = _gen(device, config, layer, S_Q + 100 * step)
    return torch.randn(batch, n_q_heads, HEAD_DIM, generator=g, device=device).to(torch.bfloat16)


def make_lengths(config: int, batch: int, lo: int, hi: int, device="cpu"):
    """Sequence lengths uniform in [lo, hi] (int32)."""
    g = _gen(device, config, 0, S_LEN)
    return torch.randint(lo, hi + 1, (batch,), generator=g, device=device, dtype=torch.int32)


def slot_permutation(config: int, layer: int, n: int, device="cpu"):
    """A seeded permutation of n slot indices (int64): scatters blocks over a shared pool."""
    return torch.randperm(n, generator=_gen(device, config, layer, S_SLOT), device=device)


def bits(x: torch.Tensor) -> torch.Tensor:
    """The 16-bit patterns of a BF16 tensor, as int16 (same storage)."""
    return x.view(torch.int16)
