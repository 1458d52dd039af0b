"""Seeded synthetic inputs for the quantized KV-cache path.

Pure data generation (no quantization or attention arithmetic): the tests,
the benchmark and the smoke check draw both the CUDA path's inputs and the
oracle's inputs from here, copying the exact same numbers to each side.

Distributions follow the workloads the source pages discuss: roughly unit
normal keys and values, keys with a few large channels that stay fixed across
tokens ("O Seu Cache KV Nao Tem um Problema de Bits...", section "Chaves: Os
Valores Extremos Vivem em Canais Fixos"), RMS-normalised keys for the hybrid
model whose keys pass a k_norm before the cache ("Asymetrie kvantizace KV
cache", section "Preneseni na Qwen3.5 a metodicka past"), and Laplace values
for the serving mix.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, device="cpu", dtype=torch.float32) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32).to(dtype)


def laplace(shape, seed, device="cpu", dtype=torch.float32) -> torch.Tensor:
    # inverse CDF of Laplace(0, 1) from uniform(-1/2, 1/2)
    u = torch.rand(shape, generator=_gen(seed, device), device=device, dtype=torch.float32) - 0.5
    u = u.clamp(-0.5 + 1e-7, 0.5 - 1e-7)
    return (-torch.sign(u) * torch.log1p(-2.0 * u.abs())).to(dtype)


def outlier_channels(H, D, per_head=0, frac=0.0, seed=0):
    """Fixed outlier channel indices per head: `per_head` random channels per
    head, or a `frac` fraction of all H*D channels.  Returns a bool mask [H][D]."""
    g = _gen(seed, "cpu")
    mask = torch.zeros((H, D), dtype=torch.bool)
    if per_head:
        for h in range(H):
            mask[h, torch.randperm(D, generator=g)[:per_head]] = True
    elif frac > 0:
        n = max(1, int(round(frac * H * D)))
        idx = torch.randperm(H * D, generator=g)[:n]
        mask.view(-1)[idx] = True
    return mask


def keys(B, T, H, D, seed, device="cpu", dtype=torch.float16, outlier_mask=None, outlier_scale=1.0,
         rmsnorm=False) -> torch.Tensor:
    """[B][T][H][D] keys: N(0,1), optional fixed outlier channels scaled up,
    optional RMS normalisation of each head vector (eps 1e-6, unit weight)."""
    k = normal((B, T, H, D), seed, device)
    if rmsnorm:
        k = k * torch.rsqrt(k.pow(2).mean(dim=-1, keepdim=True) + 1e-6)
    if outlier_mask is not None:
        m = outlier_mask.to(device)
        k = torch.where(m[None, None], k * outlier_scale, k)
    return k.to(dtype)


def values(B, T, H, D, seed, device="cpu", dtype=torch.float16, dist="normal") -> torch.Tensor:
    if dist == "laplace":
        return laplace((B, T, H, D), seed, device, dtype)
    return normal((B, T, H, D), seed, device, dtype)


def query(B, Hq, D, seed, device="cpu", dtype=torch.float16) -> torch.Tensor:
    return normal((B, Hq, D), seed, device, dtype)


def axis_study_inputs(T=1024, H=4, D=128, seed=0, outliers_per_head=2, outlier_scale=15.0, important_frac=0.05,
                      align=0.42, important_value_scale=0.1, value_channel_spread=0.5):
    """Inputs of the quantization-axis study: keys N(0,1) with fixed outlier
    channels (scaled up, the same channels for every token); a query per head;
    a small set of important tokens whose keys lean towards the query, so
    that a softmax over q.k/sqrt(D) puts most of its mass on them (sparse
    attention); values N(0,1) times a mild fixed per-channel scale drawn from
    [1 - spread, 1 + spread] (no extreme channels), except the important
    tokens' values, which are scaled down.  Returns (k [1][T][H][D],
    v [1][T][H][D], q [1][H][D], the important-token mask [T]), fp32 tensors."""
    mask = outlier_channels(H, D, per_head=outliers_per_head, seed=seed * 1000 + 1)
    k = keys(1, T, H, D, seed * 1000 + 2, dtype=torch.float32, outlier_mask=mask, outlier_scale=outlier_scale)
    q = query(1, H, D, seed * 1000 + 3, dtype=torch.float32)
    g = _gen(seed * 1000 + 4, "cpu")
    imp = torch.zeros(T, dtype=torch.bool)
    imp[torch.randperm(T, generator=g)[:max(1, int(round(important_frac * T)))]] = True
    k[0, imp] += align * q[0][None]
    v = values(1, T, H, D, seed * 1000 + 5, dtype=torch.float32)
    cs = 1.0 + value_channel_spread * (2.0 * torch.rand((H, D), generator=g) - 1.0)
    v = v * cs[None, None]
    v[0, imp] *= important_value_scale
    return k, v, q, imp


def ragged_lengths(B, lo, hi, seed) -> list:
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


@dataclass
class Workload:
    """One quantization setting of a workload (shapes + K/V tensor configs)."""
    name: str
    layers: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    lens: list
    k: tuple  # (bits, group, axis, mode)
    v: tuple
    dtype: torch.dtype = torch.float16
    key_outliers_per_head: int = 0
    key_outlier_frac: float = 0.0
    key_outlier_scale: float = 1.0
    key_rmsnorm: bool = False
    value_dist: str = "normal"
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def max_tokens(self):
        return max(self.lens)

    def layer_kv(self, layer, device="cpu", T=None):
        """Keys and values of one layer: [B][T][H][D] each (T defaults to max len)."""
        T = T or self.max_tokens
        mask = None
        if self.key_outliers_per_head or self.key_outlier_frac:
            mask = outlier_channels(self.kv_heads, self.head_dim, self.key_outliers_per_head, self.key_outlier_frac,
                                    seed=self.seed * 1000 + 17 * layer + 1)
        s = self.seed * 1000 + layer
        k = keys(self.batch, T, self.kv_heads, self.head_dim, 2 * s + 11, device, self.dtype, mask,
                 self.key_outlier_scale, self.key_rmsnorm)
        v = values(self.batch, T, self.kv_heads, self.head_dim, 2 * s + 12, device, self.dtype, self.value_dist)
        return k, v

    def layer_query(self, layer, step=0, device="cpu"):
        return query(self.batch, self.q_heads, self.head_dim, self.seed * 1000 + 500 + 7 * layer + 13 * step, device,
                     self.dtype)

    def step_kv(self, layer, step, device="cpu"):
        """One new token per sequence for decode step `step`: [B][H][D] keys and values."""
        mask = None
        if self.key_outliers_per_head or self.key_outlier_frac:
            mask = outlier_channels(self.kv_heads, self.head_dim, self.key_outliers_per_head, self.key_outlier_frac,
                                    seed=self.seed * 1000 + 17 * layer + 1)
        s = self.seed * 1000 + 900 + 31 * layer + 3 * step
        k = keys(self.batch, 1, self.kv_heads, self.head_dim, s, device, self.dtype, mask, self.key_outlier_scale,
                 self.key_rmsnorm)[:, 0]
        v = values(self.batch, 1, self.kv_heads, self.head_dim, s + 1, device, self.dtype, self.value_dist)[:, 0]
        return k.contiguous(), v.contiguous()


PT, PC = 0, 1  # per-token, per-channel
ASYM, SYM = 0, 1
WHOLE = -1


def tiny(seed=0) -> Workload:
    """1 layer, batch 1, 8 KV heads = 8 query heads, head_dim 64, 512 tokens;
    fp32 N(0,1) with 2 key channels per head x20; K 4-bit per-channel G=32,
    V 4-bit per-token G=32, asymmetric."""
    return Workload("tiny", 1, 1, 8, 8, 64, [512], (4, 32, PC, ASYM), (4, 32, PT, ASYM), torch.float32,
                    key_outliers_per_head=2, key_outlier_scale=20.0, seed=seed)


def gpt2_small(kbits=4, vbits=4, kgroup=32, vgroup=32, kaxis=PC, vaxis=PT, seed=0, batch=8, tokens=2048,
               layers=12) -> Workload:
    """GPT-2-small-shaped cache: 12 layers, batch 8, 12 heads, head_dim 64,
    2048 tokens fp16 N(0,1) plus 1% of key channels x10."""
    return Workload(f"gpt2_small_k{kbits}v{vbits}_g{kgroup}_{vgroup}", layers, batch, 12, 12, 64, [tokens] * batch,
                    (kbits, kgroup, kaxis, ASYM), (vbits, vgroup, vaxis, ASYM), torch.float16,
                    key_outlier_frac=0.01, key_outlier_scale=10.0, seed=seed)


def llama2_13b(kaxis=PC, vaxis=PT, seed=0, batch=16, sealed=4096, tail=17, layers=40) -> Workload:
    """Llama-2-13B-shaped MHA cache: 40 layers, 40 KV heads, head_dim 128,
    batch 16, 4096 + 17 tokens fp16; keys with 4 fixed outlier channels per
    head x15, values N(0,1); 2-bit G=32."""
    return Workload(f"llama2_13b_{'kc' if kaxis else 'kt'}_{'vc' if vaxis else 'vt'}", layers, batch, 40, 40, 128,
                    [sealed + tail] * batch, (2, 32, kaxis, ASYM), (2, 32, vaxis, ASYM), torch.float16,
                    key_outliers_per_head=4, key_outlier_scale=15.0, seed=seed)


def wide_gqa(variant="k4v8", kaxis=PT, seed=0, tokens=131072) -> Workload:
    """head_dim 256, 16 query heads over 2 KV heads, batch 1, 131072 tokens
    fp16; RMS-normalised keys, N(0,1) values; K4/V8 with groups of 32
    channels, or symmetric 6-bit."""
    if variant == "k4v8":
        kc = (4, 32, kaxis, ASYM)
        vc = (8, 32, PT, ASYM)
    else:
        kc = (6, 32, kaxis, SYM)
        vc = (6, 32, PT, SYM)
    return Workload(f"wide_gqa_{variant}_{'kc' if kaxis else 'kt'}", 1, 1, 16, 2, 256, [tokens], kc, vc,
                    torch.float16, key_rmsnorm=True, seed=seed)


def serving_mix(seed=0, batch=64, lo=1024, hi=32768) -> Workload:
    """64 sequences with lengths uniform in [1k, 32k], 32 query heads over 8 KV
    heads, head_dim 128; keys N(0,1), values Laplace(0,1); K 2-bit per-channel
    G=64, V 2-bit per-token G=64."""
    return Workload("serving_mix", 1, batch, 32, 8, 128, ragged_lengths(batch, lo, hi, seed * 1000 + 77),
                    (2, 64, PC, ASYM), (2, 64, PT, ASYM), torch.float16, value_dist="laplace", seed=seed)


# ------------------------------------------------------------ registry ----

GPT2_BITS = (2, 3, 4, 6, 8)
GPT2_GROUPS = (32, 64, WHOLE)


def _gname(g):
    return "whole" if g == WHOLE else str(g)


def gpt2_variant(kbits, vbits, group, reading, layers=12) -> Workload:
    """One setting of the GPT-2-small bits x group sweep.  reading "pt": keys
    and values both grouped per token along channels (groups of 32 or 64
    channels of a head, or the whole 768-channel token vector); reading "pc":
    keys grouped per channel along `group` tokens (128 tokens for the "whole"
    column, the largest per-channel group), values per token along channels as
    in "pt"."""
    if reading == "pt":
        kc, vc = (kbits, group, PT), (vbits, group, PT)
    else:
        kc, vc = (kbits, 128 if group == WHOLE else group, PC), (vbits, group, PT)
    wl = gpt2_small(kbits=kbits, vbits=vbits, kgroup=kc[1], vgroup=vc[1], kaxis=kc[2], vaxis=vc[2], layers=layers)
    wl.name = f"gpt2_small_k{kbits}v{vbits}_g{_gname(group)}_{reading}"
    return wl


def _registry():
    reg = {"tiny": lambda layers=None: tiny()}
    for rd in ("pt", "pc"):
        for b in GPT2_BITS:
            for g in GPT2_GROUPS:
                reg[f"gpt2_small_k{b}v{b}_g{_gname(g)}_{rd}"] = (
                    lambda layers=None, b=b, g=g, rd=rd: gpt2_variant(b, b, g, rd, layers or 12))
        for kb, vb in ((6, 4), (4, 6)):
            reg[f"gpt2_small_k{kb}v{vb}_g64_{rd}"] = (
                lambda layers=None, kb=kb, vb=vb, rd=rd: gpt2_variant(kb, vb, 64, rd, layers or 12))
    for ka in (PC, PT):
        for va in (PT, PC):
            name = f"llama2_13b_{'kc' if ka else 'kt'}_{'vc' if va else 'vt'}"
            reg[name] = lambda layers=None, ka=ka, va=va: llama2_13b(kaxis=ka, vaxis=va, layers=layers or 40)
    for var in ("k4v8", "sym6"):
        for ka in (PT, PC):
            reg[f"wide_gqa_{var}_{'kc' if ka else 'kt'}"] = lambda layers=None, var=var, ka=ka: wide_gqa(var, ka)
    reg["serving_mix"] = lambda layers=None: serving_mix()
    return reg


WORKLOADS = _registry()
# short names of the headline setting of each workload
ALIASES = {"gpt2_small": "gpt2_small_k4v4_g32_pc", "gpt2_small_k6v4": "gpt2_small_k6v4_g64_pt",
           "llama2_13b": "llama2_13b_kc_vt", "wide_gqa": "wide_gqa_k4v8_kt"}
GROUPS = {
    "gpt2_sweep": [n for n in WORKLOADS if n.startswith("gpt2_small")],
    "llama2_13b_axes": [n for n in WORKLOADS if n.startswith("llama2_13b")],
    "wide_gqa_all": [n for n in WORKLOADS if n.startswith("wide_gqa")],
}
GROUPS["all"] = [n for n in WORKLOADS if n != "tiny"]


def workload(name: str, layers=None) -> Workload:
    """A registered workload by name (or alias), optionally with fewer layers."""
    name = ALIASES.get(name, name)
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name}")
    return WORKLOADS[name](layers)


def workload_names(spec: str) -> list:
    """Names of a comma-separated list of workloads, aliases or groups."""
    out = []
    for part in spec.split(","):
        part = part.strip()
        if part in GROUPS:
            out += GROUPS[part]
        elif part:
            out.append(ALIASES.get(part, part))
    return out
