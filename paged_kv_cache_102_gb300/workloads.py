"""Seeded synthetic decode workloads.

This module draws inputs only: context lengths, a shuffled free-block order,
and N(0, 1) values for queries, new keys/values and the pre-filled pool.  It
holds none of the method's arithmetic (no slot mapping, no table building, no
attention), so the float64 oracle and the CUDA path can both be fed from it.

Shapes follow the pages' workloads: 16-token blocks by default and 32 as the
alternative (Ultralytics glossary "PagedAttention", section "How paging
works"; iThome "how to store the KV cache", section "PagedAttention"),
grouped-query heads and an 8-bit cache (Ultralytics glossary, section
"Related techniques"), and parallel sampling over a shared prompt (Ultralytics
glossary, section "Sharing blocks between sequences").  Request lengths are in
the range of OptiVerse "Paged KV cache" (725-1525 tokens per request).

Draw order for a seed: context lengths (numpy PCG64), then the free-block
permutation (same generator), then tensor values (a torch generator seeded
with the same seed on the target device).  ``context_lens`` are the tokens
already in the cache before the decode step's append, so the step attends over
``context_lens + 1`` tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    act_dtype: str  # "f16" | "bf16": queries, new K/V, output
    cache_dtype: str  # "f16" | "bf16" | "e4m3"
    lens: tuple  # ("fixed", values) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    pool_blocks: int = 0  # 0: 1.25 x the blocks the batch needs after its append
    partition_size: int = 512
    samples_per_prompt: int = 1  # > 1: parallel sampling over shared prompts
    divergent_tokens: tuple = (0, 0)  # per-sample extra tokens (uniform, inclusive)
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 4, 8, 8, 64, 16, "f16", "f16", ("fixed", (40, 17, 33, 1)), pool_blocks=64,
        description="4 sequences, context_lens {40,17,33,1}, 8 MHA heads, head_dim 64, block 16, "
                    "fp16 pool of 64 blocks"),
    "llama7b": Workload(
        "llama7b", 64, 32, 32, 128, 16, "bf16", "bf16", ("uniform", 128, 2048),
        description="Llama-7B-shaped decode: batch 64, 32 MHA heads, head_dim 128, bf16, block 16, "
                    "context_lens uniform in [128, 2048], pool 1.25x the blocks needed"),
    "gqa_bs16": Workload(
        "gqa_bs16", 128, 64, 8, 128, 16, "bf16", "bf16", ("lognormal", 1024, 1.0, 16, 8192),
        description="GQA decode: batch 128, 64 query heads over 8 KV heads, head_dim 128, bf16, "
                    "block 16, context_lens log-normal (median 1024, sigma 1) clipped to [16, 8192]"),
    "gqa_bs32": Workload(
        "gqa_bs32", 128, 64, 8, 128, 32, "bf16", "bf16", ("lognormal", 1024, 1.0, 16, 8192),
        description="GQA decode as gqa_bs16 with block 32"),
    "gqa_fp8": Workload(
        "gqa_fp8", 128, 64, 8, 128, 16, "bf16", "e4m3", ("lognormal", 1024, 1.0, 16, 8192),
        description="GQA decode as gqa_bs16 with an FP8-E4M3 cache (per-tensor scales from the N(0,1) data)"),
    "shared_prefix": Workload(
        "shared_prefix", 32, 32, 32, 128, 16, "f16", "f16", ("uniform_not_multiple", 1000, 1030),
        samples_per_prompt=4, divergent_tokens=(0, 256),
        description="32 prompts x 4 samples, 32 heads, head_dim 128, fp16, block 16; prompts of "
                    "1000-1030 tokens (never a multiple of 16, so the last block is partial) shared "
                    "by the 4 samples; each sample then appends 0-256 divergent tokens"),
    "fp8_13b": Workload(
        "fp8_13b", 256, 40, 40, 128, 16, "bf16", "e4m3", ("uniform", 256, 4096),
        description="13B-shaped decode with an FP8-E4M3 cache: batch 256, 40 MHA heads, head_dim "
                    "128, per-tensor scales from the N(0,1) data, bf16 q/out, context_lens uniform "
                    "in [256, 4096]"),
    # shapes at the edges of the tensor-core kernel's envelope
    "gqa_g2": Workload(
        "gqa_g2", 128, 16, 8, 128, 16, "bf16", "bf16", ("lognormal", 1024, 1.0, 16, 8192),
        description="GQA decode with 2 query heads per KV head: batch 128, 16 query heads over 8 KV heads, "
                    "head_dim 128, bf16, block 16, lengths as gqa_bs16"),
    "gqa_d64": Workload(
        "gqa_d64", 128, 64, 8, 64, 16, "bf16", "bf16", ("lognormal", 1024, 1.0, 16, 8192),
        description="GQA decode at head_dim 64: batch 128, 64 query heads over 8 KV heads, bf16, block 16, "
                    "lengths as gqa_bs16"),
    "gqa_wide": Workload(
        "gqa_wide", 4096, 64, 8, 128, 16, "bf16", "bf16", ("uniform", 64, 512),
        description="GQA decode over a wide batch: 4096 sequences, 64 query heads over 8 KV heads, head_dim "
                    "128, bf16, block 16, context_lens uniform in [64, 512]"),
    "long_gqa": Workload(
        "long_gqa", 8, 32, 8, 128, 16, "bf16", "bf16", ("fixed", (32767,) * 8),
        description="8 sequences x 32768 tokens (after the append), 32 query heads over 8 KV heads, "
                    "head_dim 128, bf16, block 16, split into 512-token partitions"),
}


def _draw_lens(wl: Workload, rng: np.random.Generator, n: int) -> np.ndarray:
    kind = wl.lens[0]
    if kind == "fixed":
        return np.asarray(wl.lens[1], dtype=np.int32)
    if kind == "uniform":
        return rng.integers(wl.lens[1], wl.lens[2], size=n, endpoint=True).astype(np.int32)
    if kind == "uniform_not_multiple":
        lo, hi = wl.lens[1], wl.lens[2]
        choices = np.asarray([x for x in range(lo, hi + 1) if x % wl.block_size != 0])
        return rng.choice(choices, size=n).astype(np.int32)
    if kind == "lognormal":
        median, sigma, lo, hi = wl.lens[1:]
        x = np.floor(np.exp(rng.normal(math.log(median), sigma, size=n)))
        return np.clip(x, lo, hi).astype(np.int32)
    raise ValueError(kind)


@dataclass
class Draw:
    workload: Workload
    seed: int
    context_lens: np.ndarray  # int32 [num_seqs]: tokens in cache before the append
    prompt_lens: np.ndarray  # shared-prefix only: int32 [num_prompts]
    divergent: np.ndarray  # shared-prefix only: int32 [num_seqs] extra tokens per sample
    num_blocks: int
    free_list: np.ndarray  # int32 [num_blocks]: seeded permutation of the pool


def draw(name_or_wl, seed: int = 0) -> Draw:
    """Draw lengths and the free-block order of a workload for ``seed``."""
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    rng = np.random.Generator(np.random.PCG64(seed))
    bs = wl.block_size
    if wl.samples_per_prompt > 1:
        prompts = _draw_lens(wl, rng, wl.batch)
        n = wl.batch * wl.samples_per_prompt
        div = rng.integers(wl.divergent_tokens[0], wl.divergent_tokens[1], size=n, endpoint=True)
        div = div.astype(np.int32)
        ctx = np.repeat(prompts, wl.samples_per_prompt).astype(np.int32) + div
        need = int(sum(-(-p // bs) for p in prompts))
        need += int(sum(-(-(c + 1) // bs) - (p // bs) for c, p in zip(ctx, np.repeat(prompts, wl.samples_per_prompt))))
    else:
        prompts = np.zeros(0, np.int32)
        ctx = _draw_lens(wl, rng, wl.batch)
        div = np.zeros(len(ctx), np.int32)
        need = int(sum(-(-(c + 1) // bs) for c in ctx))
    nb = wl.pool_blocks or int(math.ceil(1.25 * need))
    perm = rng.permutation(nb).astype(np.int32)
    return Draw(wl, seed, ctx, prompts, div, nb, perm)


def make_values(d: Draw, device="cpu", pool=True):
    """N(0, 1) tensors for a draw, on ``device``.

    Returns a dict with q [B, Hq, D], k_new, v_new [B, Hkv, D] (activation
    dtype) and, if ``pool``, the pre-filled pool k_cache, v_cache
    [NB, Hkv, bs, D].  For an E4M3 cache the pool holds E4M3 codes (uint8) of
    N(0,1)/scale clamped to +-448 and converted by torch, with per-tensor
    scales scale = amax|x| / 448 as float32 tensors ``k_scale``/``v_scale``.
    """
    wl = d.workload
    g = torch.Generator(device=device)
    g.manual_seed(d.seed)
    B = len(d.context_lens)
    act = DTYPES[wl.act_dtype]
    out = {}
    out["q"] = torch.randn(B, wl.num_q_heads, wl.head_dim, generator=g, device=device).to(act)
    out["k_new"] = torch.randn(B, wl.num_kv_heads, wl.head_dim, generator=g, device=device).to(act)
    out["v_new"] = torch.randn(B, wl.num_kv_heads, wl.head_dim, generator=g, device=device).to(act)
    if not pool:
        return out
    shape = (d.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    if wl.cache_dtype == "e4m3":
        for name in ("k", "v"):
            x = torch.empty(shape, dtype=torch.uint8, device=device)
            flat = x.view(d.num_blocks, -1)
            step = max(1, (1 << 26) // flat.shape[1])
            # pass 1 takes amax over the values; pass 2 replays the same generator stream
            state = g.get_state()
            amax = torch.zeros((), dtype=torch.float32, device=device)
            for i in range(0, d.num_blocks, step):
                vals = torch.randn(min(step, d.num_blocks - i), flat.shape[1], generator=g, device=device)
                amax = torch.maximum(amax, vals.abs().max())
            scale = (amax / 448.0).to(torch.float32)
            g.set_state(state)
            for i in range(0, d.num_blocks, step):
                vals = torch.randn(min(step, d.num_blocks - i), flat.shape[1], generator=g, device=device) / scale
                flat[i:i + vals.shape[0]] = vals.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            out[f"{name}_cache"] = x
            out[f"{name}_scale"] = scale.reshape(1)
    else:
        cd = DTYPES[wl.cache_dtype]
        for name in ("k", "v"):
            x = torch.empty(shape, dtype=cd, device=device)
            flat = x.view(d.num_blocks, -1)
            step = max(1, (1 << 26) // flat.shape[1])
            for i in range(0, d.num_blocks, step):
                n = min(step, d.num_blocks - i)
                flat[i:i + n] = torch.randn(n, flat.shape[1], generator=g, device=device).to(cd)
            out[f"{name}_cache"] = x
    return out
