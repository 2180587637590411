"""Seeded synthetic inputs for the paged decode step.

This module only draws numbers: sequence lengths, the shuffled order of the
pool's free blocks, and N(0,1) values for q, k and v.  It holds none of the
step's arithmetic (no block tables, no slots, no attention), so the CUDA path
and the CPU oracle can both take their inputs from it.

Workloads (shapes from the pages' running examples):
  tiny           4 sequences with context {1,17,100,33}: prior lengths
                 {0,16,99,32} plus one new token each; 4 q / 2 kv heads,
                 head_dim 64, fp16, 64-block pool in a seeded random order,
                 scale 1/8.
  opt13b         one OPT-13B layer (MHA 40 x 128, fp16): 64 sequences with
                 context uniform in [128, 2048], 16,384-block shuffled pool.
  gqa_long       GQA 32 q / 8 kv heads, head_dim 128, bf16, 256 sequences,
                 context = clip(round(LogNormal(ln 4096, 1.0)), 64, 32768),
                 shuffled pool of 1.1 x the blocks needed (+ growth room).
  shared_prefix  128 sequences sharing a 1024-token prefix (64 blocks) plus a
                 private suffix uniform in [64, 512] tokens; GQA 32/8, bf16.
  trace          continuous-batching schedule: Poisson(8) arrivals per step,
                 prompts uniform [64, 1024], output lengths geometric with
                 mean 200 capped at 2048; 40 GiB pool of 64 KiB blocks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass
class DecodeWorkload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f16" or "bf16"
    scale: float
    prior_lens: np.ndarray          # int32 [S]: tokens in the cache before this step
    new_tokens: np.ndarray          # int32 [S]: tokens appended this step
    num_blocks: int                 # pool size in blocks
    free_order: np.ndarray          # int32 [num_blocks]: seeded shuffled pool order
    max_blocks_per_seq: int
    block_size: int = BLOCK_SIZE
    shared_prefix_tokens: int = 0   # tokens every sequence shares (shared_prefix only)
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(len(self.prior_lens))

    @property
    def is_bf16(self) -> bool:
        return self.dtype == "bf16"


def _shuffled(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.permutation(n).astype(np.int32)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def tiny(seed: int = 0) -> DecodeWorkload:
    rng = np.random.default_rng(seed)
    prior = np.array([0, 16, 99, 32], dtype=np.int32)
    return DecodeWorkload("tiny", 4, 2, 64, "f16", 1.0 / 8.0, prior,
                          np.ones(4, dtype=np.int32), 64, _shuffled(rng, 64),
                          max_blocks_per_seq=8, seed=seed)


def opt13b(seed: int = 0) -> DecodeWorkload:
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 2048, size=64, endpoint=True).astype(np.int32)
    return DecodeWorkload("opt13b", 40, 40, 128, "f16", 1.0 / math.sqrt(128), ctx - 1,
                          np.ones(64, dtype=np.int32), 16384, _shuffled(rng, 16384),
                          max_blocks_per_seq=_ceil_div(2048, BLOCK_SIZE) + 4, seed=seed)


def gqa_long(seed: int = 0, num_seqs: int = 256, growth_tokens: int = 64) -> DecodeWorkload:
    """GQA 32/8 long-context decode.  ``growth_tokens`` leaves table and pool room
    for that many further decode steps per sequence."""
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(rng.lognormal(math.log(4096.0), 1.0, size=num_seqs)), 64, 32768)
    ctx = ctx.astype(np.int32)
    need = int(sum(_ceil_div(int(n) + growth_tokens, BLOCK_SIZE) for n in ctx))
    num_blocks = int(math.ceil(1.1 * need))
    maxb = _ceil_div(32768 + growth_tokens, BLOCK_SIZE)
    return DecodeWorkload("gqa_long", 32, 8, 128, "bf16", 1.0 / math.sqrt(128), ctx - 1,
                          np.ones(num_seqs, dtype=np.int32), num_blocks,
                          _shuffled(rng, num_blocks), max_blocks_per_seq=maxb, seed=seed,
                          extra={"growth_tokens": growth_tokens})


def shared_prefix(seed: int = 0, growth_tokens: int = 64) -> DecodeWorkload:
    rng = np.random.default_rng(seed)
    prefix = 1024
    suffix = rng.integers(64, 512, size=128, endpoint=True).astype(np.int32)
    need = _ceil_div(prefix, BLOCK_SIZE) + int(
        sum(_ceil_div(int(x) + growth_tokens, BLOCK_SIZE) for x in suffix))
    num_blocks = int(math.ceil(1.1 * need))
    maxb = _ceil_div(prefix + 512 + growth_tokens, BLOCK_SIZE)
    # suffix counts the private tokens including this step's new one
    return DecodeWorkload("shared_prefix", 32, 8, 128, "bf16", 1.0 / math.sqrt(128),
                          prefix + suffix - 1, np.ones(128, dtype=np.int32), num_blocks,
                          _shuffled(rng, num_blocks), max_blocks_per_seq=maxb,
                          shared_prefix_tokens=prefix, seed=seed)


def small_random(seed: int, num_seqs: int, max_len: int, num_q_heads: int,
                 num_kv_heads: int, head_dim: int, dtype: str,
                 include_empty: bool = False) -> DecodeWorkload:
    """Randomised small shapes for parity sweeps: lengths uniform in [1, max_len]
    (optionally with some zero-length sequences), pool 25% larger than needed."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, max_len, size=num_seqs, endpoint=True).astype(np.int32)
    new = np.ones(num_seqs, dtype=np.int32)
    if include_empty:
        empty = rng.random(num_seqs) < 0.2
        ctx[empty] = 0
        new[empty] = 0
    need = int(sum(_ceil_div(int(n), BLOCK_SIZE) for n in ctx)) + 1
    num_blocks = int(math.ceil(1.25 * need)) + 4
    maxb = _ceil_div(max_len, BLOCK_SIZE) + 1
    return DecodeWorkload(f"random{seed}", num_q_heads, num_kv_heads, head_dim, dtype,
                          1.0 / math.sqrt(head_dim), ctx - new, new, num_blocks,
                          _shuffled(rng, num_blocks), max_blocks_per_seq=maxb, seed=seed)


CONFIGS = {"tiny": tiny, "opt13b": opt13b, "gqa_long": gqa_long,
           "shared_prefix": shared_prefix}


# --------------------------------------------------------------------- values
def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) values as fp16 or bf16 bit patterns (uint16)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(x)
    raise ValueError(dtype)


def host_values(w: DecodeWorkload, seed_offset: int = 1000) -> dict:
    """Host (numpy) values for a workload, as uint16 bit patterns.

    q        [S][Hq][D]              query of this step
    k_prompt [sum prior - shared][Hkv][D]  K rows of the tokens already cached,
             sequence after sequence (the shared prefix, if any, is its own
             array ``k_shared`` [shared_prefix_tokens][Hkv][D])
    k_new    [sum new][Hkv][D]       K rows of this step's tokens
    (and the same for v)
    """
    rng = np.random.default_rng(w.seed + seed_offset)
    S, hq, hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    private = int(np.sum(w.prior_lens)) - S * w.shared_prefix_tokens
    out = {
        "q": normal_bits(rng, (S, hq, d), w.dtype),
        "k_prompt": normal_bits(rng, (private, hkv, d), w.dtype),
        "v_prompt": normal_bits(rng, (private, hkv, d), w.dtype),
        "k_new": normal_bits(rng, (int(np.sum(w.new_tokens)), hkv, d), w.dtype),
        "v_new": normal_bits(rng, (int(np.sum(w.new_tokens)), hkv, d), w.dtype),
    }
    if w.shared_prefix_tokens:
        out["k_shared"] = normal_bits(rng, (w.shared_prefix_tokens, hkv, d), w.dtype)
        out["v_shared"] = normal_bits(rng, (w.shared_prefix_tokens, hkv, d), w.dtype)
    return out


def device_values(w: DecodeWorkload, device, seed_offset: int = 1000) -> dict:
    """Same arrays as :func:`host_values` (same shapes, same N(0,1) law), drawn on
    the GPU with torch's seeded generator for workloads too big to draw on the
    host quickly.  Returned as torch tensors of the workload dtype."""
    import torch
    tdt = torch.bfloat16 if w.is_bf16 else torch.float16
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + seed_offset)
    S, hq, hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    private = int(np.sum(w.prior_lens)) - S * w.shared_prefix_tokens
    n_new = int(np.sum(w.new_tokens))

    def draw(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(tdt)

    out = {"q": draw(S, hq, d), "k_prompt": draw(private, hkv, d),
           "v_prompt": draw(private, hkv, d), "k_new": draw(n_new, hkv, d),
           "v_new": draw(n_new, hkv, d)}
    if w.shared_prefix_tokens:
        out["k_shared"] = draw(w.shared_prefix_tokens, hkv, d)
        out["v_shared"] = draw(w.shared_prefix_tokens, hkv, d)
    return out


# ---------------------------------------------------------------------- trace
@dataclass
class TraceSchedule:
    """Arrivals of a continuous-batching run: for each step, the requests that
    arrive, each with a prompt length and an output length."""
    steps: int
    arrivals: list                  # per step: list of (prompt_len, output_len)
    max_running: int
    num_blocks: int
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    dtype: str = "bf16"
    block_size: int = BLOCK_SIZE
    seed: int = 0


def trace(seed: int = 5, steps: int = 500, rate: float = 8.0, max_running: int = 512,
          pool_bytes: int = 40 * 2**30) -> TraceSchedule:
    rng = np.random.default_rng(seed)
    block_bytes = 2 * 8 * BLOCK_SIZE * 128 * 2        # K+V of one 16-token block, 8 kv heads, bf16
    arrivals = []
    for _ in range(steps):
        k = int(rng.poisson(rate))
        prompts = rng.integers(64, 1024, size=k, endpoint=True)
        outs = np.minimum(rng.geometric(1.0 / 200.0, size=k), 2048)
        arrivals.append([(int(p), int(o)) for p, o in zip(prompts, outs)])
    return TraceSchedule(steps, arrivals, max_running, pool_bytes // block_bytes, seed=seed)
