"""Seeded synthetic decode workloads (inputs only -- none of the method's arithmetic).

Both the CUDA path and the CPU oracle are fed from here.  A workload is one
decode step of one layer: a query per sequence, the new token's K/V, a paged KV
pool holding each sequence's history, block tables, context lengths and the
slot mapping for the new token; the beam workload also carries copy-on-write
block pairs and swap-out / swap-in pairs.

The pool is generated as an opaque array of ``num_blocks`` chunks of
``2 * block_size * head_size`` elements per kv head: every element is drawn
from the workload's value distribution, so the generator needs no knowledge of
where inside a chunk a given (slot, dim) lives.  Blocks that no table uses can
be filled with NaN, so any stray read shows up in the output.

Shapes and distributions follow the five decode workloads the cache is
measured on (tiny MHA, Llama-2-7B-shaped MHA, Llama-3-8B-shaped GQA,
long-context 70B-shaped GQA, beam search with a shared prompt).  Metadata is
drawn with numpy's PCG64 (identical on every machine); pool values with a
seeded torch generator on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Config:
    name: str
    index: int              # seed = 1000 + index
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: str              # "f16" | "bf16"
    values: str             # "uniform" (U[-1, 1]) | "normal" (N(0, 1))
    ctx: tuple              # ("uniform", lo, hi) | ("lognormal", median, sigma, cap) | ("beam", prompt, tail_max)
    pool_blocks: int = 0    # fixed pool size; 0 -> 1.2 x the blocks the tables need
    beams: int = 1          # beams per prompt group (beam workload)
    swap_fraction: float = 0.0
    kv_int8: bool = False   # cache stored as 8-bit codes + scales (q/out/K/V stay `dtype`)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def ctx_cap(self) -> int:
        kind = self.ctx[0]
        if kind == "uniform":
            return self.ctx[2]
        if kind == "lognormal":
            return self.ctx[3]
        return self.ctx[1] + self.ctx[2] + 1


CONFIGS = {
    c.name: c for c in [
        Config("tiny", 0, 4, 4, 4, 64, 16, "f16", "uniform", ("uniform", 1, 100), pool_blocks=64),
        Config("7b", 1, 64, 32, 32, 128, 16, "f16", "normal", ("uniform", 512, 4096)),
        Config("8b", 2, 256, 32, 8, 128, 16, "bf16", "normal", ("lognormal", 1024, 0.8, 8192)),
        Config("70b", 3, 8, 64, 8, 128, 32, "bf16", "normal", ("uniform", 32768, 131072)),
        Config("beam", 4, 128, 32, 8, 128, 16, "bf16", "normal", ("beam", 2048, 256), beams=4,
               swap_fraction=0.10),
        # token-granular paging (block_size 1) on the Llama-2-7B-shaped layer
        Config("7b_bs1", 5, 64, 32, 32, 128, 1, "f16", "normal", ("uniform", 512, 4096)),
        # 8-bit KV cache on the 7B- and 8B-shaped layers
        Config("7b_int8", 6, 64, 32, 32, 128, 16, "f16", "normal", ("uniform", 512, 4096), kv_int8=True),
        Config("8b_int8", 7, 256, 32, 8, 128, 16, "bf16", "normal", ("lognormal", 1024, 0.8, 8192), kv_int8=True),
    ]
}


@dataclass
class Workload:
    cfg: Config
    num_blocks: int
    q: torch.Tensor                  # [S, Hq, D]
    key: torch.Tensor                # [S, Hkv, D]  new token's K
    value: torch.Tensor              # [S, Hkv, D]  new token's V
    kv_cache: torch.Tensor           # [NB, Hkv, 2 * bs * D] opaque chunks (16-bit caches; None for 8-bit)
    block_tables: torch.Tensor       # int32 [S, max_blocks_per_seq], unused entries = -1
    context_lens: torch.Tensor       # int32 [S], includes the new token
    slot_mapping: torch.Tensor       # int64 [S]
    max_context_len: int
    scale: float
    # host-side copies of the metadata (numpy)
    block_tables_np: np.ndarray = None
    context_lens_np: np.ndarray = None
    slot_mapping_np: np.ndarray = None
    used_blocks: np.ndarray = None   # physical blocks referenced by the tables
    # beam workload extras (host int64 [n, 2] (src, dst) pairs)
    block_tables_before_cow_np: np.ndarray = None
    copy_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    swap_out_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    swap_in_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    host_blocks: int = 0
    # sequences sharing their first blocks physically (beam groups): group g is
    # sequences group_start[g] .. group_start[g+1]-1, whose first prefix_lens[g]
    # tokens sit in the same blocks (device int32 tensors; None: no groups)
    group_start: torch.Tensor = None
    prefix_lens: torch.Tensor = None
    group_start_np: np.ndarray = None
    prefix_lens_np: np.ndarray = None
    # 8-bit caches: the history as logical 16-bit values [NB, Hkv, 2 (K, V), bs, D];
    # every slot of every block holds a drawn vector, quantised by whichever side
    # builds the cache from it
    kv_logical: torch.Tensor = None

    @property
    def dtype(self) -> torch.dtype:
        return DTYPES[self.cfg.dtype]


def draw_context_lens(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    kind = cfg.ctx[0]
    S = cfg.num_seqs
    if kind == "uniform":
        return rng.integers(cfg.ctx[1], cfg.ctx[2] + 1, size=S).astype(np.int32)
    if kind == "lognormal":
        median, sigma, cap = cfg.ctx[1:]
        x = np.rint(rng.lognormal(mean=math.log(median), sigma=sigma, size=S))
        return np.clip(x, 1, cap).astype(np.int32)
    prompt, tail_max = cfg.ctx[1:]
    tails = rng.integers(0, tail_max + 1, size=S)
    return (prompt + tails + 1).astype(np.int32)


def fill_values(t: torch.Tensor, values: str, gen: torch.Generator, chunk: int = 1 << 26) -> None:
    """Fill a 16-bit tensor in place with U[-1, 1] or N(0, 1) draws, chunk by chunk."""
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        if values == "uniform":
            x = torch.rand(n, generator=gen, device=t.device, dtype=torch.float32) * 2 - 1
        else:
            x = torch.randn(n, generator=gen, device=t.device, dtype=torch.float32)
        flat[i:i + n].copy_(x)


def make_workload(name_or_cfg, device="cpu", seed: int | None = None, nan_unused: bool = False,
                  num_seqs: int | None = None, max_context_len: int | None = None) -> Workload:
    """Build one decode step of the named workload on ``device``.

    num_seqs / max_context_len optionally shrink a workload (first sequences, contexts
    clipped) for fast CPU-side checks; the full shapes are the defaults.
    """
    cfg = CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    if num_seqs is not None:
        cfg = Config(**{**cfg.__dict__, "num_seqs": num_seqs})
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    S, Hq, Hkv, D, bs = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    ctx = draw_context_lens(cfg, rng)
    if max_context_len is not None:
        ctx = np.minimum(ctx, max_context_len).astype(np.int32)
    nblk = (ctx + bs - 1) // bs
    cap = cfg.ctx_cap if max_context_len is None else min(cfg.ctx_cap, max_context_len)
    width = (cap + bs - 1) // bs

    # Logical block lists; the beam workload shares prompt blocks within a group
    # and gives every beam one copy-on-write (old last block -> fresh block).
    if cfg.ctx[0] == "beam":
        prompt_blocks = cfg.ctx[1] // bs
        groups = S // cfg.beams
        n_shared = groups * prompt_blocks
        n_private = int(sum(nblk - prompt_blocks))   # includes each beam's old last block
        needed = n_shared + n_private + S            # + one fresh CoW block per beam
    else:
        needed = int(nblk.sum())
    NB = cfg.pool_blocks or int(math.ceil(1.2 * needed))
    assert NB >= needed, "pool too small for the workload"
    perm = rng.permutation(NB).astype(np.int64)

    tables = np.full((S, width), -1, dtype=np.int32)
    before = None
    copy_pairs = np.zeros((0, 2), np.int64)
    if cfg.ctx[0] == "beam":
        shared = perm[:n_shared].reshape(groups, prompt_blocks)
        nxt = n_shared
        before = np.full((S, width), -1, dtype=np.int32)
        pairs = []
        for s in range(S):
            g = s // cfg.beams
            priv = perm[nxt:nxt + nblk[s] - prompt_blocks]
            nxt += nblk[s] - prompt_blocks
            row = np.concatenate([shared[g], priv])
            before[s, :nblk[s]] = row
            fresh = perm[n_shared + n_private + s]
            pairs.append((row[-1], fresh))
            row = row.copy()
            row[-1] = fresh
            tables[s, :nblk[s]] = row
        copy_pairs = np.asarray(pairs, dtype=np.int64)
    else:
        nxt = 0
        for s in range(S):
            tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
            nxt += nblk[s]

    pos = ctx.astype(np.int64) - 1
    slots = tables[np.arange(S), pos // bs].astype(np.int64) * bs + pos % bs

    used = np.unique(tables[tables >= 0])
    swap_out = swap_in = np.zeros((0, 2), np.int64)
    host_blocks = 0
    if cfg.swap_fraction > 0:
        n_swap = int(round(cfg.swap_fraction * used.size))
        picked = rng.choice(used, size=n_swap, replace=False).astype(np.int64)
        host_ids = np.arange(n_swap, dtype=np.int64)
        swap_out = np.stack([picked, host_ids], axis=1)
        swap_in = np.stack([host_ids, picked], axis=1)
        host_blocks = n_swap

    dt = DTYPES[cfg.dtype]
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.empty((S, Hq, D), dtype=dt, device=dev)
    key = torch.empty((S, Hkv, D), dtype=dt, device=dev)
    value = torch.empty((S, Hkv, D), dtype=dt, device=dev)
    pool = torch.empty((NB, Hkv, 2 * bs * D), dtype=dt, device=dev)
    for t in (q, key, value, pool):
        fill_values(t, cfg.values, gen)
    logical = None
    if cfg.kv_int8:
        logical, pool = pool.view(NB, Hkv, 2, bs, D), None
        nan_unused = False      # an 8-bit cache has no NaN codes to plant
    if nan_unused:
        keep = np.zeros(NB, dtype=bool)
        keep[used] = True
        if copy_pairs.size:
            keep[copy_pairs[:, 0]] = True
        unused = torch.from_numpy(np.nonzero(~keep)[0]).to(dev)
        if unused.numel():
            pool[unused] = float("nan")

    group_start = prefix_lens = None
    if cfg.ctx[0] == "beam":
        group_start = np.arange(0, S + 1, cfg.beams, dtype=np.int32)
        prefix_lens = np.full(S // cfg.beams, cfg.ctx[1], dtype=np.int32)   # the shared prompt blocks
    return Workload(
        cfg=cfg, num_blocks=NB, q=q, key=key, value=value, kv_cache=pool,
        block_tables=torch.from_numpy(tables).to(dev),
        context_lens=torch.from_numpy(ctx).to(dev),
        slot_mapping=torch.from_numpy(slots).to(dev),
        max_context_len=int(cap), scale=1.0 / math.sqrt(D),
        block_tables_np=tables, context_lens_np=ctx, slot_mapping_np=slots, used_blocks=used,
        block_tables_before_cow_np=before, copy_pairs=copy_pairs,
        swap_out_pairs=swap_out, swap_in_pairs=swap_in, host_blocks=host_blocks, kv_logical=logical,
        group_start=None if group_start is None else torch.from_numpy(group_start).to(dev),
        prefix_lens=None if prefix_lens is None else torch.from_numpy(prefix_lens).to(dev),
        group_start_np=group_start, prefix_lens_np=prefix_lens,
    )


def as_u16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit pattern of a CPU/GPU fp16/bf16 tensor as a numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ------------------------------------------------------------------ prefill / extend

@dataclass(frozen=True)
class PrefillConfig:
    name: str
    index: int              # seed = 2000 + index
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: str
    q_len: int              # new tokens per sequence (a prompt, or a chunk of one)
    prefix: tuple           # cached tokens before them: ("fixed", n) | ("uniform", lo, hi)

    @property
    def seed(self) -> int:
        return 2000 + self.index


PREFILL_CONFIGS = {
    c.name: c for c in [
        # whole prompts: 16 x 2048 tokens on a Llama-3-8B-shaped layer
        PrefillConfig("prefill_8b", 0, 16, 32, 8, 128, 16, "bf16", 2048, ("fixed", 0)),
        # chunked prefill: 512-token chunks over cached prefixes of 512..3584 tokens
        PrefillConfig("extend_8b", 1, 32, 32, 8, 128, 16, "bf16", 512, ("uniform", 512, 3584)),
        # whole prompts on a Llama-2-7B-shaped (MHA) layer
        PrefillConfig("prefill_7b", 2, 8, 32, 32, 128, 16, "f16", 2048, ("fixed", 0)),
        # small case for parity tests
        PrefillConfig("prefill_tiny", 3, 3, 8, 2, 128, 16, "bf16", 100, ("uniform", 0, 300)),
    ]
}


@dataclass
class PrefillWorkload:
    cfg: PrefillConfig
    num_blocks: int
    q: torch.Tensor                  # [T, Hq, D] packed new tokens
    key: torch.Tensor                # [T, Hkv, D] their K
    value: torch.Tensor              # [T, Hkv, D] their V
    kv_cache: torch.Tensor           # [NB, Hkv, 2 * bs * D] opaque chunks (history)
    block_tables: torch.Tensor       # int32 [S, W]
    context_lens: torch.Tensor       # int32 [S] = prefix + q_len
    query_start_loc: torch.Tensor    # int32 [S + 1]
    slot_mapping: torch.Tensor       # int64 [T] slots of the new tokens
    max_query_len: int
    scale: float
    block_tables_np: np.ndarray = None
    context_lens_np: np.ndarray = None
    query_start_loc_np: np.ndarray = None
    slot_mapping_np: np.ndarray = None

    @property
    def dtype(self) -> torch.dtype:
        return DTYPES[self.cfg.dtype]


def make_prefill_workload(name_or_cfg, device="cpu", seed: int | None = None) -> PrefillWorkload:
    cfg = PREFILL_CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    S, Hq, Hkv, D, bs = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    if cfg.prefix[0] == "fixed":
        prefix = np.full(S, cfg.prefix[1], dtype=np.int64)
    else:
        prefix = rng.integers(cfg.prefix[1], cfg.prefix[2] + 1, size=S)
    ctx = (prefix + cfg.q_len).astype(np.int32)
    nblk = (ctx + bs - 1) // bs
    width = int(nblk.max())
    NB = int(math.ceil(1.2 * int(nblk.sum())))
    perm = rng.permutation(NB).astype(np.int64)
    tables = np.full((S, width), -1, dtype=np.int32)
    nxt = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
        nxt += nblk[s]
    qsl = np.concatenate([[0], np.cumsum(np.full(S, cfg.q_len))]).astype(np.int32)
    pos = np.concatenate([np.arange(prefix[s], ctx[s]) for s in range(S)]).astype(np.int64)
    seq = np.repeat(np.arange(S), cfg.q_len)
    slots = tables[seq, pos // bs].astype(np.int64) * bs + pos % bs
    T = int(qsl[-1])
    dt = DTYPES[cfg.dtype]
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.empty((T, Hq, D), dtype=dt, device=dev)
    key = torch.empty((T, Hkv, D), dtype=dt, device=dev)
    value = torch.empty((T, Hkv, D), dtype=dt, device=dev)
    pool = torch.empty((NB, Hkv, 2 * bs * D), dtype=dt, device=dev)
    for t in (q, key, value, pool):
        fill_values(t, "normal", gen)
    return PrefillWorkload(
        cfg=cfg, num_blocks=NB, q=q, key=key, value=value, kv_cache=pool,
        block_tables=torch.from_numpy(tables).to(dev), context_lens=torch.from_numpy(ctx).to(dev),
        query_start_loc=torch.from_numpy(qsl).to(dev), slot_mapping=torch.from_numpy(slots).to(dev),
        max_query_len=cfg.q_len, scale=1.0 / math.sqrt(D),
        block_tables_np=tables, context_lens_np=ctx, query_start_loc_np=qsl, slot_mapping_np=slots,
    )
