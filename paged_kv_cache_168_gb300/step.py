"""One decode step of one layer over a workload, through the C ABI.

Order within a step (what a scheduler's output asks the cache engine for, then
the attention layer): swap_out -> swap_in -> copy_blocks (copy-on-write) ->
reshape_and_cache (the new token's K/V) -> paged decode.  All buffers (output,
workspace, pinned host pool, error word) are allocated once here, outside the
step; the step itself only launches kernels on one stream.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib
from .workloads import Workload


def unique_kv_tokens(block_tables: np.ndarray, context_lens: np.ndarray, block_size: int) -> int:
    """Distinct cache slots one decode step reads: for each physical block, the
    most tokens any sequence attends in it.  Blocks that several sequences share
    (a beam group's prompt) count once, which is what HBM must deliver when the
    other readers hit L2."""
    ctx = context_lens.astype(np.int64)
    nblk = -(-ctx // block_size)
    j = np.arange(block_tables.shape[1])[None, :]
    valid = j < nblk[:, None]
    tokens = np.clip(ctx[:, None] - j * block_size, 0, block_size)[valid]
    phys = block_tables[valid].astype(np.int64)
    if phys.size == 0:
        return 0
    best = np.zeros(int(phys.max()) + 1, np.int64)
    np.maximum.at(best, phys, tokens)
    return int(best.sum())


class DecodeStep:
    """One decode step over a workload.  For an 8-bit cache the pool is built
    here (outside any timed step) by writing the workload's logical history into
    every slot of every block with pa_reshape_and_cache, which quantises it."""

    def __init__(self, w: Workload, partition_size: int = 0, stream: torch.cuda.Stream | None = None,
                 nvtx: bool = False, shared_prefix: bool | None = None):
        cfg = w.cfg
        dev = w.q.device
        self.w = w
        self.stream = stream or torch.cuda.current_stream(dev)
        self.nvtx = nvtx                 # an NVTX range around every library call (for profilers)
        self.desc = _lib.CacheDesc(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, w.dtype,
                                   kv_int8=cfg.kv_int8)
        self.block_bytes = _lib.cache_bytes(self.desc) // w.num_blocks
        if cfg.kv_int8:
            self.kv_cache = torch.zeros(_lib.cache_bytes(self.desc), dtype=torch.uint8, device=dev)
            self.fill_from_logical(w.kv_logical)
        else:
            self.kv_cache = w.kv_cache
        self.partition_size = partition_size
        self.out = torch.empty_like(w.q)
        # a workload whose sequences share their first blocks (beam groups) is
        # decoded with pa_decode_shared_prefix, which reads those blocks once
        self.shared_prefix = (w.group_start is not None) if shared_prefix is None else shared_prefix
        if self.shared_prefix:
            nbytes = _lib.decode_shared_prefix_workspace_bytes(self.desc, cfg.num_seqs, cfg.num_q_heads,
                                                               self.num_groups, w.max_context_len, partition_size)
        else:
            nbytes = _lib.decode_workspace_bytes(self.desc, cfg.num_seqs, cfg.num_q_heads, w.max_context_len,
                                                 partition_size)
        self.workspace = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.host_pool = None
        if w.host_blocks:
            self.host_desc = _lib.CacheDesc(w.host_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size,
                                            w.dtype, kv_int8=cfg.kv_int8)
            self.host_pool = torch.empty(w.host_blocks * self.block_bytes, dtype=torch.uint8).pin_memory()

    def fill_from_logical(self, logical: torch.Tensor, chunk_blocks: int = 4096):
        """Write logical K/V [NB, Hkv, 2, bs, D] into slot b * bs + t of every block b."""
        NB, Hkv, _, bs, D = logical.shape
        for b0 in range(0, NB, chunk_blocks):
            part = logical[b0:b0 + chunk_blocks]
            n = part.shape[0] * bs
            key = part[:, :, 0].permute(0, 2, 1, 3).reshape(n, Hkv, D).contiguous()
            value = part[:, :, 1].permute(0, 2, 1, 3).reshape(n, Hkv, D).contiguous()
            slots = torch.arange(b0 * bs, b0 * bs + n, dtype=torch.int64, device=logical.device)
            _lib.reshape_and_cache(self.kv_cache, self.desc, key, value, slots, stream=self.stream)

    @property
    def num_groups(self) -> int:
        return 0 if self.w.group_start is None else int(self.w.prefix_lens.shape[0])

    def partition(self) -> int:
        """The partition size the decode call takes."""
        cfg = self.w.cfg
        if self.shared_prefix:
            return _lib.decode_shared_prefix_partition_size(self.desc, cfg.num_seqs, cfg.num_q_heads, self.num_groups,
                                                            self.w.max_context_len, self.partition_size)
        return _lib.decode_partition_size(self.desc, cfg.num_seqs, self.w.max_context_len, self.partition_size)

    def _range(self, name):
        if self.nvtx:
            torch.cuda.nvtx.range_push(name)

    def _end(self):
        if self.nvtx:
            torch.cuda.nvtx.range_pop()

    def cache_ops(self):
        w, s = self.w, self.stream
        if self.host_pool is not None:
            self._range("pa_swap_blocks out")
            _lib.swap_blocks(self.host_pool, self.host_desc, self.kv_cache, self.desc, 0, w.swap_out_pairs, stream=s)
            self._end()
            self._range("pa_swap_blocks in")
            _lib.swap_blocks(self.kv_cache, self.desc, self.host_pool, self.host_desc, 1, w.swap_in_pairs, stream=s)
            self._end()
        if w.copy_pairs.shape[0]:
            self._range("pa_copy_blocks")
            _lib.copy_blocks(self.kv_cache, self.desc, w.copy_pairs, stream=s)
            self._end()
        self._range("pa_reshape_and_cache")
        _lib.reshape_and_cache(self.kv_cache, self.desc, w.key, w.value, w.slot_mapping, dev_err=self.dev_err,
                               stream=s)
        self._end()

    def attention(self, q=None, out=None):
        w = self.w
        if self.shared_prefix:
            self._range("pa_decode_shared_prefix")
            _lib.decode_shared_prefix(self.out if out is None else out, w.q if q is None else q, self.kv_cache,
                                      self.desc, w.block_tables, w.context_lens, w.max_context_len, w.scale,
                                      w.group_start, w.prefix_lens, self.workspace, self.partition_size,
                                      dev_err=self.dev_err, stream=self.stream)
        else:
            self._range("pa_decode")
            _lib.decode(self.out if out is None else out, w.q if q is None else q, self.kv_cache, self.desc,
                        w.block_tables, w.context_lens, w.max_context_len, w.scale, self.workspace,
                        self.partition_size, dev_err=self.dev_err, stream=self.stream)
        self._end()

    def __call__(self):
        self.cache_ops()
        self.attention()
        return self.out

    def kernel_launches(self) -> int:
        """Kernels one step launches."""
        w, cfg = self.w, self.w.cfg
        n = 1                                                   # reshape_and_cache
        per = 1024                                              # pairs per copy launch
        if self.host_pool is not None:
            n += -(-w.swap_out_pairs.shape[0] // per) + -(-w.swap_in_pairs.shape[0] // per)
        if w.copy_pairs.shape[0]:
            n += -(-w.copy_pairs.shape[0] // per)
        if self.shared_prefix and self.num_groups > 0:
            return n + 2                                        # decode + merge
        P = self.partition()
        n += 1 + (1 if -(-w.max_context_len // P) > 1 else 0)   # decode (+ merge)
        return n

    def algorithmic_bytes(self) -> dict:
        """Bytes the method must move per step (what each kernel reads + writes)."""
        w, cfg = self.w, self.w.cfg
        esz = 2
        in_tok = 2 * cfg.num_kv_heads * cfg.head_size * esz        # one token's K and V, 16-bit
        # one token's K and V as stored: 16-bit, or 8-bit codes + two fp32 scales per kv head
        kv_tok = cfg.num_kv_heads * (2 * cfg.head_size + 8) if cfg.kv_int8 else in_tok
        ctx = w.context_lens_np.astype("int64")
        nblk = -(-ctx // cfg.block_size)
        decode = int(ctx.sum()) * kv_tok + 2 * cfg.num_seqs * cfg.num_q_heads * cfg.head_size * esz \
            + 4 * int(nblk.sum()) + 4 * cfg.num_seqs
        reshape = cfg.num_seqs * (in_tok + kv_tok) + 8 * cfg.num_seqs
        block_bytes = self.block_bytes
        copy = 2 * w.copy_pairs.shape[0] * block_bytes
        swap = (w.swap_out_pairs.shape[0] + w.swap_in_pairs.shape[0]) * block_bytes * 2
        unique = unique_kv_tokens(w.block_tables_np, w.context_lens_np, cfg.block_size) * kv_tok
        # the same decode bytes with each shared physical block's tokens counted
        # once (what HBM must deliver; equal to `decode` when nothing is shared)
        decode_unique = decode - int(ctx.sum()) * kv_tok + unique
        return {"decode": decode, "decode_unique": decode_unique, "decode_kv": int(ctx.sum()) * kv_tok,
                "decode_kv_unique": unique, "reshape": reshape, "copy": copy, "swap": swap,
                "total": decode_unique + reshape + copy + swap}


class PrefillStep:
    """One prefill / extend step of one layer: reshape_and_cache of every new
    token, then causal attention of the new tokens over the paged cache."""

    def __init__(self, w, stream: torch.cuda.Stream | None = None):
        cfg = w.cfg
        self.w = w
        self.stream = stream or torch.cuda.current_stream(w.q.device)
        self.desc = _lib.CacheDesc(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, w.dtype)
        self.kv_cache = w.kv_cache
        self.out = torch.empty_like(w.q)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=w.q.device)

    def cache_ops(self):
        w = self.w
        _lib.reshape_and_cache(self.kv_cache, self.desc, w.key, w.value, w.slot_mapping, dev_err=self.dev_err,
                               stream=self.stream)

    def attention(self, q=None, out=None):
        w = self.w
        _lib.prefill(self.out if out is None else out, w.q if q is None else q, self.kv_cache, self.desc,
                     w.block_tables, w.context_lens, w.query_start_loc, w.max_query_len, w.scale,
                     dev_err=self.dev_err, stream=self.stream)

    def __call__(self):
        self.cache_ops()
        self.attention()
        return self.out

    def kernel_launches(self) -> int:
        return 2

    def flops(self) -> int:
        """Causal attention FLOPs: 4 * D per (query row, attended position)."""
        cfg = self.w.cfg
        ctx = self.w.context_lens_np.astype(np.int64)
        q_len = np.diff(self.w.query_start_loc_np).astype(np.int64)
        # sum over j < q_len of (ctx - q_len + j + 1)
        attended = q_len * (ctx - q_len) + q_len * (q_len + 1) // 2
        return int(4 * cfg.head_size * cfg.num_q_heads * attended.sum())

    def algorithmic_bytes(self) -> int:
        """Bytes the step must move at least: new K/V read + written, q read, out written,
        and each sequence's KV once per kv head."""
        w, cfg = self.w, self.w.cfg
        T = int(self.w.query_start_loc_np[-1])
        kv_tok = 2 * cfg.num_kv_heads * cfg.head_size * 2
        return int(2 * T * kv_tok + 2 * T * cfg.num_q_heads * cfg.head_size * 2
                   + int(w.context_lens_np.astype(np.int64).sum()) * kv_tok)
