"""Test-side helpers: build paged pools from logical per-sequence K/V with the oracle.

Everything here runs on the CPU through ``oracle`` (the fp64 reference); the CUDA
library is never used to build an expected value.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float data to fp16/bf16 (round-to-nearest-even) and return the raw bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(TORCH_DT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(TORCH_DT[dtype])
    return t.to(torch.float64).numpy()


class Paged:
    """Logical K/V for S sequences written into a NaN-filled paged pool."""

    def __init__(self, rng, S, Hq, Hkv, D, bs, ctx, dtype="f16", num_blocks=None,
                 values="normal", width=None, perm=None):
        self.S, self.Hq, self.Hkv, self.D, self.bs, self.dtype = S, Hq, Hkv, D, bs, dtype
        self.ctx = np.asarray(ctx, dtype=np.int32)
        nblk = (self.ctx + bs - 1) // bs
        need = int(nblk.sum())
        self.num_blocks = num_blocks or max(need + 3, 1)
        self.width = width or max(int(nblk.max()) if S else 1, 1)
        self.geom = oracle.Geom(self.num_blocks, bs, Hkv, D, dtype)
        draw = (lambda *s: rng.uniform(-1, 1, s)) if values == "uniform" else (lambda *s: rng.standard_normal(s))
        # logical data, already rounded to the storage type
        self.K = [bits_to_f64(to_bits(draw(c, Hkv, D), dtype), dtype) for c in self.ctx]
        self.V = [bits_to_f64(to_bits(draw(c, Hkv, D), dtype), dtype) for c in self.ctx]
        self.q_bits = to_bits(draw(S, Hq, D), dtype)
        self.q = bits_to_f64(self.q_bits, dtype)
        perm = rng.permutation(self.num_blocks) if perm is None else np.asarray(perm)
        self.tables = np.full((S, self.width), -1, dtype=np.int32)
        nxt = 0
        for s in range(S):
            self.tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
            nxt += nblk[s]
        self.pool = np.full(self.geom.layer_elems, NAN_BITS[dtype], dtype=np.uint16)
        self.write_all()

    def write_all(self):
        for s in range(self.S):
            c = int(self.ctx[s])
            if c == 0:
                continue
            t = np.arange(c)
            slots = self.tables[s, t // self.bs].astype(np.int64) * self.bs + t % self.bs
            err = oracle.reshape_and_cache(self.pool, self.geom, to_bits(self.K[s], self.dtype),
                                           to_bits(self.V[s], self.dtype), slots)
            assert err == 0

    def expected_contiguous(self, scale):
        """Reference via torch's fp64 scaled_dot_product_attention on the logical arrays
        (kv head of query head h is h // (Hq // Hkv))."""
        G = self.Hq // self.Hkv
        out = np.zeros((self.S, self.Hq, self.D))
        for s in range(self.S):
            if self.ctx[s] == 0:
                continue
            q = torch.from_numpy(self.q[s]).unsqueeze(1)                       # [Hq, 1, D]
            K = torch.from_numpy(self.K[s]).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, ctx, D]
            V = torch.from_numpy(self.V[s]).permute(1, 0, 2).repeat_interleave(G, 0)
            o = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
            out[s] = o[:, 0, :].numpy()
        return out


class RingPaged:
    """Sequences written token by token into ring block tables (a sliding-window
    cache): token t goes to slot t % bs of block ring_table[(t / bs) % ring], so
    later tokens overwrite the ring's oldest block."""

    def __init__(self, rng, S, Hq, Hkv, D, bs, ctx, ring, dtype="bf16", num_blocks=None):
        self.S, self.Hq, self.Hkv, self.D, self.bs, self.dtype, self.ring = S, Hq, Hkv, D, bs, dtype, ring
        self.ctx = np.asarray(ctx, dtype=np.int32)
        self.num_blocks = num_blocks or S * ring + 3
        self.geom = oracle.Geom(self.num_blocks, bs, Hkv, D, dtype)
        self.K = [bits_to_f64(to_bits(rng.standard_normal((c, Hkv, D)), dtype), dtype) for c in self.ctx]
        self.V = [bits_to_f64(to_bits(rng.standard_normal((c, Hkv, D)), dtype), dtype) for c in self.ctx]
        self.q_bits = to_bits(rng.standard_normal((S, Hq, D)), dtype)
        self.q = bits_to_f64(self.q_bits, dtype)
        perm = rng.permutation(self.num_blocks)
        self.tables = perm[:S * ring].reshape(S, ring).astype(np.int32)
        self.pool = np.full(self.geom.layer_elems, NAN_BITS[dtype], dtype=np.uint16)
        for s in range(S):
            t = np.arange(int(self.ctx[s]))
            slots = self.tables[s, (t // bs) % ring].astype(np.int64) * bs + t % bs
            assert oracle.reshape_and_cache(self.pool, self.geom, to_bits(self.K[s], dtype),
                                            to_bits(self.V[s], dtype), slots) == 0

    def expected_window(self, scale, window):
        """torch fp64 SDPA over the last `window` logical tokens of each sequence."""
        G = self.Hq // self.Hkv
        out = np.zeros((self.S, self.Hq, self.D))
        for s in range(self.S):
            c = int(self.ctx[s])
            lo = max(0, c - window)
            q = torch.from_numpy(self.q[s]).unsqueeze(1)
            K = torch.from_numpy(self.K[s][lo:c]).permute(1, 0, 2).repeat_interleave(G, 0)
            V = torch.from_numpy(self.V[s][lo:c]).permute(1, 0, 2).repeat_interleave(G, 0)
            out[s] = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)[:, 0, :].numpy()
        return out


def i8_pool_case(rng, ctx, Hq, Hkv, bs, dtype):
    """An 8-bit pool the oracle writes from random N(0,1) K/V of each sequence
    (head_size 128), blocks placed by a random permutation; unused blocks stay
    zero.  Returns (q_bits [S, Hq, 128], pool bytes, geom, tables, ctx)."""
    ctx = np.asarray(ctx, np.int32)
    nblk = -(-ctx // bs)
    nb = int(nblk.sum()) + 3
    g = oracle.Geom(nb, bs, Hkv, 128, dtype)
    pool = np.zeros(nb * oracle.i8_block_bytes(g), np.uint8)
    tables = np.full((len(ctx), max(int(nblk.max()), 1)), -1, np.int32)
    perm = rng.permutation(nb)
    at = 0
    for s, c in enumerate(ctx):
        tables[s, :nblk[s]] = perm[at:at + nblk[s]]
        at += nblk[s]
        if c == 0:
            continue
        t = np.arange(c)
        slots = tables[s, t // bs].astype(np.int64) * bs + t % bs
        x = rng.standard_normal((2, c, Hkv, 128))
        assert oracle.reshape_and_cache_i8(pool, g, to_bits(x[0], dtype), to_bits(x[1], dtype), slots) == 0
    q_bits = to_bits(rng.standard_normal((len(ctx), Hq, 128)), dtype)
    return q_bits, pool, g, tables, ctx


class SharedPaged:
    """Groups of sequences whose first blocks are the same physical blocks, as
    beams of one prompt after copy-on-write: group g has a prompt of prompt_len
    tokens; its floor(prompt_len / bs) whole blocks appear at the start of every
    member's table row, and the rest of each member's context (a partial prompt
    block included, as a copy) sits in the member's own blocks.  Every member's
    context holds the prompt's tokens first (as far as its length goes), then
    its own.  `groups` is a list of (prompt_len, [member context lengths]);
    all sequences are consecutive, group after group.  The pool is written by
    the oracle into NaN-filled memory."""

    def __init__(self, rng, groups, Hq, Hkv, D, bs, dtype="bf16"):
        self.Hq, self.Hkv, self.D, self.bs, self.dtype = Hq, Hkv, D, bs, dtype
        ctx = [c for _, members in groups for c in members]
        self.S = len(ctx)
        self.ctx = np.asarray(ctx, np.int32)
        self.group_start = np.cumsum([0] + [len(m) for _, m in groups]).astype(np.int32)
        self.prompt_lens = np.asarray([p for p, _ in groups], np.int32)
        nblk = -(-self.ctx // bs)
        shared = [p // bs for p, _ in groups]
        need = sum(shared) + int(sum(max(0, int(n) - 0) for n in nblk))
        self.num_blocks = need + 3
        self.width = max(int(nblk.max()), 1)
        self.geom = oracle.Geom(self.num_blocks, bs, Hkv, D, dtype)
        perm = iter(rng.permutation(self.num_blocks).tolist())
        self.tables = np.full((self.S, self.width), -1, np.int32)
        draw = lambda *s: bits_to_f64(to_bits(rng.standard_normal(s), dtype), dtype)
        self.K, self.V = [None] * self.S, [None] * self.S
        s = 0
        for (plen, members), nsh in zip(groups, shared):
            pk, pv = draw(plen, Hkv, D), draw(plen, Hkv, D)
            ids = [next(perm) for _ in range(nsh)]
            for c in members:
                own = max(0, c - plen)
                self.K[s] = np.concatenate([pk[:min(c, plen)], draw(own, Hkv, D)])
                self.V[s] = np.concatenate([pv[:min(c, plen)], draw(own, Hkv, D)])
                nb = -(-c // bs)
                row = ids[:min(nsh, nb)] + [next(perm) for _ in range(nb - min(nsh, nb))]
                self.tables[s, :nb] = row
                s += 1
        self.q_bits = to_bits(rng.standard_normal((self.S, Hq, D)), dtype)
        self.pool = np.full(self.geom.layer_elems, NAN_BITS[dtype], dtype=np.uint16)
        for s in range(self.S):
            c = int(self.ctx[s])
            if c == 0:
                continue
            t = np.arange(c)
            slots = self.tables[s, t // bs].astype(np.int64) * bs + t % bs
            assert oracle.reshape_and_cache(self.pool, self.geom, to_bits(self.K[s], dtype),
                                            to_bits(self.V[s], dtype), slots) == 0
