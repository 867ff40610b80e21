"""Pins of the fp64 CPU oracle against things other than itself.

Each test ties the oracle to a fact the pages or mathematics fix: library
routines (numpy / torch conversions, torch's scaled_dot_product_attention on
unpaged data, numpy fancy-index assignment), closed forms, invariants and the
pages' worked examples.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_helpers import NAN_BITS, Paged, RingPaged, bits_to_f64, to_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- element decoding

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_16bit_pattern_decodes_like_the_library(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits_to_f64(bits, dtype)
    got = np.array([oracle.elem_to_double(int(b), dtype) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- layout

@pytest.mark.parametrize("bs,D", [(1, 64), (8, 64), (16, 128), (32, 128), (16, 64)])
def test_layout_is_a_bijection_onto_each_block(bs, D):
    Hkv, NB = 3, 2
    g = oracle.Geom(NB, bs, Hkv, D)
    offs = [oracle.cache_offset(g, b, h, p, t, d)
            for b in range(NB) for h in range(Hkv) for p in range(2)
            for t in range(bs) for d in range(D)]
    assert sorted(offs) == list(range(NB * Hkv * 2 * bs * D))
    # every (block, kv head) owns one contiguous chunk of 2*bs*D elements
    chunk = 2 * bs * D
    for b in range(NB):
        for h in range(Hkv):
            o = [oracle.cache_offset(g, b, h, p, t, d) for p in range(2) for t in range(bs) for d in range(D)]
            assert min(o) == (b * Hkv + h) * chunk and max(o) == (b * Hkv + h + 1) * chunk - 1


def test_layout_keeps_16_byte_pieces_whole():
    # 8 consecutive dims starting at a multiple of 8 are 8 consecutive elements
    g = oracle.Geom(4, 16, 2, 128)
    for t in (0, 5, 15):
        for d0 in range(0, 128, 8):
            o = [oracle.cache_offset(g, 3, 1, 1, t, d0 + e) for e in range(8)]
            assert o == list(range(o[0], o[0] + 8)) and o[0] % 8 == 0


def test_reshape_then_gather_round_trips():
    rng = np.random.default_rng(0)
    p = Paged(rng, S=3, Hq=4, Hkv=2, D=64, bs=16, ctx=[1, 17, 40])
    for s in range(p.S):
        for h in range(p.Hkv):
            K, V = oracle.gather(p.pool, p.geom, p.tables[s], int(p.ctx[s]), h)
            assert np.array_equal(K, p.K[s][:, h, :]) and np.array_equal(V, p.V[s][:, h, :])


def test_reshape_skips_minus_one_and_flags_bad_slots():
    g = oracle.Geom(2, 8, 1, 64)
    pool = np.zeros(g.layer_elems, dtype=np.uint16)
    k = np.full((3, 1, 64), 0x3C00, dtype=np.uint16)
    err = oracle.reshape_and_cache(pool, g, k, k, np.array([-1, 5, 16]))
    assert err == oracle.ERR_SLOT
    K, _ = oracle.gather(pool, g, np.array([0, 1], np.int32), 8, 0)
    assert np.all(K[5] == 1.0) and np.all(np.delete(K, 5, axis=0) == 0.0)


# ---------------------------------------------------------------- attention

def test_contiguous_attention_matches_softmax_definition():
    from scipy.special import softmax
    rng = np.random.default_rng(1)
    for ctx, D in [(1, 8), (7, 64), (100, 128)]:
        q, K, V = rng.standard_normal(D), rng.standard_normal((ctx, D)), rng.standard_normal((ctx, D))
        scale = 1 / math.sqrt(D)
        ref = softmax(scale * (K @ q)) @ V
        assert np.allclose(oracle.contiguous_attention(q, K, V, scale), ref, rtol=1e-12, atol=1e-13)


def test_closed_forms():
    rng = np.random.default_rng(2)
    D = 16
    V = rng.standard_normal((5, D))
    K = rng.standard_normal((5, D))
    # one token: the output is that token's value exactly
    assert np.array_equal(oracle.contiguous_attention(rng.standard_normal(D), K[:1], V[:1], 0.3), V[0])
    # zero query (or equal keys): uniform weights, the mean of V
    assert np.allclose(oracle.contiguous_attention(np.zeros(D), K, V, 0.3), V.mean(0), atol=1e-15)
    Keq = np.tile(K[:1], (5, 1))
    assert np.allclose(oracle.contiguous_attention(rng.standard_normal(D), Keq, V, 0.3), V.mean(0), atol=1e-14)
    # two tokens: weights are the logistic function of the score difference
    q = rng.standard_normal(D)
    z = 0.7 * (K[:2] @ q)
    w0 = 1 / (1 + math.exp(z[1] - z[0]))
    assert np.allclose(oracle.contiguous_attention(q, K[:2], V[:2], 0.7), w0 * V[0] + (1 - w0) * V[1],
                       rtol=1e-13, atol=1e-15)
    # one score larger by >= 50: the output is that token's value
    q = np.zeros(D); q[0] = 1.0
    Kd = np.zeros((5, D)); Kd[3, 0] = 60.0
    assert np.allclose(oracle.contiguous_attention(q, Kd, V, 1.0), V[3], atol=1e-20)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,D,bs", [(4, 4, 64, 16), (8, 1, 64, 8), (8, 2, 128, 32), (6, 3, 64, 1)])
def test_paged_decode_equals_unpaged_sdpa(dtype, Hq, Hkv, D, bs):
    rng = np.random.default_rng(3)
    ctx = [1, bs - 1 if bs > 1 else 2, bs, bs + 1, 37, 100]
    p = Paged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype)
    scale = 1 / math.sqrt(D)
    out, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale)
    assert err == 0
    assert np.allclose(out, p.expected_contiguous(scale), rtol=1e-12, atol=1e-12)


def test_decode_selected_pairs_match_full_run():
    rng = np.random.default_rng(4)
    p = Paged(rng, S=4, Hq=8, Hkv=2, D=64, bs=16, ctx=[3, 50, 16, 77])
    full, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125)
    sel = np.array([[3, 7], [0, 0], [2, 5]], np.int32)
    part, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125, sel=sel)
    assert np.array_equal(part, full[sel[:, 0], sel[:, 1]])


def test_decode_zero_context_and_error_cases():
    rng = np.random.default_rng(5)
    p = Paged(rng, S=3, Hq=2, Hkv=1, D=64, bs=8, ctx=[0, 9, 20])
    out, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.1)
    assert err == 0 and np.all(out[0] == 0) and np.all(np.isfinite(out))
    bad = p.tables.copy()
    bad[1, 1] = p.num_blocks          # out-of-range block id
    out2, err2 = oracle.decode(p.q_bits, p.pool, p.geom, bad, p.ctx, 0.1)
    assert err2 == oracle.ERR_BLOCK_ID and np.all(out2[1] == 0) and np.array_equal(out2[2], out[2])
    ctx = p.ctx.copy()
    ctx[2] = p.width * p.bs + 1       # beyond the table row
    out3, err3 = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, ctx, 0.1, max_context_len=10**6)
    assert err3 == oracle.ERR_CONTEXT and np.all(out3[2] == 0)


# ---------------------------------------------------------------- invariants

def test_invariant_under_physical_block_permutation():
    rng = np.random.default_rng(6)
    p1 = Paged(rng, S=3, Hq=4, Hkv=2, D=64, bs=16, ctx=[5, 33, 64], num_blocks=12)
    rng2 = np.random.default_rng(6)
    p2 = Paged(rng2, S=3, Hq=4, Hkv=2, D=64, bs=16, ctx=[5, 33, 64], num_blocks=12,
               perm=np.arange(12)[::-1])
    o1, _ = oracle.decode(p1.q_bits, p1.pool, p1.geom, p1.tables, p1.ctx, 0.125)
    o2, _ = oracle.decode(p2.q_bits, p2.pool, p2.geom, p2.tables, p2.ctx, 0.125)
    assert not np.array_equal(p1.tables, p2.tables)
    assert np.array_equal(o1, o2)


def test_invariant_under_block_size():
    outs = []
    for bs in (1, 8, 16, 32):
        rng = np.random.default_rng(7)
        p = Paged(rng, S=3, Hq=4, Hkv=2, D=64, bs=bs, ctx=[1, 45, 70])
        o, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125)
        outs.append(o)
    for o in outs[1:]:
        assert np.allclose(o, outs[0], rtol=1e-12, atol=1e-12)


def test_shared_prefix_equals_unshared_copy():
    rng = np.random.default_rng(8)
    p = Paged(rng, S=2, Hq=4, Hkv=2, D=64, bs=16, ctx=[40, 40], num_blocks=12)
    # sequence 1 gets sequence 0's first two blocks (its prefix) shared, not copied
    p.K[1][:32] = p.K[0][:32]
    p.V[1][:32] = p.V[0][:32]
    p.write_all()
    shared = p.tables.copy()
    shared[1, :2] = shared[0, :2]
    o_copy, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125)
    o_shared, _ = oracle.decode(p.q_bits, p.pool, p.geom, shared, p.ctx, 0.125)
    assert np.array_equal(o_copy, o_shared)


def test_nan_in_unused_blocks_and_tail_slots_never_reaches_output():
    rng = np.random.default_rng(9)
    p = Paged(rng, S=4, Hq=4, Hkv=4, D=64, bs=16, ctx=[1, 15, 17, 31], num_blocks=20)
    assert np.isnan(bits_to_f64(p.pool, "f16")).any()      # tails and spare blocks are NaN
    out, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125)
    assert err == 0 and np.all(np.isfinite(out))


# ---------------------------------------------------------------- partitions + merge

@pytest.mark.parametrize("P", [16, 32, 512, 4096])
def test_partitions_merged_by_lse_equal_single_pass(P):
    rng = np.random.default_rng(10)
    p = Paged(rng, S=3, Hq=4, Hkv=2, D=64, bs=16, ctx=[1, 700, 1300])
    scale = 0.125
    full, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale)
    for s in range(p.S):
        for h in range(p.Hq):
            m, l, o = oracle.partition_stats(p.q_bits[s, h], p.pool, p.geom, p.tables[s],
                                             int(p.ctx[s]), h // 2, scale, P)
            assert len(m) == -(-int(p.ctx[s]) // P)
            merged = oracle.merge_partitions(m, l, o)
            assert np.allclose(merged, full[s, h], rtol=1e-12, atol=1e-13)


def test_partition_stats_closed_form():
    # two partitions of one token each: m_p = score, l_p = 1, o_p = v_p
    g = oracle.Geom(1, 8, 1, 64)
    rng = np.random.default_rng(11)
    K = to_bits(rng.standard_normal((2, 1, 64)), "f16")
    V = to_bits(rng.standard_normal((2, 1, 64)), "f16")
    pool = np.zeros(g.layer_elems, dtype=np.uint16)
    oracle.reshape_and_cache(pool, g, K, V, np.array([0, 1]))
    q = to_bits(rng.standard_normal(64), "f16")
    m, l, o = oracle.partition_stats(q, pool, g, np.array([0], np.int32), 2, 0, 0.5, 1)
    Kd, Vd, qd = bits_to_f64(K, "f16")[:, 0], bits_to_f64(V, "f16")[:, 0], bits_to_f64(q, "f16")
    assert np.allclose(m, 0.5 * Kd @ qd, rtol=1e-14) and np.array_equal(l, [1.0, 1.0])
    assert np.array_equal(o, Vd)


# ---------------------------------------------------------------- copy / swap

def test_copy_blocks_reads_every_source_before_writing():
    g = oracle.Geom(6, 8, 2, 64, num_layers=2)
    rng = np.random.default_rng(12)
    pool = rng.integers(0, 1 << 16, size=2 * g.layer_elems, dtype=np.uint32).astype(np.uint16)
    pairs = np.array([[0, 1], [1, 2], [4, 3]])
    ref = pool.reshape(2, 6, -1).copy()
    ref[:, pairs[:, 1]] = ref[:, pairs[:, 0]]        # numpy reads the right side first
    assert oracle.copy_blocks(pool, g, pairs) == 0
    assert np.array_equal(pool.reshape(2, 6, -1), ref)
    # idempotent for pairs whose destinations are not sources
    pool2 = pool.copy()
    oracle.copy_blocks(pool2, g, np.array([[4, 3], [0, 5]]))
    again = pool2.copy()
    oracle.copy_blocks(again, g, np.array([[4, 3], [0, 5]]))
    assert np.array_equal(again, pool2)
    assert oracle.copy_blocks(pool, g, np.array([[0, 6]])) == oracle.ERR_BLOCK_ID


def test_swap_round_trip_is_identity():
    gd = oracle.Geom(10, 16, 2, 64, num_layers=3)
    gh = oracle.Geom(4, 16, 2, 64, num_layers=3)
    rng = np.random.default_rng(13)
    dev = rng.integers(0, 1 << 16, size=3 * gd.layer_elems, dtype=np.uint32).astype(np.uint16)
    host = np.zeros(3 * gh.layer_elems, dtype=np.uint16)
    out_pairs = np.array([[7, 0], [2, 3], [9, 1]])
    assert oracle.swap_blocks(host, gh, dev, gd, out_pairs) == 0
    saved = dev.copy()
    dev.reshape(3, 10, -1)[:, [7, 2, 9]] = 0
    assert oracle.swap_blocks(dev, gd, host, gh, out_pairs[:, ::-1].copy()) == 0
    assert np.array_equal(dev, saved)
    assert np.array_equal(host.reshape(3, 4, -1)[:, 3], saved.reshape(3, 10, -1)[:, 2])


# ---------------------------------------------------------------- the pages' worked examples

class MiniBlockManager:
    """Reference counts and copy-on-write on append, as the vLLM block manager
    (append_slots) and the mlqm.cn CoW example describe them."""

    def __init__(self, tables, refs, free):
        self.tables = {k: list(v) for k, v in tables.items()}
        self.refs = {int(k): v for k, v in refs.items()}
        self.free = list(free)

    def append_slot(self, seq):
        last = self.tables[seq][-1]
        if self.refs[last] == 1:
            return []
        new = self.free.pop(0)
        self.refs[new] = 1
        self.refs[last] -= 1
        self.tables[seq][-1] = new
        return [(last, new)]


def test_cow_worked_example_block_bookkeeping_and_bytes():
    ex = json.load(open(os.path.join(GOLDEN, "cow_worked_example.json")))
    bs = ex["block_size"]
    mgr = MiniBlockManager(ex["initial_tables"], ex["initial_ref_counts"], ex["free_blocks_in_order"])
    g = oracle.Geom(6, bs, 2, 64)
    rng = np.random.default_rng(14)
    n_prompt = ex["prompt_tokens"]
    pk = to_bits(rng.standard_normal((n_prompt, 2, 64)), "f16")
    pv = to_bits(rng.standard_normal((n_prompt, 2, 64)), "f16")
    pool = np.full(g.layer_elems, NAN_BITS["f16"], dtype=np.uint16)
    t = np.arange(n_prompt)
    oracle.reshape_and_cache(pool, g, pk, pv, np.array([0, 1])[t // bs] * bs + t % bs)
    new_k, new_v = {}, {}
    for seq in ex["write_order"]:
        pairs = mgr.append_slot(seq)
        assert pairs == [tuple(p) for p in ex["expected_copy_pairs"][seq]]
        if pairs:
            assert oracle.copy_blocks(pool, g, np.array(pairs)) == 0
        off = ex["expected_new_token_position"]["block_offset"]
        assert off == n_prompt % bs
        new_k[seq] = to_bits(rng.standard_normal((1, 2, 64)), "f16")
        new_v[seq] = to_bits(rng.standard_normal((1, 2, 64)), "f16")
        slot = mgr.tables[seq][-1] * bs + off
        assert oracle.reshape_and_cache(pool, g, new_k[seq], new_v[seq], np.array([slot])) == 0
    assert mgr.tables == ex["expected_tables"]
    assert mgr.refs == {int(k): v for k, v in ex["expected_ref_counts"].items()}
    # every sequence now sees the intact prompt followed by its own new token
    for seq in ex["write_order"]:
        K, V = oracle.gather(pool, g, np.array(mgr.tables[seq], np.int32), n_prompt + 1, 1)
        assert np.array_equal(K[:n_prompt], bits_to_f64(pk[:, 1], "f16"))
        assert np.array_equal(K[n_prompt], bits_to_f64(new_k[seq][0, 1], "f16"))
        assert np.array_equal(V[n_prompt], bits_to_f64(new_v[seq][0, 1], "f16"))


def test_kv_size_formula_llama13b():
    # "2 (K,V) x batch x seq x layers x heads x head_dim x 2 bytes": a LLaMA-13B
    # request of 8192 tokens needs about 6 GB.  In blocks of 16 tokens:
    g = oracle.Geom(num_blocks=8192 // 16, block_size=16, num_kv_heads=40, head_size=128)
    total = g.layer_elems * 2 * 40                  # 40 layers, 2 bytes per element
    assert total == 2 * 1 * 8192 * 40 * 40 * 128 * 2
    assert 6.0 <= total / 2**30 <= 7.0              # 6.25 GiB: "about 6 GB"


def test_paging_wastes_at_most_one_partial_block_per_sequence():
    from paged_kv_cache_168_gb300.workloads import CONFIGS, draw_context_lens
    for cfg in CONFIGS.values():
        ctx = draw_context_lens(cfg, np.random.Generator(np.random.PCG64(cfg.seed)))
        slots = -(-ctx // cfg.block_size) * cfg.block_size
        assert np.all(slots - ctx <= cfg.block_size - 1)       # at most 15 tokens at block 16
        if cfg.name in ("7b", "8b", "70b", "beam"):
            assert (slots - ctx).sum() / slots.sum() < 0.04   # "under 4%" waste


# ---------------------------------------------------------------- sliding window over ring tables

def test_window_start_closed_forms():
    assert oracle.window_start(40, 16, 0, 0) == 0
    assert oracle.window_start(5, 16, 10, 0) == 0
    assert oracle.window_start(40, 16, 32, 0) == 8
    assert oracle.window_start(40, 16, 32, 3) == 8      # ring of 3 blocks holds [0, 48): the window rules
    assert oracle.window_start(40, 16, 32, 2) == 16     # ring of ceil(32/16) blocks only holds [16, 40)
    assert oracle.window_start(33, 16, 0, 1) == 32      # a one-block ring holds just the current block


def test_window_covering_the_context_equals_plain_decode():
    rng = np.random.default_rng(20)
    p = Paged(rng, S=3, Hq=4, Hkv=2, D=64, bs=16, ctx=[5, 40, 77])
    plain, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125)
    wide, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125, window=77)
    assert err == 0 and np.array_equal(plain, wide)


def test_window_of_one_token_returns_the_last_value():
    rng = np.random.default_rng(21)
    p = Paged(rng, S=2, Hq=4, Hkv=2, D=64, bs=8, ctx=[9, 30])
    out, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.3, window=1)
    assert err == 0
    for s in range(2):
        for h in range(4):
            assert np.array_equal(out[s, h], p.V[s][p.ctx[s] - 1, h // 2])


@pytest.mark.parametrize("bs,W", [(16, 32), (16, 20), (8, 8), (1, 5), (32, 100)])
def test_ring_cache_window_equals_sdpa_on_last_tokens(bs, W):
    from paged_helpers import RingPaged
    rng = np.random.default_rng(22)
    ring = -(-(W - 1) // bs) + 1                       # enough blocks for an exact window
    p = RingPaged(rng, S=4, Hq=8, Hkv=2, D=64, bs=bs, ctx=[3, W, W + 7, 5 * W + 3], ring=ring)
    out, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 0.125, max_context_len=10 ** 6,
                             window=W, ring=ring)
    assert err == 0
    assert np.allclose(out, p.expected_window(0.125, W), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- 8-bit KV cache

def _i8_pool(geom, num_blocks):
    return np.zeros(oracle.i8_block_bytes(geom) * num_blocks, dtype=np.uint8)


def _read_i8(pool, geom, block, head, part, t):
    """(codes, scale) of one stored vector, read by the chunk description
    [K codes | V codes | K scales | V scales] (each scale area padded to 16 bytes;
    16-byte pieces of a code row swizzled by the slot's row index mod 8)."""
    bs, D = geom.block_size, geom.head_size
    chunk = oracle.i8_block_bytes(geom) // geom.num_kv_heads
    base = (block * geom.num_kv_heads + head) * chunk
    row = pool[base + (part * bs + t) * D: base + (part * bs + t + 1) * D].view(np.int8)
    pos = (((np.arange(D) >> 4) ^ (t & 7)) << 4) | (np.arange(D) & 15)   # piece c of the row at c ^ (t % 8)
    codes = row[pos]
    sbytes = -(-bs * 4 // 16) * 16
    off = base + 2 * bs * D + part * sbytes + t * 4
    return codes, float(pool[off:off + 4].view(np.float32)[0])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_i8_quantisation_properties(dtype):
    rng = np.random.default_rng(30)
    g = oracle.Geom(4, 16, 2, 128, dtype)
    pool = _i8_pool(g, 4)
    x = rng.standard_normal((20, 2, 128)) * rng.uniform(0.01, 100, (20, 2, 1))
    x[3, 1] = 0.0                                       # an all-zero vector
    k = to_bits(x, dtype)
    v = to_bits(-x, dtype)
    slots = rng.choice(64, 20, replace=False)
    assert oracle.reshape_and_cache_i8(pool, g, k, v, slots) == 0
    kd, vd = bits_to_f64(k, dtype), bits_to_f64(v, dtype)
    for i, slot in enumerate(slots):
        for h in range(2):
            for part, src in ((0, kd), (1, vd)):
                codes, scale = _read_i8(pool, g, slot // 16, h, part, slot % 16)
                vec = src[i, h]
                amax = np.abs(vec).max()
                if amax == 0:
                    assert scale == 0 and np.all(codes == 0)
                    continue
                assert np.isclose(scale, amax / 127, rtol=1e-6)
                assert np.abs(codes).max() == 127 and codes[np.argmax(np.abs(vec))] == np.sign(vec[np.argmax(np.abs(vec))]) * 127
                assert np.all(np.abs(vec - codes * scale) <= scale * 0.5 * (1 + 1e-5))


def _np_i8_quantise(vec: np.ndarray):
    """numpy binary32 restatement of the 8-bit reading (FAQ page, TurboMind
    section, "8bit KV Cache"): amax = max|x|; the quotient 127 / amax is rounded
    to binary32 first, each x is multiplied by it (binary32) and rounded half to
    even (np.rint), then clipped to +-127; scale = amax / 127 in binary32."""
    v = vec.astype(np.float32)
    amax = np.float32(np.max(np.abs(v)))
    if amax == 0:
        return np.zeros(v.shape, np.int8), np.float32(0)
    inv = np.float32(127) / amax
    return np.clip(np.rint(v * inv), -127, 127).astype(np.int8), np.float32(amax / np.float32(127))


def _i8_discriminating_vectors(dtype, want=24):
    """Vectors (exactly representable in `dtype`) on which the plausible wrong
    arrangements of the quantiser give other bytes than the reading:
      * exact ties x * (127 / amax) = k + 1/2 of both signs (amax = 127 / 2^j
        makes the quotient a power of two): half-away-from-zero rounding differs;
      * pairs (amax, x) where (x * 127) / amax and x * (127 / amax) round to
        different integers (a one-ulp difference across a half-integer);
      * maxima where amax * (1 / 127) is not amax / 127."""
    tdt = TORCH_DT16[dtype]

    def rep(a):
        return torch.from_numpy(np.asarray(a, np.float32)).to(tdt).to(torch.float32).numpy()

    vecs = []
    for j in range(4):
        amax = np.float32(127.0 / 2 ** j)
        half = np.float32(0.5 / 2 ** j)                  # x * 2^j = k + 1/2  for x = (2k + 1) * half
        ks = np.array([0, 1, 2, 3, 10, 41, 100, 125, 126])
        xs = ((2 * ks + 1) * half).astype(np.float32)
        xs = xs[xs < amax]
        v = np.zeros(128, np.float32)
        v[0] = amax
        v[1:1 + xs.size] = xs
        v[64:64 + xs.size] = -xs
        vecs.append(rep(v))
    rng = np.random.default_rng(7)
    amax = rep(rng.uniform(0.01, 1000, 40000))
    k = rng.integers(0, 127, amax.size)
    x0 = torch.from_numpy(((k + 0.5) * amax.astype(np.float64) / 127).astype(np.float32)).to(tdt)
    order_pairs = []
    for d in range(-3, 4):                               # neighbours of the tie point, in ulps of dtype
        x = (x0.view(torch.int16) + d).view(tdt).to(torch.float32).numpy()
        ok = np.isfinite(x) & (np.abs(x) <= amax)
        inv = np.float32(127) / amax
        diff = ok & (np.rint(x * inv) != np.rint((x * np.float32(127)) / amax))
        order_pairs += list(zip(amax[diff], x[diff]))
    for a, x in order_pairs[:want]:
        v = np.zeros(128, np.float32)
        v[0], v[1], v[2] = a, x, -x
        v[3:] = rep(rng.uniform(-1, 1, 125) * a)
        vecs.append(rep(v))
    scale_diff = amax[(amax / np.float32(127)) != (amax * (np.float32(1) / np.float32(127)))]
    for a in scale_diff[:want]:
        v = rep(rng.uniform(-1, 1, 128) * a)
        v[5] = -a
        vecs.append(rep(v))
    return np.stack(vecs)


TORCH_DT16 = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_i8_quantiser_bytes_equal_numpy_binary32(dtype):
    """The oracle's 8-bit writer stores exactly the codes and scales of an
    independent numpy binary32 computation of the reading, on inputs chosen so
    that half-away-from-zero rounding, the order x * 127 / amax, or a scale of
    amax * (1 / 127) would each change some byte."""
    vecs = _i8_discriminating_vectors(dtype)
    n = vecs.shape[0]
    bs, hkv = 16, 1
    nb = -(-n // bs)
    g = oracle.Geom(nb, bs, hkv, 128, dtype)
    pool = _i8_pool(g, nb)
    bits = to_bits(vecs.reshape(n, 1, 128), dtype)
    assert np.array_equal(bits_to_f64(bits, dtype).reshape(n, 128), vecs.astype(np.float64))   # exact inputs
    slots = np.arange(n, dtype=np.int64)
    assert oracle.reshape_and_cache_i8(pool, g, bits, bits, slots) == 0
    half_away = order = scale_mul = 0
    for i in range(n):
        want_codes, want_scale = _np_i8_quantise(vecs[i])
        for part in (0, 1):
            codes, scale = _read_i8(pool, g, i // bs, 0, part, i % bs)
            assert np.array_equal(codes, want_codes), (i, part)
            assert np.float32(scale).view(np.uint32) == want_scale.view(np.uint32), (i, part)
        # the fixture discriminates: count the elements each wrong arrangement changes
        v = vecs[i].astype(np.float32)
        amax = np.float32(np.max(np.abs(v)))
        y = v * (np.float32(127) / amax)
        half_away += int(np.sum(np.clip(np.trunc(y + np.copysign(np.float32(0.5), y)), -127, 127) != want_codes))
        order += int(np.sum(np.clip(np.rint((v * np.float32(127)) / amax), -127, 127) != want_codes))
        scale_mul += int(amax * (np.float32(1) / np.float32(127)) != want_scale)
    assert half_away > 0 and order > 0 and scale_mul > 0, (half_away, order, scale_mul)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_i8_decode_on_grid_values_equals_16bit_decode(dtype):
    # values code * 2^-6 with one code of +-127 per vector are stored exactly by
    # the 8-bit cache (scale = 2^-6), so its decode equals the 16-bit decode
    rng = np.random.default_rng(31)
    S, Hq, Hkv, D, bs = 4, 8, 2, 128, 16
    ctx = [1, 17, 40, 90]
    p = Paged(rng, S=S, Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype)
    g = oracle.Geom(p.num_blocks, bs, Hkv, D, dtype)
    pool = _i8_pool(g, p.num_blocks)
    for s in range(S):
        c = ctx[s]
        codes = rng.integers(-127, 128, (2, c, Hkv, D))
        codes[:, :, :, 0] = 127
        vals = codes * 2.0 ** -6
        p.K[s], p.V[s] = vals[0], vals[1]
        t = np.arange(c)
        slots = p.tables[s, t // bs].astype(np.int64) * bs + t % bs
        assert oracle.reshape_and_cache_i8(pool, g, to_bits(vals[0], dtype), to_bits(vals[1], dtype), slots) == 0
    p.write_all()
    scale = 1 / math.sqrt(D)
    ref, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale)
    got, err = oracle.decode_i8(p.q_bits, pool, g, p.tables, p.ctx, scale)
    assert err == 0
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(got, p.expected_contiguous(scale), rtol=1e-12, atol=1e-12)


def test_byte_block_copy_matches_numpy():
    rng = np.random.default_rng(32)
    pool = rng.integers(0, 256, 7 * 300, dtype=np.uint8)
    ref = pool.reshape(7, 300).copy()
    ref[[5, 2]] = ref[[0, 1]]
    assert oracle.copy_blocks_bytes(pool, 300, 7, np.array([[0, 5], [1, 2]])) == 0
    assert np.array_equal(pool.reshape(7, 300), ref)


# ---------------------------------------------------------------- prefill / extend

def _prefill_case(rng, q_lens, ctx, Hq=4, Hkv=2, D=64, bs=16, dtype="f16"):
    """Paged history for each sequence, plus its last q_len tokens as packed queries."""
    p = Paged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q_bits = to_bits(rng.standard_normal((int(qsl[-1]), Hq, D)), dtype)
    return p, qsl, q_bits


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_of_whole_prompts_equals_causal_sdpa(dtype):
    rng = np.random.default_rng(40)
    ctx = [1, 17, 40, 33]
    p, qsl, qb = _prefill_case(rng, ctx, ctx, dtype=dtype)      # q_len == ctx: a prompt from scratch
    got, err = oracle.prefill(qb, p.pool, p.geom, p.tables, p.ctx, qsl, 0.125)
    assert err == 0
    q = bits_to_f64(qb, dtype)
    for s, c in enumerate(ctx):
        qs = torch.from_numpy(q[qsl[s]:qsl[s + 1]]).permute(1, 0, 2)                        # [Hq, c, D]
        K = torch.from_numpy(p.K[s]).permute(1, 0, 2).repeat_interleave(2, 0)
        V = torch.from_numpy(p.V[s]).permute(1, 0, 2).repeat_interleave(2, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, K, V, is_causal=True, scale=0.125)
        assert np.allclose(got[qsl[s]:qsl[s + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_extend_rows_equal_decodes_at_their_positions():
    rng = np.random.default_rng(41)
    ctx, q_lens = [50, 20, 130, 9], [7, 20, 1, 3]
    p, qsl, qb = _prefill_case(rng, q_lens, ctx, Hq=8, Hkv=2, D=128, bs=8, dtype="bf16")
    got, err = oracle.prefill(qb, p.pool, p.geom, p.tables, p.ctx, qsl, 0.09)
    assert err == 0
    for s in range(len(ctx)):
        for j in range(q_lens[s]):
            pos = ctx[s] - q_lens[s] + j
            tok = qsl[s] + j
            ref, e = oracle.decode(qb[tok:tok + 1], p.pool, p.geom, p.tables[s:s + 1],
                                   np.array([pos + 1], np.int32), 0.09)
            assert e == 0 and np.allclose(got[tok], ref[0], rtol=1e-13, atol=1e-13)


def test_chunked_prefill_equals_one_shot_prefill():
    rng = np.random.default_rng(42)
    total = 45
    p, qsl, qb = _prefill_case(rng, [total], [total], Hq=2, Hkv=1)
    whole, e = oracle.prefill(qb, p.pool, p.geom, p.tables, p.ctx, qsl, 0.2)
    assert e == 0
    done = 0
    for chunk in (16, 16, 13):          # the same prompt in three chunks over a growing context
        part, e = oracle.prefill(qb[done:done + chunk], p.pool, p.geom, p.tables, np.array([done + chunk], np.int32),
                                 np.array([0, chunk], np.int32), 0.2)
        assert e == 0 and np.allclose(part, whole[done:done + chunk], rtol=1e-13, atol=1e-13)
        done += chunk


def test_prefill_with_identical_keys_averages_the_causal_prefix():
    # every key equal -> uniform weights over the attended positions: query j of a
    # chunk at position ctx - q_len + j gets the mean of V[0 .. that position]
    rng = np.random.default_rng(43)
    ctx, q_len = 30, 6
    p = Paged(rng, S=1, Hq=1, Hkv=1, D=64, bs=16, ctx=[ctx], dtype="f16")
    p.K[0][:] = p.K[0][0]
    p.write_all()
    qb = to_bits(rng.standard_normal((q_len, 1, 64)), "f16")
    got, e = oracle.prefill(qb, p.pool, p.geom, p.tables, p.ctx, np.array([0, q_len], np.int32), 0.3)
    assert e == 0
    for j in range(q_len):
        pos = ctx - q_len + j
        assert np.allclose(got[j, 0], p.V[0][:pos + 1, 0].mean(axis=0), rtol=1e-12, atol=1e-12)


def test_prefill_error_cases():
    rng = np.random.default_rng(44)
    p, qsl, qb = _prefill_case(rng, [5, 3, 2], [20, 2, 40])       # second sequence: q_len 3 > ctx 2
    got, err = oracle.prefill(qb, p.pool, p.geom, p.tables, p.ctx, qsl, 0.1)
    assert err == oracle.ERR_CONTEXT and np.all(got[5:8] == 0) and np.any(got[:5] != 0)
    tables = p.tables.copy()
    tables[2, 1] = p.num_blocks + 1
    got, err = oracle.prefill(qb, p.pool, p.geom, tables, p.ctx, qsl, 0.1)
    assert err & oracle.ERR_BLOCK_ID and np.all(got[8:] == 0) and np.any(got[:5] != 0)
    # a sequence with no new tokens contributes no rows
    got, err = oracle.prefill(qb[:5], p.pool, p.geom, p.tables[:2], p.ctx[:2], np.array([0, 5, 5], np.int32), 0.1)
    assert err == 0 and got.shape == (5, 4, 64)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs,W,exact", [(16, 40, True), (16, 40, False), (8, 100, True), (4, 9, True)])
def test_i8_window_on_grid_values_equals_16bit_window(dtype, bs, W, exact):
    # ring tables written token by token (older blocks overwritten): on values the
    # 8-bit cache stores exactly, its window decode equals the pinned 16-bit window
    # decode, and with an exact ring both equal attention over the last W tokens
    rng = np.random.default_rng(33 + bs + W)
    ring = -(-(W - 1) // bs) + 1 if exact else -(-W // bs)
    ctx = [1, W - 1, W, W + 1, 3 * W + 5]
    p = RingPaged(rng, S=len(ctx), Hq=8, Hkv=2, D=128, bs=bs, ctx=ctx, ring=ring, dtype=dtype)
    g8 = oracle.Geom(p.num_blocks, bs, 2, 128, dtype)
    pool8 = _i8_pool(g8, p.num_blocks)
    p.pool[:] = 0
    for s, c in enumerate(ctx):
        codes = rng.integers(-127, 128, (2, c, 2, 128))
        codes[:, :, :, 0] = 127
        vals = codes * 2.0 ** -6
        p.K[s], p.V[s] = vals[0], vals[1]
        t = np.arange(c)
        slots = p.tables[s, (t // bs) % ring].astype(np.int64) * bs + t % bs
        kb, vb = to_bits(vals[0], dtype), to_bits(vals[1], dtype)
        assert oracle.reshape_and_cache(p.pool, p.geom, kb, vb, slots) == 0
        assert oracle.reshape_and_cache_i8(pool8, g8, kb, vb, slots) == 0
    scale = 1 / math.sqrt(128)
    ref, e1 = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, window=W, ring=ring)
    got, e2 = oracle.decode_i8(p.q_bits, pool8, g8, p.tables, p.ctx, scale, window=W, ring=ring)
    assert e1 == 0 and e2 == 0
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    if exact:
        assert np.allclose(got, p.expected_window(scale, W), rtol=1e-12, atol=1e-12)
