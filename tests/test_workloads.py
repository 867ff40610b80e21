"""The seeded workload generator: shapes, determinism and table/slot consistency."""
import numpy as np
import pytest
import torch

from paged_kv_cache_168_gb300.workloads import CONFIGS, make_workload


def test_tiny_shapes_and_determinism():
    a = make_workload("tiny")
    b = make_workload("tiny")
    assert a.q.shape == (4, 4, 64) and a.kv_cache.shape == (64, 4, 2 * 16 * 64)
    assert torch.equal(a.kv_cache, b.kv_cache) and np.array_equal(a.block_tables_np, b.block_tables_np)
    assert a.kv_cache.dtype == torch.float16 and float(a.kv_cache.abs().max()) <= 1.0
    assert 1 <= a.context_lens_np.min() and a.context_lens_np.max() <= 100


@pytest.mark.parametrize("name", ["tiny", "7b", "8b", "beam"])
def test_tables_slots_and_pool_sizing(name):
    cfg = CONFIGS[name]
    w = make_workload(name, num_seqs=None if name in ("tiny", "beam") else 16)
    S, bs = w.cfg.num_seqs, cfg.block_size
    ctx, bt = w.context_lens_np, w.block_tables_np
    nblk = -(-ctx // bs)
    for s in range(S):
        assert np.all(bt[s, :nblk[s]] >= 0) and np.all(bt[s, nblk[s]:] == -1)
        pos = ctx[s] - 1
        assert w.slot_mapping_np[s] == bt[s, pos // bs] * bs + pos % bs
    if name != "beam":
        used = bt[bt >= 0]
        assert len(np.unique(used)) == used.size           # no block shared
    else:
        # 4 beams of a group share their 128 prompt blocks, and nothing else
        for g in range(S // 4):
            rows = bt[4 * g:4 * g + 4]
            assert np.all(rows[:, :128] == rows[0, :128])
        assert len(np.unique(bt[:, 128:][bt[:, 128:] >= 0])) == (bt[:, 128:] >= 0).sum()
        assert w.copy_pairs.shape == (S, 2)
        assert np.array_equal(w.copy_pairs[:, 1], bt[np.arange(S), nblk - 1])
        assert abs(w.swap_out_pairs.shape[0] - 0.1 * w.used_blocks.size) <= 1
        assert np.array_equal(w.swap_in_pairs, w.swap_out_pairs[:, ::-1])
    assert w.num_blocks >= len(np.unique(bt[bt >= 0]))


def test_nan_unused_blocks():
    w = make_workload("tiny", nan_unused=True)
    used = set(w.used_blocks.tolist())
    for b in range(w.num_blocks):
        assert bool(torch.isnan(w.kv_cache[b]).all()) == (b not in used)


def test_prefill_workloads_are_seeded_and_consistent():
    from paged_kv_cache_168_gb300.workloads import PREFILL_CONFIGS, make_prefill_workload
    for name in PREFILL_CONFIGS:
        a, b = make_prefill_workload(name), make_prefill_workload(name)
        assert torch.equal(a.q, b.q) and np.array_equal(a.slot_mapping_np, b.slot_mapping_np)
        cfg = a.cfg
        qsl, ctx, bs = a.query_start_loc_np, a.context_lens_np, cfg.block_size
        assert qsl[0] == 0 and np.all(np.diff(qsl) == cfg.q_len) and a.q.shape[0] == qsl[-1]
        # the new tokens are each sequence's last q_len positions, in its own blocks
        for s in range(cfg.num_seqs):
            pos = np.arange(ctx[s] - cfg.q_len, ctx[s])
            want = a.block_tables_np[s, pos // bs].astype(np.int64) * bs + pos % bs
            assert np.array_equal(a.slot_mapping_np[qsl[s]:qsl[s + 1]], want)
        used = a.block_tables_np[a.block_tables_np >= 0]
        assert np.unique(used).size == used.size and used.max() < a.num_blocks


def test_unique_kv_tokens_counts_a_shared_block_once():
    from paged_kv_cache_168_gb300.step import unique_kv_tokens
    bs = 4
    # seqs 0 and 1 share blocks 5 and 6 (8 tokens); seq 0 then has 3 tokens in
    # block 1, seq 1 has 4 in block 2 and 1 in block 3; seq 2 is empty
    tables = np.array([[5, 6, 1, -1], [5, 6, 2, 3], [-1, -1, -1, -1]], np.int32)
    ctx = np.array([11, 13, 0], np.int32)
    assert unique_kv_tokens(tables, ctx, bs) == 8 + 3 + 4 + 1
    # a block that two sequences fill to different depths counts its deeper use
    tables2 = np.array([[7, -1], [7, 8]], np.int32)
    assert unique_kv_tokens(tables2, np.array([3, 5], np.int32), bs) == 4 + 1
    # without sharing, unique equals the logical count
    w = make_workload("tiny")
    assert unique_kv_tokens(w.block_tables_np, w.context_lens_np, w.cfg.block_size) == int(w.context_lens_np.sum())
    beam = make_workload("beam")
    u = unique_kv_tokens(beam.block_tables_np, beam.context_lens_np, beam.cfg.block_size)
    groups = beam.cfg.num_seqs // beam.cfg.beams
    assert u < int(beam.context_lens_np.sum())
    assert u >= groups * beam.cfg.ctx[1]          # every group's shared prompt, once
