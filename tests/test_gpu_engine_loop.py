"""End to end: the host block manager drives the device calls through several
decode steps -- prompt writes, parallel-sampling forks with copy-on-write,
sliding-window ring tables, swap out / in -- while the oracle replays the same
cache operations on the CPU.  Pools must agree bit for bit after every step and
attention within the usual tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import assert_attention_close, desc_of, dev_to_u16, ensure_built, u16_to_dev
from paged_helpers import NAN_BITS, to_bits
from paged_kv_cache_168_gb300._lib import BlockManager

pytestmark = pytest.mark.gpu

BS, HKV, HQ, D, DT = 16, 2, 8, 128, "bf16"


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


class Engine:
    def __init__(self, rng, num_blocks, num_cpu=0, window=0, caching=False):
        self.rng = rng
        self.bm = BlockManager(BS, num_blocks, num_cpu, sliding_window=window, prefix_caching=caching)
        self.geom = oracle.Geom(num_blocks, BS, HKV, D, DT)
        self.host_pool = np.full(self.geom.layer_elems, NAN_BITS[DT], dtype=np.uint16)   # oracle's device pool
        self.dev_pool = u16_to_dev(self.host_pool, DT)
        self.desc = desc_of(num_blocks, BS, HKV, D, DT)
        if num_cpu:
            self.hgeom = oracle.Geom(num_cpu, BS, HKV, D, DT)
            self.ocpu = np.zeros(self.hgeom.layer_elems, dtype=np.uint16)
            self.pinned = torch.zeros(self.hgeom.layer_elems, dtype=torch.bfloat16).pin_memory()
            self.hdesc = desc_of(num_cpu, BS, HKV, D, DT)

    def write(self, slots):
        k = to_bits(self.rng.standard_normal((len(slots), HKV, D)), DT)
        v = to_bits(self.rng.standard_normal((len(slots), HKV, D)), DT)
        sm = np.asarray(slots, np.int64)
        pkv.reshape_and_cache(self.dev_pool, self.desc, u16_to_dev(k, DT), u16_to_dev(v, DT),
                              torch.from_numpy(sm).cuda())
        assert oracle.reshape_and_cache(self.host_pool, self.geom, k, v, sm) == 0

    def prompt(self, sid, tokens):
        self.bm.allocate(sid, tokens)
        table, n = self.bm.block_table(sid)
        t = np.arange(n)
        self.write(table[(t // BS)].astype(np.int64) * BS + t % BS)

    def step(self, sids, token=7):
        slots, pairs = [], []
        for sid in sids:
            slot, cow = self.bm.append_slot(sid, token)
            slots.append(slot)
            if cow:
                pairs.append(cow)
        if pairs:
            pkv.copy_blocks(self.dev_pool, self.desc, pairs)
            assert oracle.copy_blocks(self.host_pool, self.geom, np.array(pairs)) == 0
        self.write(slots)
        return pairs

    def check_pool(self):
        assert np.array_equal(dev_to_u16(self.dev_pool), self.host_pool)

    def decode(self, sids, window=0, ring=0):
        tabs = [self.bm.block_table(s) for s in sids]
        width = ring or max(len(t) for t, _ in tabs)
        tables = np.full((len(sids), width), -1, np.int32)
        for i, (t, _) in enumerate(tabs):
            tables[i, :min(width, len(t))] = t[:width]
        ctx = np.array([n for _, n in tabs], np.int32)
        q = to_bits(self.rng.standard_normal((len(sids), HQ, D)), DT)
        scale = 1 / math.sqrt(D)
        ref, err = oracle.decode(q, self.host_pool, self.geom, tables, ctx, scale, max_context_len=int(ctx.max()),
                                 window=window, ring=ring)
        assert err == 0
        out = torch.empty((len(sids), HQ, D), dtype=torch.bfloat16, device="cuda")
        mx = int(ctx.max())
        span = pkv.decode_window_span(mx, BS, window, ring)
        nbytes = pkv.decode_workspace_bytes(self.desc, len(sids), HQ, span, 128)
        ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
        pkv.decode_window(out, u16_to_dev(q, DT), self.dev_pool, self.desc, torch.from_numpy(tables).cuda(),
                          torch.from_numpy(ctx).cuda(), mx, scale, window, ring, ws, 128)
        assert_attention_close(out, ref, "engine step")


def test_parallel_sampling_with_copy_on_write():
    eng = Engine(np.random.default_rng(400), num_blocks=64)
    eng.prompt(0, list(range(37)))
    eng.bm.fork(0, 1)
    eng.bm.fork(0, 2)
    cow_seen = 0
    for _ in range(20):
        cow_seen += len(eng.step([0, 1, 2]))
        eng.check_pool()
        eng.decode([0, 1, 2])
    assert cow_seen == 2        # the shared partial prompt block is copied for two of the three samples


def test_sliding_window_wraps_through_the_ring():
    eng = Engine(np.random.default_rng(401), num_blocks=32, window=40)
    ring = -(-40 // BS)
    eng.prompt(0, list(range(20)))
    eng.prompt(1, list(range(3)))
    for i in range(70):
        eng.step([0, 1])
        if i % 7 == 0:
            eng.check_pool()
            eng.decode([0, 1], window=40, ring=ring)


def test_prefix_cache_and_swap_round_trip():
    eng = Engine(np.random.default_rng(402), num_blocks=48, num_cpu=16, caching=True)
    prompt = [int(x) for x in np.random.default_rng(0).integers(0, 5, 40)]
    eng.prompt(0, prompt)
    eng.bm.allocate(1, prompt[:32] + [9, 9, 9])        # shares the first two full blocks
    t0, t1 = eng.bm.block_table(0)[0], eng.bm.block_table(1)[0]
    assert t0[:2].tolist() == t1[:2].tolist()
    n = eng.bm.block_table(1)[1]
    eng.write([int(t1[2]) * BS + t % BS for t in range(32, n)])   # only the unshared tail is written
    for _ in range(5):
        eng.step([0, 1])
    eng.decode([0, 1])
    pairs_out = eng.bm.swap_out([1])
    pkv.swap_blocks(eng.pinned, eng.hdesc, eng.dev_pool, eng.desc, 0, pairs_out)
    torch.cuda.synchronize()
    assert oracle.swap_blocks(eng.ocpu, eng.hgeom, eng.host_pool, eng.geom, pairs_out) == 0
    assert np.array_equal(eng.pinned.view(torch.int16).numpy().view(np.uint16), eng.ocpu)
    eng.step([0])
    pairs_in = eng.bm.swap_in([1])
    pkv.swap_blocks(eng.dev_pool, eng.desc, eng.pinned, eng.hdesc, 1, pairs_in)
    assert oracle.swap_blocks(eng.host_pool, eng.geom, eng.ocpu, eng.hgeom, pairs_in) == 0
    eng.check_pool()
    for _ in range(3):
        eng.step([0, 1])
    eng.check_pool()
    eng.decode([0, 1])
