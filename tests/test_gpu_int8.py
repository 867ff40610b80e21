"""8-bit KV cache on the GPU against the oracle.

The writer (pa_reshape_and_cache into an 8-bit pool) must produce the oracle's
bytes exactly: codes and fp32 scales are integer / IEEE decisions both sides
take in fp32.  Decode over an 8-bit pool the oracle built is compared with the
oracle's fp64 decode of code * scale within the attention tolerance.  Block
copies and swaps of 8-bit pools are compared bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import TORCH_DT, assert_attention_close, ensure_built, u16_to_dev
from paged_helpers import to_bits
from paged_kv_cache_168_gb300.step import DecodeStep
from paged_kv_cache_168_gb300.workloads import as_u16, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    """Which 8-bit decode runs: the default dispatch (tensor cores with converter
    warps from 4 query heads per kv head, CUDA cores below) or the CUDA-core
    kernel everywhere (PAGEDKV_DECODE_KERNEL=simt)."""
    if request.param == "simt":
        monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PAGEDKV_DECODE_KERNEL", raising=False)
    return request.param


def i8_desc(nb, bs, hkv, dtype):
    return pkv.CacheDesc(nb, bs, hkv, 128, TORCH_DT[dtype], kv_int8=True)


def pool_to_dev(pool: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(pool).cuda()


def special_vectors(dtype):
    """Vectors whose quantisation hits the edge cases: ties at amax 127 (x * 1.0
    exactly half-way), an all-zero vector, a single spike, tiny and large scales."""
    v = np.zeros((6, 128))
    v[0, 0] = 127.0
    v[0, 1:9] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5]     # round-half-even both ways
    v[2, 17] = -3.0                                                    # one spike: code -127, rest 0
    v[3] = np.linspace(-1e-3, 1e-3, 128)
    v[4] = np.linspace(-6e4, 6e4, 128) if dtype == "f16" else np.linspace(-1e30, 1e30, 128)
    v[5] = 1.0                                                         # constant: all codes 127
    return v


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32])
def test_writer_bytes_equal_oracle(bs, dtype):
    rng = np.random.default_rng(500 + bs)
    hkv, n = 3, 150
    nb = max(40, -(-2 * n // bs))
    g = oracle.Geom(nb, bs, hkv, 128, dtype)
    init = rng.integers(0, 256, nb * oracle.i8_block_bytes(g), dtype=np.uint8)   # stale bytes in the pool
    slots = rng.choice(nb * bs, n, replace=False).astype(np.int64)
    slots[13::17] = -1
    x = np.clip(rng.standard_normal((2, n, hkv, 128)) * rng.lognormal(0, 2, (2, n, hkv, 1)), -3e4, 3e4)
    sp = special_vectors(dtype)
    x[0, :6, 0], x[1, 6:12, 1] = sp, sp
    k, v = to_bits(x[0], dtype), to_bits(x[1], dtype)
    ref = init.copy()
    assert oracle.reshape_and_cache_i8(ref, g, k, v, slots) == 0
    dev = pool_to_dev(init.copy())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(dev, i8_desc(nb, bs, hkv, dtype), u16_to_dev(k, dtype), u16_to_dev(v, dtype),
                          torch.from_numpy(slots).cuda(), dev_err=err)
    assert pkv.read_device_errors(err) == 0
    got = dev.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError(f"{bad.size} bytes differ, first at {bad[:8]}: gpu {got[bad[:8]]} oracle {ref[bad[:8]]}")


def test_writer_strided_inputs_and_bad_slot():
    rng = np.random.default_rng(510)
    nb, bs, hkv, dtype = 8, 16, 2, "bf16"
    g = oracle.Geom(nb, bs, hkv, 128, dtype)
    # key / value rows live inside a wider [n, 3 * hkv * 128] buffer (a fused qkv projection)
    n = 10
    big = to_bits(rng.standard_normal((n, 3, hkv, 128)), dtype)
    slots = np.array([3, 5, nb * bs, 7, -1, 100, 2, 9, 11, 12], np.int64)     # one slot out of range
    ref = np.zeros(nb * oracle.i8_block_bytes(g), np.uint8)
    assert oracle.reshape_and_cache_i8(ref, g, big[:, 1], big[:, 2], slots) == oracle.ERR_SLOT
    dev = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    bigd = u16_to_dev(big, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(dev, i8_desc(nb, bs, hkv, dtype), bigd[:, 1], bigd[:, 2], torch.from_numpy(slots).cuda(),
                          dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_SLOT
    assert np.array_equal(dev.cpu().numpy(), ref)


class I8Case:
    """Sequences' logical K/V written by the oracle into an 8-bit pool."""

    def __init__(self, rng, S, Hq, Hkv, bs, ctx, dtype, width=None):
        self.S, self.Hq, self.Hkv, self.bs, self.dtype = S, Hq, Hkv, bs, dtype
        self.ctx = np.asarray(ctx, np.int32)
        nblk = -(-self.ctx // bs)
        self.nb = int(nblk.sum()) + 3
        self.width = width or max(int(nblk.max()), 1)
        self.geom = oracle.Geom(self.nb, bs, Hkv, 128, dtype)
        self.pool = rng.integers(0, 256, self.nb * oracle.i8_block_bytes(self.geom), dtype=np.uint8)
        perm = rng.permutation(self.nb)
        self.tables = np.full((S, self.width), -1, np.int32)
        nxt = 0
        for s in range(S):
            self.tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
            nxt += nblk[s]
            c = int(self.ctx[s])
            if c == 0:
                continue
            t = np.arange(c)
            slots = self.tables[s, t // bs].astype(np.int64) * bs + t % bs
            x = rng.standard_normal((2, c, Hkv, 128))
            assert oracle.reshape_and_cache_i8(self.pool, self.geom, to_bits(x[0], dtype), to_bits(x[1], dtype),
                                               slots) == 0
        self.q_bits = to_bits(rng.standard_normal((S, Hq, 128)), dtype)

    def run(self, P=0, tables=None, err=None):
        tables = self.tables if tables is None else tables
        mx = max(int(self.ctx.max()), 1)
        q = u16_to_dev(self.q_bits, self.dtype)
        out = torch.full_like(q, float("nan"))
        desc = i8_desc(self.nb, self.bs, self.Hkv, self.dtype)
        nbytes = pkv.decode_workspace_bytes(desc, self.S, self.Hq, mx, P)
        ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
        pkv.decode(out, q, pool_to_dev(self.pool), desc,
                   torch.from_numpy(tables).cuda(), torch.from_numpy(self.ctx).cuda(), mx, 1 / math.sqrt(128), ws, P,
                   dev_err=err)
        return out

    def expected(self, tables=None):
        tables = self.tables if tables is None else tables
        return oracle.decode_i8(self.q_bits, self.pool, self.geom, tables, self.ctx, 1 / math.sqrt(128),
                                max_context_len=max(int(self.ctx.max()), 1))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [1, 4, 16, 32])
def test_decode_matches_oracle(bs, G, dtype, kernel):
    rng = np.random.default_rng(520 + bs * 10 + G)
    ctx = [1, 2, 63, 64, 65, 511, 512, 513, 1100, 0, 300]
    case = I8Case(rng, len(ctx), 2 * G, 2, bs, ctx, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = case.run(err=err)
    assert pkv.read_device_errors(err) == 0
    ref, e = case.expected()
    assert e == 0
    assert_attention_close(out, ref, f"int8 decode ({kernel}) bs={bs} G={G} {dtype}")


@pytest.mark.parametrize("P", [128, 256, 1024, 4096, 8192])
def test_decode_partition_sizes(P, kernel):
    rng = np.random.default_rng(540 + P)
    ctx = [129, 3000, 1024, 1025, 7, 9000]
    case = I8Case(rng, len(ctx), 8, 2, 16, ctx, "bf16")
    ref, e = case.expected()
    assert e == 0
    assert_attention_close(case.run(P=P), ref, f"int8 decode P={P}")


def test_decode_remainders_of_every_length_class(kernel):
    # a remainder of P - 1 tokens has P / 128 tiles: the top ordering class
    P = 8192
    rng = np.random.default_rng(545)
    ctx = [P - 1, 2 * P - 1, P - 127, P - 129, 3, P]
    case = I8Case(rng, len(ctx), 8, 2, 16, ctx, "f16")
    ref, e = case.expected()
    assert e == 0
    assert_attention_close(case.run(P=P), ref, "int8 decode, remainder classes")


@pytest.mark.parametrize("S", [1024, 1025])
def test_decode_at_the_tensor_core_sequence_limit(S):
    # 1024 sequences is the most the 8-bit tensor-core decode takes; one more
    # goes to the CUDA-core 8-bit kernel
    rng = np.random.default_rng(548 + S)
    ctx = rng.integers(0, 40, size=S)
    ctx[::97] = 0
    case = I8Case(rng, S, 2, 1, 16, list(ctx), "bf16")
    ref, e = case.expected()
    assert e == 0
    assert_attention_close(case.run(), ref, f"int8 decode, S={S} at the tensor-core limit")


def test_decode_bad_block_id_zeroes_the_item(kernel):
    rng = np.random.default_rng(550)
    ctx = [40, 900, 200]
    case = I8Case(rng, 3, 4, 2, 16, ctx, "f16")
    tables = case.tables.copy()
    tables[0, 1] = case.nb + 5          # single-partition sequence
    tables[1, 40] = -3                  # second partition of a two-partition sequence
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = case.run(tables=tables, err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_BLOCK_ID
    ref, e = case.expected(tables)
    assert e == oracle.ERR_BLOCK_ID
    assert bool((out[:2] == 0).all())
    assert_attention_close(out[2:], ref[2:], "int8 decode, good sequence beside bad ones")


@pytest.mark.parametrize("bs", [2, 16])
def test_copy_and_swap_blocks_bit_exact(bs):
    rng = np.random.default_rng(560 + bs)
    nb, hkv, layers = 12, 2, 2
    g = oracle.Geom(nb, bs, hkv, 128, "f16")
    bb = oracle.i8_block_bytes(g)
    pool = rng.integers(0, 256, layers * nb * bb, dtype=np.uint8)
    desc = pkv.CacheDesc(nb, bs, hkv, 128, torch.float16, num_layers=layers, kv_int8=True)
    dev = pool_to_dev(pool.copy())
    pairs = np.array([[0, 5], [3, 7], [11, 1]])
    pkv.copy_blocks(dev, desc, pairs)
    assert oracle.copy_blocks_bytes(pool, bb, nb, pairs, num_layers=layers) == 0
    assert np.array_equal(dev.cpu().numpy(), pool)
    hdesc = pkv.CacheDesc(4, bs, hkv, 128, torch.float16, num_layers=layers, kv_int8=True)
    host = torch.zeros(layers * 4 * bb, dtype=torch.uint8).pin_memory()
    out_pairs = np.array([[5, 0], [9, 3]])
    pkv.swap_blocks(host, hdesc, dev, desc, 0, out_pairs)
    torch.cuda.synchronize()
    for layer in range(layers):
        for src, dst in out_pairs:
            a = host.numpy()[(layer * 4 + dst) * bb:(layer * 4 + dst + 1) * bb]
            b = pool[(layer * nb + src) * bb:(layer * nb + src + 1) * bb]
            assert np.array_equal(a, b)
    pkv.swap_blocks(dev, desc, host, hdesc, 1, np.array([[0, 10], [3, 2]]))
    for layer in range(layers):
        for src, dst in ((0, 10), (3, 2)):
            pool[(layer * nb + dst) * bb:(layer * nb + dst + 1) * bb] = \
                host.numpy()[(layer * 4 + src) * bb:(layer * 4 + src + 1) * bb]
    assert np.array_equal(dev.cpu().numpy(), pool)


@pytest.mark.parametrize("name", ["7b_int8", "8b_int8"])
def test_full_size_step_matches_oracle(name):
    """The benchmarked step (the library builds the 8-bit pool from the logical
    history, writes the new token, decodes) against the oracle building its own
    pool from the same logical history: bytes of every block any sequence uses,
    and every output row."""
    w = make_workload(name, device="cuda")
    cfg = w.cfg
    step = DecodeStep(w)
    out = step()
    torch.cuda.synchronize()
    assert pkv.read_device_errors(step.dev_err) == 0
    g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, 128, cfg.dtype)
    bb = oracle.i8_block_bytes(g)
    ctx = w.context_lens_np
    seqs = list(range(cfg.num_seqs))
    bs = cfg.block_size
    blocks = np.unique(np.concatenate([w.block_tables_np[s, :-(-int(ctx[s]) // bs)] for s in seqs]))
    # oracle pool: the sampled sequences' blocks from the logical history, then the step's new tokens
    pool = np.zeros(w.num_blocks * bb, np.uint8)
    part = w.kv_logical[torch.from_numpy(blocks).cuda()]
    n = blocks.size * bs
    key = as_u16(part[:, :, 0].permute(0, 2, 1, 3).reshape(n, cfg.num_kv_heads, 128))
    value = as_u16(part[:, :, 1].permute(0, 2, 1, 3).reshape(n, cfg.num_kv_heads, 128))
    slots = (blocks[:, None].astype(np.int64) * bs + np.arange(bs)).reshape(-1)
    assert oracle.reshape_and_cache_i8(pool, g, key, value, slots) == 0
    assert oracle.reshape_and_cache_i8(pool, g, as_u16(w.key), as_u16(w.value), w.slot_mapping_np) == 0
    gpu_pool = step.kv_cache.cpu().numpy().reshape(w.num_blocks, bb)
    used = gpu_pool[blocks] == pool.reshape(w.num_blocks, bb)[blocks]
    assert used.all(), f"{int((~used.all(axis=1)).sum())} blocks differ, first {blocks[~used.all(axis=1)][0]}"
    ref, e = oracle.decode_i8(as_u16(w.q), pool, g, w.block_tables_np, ctx, w.scale,
                              max_context_len=w.max_context_len)
    assert e == 0
    assert_attention_close(out, ref, f"full-size {name}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("bs,W,exact", [(16, 40, True), (16, 200, False), (8, 100, True), (1, 30, True)])
def test_window_ring_decode_matches_oracle(bs, W, exact, G, dtype, kernel):
    # sliding-window decode over an 8-bit cache whose ring tables were written
    # token by token (older blocks overwritten; the pool starts as random bytes)
    rng = np.random.default_rng(570 + bs * 10 + W + G)
    ring = -(-(W - 1) // bs) + 1 if exact else -(-W // bs)
    ctx = np.asarray([1, W - 1, W, W + 1, 3 * W + 5, 700, 0], np.int32)
    S, Hkv = len(ctx), 2
    nb = S * ring + 3
    geom = oracle.Geom(nb, bs, Hkv, 128, dtype)
    pool = rng.integers(0, 256, nb * oracle.i8_block_bytes(geom), dtype=np.uint8)
    tables = rng.permutation(nb)[:S * ring].reshape(S, ring).astype(np.int32)
    for s, c in enumerate(ctx):
        if c == 0:
            continue
        t = np.arange(c)
        slots = tables[s, (t // bs) % ring].astype(np.int64) * bs + t % bs
        x = rng.standard_normal((2, c, Hkv, 128))
        assert oracle.reshape_and_cache_i8(pool, geom, to_bits(x[0], dtype), to_bits(x[1], dtype), slots) == 0
    q_bits = to_bits(rng.standard_normal((S, G * Hkv, 128)), dtype)
    mx = int(ctx.max())
    ref, e = oracle.decode_i8(q_bits, pool, geom, tables, ctx, 1 / math.sqrt(128), max_context_len=mx,
                              window=W, ring=ring)
    assert e == 0
    q = u16_to_dev(q_bits, dtype)
    out = torch.full_like(q, float("nan"))
    span = pkv.decode_window_span(mx, bs, W, ring)
    nbytes = pkv.decode_workspace_bytes(i8_desc(nb, bs, Hkv, dtype), S, G * Hkv, span, 128)
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.decode_window(out, q, pool_to_dev(pool), i8_desc(nb, bs, Hkv, dtype), torch.from_numpy(tables).cuda(),
                      torch.from_numpy(ctx).cuda(), mx, 1 / math.sqrt(128), W, ring, ws, 128, dev_err=err)
    assert pkv.read_device_errors(err) == 0
    assert_attention_close(out, ref, f"int8 window ({kernel}) bs={bs} W={W} ring={ring} G={G} {dtype}")
