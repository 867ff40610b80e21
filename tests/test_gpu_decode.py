"""GPU parity of paged decode attention against the fp64 CPU oracle.

Pools are built by the oracle (reshape_and_cache of every history token) into
NaN-filled memory, so any read of an unused block or a tail slot poisons the
output.  Elementwise bound: |gpu - oracle| <= 2e-3 + 1e-2 |oracle|."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import assert_attention_close, ensure_built, paged_to_dev, run_decode
from paged_helpers import Paged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


def check(p, P=0, max_ctx=None, what=""):
    scale = 1 / math.sqrt(p.D)
    max_ctx = max_ctx or max(int(p.ctx.max()), 1)
    ref, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, max_context_len=max_ctx)
    assert err == 0
    q, pool, tables, ctx, desc = paged_to_dev(p)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_decode(q, pool, desc, tables, ctx, max_ctx, scale, P, dev_err)
    assert pkv.read_device_errors(dev_err) == 0
    assert_attention_close(out, ref, what)
    return out


def ctx_cases(bs, P):
    return [1, max(bs - 1, 2), bs, bs + 1, P - 1, P, P + 1, 2 * P + 7, 3]


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    """Which decode kernel serves head_size 128: the tensor-core one (default) or
    the CUDA-core one (selected through PAGEDKV_DECODE_KERNEL=simt)."""
    if request.param == "simt":
        monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PAGEDKV_DECODE_KERNEL", raising=False)
    return request.param


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 1), (32, 8), (64, 8), (4, 2), (16, 1)])
def test_decode_sweep(dtype, bs, D, Hq, Hkv, kernel):
    if (D == 64 or bs < 8) and kernel == "tc":
        pytest.skip("head_size 64 and block sizes below 8 are served by the CUDA-core kernel only")
    if Hq // Hkv == 16 and (D != 128 or kernel != "tc"):
        pytest.skip("16 query heads per kv head: tensor-core kernel (head_size 128, block_size >= 8) only")
    rng = np.random.default_rng(zlib.crc32(repr((dtype, bs, D, Hq, Hkv)).encode()))
    P = 128
    ctx = ctx_cases(bs, P)
    p = Paged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype)
    check(p, P=P, what=f"{kernel} {dtype} bs{bs} D{D} {Hq}/{Hkv}")


def test_both_kernels_agree_on_many_sequences(monkeypatch):
    # more items than SMs, so every persistent CTA walks several items and tiles
    rng = np.random.default_rng(210)
    ctx = list(rng.integers(1, 700, size=300))
    p = Paged(rng, S=len(ctx), Hq=8, Hkv=2, D=128, bs=16, ctx=ctx, dtype="bf16")
    out_tc = check(p, P=256, what="tc many")
    monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")
    out_simt = check(p, P=256, what="simt many")
    assert_attention_close(out_tc, out_simt.to(torch.float64).cpu().numpy(), "tc vs simt")


@pytest.mark.parametrize("P", [128, 256, 512, 8192])
def test_partition_size_does_not_change_the_result(P, kernel):
    rng = np.random.default_rng(200)
    ctx = [1, 127, 128, 129, 700, 2049, 3000]
    p = Paged(rng, S=len(ctx), Hq=8, Hkv=2, D=128, bs=16, ctx=ctx, dtype="bf16")
    check(p, P=P, what=f"P={P}")


@pytest.mark.parametrize("P", [4096, 8192])
def test_remainders_of_every_length_class(P, kernel):
    # remainder partitions of P - 1 tokens have P / 128 tiles: the top class of
    # the tensor-core kernel's longest-first item order
    rng = np.random.default_rng(230 + P // 1024)
    ctx = [P - 1, 2 * P - 1, P - 127, P - 128, P - 129, P + 1, 1, P, 3 * P - 5]
    p = Paged(rng, S=len(ctx), Hq=8, Hkv=2, D=128, bs=16, ctx=ctx, dtype="bf16")
    check(p, P=P, what=f"remainder classes P={P}")


def test_tiny_config_end_to_end():
    w = pytest.importorskip("paged_kv_cache_168_gb300.workloads").make_workload("tiny", device="cuda",
                                                                                nan_unused=True)
    from gpu_helpers import desc_of, dev_to_u16
    from paged_kv_cache_168_gb300.workloads import as_u16
    cfg = w.cfg
    g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
    pool = as_u16(w.kv_cache).reshape(-1)
    desc = desc_of(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
    pkv.reshape_and_cache(w.kv_cache, desc, w.key, w.value, w.slot_mapping)
    oracle.reshape_and_cache(pool, g, as_u16(w.key), as_u16(w.value), w.slot_mapping_np)
    assert np.array_equal(dev_to_u16(w.kv_cache).reshape(-1), pool)
    out = run_decode(w.q, w.kv_cache, desc, w.block_tables, w.context_lens, w.max_context_len, w.scale)
    ref, err = oracle.decode(as_u16(w.q), pool, g, w.block_tables_np, w.context_lens_np, w.scale,
                             max_context_len=w.max_context_len)
    assert err == 0
    assert_attention_close(out, ref, "tiny")


def test_physical_placement_gives_bit_identical_output(kernel):
    outs = []
    for perm in (None, np.arange(40)[::-1].copy(), np.random.default_rng(9).permutation(40)):
        rng = np.random.default_rng(201)
        p = Paged(rng, S=4, Hq=16, Hkv=4, D=128, bs=16, ctx=[5, 160, 300, 33], num_blocks=40, dtype="bf16",
                  perm=perm)
        q, pool, tables, ctx, desc = paged_to_dev(p)
        outs.append(run_decode(q, pool, desc, tables, ctx, 300, 0.088, P=128))
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_block_size_gives_matching_output():
    for bs in (1, 2, 4, 8, 16, 32):
        rng = np.random.default_rng(202)
        p = Paged(rng, S=3, Hq=8, Hkv=2, D=64, bs=bs, ctx=[1, 200, 513], dtype="f16")
        check(p, P=256, what=f"bs={bs}")


def test_shared_prefix_blocks_equal_unshared_copies(kernel):
    rng = np.random.default_rng(203)
    p = Paged(rng, S=2, Hq=8, Hkv=8, D=128, bs=16, ctx=[300, 300], num_blocks=48, dtype="f16")
    p.K[1][:256] = p.K[0][:256]
    p.V[1][:256] = p.V[0][:256]
    p.q_bits[1] = p.q_bits[0]
    p.write_all()
    shared = p.tables.copy()
    shared[1, :16] = shared[0, :16]
    q, pool, tables, ctx, desc = paged_to_dev(p)
    a = run_decode(q, pool, desc, tables, ctx, 300, 0.088, P=128)
    b = run_decode(q, pool, desc, torch.from_numpy(shared).cuda(), ctx, 300, 0.088, P=128)
    assert torch.equal(a, b)


def test_bad_block_ids_among_many_items(kernel):
    # several items per persistent CTA, so an item's ids are checked while the
    # item before it streams: bad ids in first, middle and last partitions
    rng = np.random.default_rng(206)
    S = 300
    ctx = rng.integers(1, 600, size=S)
    bad = {7: 0, 55: None, 123: None, 250: 0, 299: None}     # sequence -> table entry (None: the last)
    for s_ in bad:
        ctx[s_] = max(int(ctx[s_]), 300)
    p = Paged(rng, S=S, Hq=4, Hkv=2, D=128, bs=16, ctx=list(ctx), dtype="f16")
    scale = 1 / math.sqrt(128)
    mx = int(p.ctx.max())
    ref, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, max_context_len=mx)
    q, pool, tables, ctx_d, desc = paged_to_dev(p)
    bad_tables = tables.clone()
    for i, (s_, e) in enumerate(bad.items()):
        e = (int(p.ctx[s_]) - 1) // 16 if e is None else e
        if s_ == 55:
            e = 10                                            # a middle partition (P = 128: 8 blocks each)
        bad_tables[s_, e] = -1 - i if i % 2 else p.num_blocks + i
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_decode(q, pool, desc, bad_tables, ctx_d, mx, scale, P=128, dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_BLOCK_ID
    rows = sorted(bad)
    assert torch.all(out[rows] == 0)
    good = [s_ for s_ in range(S) if s_ not in bad]
    assert_attention_close(out[good], ref[good], f"{kernel}: sequences beside bad ones")


@pytest.mark.parametrize("D", [64, 128])
def test_zero_context_rows_are_zero(D, kernel):
    rng = np.random.default_rng(204)
    p = Paged(rng, S=3, Hq=4, Hkv=4, D=D, bs=16, ctx=[0, 20, 0], dtype="f16")
    out = check(p, P=128)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)


def test_device_errors_skip_the_item_and_zero_its_output(kernel):
    rng = np.random.default_rng(205)
    p = Paged(rng, S=4, Hq=8, Hkv=2, D=128, bs=16, ctx=[40, 600, 50, 300], dtype="bf16", width=40)
    scale = 0.088
    ref, _ = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, max_context_len=640)
    q, pool, tables, ctx, desc = paged_to_dev(p)
    bad_tables = tables.clone()
    bad_tables[1, 30] = p.num_blocks          # inside ctx of sequence 1 (a later partition)
    bad_tables[2, 1] = -5                     # sequence 2 (single partition)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_decode(q, pool, desc, bad_tables, ctx, 640, scale, P=128, dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_BLOCK_ID
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    assert_attention_close(out[[0, 3]], ref[[0, 3]], "untouched sequences")
    # a context longer than the table row (or than max_context_len) is flagged and zeroed
    long_ctx = ctx.clone()
    long_ctx[3] = 40 * 16 + 1
    out = run_decode(q, pool, desc, tables, long_ctx, 700, scale, P=128, dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_CONTEXT
    assert torch.all(out[3] == 0)
    assert_attention_close(out[:3], ref[:3], "other sequences")
    out = run_decode(q, pool, desc, tables, ctx, 512, scale, P=128, dev_err=err)   # 600 > 512
    assert pkv.read_device_errors(err) == pkv.DEVERR_CONTEXT and torch.all(out[1] == 0)


@pytest.mark.parametrize("D", [64, 128])
def test_entries_past_the_context_are_never_read(D, kernel):
    # table padding of -1 (already in every Paged case) plus garbage ids past ceil(ctx/bs)
    rng = np.random.default_rng(206)
    p = Paged(rng, S=2, Hq=4, Hkv=4, D=D, bs=16, ctx=[17, 100], dtype="f16", width=12)
    p.tables[0, 2:] = 10 ** 6
    check(p, P=128)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (64, 8)])
def test_decode_tiles_with_far_apart_maxima(dtype, Hq, Hkv, kernel):
    # keys of every other 128-token tile scaled by 8 (exact in fp16/bf16): the
    # score maxima of consecutive tiles differ by tens of base-2 units, so the
    # running maximum jumps between tiles and, with two softmax groups taking
    # alternate tiles, one group's share of an item all but vanishes in the merge
    rng = np.random.default_rng(zlib.crc32(repr(("far", dtype, Hq, Hkv)).encode()))
    ctx = [128 * 5 + 17, 300, 129, 1000, 384, 2048]
    p = Paged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=128, bs=16, ctx=ctx, dtype=dtype)
    for s, c in enumerate(ctx):
        hot = (np.arange(c) // 128) % 2 == s % 2
        p.K[s][hot] *= 8.0
    p.write_all()
    check(p, P=512, what=f"{kernel} far-apart maxima {dtype} {Hq}/{Hkv}")


@pytest.mark.parametrize("S", [8192, 8193])
def test_decode_at_the_tensor_core_sequence_limit(S):
    # 8192 sequences is the most the tensor-core decode takes (its item-order
    # tables live in shared memory); one more goes to the CUDA-core kernel
    rng = np.random.default_rng(320 + S)
    ctx = rng.integers(0, 48, size=S)
    ctx[::501] = 0
    p = Paged(rng, S=S, Hq=2, Hkv=1, D=128, bs=16, ctx=list(ctx), dtype="f16")
    check(p, what=f"S={S} at the tensor-core limit")


@pytest.mark.parametrize("S,Hq,Hkv,dtype", [(700, 8, 2, "bf16"), (1100, 4, 4, "f16")])
def test_decode_many_sequences_item_order(S, Hq, Hkv, dtype):
    # more than 512 sequences (the tensor-core decode's 2-stage ring) with
    # contexts of every partition class, zeros included: every item of the
    # longest-first, snake-ordered walk must be served exactly once
    rng = np.random.default_rng(300 + S)
    ctx = rng.integers(0, 600, size=S)
    ctx[::97] = 0
    ctx[5::89] = 128 * rng.integers(1, 5, size=len(ctx[5::89]))   # whole partitions, no remainder
    p = Paged(rng, S=S, Hq=Hq, Hkv=Hkv, D=128, bs=16, ctx=list(ctx), dtype=dtype)
    check(p, P=128, what=f"many sequences S={S}")
