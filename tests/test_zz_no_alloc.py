"""pa_decode_static_workspace: decode for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc where they run decode -- a
plugin inside a framework whose allocator owns all device memory, a serving loop
that forbids allocation once it is running, a binding from another language that
cannot keep a device buffer alive between calls.  For them the library offers an
entry point that takes no workspace and uses a fixed array in its own device
memory instead.  These tests call it through the C ABI and check that it gives
the same output as pa_decode with a caller-allocated workspace (and the fp64
oracle's within the attention tolerance), on two calls in a row (the second
call must not be disturbed by what the first left in the shared array), for
16-bit and 8-bit caches and the default partition size, and that shapes too
large for the array are refused.

This file is named so that pytest collects it last."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import TORCH_DT, assert_attention_close, ensure_built, paged_to_dev, run_decode, u16_to_dev
from paged_helpers import Paged, i8_pool_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


def _case(seed, ctx, Hq=8, Hkv=2, D=128, bs=16, dtype="bf16"):
    p = Paged(np.random.default_rng(seed), S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype)
    return p, paged_to_dev(p)


def _i8_case(seed, ctx, Hq=8, Hkv=2, bs=16, dtype="bf16"):
    """An 8-bit pool the oracle writes from random K/V, random block placement."""
    q_bits, pool, g, tables, ctx = i8_pool_case(np.random.default_rng(seed), ctx, Hq, Hkv, bs, dtype)
    desc = pkv.CacheDesc(g.num_blocks, bs, Hkv, 128, TORCH_DT[dtype], kv_int8=True)
    dev = (u16_to_dev(q_bits, dtype), torch.from_numpy(pool).cuda(), torch.from_numpy(tables).cuda(),
           torch.from_numpy(ctx).cuda(), desc)
    return (q_bits, pool, g, tables, ctx), dev


def _static(q, pool, desc, tables, ctx, max_ctx, scale, P):
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv._lib.decode_static_workspace(out, q, pool, desc, tables, ctx, max_ctx, scale, P, dev_err=err)
    torch.cuda.synchronize()
    assert pkv.read_device_errors(err) == 0
    return out


def test_static_workspace_matches_caller_workspace_and_oracle_on_two_calls():
    """Two calls in a row with different data (the second must not be disturbed
    by what the first left in the shared array), each equal to pa_decode with a
    caller workspace and within the attention tolerance of the fp64 oracle."""
    P = 128
    cases = [_case(300, [1, 127, 129, 700, 2049, 3000]),
             _case(301, [3000, 5, 1500, 256, 257, 999], Hq=16, Hkv=16, D=64, bs=8, dtype="f16")]
    for p, (q, pool, tables, ctx, desc) in cases:
        max_ctx = int(p.ctx.max())
        scale = 1 / math.sqrt(p.D)
        need = pkv.decode_workspace_bytes(desc, p.S, p.Hq, max_ctx, P)
        assert 0 < need <= pkv._lib.STATIC_WORKSPACE_BYTES     # the shared array is really used
        ref = run_decode(q, pool, desc, tables, ctx, max_ctx, scale, P)
        out = _static(q, pool, desc, tables, ctx, max_ctx, scale, P)
        assert_attention_close(out, ref.to(torch.float64).cpu().numpy(), "static workspace vs caller workspace")
        want, e = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, max_context_len=max_ctx)
        assert e == 0
        assert_attention_close(out, want, "static workspace vs oracle")


def test_static_workspace_default_partition_and_8bit_cache():
    """The default partition size (here still several partitions per sequence)
    and an 8-bit cache, whose kernels lay out their partial results differently;
    two calls in a row, against pa_decode with a caller workspace and the oracle."""
    scale = 1 / math.sqrt(128)
    p, (q, pool, tables, ctx, desc) = _case(302, [5000, 1, 4097, 640, 2500])
    max_ctx = int(p.ctx.max())
    assert pkv.decode_partition_size(desc, p.S, max_ctx, 0) < max_ctx            # more than one partition
    assert pkv.decode_workspace_bytes(desc, p.S, p.Hq, max_ctx, 0) > 0
    (qb, hpool, g, htables, hctx), (q8, pool8, tables8, ctx8, desc8) = _i8_case(303, [3000, 17, 1029, 2049])
    max8 = int(hctx.max())
    assert pkv.decode_workspace_bytes(desc8, len(hctx), 8, max8, 512) > 0
    for _ in range(2):
        out = _static(q, pool, desc, tables, ctx, max_ctx, scale, 0)
        ref = run_decode(q, pool, desc, tables, ctx, max_ctx, scale, 0)
        assert_attention_close(out, ref.to(torch.float64).cpu().numpy(), "static workspace, default partition")
        want, e = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, scale, max_context_len=max_ctx)
        assert e == 0
        assert_attention_close(out, want, "static workspace, default partition, vs oracle")
        out8 = _static(q8, pool8, desc8, tables8, ctx8, max8, scale, 512)
        ref8 = run_decode(q8, pool8, desc8, tables8, ctx8, max8, scale, 512)
        assert_attention_close(out8, ref8.to(torch.float64).cpu().numpy(), "static workspace, 8-bit cache")
        want8, e = oracle.decode_i8(qb, hpool, g, htables, hctx, scale, max_context_len=max8)
        assert e == 0
        assert_attention_close(out8, want8, "static workspace, 8-bit cache, vs oracle")


def test_static_workspace_refuses_shapes_beyond_its_size():
    S, Hq, D, max_ctx, P = 2048, 64, 128, 8192, 128
    desc = pkv.CacheDesc(1, 16, 8, D, torch.float16)
    assert pkv.decode_workspace_bytes(desc, S, Hq, max_ctx, P) > pkv._lib.STATIC_WORKSPACE_BYTES
    q = torch.zeros((S, Hq, D), dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    pool = torch.zeros(8 * 2 * 16 * D, dtype=torch.float16, device="cuda")
    tables = torch.zeros((S, 1), dtype=torch.int32, device="cuda")
    ctx = torch.zeros(S, dtype=torch.int32, device="cuda")     # even if launched, nothing would be read
    with pytest.raises(pkv.PagedKVError) as e:
        pkv._lib.decode_static_workspace(out, q, pool, desc, tables, ctx, max_ctx, 0.088, P)
    assert e.value.status == pkv.PA_ERR_WORKSPACE_TOO_SMALL
    assert "PA_STATIC_WORKSPACE_BYTES" in str(e.value)
