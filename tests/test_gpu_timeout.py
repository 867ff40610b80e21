"""The bounded waits of the CUDA-core decode kernels, made to run out.

Every wait inside the kernels is bounded; when one runs out the CTA reports
PA_DEVERR_TIMEOUT, waits (with the full bound) for the bulk copies it issued,
and abandons its item: a single-partition item writes zero rows, a partition
of a longer context marks itself invalid so that the merge writes zero rows.
PAGEDKV_WAIT_POLLS=n makes the ordinary waits of the CUDA-core decode kernels
(16-bit and 8-bit caches) give up after n non-suspending polls, so with n = 1
they run out during an ordinary call.  The test checks that the error word
says so, that every output row is either the correct result or zeros, and
that the next call without the limit, on the same device, is correct again:
the abandoning CTAs left nothing in flight and the context stays usable."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import ATOL, RTOL, TORCH_DT, assert_attention_close, ensure_built, paged_to_dev, u16_to_dev
from paged_helpers import Paged, i8_pool_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


def _rows_zero_or_correct(out: torch.Tensor, ref: np.ndarray, what: str) -> int:
    """Every (sequence, head) row is all zeros (abandoned) or within the attention
    tolerance of the oracle; returns the number of zero rows."""
    g = out.detach().to(torch.float64).cpu().numpy().reshape(ref.shape)
    zero = (g == 0).all(axis=-1)
    close = (np.abs(g - ref) <= ATOL + RTOL * np.abs(ref)).all(axis=-1)
    bad = ~(zero | close)
    assert not bad.any(), f"{what}: {int(bad.sum())} rows neither zero nor correct"
    return int(zero.sum())


def _case(kind):
    rng = np.random.default_rng(880 if kind == "f16" else 881)
    ctx = [4096, 3000, 2049, 1024, 700, 129, 17, 1]
    if kind == "f16":
        p = Paged(rng, S=len(ctx), Hq=8, Hkv=2, D=128, bs=16, ctx=ctx, dtype="f16")
        q, pool, tables, ctxd, desc = paged_to_dev(p)
        ref, e = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 1 / math.sqrt(128),
                               max_context_len=max(ctx))
    else:
        q_bits, hpool, g, htables, hctx = i8_pool_case(rng, ctx, 8, 2, 16, "bf16")
        q, pool, tables, ctxd = (u16_to_dev(q_bits, "bf16"), torch.from_numpy(hpool).cuda(),
                                 torch.from_numpy(htables).cuda(), torch.from_numpy(hctx).cuda())
        desc = pkv.CacheDesc(g.num_blocks, 16, 2, 128, TORCH_DT["bf16"], kv_int8=True)
        ref, e = oracle.decode_i8(q_bits, hpool, g, htables, hctx, 1 / math.sqrt(128), max_context_len=max(ctx))
    assert e == 0
    return (q, pool, tables, ctxd, desc), ref, max(ctx)


def _run(dev, max_ctx, P):
    q, pool, tables, ctx, desc = dev
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(max(pkv.decode_workspace_bytes(desc, q.shape[0], q.shape[1], max_ctx, P) // 4, 4),
                     dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.decode(out, q, pool, desc, tables, ctx, max_ctx, 1 / math.sqrt(128), ws, P, dev_err=err)
    torch.cuda.synchronize()
    return out, pkv.read_device_errors(err)


@pytest.mark.parametrize("cache", ["f16", "bf16-int8"])
@pytest.mark.parametrize("P", [512, 4096])
def test_waits_run_out_and_the_context_stays_usable(cache, P, monkeypatch):
    monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")      # the CUDA-core kernels
    dev, ref, max_ctx = _case(cache)
    monkeypatch.setenv("PAGEDKV_WAIT_POLLS", "1")
    timeouts = zero_rows = 0
    for _ in range(3):
        out, bits = _run(dev, max_ctx, P)
        assert bits & ~pkv.DEVERR_TIMEOUT == 0, f"unexpected device error bits {bits:#x}"
        timeouts += bool(bits & pkv.DEVERR_TIMEOUT)
        zero_rows += _rows_zero_or_correct(out, ref, f"{cache} P={P} with one-poll waits")
    assert timeouts > 0, "no wait ran out"
    assert zero_rows > 0, "a timeout was reported but no item was abandoned"
    monkeypatch.delenv("PAGEDKV_WAIT_POLLS")
    out, bits = _run(dev, max_ctx, P)
    assert bits == 0
    assert_attention_close(out, ref, f"{cache} P={P} after the timeouts")
