"""GPU parity of sliding-window decode (pa_decode_window) against the fp64 oracle,
on caches written token by token into ring block tables (stale tokens of older
blocks and never-written NaN slots must both stay outside the attended set) and
on linear tables."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import assert_attention_close, desc_of, ensure_built, u16_to_dev
from paged_helpers import Paged, RingPaged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    if request.param == "simt":
        monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PAGEDKV_DECODE_KERNEL", raising=False)
    return request.param


def run_window(p, window, ring, P=0, max_ctx=None, dev_err=None):
    max_ctx = max_ctx or int(p.ctx.max())
    q = u16_to_dev(p.q_bits, p.dtype)
    pool = u16_to_dev(p.pool, p.dtype)
    tables = torch.from_numpy(np.ascontiguousarray(p.tables)).cuda()
    ctx = torch.from_numpy(p.ctx).cuda()
    desc = desc_of(p.num_blocks, p.bs, p.Hkv, p.D, p.dtype)
    span = pkv.decode_window_span(max_ctx, p.bs, window, ring)
    nbytes = pkv.decode_workspace_bytes(desc, p.S, p.Hq, span, P)
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
    out = torch.full_like(q, float("nan"))
    pkv.decode_window(out, q, pool, desc, tables, ctx, max_ctx, 1 / math.sqrt(p.D), window, ring, ws, P,
                      dev_err=dev_err)
    return out


def check(p, window, ring, P=0, what=""):
    max_ctx = int(p.ctx.max())
    ref, err = oracle.decode(p.q_bits, p.pool, p.geom, p.tables, p.ctx, 1 / math.sqrt(p.D),
                             max_context_len=max_ctx, window=window, ring=ring)
    assert err == 0
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_window(p, window, ring, P, dev_err=dev_err)
    assert pkv.read_device_errors(dev_err) == 0
    assert_attention_close(out, ref, what)
    return out


@pytest.mark.parametrize("bs,W,exact", [(16, 32, True), (16, 32, False), (16, 20, True), (8, 200, True),
                                        (32, 100, False), (1, 40, True), (4, 9, True)])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 128), (32, 8, 128), (8, 2, 64)])
def test_ring_tables(bs, W, exact, Hq, Hkv, D, kernel):
    if kernel == "tc" and (bs < 8 or D != 128):
        pytest.skip("tensor-core kernel: head_size 128, block_size >= 8")
    ring = -(-(W - 1) // bs) + 1 if exact else -(-W // bs)     # exact window, or the page's ceil(W / bs)
    rng = np.random.default_rng(300 + bs * 7 + W)
    ctx = [1, 3, W - 1, W, W + 1, 3 * W + 5, 700]
    p = RingPaged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, ring=ring, dtype="bf16")
    check(p, W, ring, P=128, what=f"{kernel} ring bs{bs} W{W} ring{ring}")


@pytest.mark.parametrize("W", [1, 17, 129, 700])
def test_window_on_linear_tables(W, kernel):
    rng = np.random.default_rng(310 + W)
    p = Paged(rng, S=5, Hq=16, Hkv=4, D=128, bs=16, ctx=[2, 100, 300, 641, 1000], dtype="f16")
    check(p, W, 0, P=256, what=f"{kernel} linear W{W}")


def test_window_wider_than_the_context_is_plain_decode(kernel):
    rng = np.random.default_rng(320)
    p = Paged(rng, S=3, Hq=8, Hkv=2, D=128, bs=16, ctx=[9, 300, 515], dtype="bf16")
    a = run_window(p, 0, 0, P=128)
    b = run_window(p, 10 ** 6, 0, P=128)
    assert torch.equal(a, b)


def test_bad_ring_entry_sets_the_error_bit(kernel):
    rng = np.random.default_rng(330)
    p = RingPaged(rng, S=2, Hq=8, Hkv=8, D=128, bs=16, ctx=[100, 200], ring=3, dtype="bf16")
    p.tables[1, 2] = -4
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_window(p, 40, 3, P=128, dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_BLOCK_ID
    assert torch.all(out[1] == 0) and bool(torch.isfinite(out[0]).all())


def test_window_arguments_are_validated():
    rng = np.random.default_rng(340)
    p = RingPaged(rng, S=1, Hq=8, Hkv=8, D=128, bs=16, ctx=[10], ring=2, dtype="bf16")
    with pytest.raises(pkv.PagedKVError):
        run_window(p, -1, 0)
    with pytest.raises(pkv.PagedKVError):
        run_window(p, 16, 3)          # ring longer than the table row
