"""Causal prefill / extend over the paged cache (pa_prefill) against the oracle.

Pools are built by the oracle (NaN everywhere no written slot is, so a stray
read poisons the output); each case mixes whole prompts and extends whose
lengths straddle the 128-token tiles, sequences with no new tokens and
single-token queries."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
import gpu_helpers
from gpu_helpers import ensure_built, paged_to_dev, u16_to_dev
from paged_helpers import Paged, to_bits

pytestmark = pytest.mark.gpu


def assert_attention_close(got, ref, what=""):
    """The combined attention bound only (no separate fp16 max-rel bound): the
    fp16 PV product takes the weights as one fp16 operand."""
    return gpu_helpers.assert_attention_close(got, ref, what, strict_fp16=False)


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


class PrefillCase:
    def __init__(self, rng, q_lens, ctx, Hq, Hkv, D, bs, dtype, values="normal"):
        self.p = Paged(rng, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, bs=bs, ctx=ctx, dtype=dtype, values=values)
        self.q_lens = np.asarray(q_lens, np.int32)
        self.qsl = np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)
        self.T = int(self.qsl[-1])
        self.q_bits = to_bits(rng.standard_normal((self.T, Hq, D)) if values == "normal"
                              else rng.uniform(-1, 1, (self.T, Hq, D)), dtype)

    def run(self, scale, max_query_len=None, tables=None, err=None):
        p = self.p
        _, pool, tab, ctx, desc = paged_to_dev(p)
        if tables is not None:
            tab = torch.from_numpy(tables).cuda()
        q = u16_to_dev(self.q_bits, p.dtype)
        out = torch.full_like(q, float("nan"))
        mq = int(self.q_lens.max()) if max_query_len is None else max_query_len
        pkv.prefill(out, q, pool, desc, tab, ctx, torch.from_numpy(self.qsl).cuda(), mq, scale, dev_err=err)
        return out

    def expected(self, scale, tables=None):
        p = self.p
        return oracle.prefill(self.q_bits, p.pool, p.geom, p.tables if tables is None else tables, p.ctx, self.qsl,
                              scale)


MIX = ([1, 5, 127, 128, 129, 17, 64, 0, 1, 40],            # q_len
       [1, 5, 127, 128, 129, 400, 320, 50, 1000, 40])       # ctx


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_prefill_matches_oracle(G, D, dtype):
    rng = np.random.default_rng(600 + G * 10 + D)
    case = PrefillCase(rng, *MIX, Hq=2 * G, Hkv=2, D=D, bs=16, dtype=dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(D)
    out = case.run(scale, err=err)
    assert pkv.read_device_errors(err) == 0
    ref, e = case.expected(scale)
    assert e == 0
    assert_attention_close(out, ref, f"prefill G={G} D={D} {dtype}")


@pytest.mark.parametrize("bs", [8, 32])
def test_prefill_block_sizes(bs):
    rng = np.random.default_rng(620 + bs)
    case = PrefillCase(rng, [200, 33, 300], [200, 700, 301], Hq=8, Hkv=2, D=128, bs=bs, dtype="bf16")
    out = case.run(0.088)
    ref, e = case.expected(0.088)
    assert e == 0
    assert_attention_close(out, ref, f"prefill bs={bs}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_large_scores_take_the_rescale_path(dtype):
    # scale 1 on N(0,1) data: scores spread over tens of units, so the running
    # maximum grows by more than 2^8 across tiles and O is rescaled in TMEM
    rng = np.random.default_rng(630)
    case = PrefillCase(rng, [600, 130], [900, 130], Hq=4, Hkv=1, D=128, bs=16, dtype=dtype)
    out = case.run(1.0)
    ref, e = case.expected(1.0)
    assert e == 0
    assert_attention_close(out, ref, f"prefill, large scores, {dtype}")


def test_prefill_error_rows():
    rng = np.random.default_rng(640)
    case = PrefillCase(rng, [10, 6, 3, 300], [50, 4, 60, 300], Hq=4, Hkv=2, D=128, bs=16, dtype="f16")
    tables = case.p.tables.copy()
    tables[2, 3] = case.p.num_blocks + 7          # the third sequence reads block 3 (positions 48..59)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = case.run(0.1, tables=tables, err=err)
    bits = pkv.read_device_errors(err)
    assert bits == pkv.DEVERR_CONTEXT | pkv.DEVERR_BLOCK_ID
    ref, e = case.expected(0.1, tables=tables)
    assert e == oracle.ERR_CONTEXT | oracle.ERR_BLOCK_ID
    qsl = case.qsl
    assert bool((out[qsl[1]:qsl[3]] == 0).all())          # q_len > ctx, and the bad block id
    assert_attention_close(out[:qsl[1]], ref[:qsl[1]], "rows beside the bad sequences")
    assert_attention_close(out[qsl[3]:], ref[qsl[3]:], "rows beside the bad sequences")
    # max_query_len below a sequence's q_len: that sequence's rows are zeroed
    err.zero_()
    out = case.run(0.1, max_query_len=100, err=err)
    assert pkv.read_device_errors(err) & pkv.DEVERR_CONTEXT
    assert bool((out[qsl[3]:] == 0).all())
    ref, _ = case.expected(0.1)
    assert_attention_close(out[:qsl[1]], ref[:qsl[1]], "short sequences with a small max_query_len")


@pytest.mark.parametrize("name", ["prefill_tiny", "prefill_8b", "extend_8b", "prefill_7b"])
def test_full_size_prefill_step_matches_oracle(name):
    """The benchmarked step (reshape_and_cache of every new token, then pa_prefill)
    against the oracle: the whole pool bit for bit, and attention on every
    (token, head) row."""
    from paged_kv_cache_168_gb300.step import PrefillStep
    from paged_kv_cache_168_gb300.workloads import as_u16, make_prefill_workload
    w = make_prefill_workload(name, device="cuda")
    cfg = w.cfg
    g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
    pool = as_u16(w.kv_cache).reshape(-1)
    step = PrefillStep(w)
    out = step()
    torch.cuda.synchronize()
    assert pkv.read_device_errors(step.dev_err) == 0
    assert oracle.reshape_and_cache(pool, g, as_u16(w.key), as_u16(w.value), w.slot_mapping_np) == 0
    assert np.array_equal(as_u16(w.kv_cache).reshape(-1), pool)
    q = as_u16(w.q)
    qsl, ctx = w.query_start_loc_np, w.context_lens_np
    ref, e = oracle.prefill(q, pool, g, w.block_tables_np, ctx, qsl, w.scale)
    assert e == 0
    assert_attention_close(out, ref, f"full-size {name}")
