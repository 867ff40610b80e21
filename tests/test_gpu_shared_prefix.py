"""pa_decode_shared_prefix on the GPU against the fp64 oracle.

Groups of sequences whose first blocks are the same physical blocks (beams of
one prompt after copy-on-write, mlqm.cn article section 二.2.2) are decoded with
each group's shared blocks streamed once for all its members.  The result must
be pa_decode's: every output row is compared with the oracle's plain decode of
each sequence through its own table row.  Cases: every query-head grouping the
kernel serves (1, 2, 4, 8 heads per kv head), block sizes 8 / 16 / 32, prompts
that are not whole blocks, groups larger than one tensor-core item's members,
a group of one, a member whose context is exactly the prompt, an empty prompt,
sequences in no group, partitions shorter than the prompt; then the checks the
kernel makes (a member whose table differs inside the prefix, group starts out
of order), the shapes that fall back to pa_decode, and the beam workload."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import TORCH_DT, assert_attention_close, ensure_built, u16_to_dev
from paged_helpers import SharedPaged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


def _dev(sp):
    q = u16_to_dev(sp.q_bits, sp.dtype)
    pool = u16_to_dev(sp.pool, sp.dtype)
    desc = pkv.CacheDesc(sp.num_blocks, sp.bs, sp.Hkv, sp.D, TORCH_DT[sp.dtype])
    return q, pool, desc


def run_shared(sp, q, pool, desc, tables, group_start, prefix_lens, P=0, max_ctx=None):
    S, Hq = q.shape[0], q.shape[1]
    max_ctx = max_ctx or max(int(sp.ctx.max()), 1)
    G = len(prefix_lens)
    nbytes = pkv.decode_shared_prefix_workspace_bytes(desc, S, Hq, G, max_ctx, P)
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.decode_shared_prefix(out, q, pool, desc, torch.from_numpy(np.ascontiguousarray(tables)).cuda(),
                             torch.from_numpy(sp.ctx).cuda(), max_ctx, 1 / math.sqrt(sp.D),
                             torch.from_numpy(np.asarray(group_start, np.int32)).cuda(),
                             torch.from_numpy(np.asarray(prefix_lens, np.int32)).cuda(), ws, P, dev_err=err)
    torch.cuda.synchronize()
    return out, pkv.read_device_errors(err)


def oracle_ref(sp, tables=None):
    ref, e = oracle.decode(sp.q_bits, sp.pool, sp.geom, sp.tables if tables is None else tables, sp.ctx,
                           1 / math.sqrt(sp.D), max_context_len=max(int(sp.ctx.max()), 1))
    assert e == 0
    return ref


GROUPS = [
    (2048, [2049, 2100, 2300, 2049]),        # four beams of one prompt
    (100, [150, 101, 300]),                  # a prompt that is not whole blocks
    (300, [310]),                            # a group of one: shares nothing
    (1000, [1001, 1500, 1200, 1100, 1050]),  # more members than one item takes (G >= 4)
    (64, [64, 69]),                          # a member whose context is exactly the prompt
    (0, [77, 9]),                            # nothing shared
    (700, [740]), (40, [41]),                # two sequences in no declared group
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("P", [0, 256])
def test_shared_prefix_matches_oracle(dtype, bs, Hq, Hkv, P):
    rng = np.random.default_rng(zlib.crc32(repr((dtype, bs, Hq, Hkv, P)).encode()))
    sp = SharedPaged(rng, GROUPS, Hq, Hkv, 128, bs, dtype)
    q, pool, desc = _dev(sp)
    # declare the first six groups; the last two sequences are in none
    gs, pl = sp.group_start[:7], sp.prompt_lens[:6]
    out, bits = run_shared(sp, q, pool, desc, sp.tables, gs, pl, P)
    assert bits == 0
    assert_attention_close(out, oracle_ref(sp), f"shared prefix {dtype} bs{bs} {Hq}/{Hkv} P{P}")


def test_declared_prefix_longer_than_shared_blocks_is_cut_to_the_group():
    # prefix_lens beyond the shortest member, or not whole blocks: the kernel
    # takes whole blocks up to the shortest member's context
    rng = np.random.default_rng(31)
    sp = SharedPaged(rng, [(512, [512, 600, 530]), (200, [260, 230])], 32, 8, 128, 16, "bf16")
    q, pool, desc = _dev(sp)
    out, bits = run_shared(sp, q, pool, desc, sp.tables, sp.group_start, [10**6, 200], 256)
    assert bits == 0
    assert_attention_close(out, oracle_ref(sp), "declared prefix cut to the group")


def test_member_with_other_blocks_inside_the_prefix_gets_zero_rows():
    rng = np.random.default_rng(32)
    sp = SharedPaged(rng, [(1024, [1100, 1050, 1200, 1030]), (512, [600, 700])], 32, 8, 128, 16, "bf16")
    q, pool, desc = _dev(sp)
    tables = sp.tables.copy()
    # member 2 of group 0 points its block 5 at a block with other data (its own tail block)
    tables[2, 5] = tables[2, 70]
    out, bits = run_shared(sp, q, pool, desc, tables, sp.group_start, sp.prompt_lens, 512)
    assert bits == pkv.DEVERR_PREFIX
    assert bool((out[2] == 0).all())
    ref = oracle_ref(sp)
    keep = [s for s in range(sp.S) if s != 2]
    assert_attention_close(out[keep], ref[keep], "members beside the mismatched one")


def test_group_starts_out_of_order_are_ignored():
    rng = np.random.default_rng(33)
    sp = SharedPaged(rng, [(512, [600, 530]), (256, [300, 280, 260])], 8, 8, 128, 16, "f16")
    q, pool, desc = _dev(sp)
    out, bits = run_shared(sp, q, pool, desc, sp.tables, [0, 4, 2], [512, 256], 256)
    assert bits == pkv.DEVERR_PREFIX
    assert_attention_close(out, oracle_ref(sp), "group starts out of order: no sharing")


@pytest.mark.parametrize("case", ["head64", "bs4", "simt", "many"])
def test_shapes_outside_the_kernel_fall_back_to_plain_decode(case, monkeypatch):
    rng = np.random.default_rng(34)
    D, bs, groups = 128, 16, [(300, [310, 400, 350]), (64, [100, 70])]
    if case == "head64":
        D = 64
    elif case == "bs4":
        bs = 4
    elif case == "simt":
        monkeypatch.setenv("PAGEDKV_DECODE_KERNEL", "simt")
    else:
        groups = [(64, [70, 80])] * 81           # 162 sequences: above the kernel's limit
    sp = SharedPaged(rng, groups, 16, 4, D, bs, "bf16")
    q, pool, desc = _dev(sp)
    out, bits = run_shared(sp, q, pool, desc, sp.tables, sp.group_start, sp.prompt_lens, 256)
    assert bits == 0
    assert_attention_close(out, oracle_ref(sp), f"fallback {case}")


def test_the_largest_batch_the_kernel_serves():
    # 160 sequences (40 groups of 4): the kernel's item tables at their largest
    rng = np.random.default_rng(35)
    groups = [(int(rng.integers(16, 400)), [int(c) for c in rng.integers(400, 700, 4)]) for _ in range(40)]
    sp = SharedPaged(rng, groups, 32, 8, 128, 16, "bf16")
    assert sp.S == 160
    q, pool, desc = _dev(sp)
    out, bits = run_shared(sp, q, pool, desc, sp.tables, sp.group_start, sp.prompt_lens, 0)
    assert bits == 0
    assert_attention_close(out, oracle_ref(sp), "160 sequences in groups")


def test_beam_workload_shared_prefix_equals_plain_decode():
    from paged_kv_cache_168_gb300.step import DecodeStep
    from paged_kv_cache_168_gb300.workloads import make_workload
    w = make_workload("beam", device="cuda", nan_unused=True)
    a = DecodeStep(w, shared_prefix=True)
    b = DecodeStep(w, shared_prefix=False)
    a.cache_ops()
    a.attention()
    b.attention()
    torch.cuda.synchronize()
    assert pkv.read_device_errors(a.dev_err) == 0 and pkv.read_device_errors(b.dev_err) == 0
    assert_attention_close(a.out, b.out.to(torch.float64).cpu().numpy(), "beam: shared prefix vs plain decode")
