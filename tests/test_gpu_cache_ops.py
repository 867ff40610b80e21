"""GPU parity of the cache operations: every result is compared bit for bit with
the fp64 CPU oracle on the WHOLE pool (untouched regions must stay unchanged)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import desc_of, dev_to_u16, ensure_built, u16_to_dev
from paged_helpers import NAN_BITS, to_bits

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


def random_pool(rng, geom):
    n = geom.layer_elems * geom.num_layers
    return rng.integers(0, 1 << 16, size=n, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("bs,Hkv,D,dtype", [(16, 4, 64, "f16"), (8, 1, 128, "bf16"), (32, 8, 128, "bf16"),
                                            (16, 32, 128, "f16")])
def test_reshape_and_cache_bit_exact(bs, Hkv, D, dtype):
    rng = np.random.default_rng(100)
    NB, N = 37, 50
    g = oracle.Geom(NB, bs, Hkv, D, dtype)
    pool = random_pool(rng, g)
    key = to_bits(rng.standard_normal((N, Hkv, D)), dtype)
    val = to_bits(rng.standard_normal((N, Hkv, D)), dtype)
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[[3, 17, 40]] = -1                                    # padding tokens are skipped
    dpool = u16_to_dev(pool, dtype)
    dkey, dval = u16_to_dev(key, dtype), u16_to_dev(val, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(dpool, desc_of(NB, bs, Hkv, D, dtype), dkey, dval,
                          torch.from_numpy(slots).cuda(), dev_err=err)
    assert oracle.reshape_and_cache(pool, g, key, val, slots) == 0
    assert np.array_equal(dev_to_u16(dpool), pool)
    assert pkv.read_device_errors(err) == 0


def test_reshape_strided_key_and_layer():
    # key/value rows with a token stride larger than Hkv*D (e.g. slices of a fused QKV tensor), layer 1 of 2
    rng = np.random.default_rng(101)
    NB, bs, Hkv, D, N = 9, 16, 2, 64, 7
    g = oracle.Geom(NB, bs, Hkv, D, "f16", num_layers=2)
    pool = random_pool(rng, g)
    qkv = to_bits(rng.standard_normal((N, 3 * Hkv * D)), "f16")
    dqkv = u16_to_dev(qkv, "f16")
    key = dqkv[:, Hkv * D:2 * Hkv * D].view(N, Hkv, D)
    val = dqkv[:, 2 * Hkv * D:].view(N, Hkv, D)
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    dpool = u16_to_dev(pool, "f16")
    pkv.reshape_and_cache(dpool, desc_of(NB, bs, Hkv, D, "f16", num_layers=2), key, val,
                          torch.from_numpy(slots).cuda(), layer=1)
    layer1 = pool[g.layer_elems:]
    kb = np.ascontiguousarray(qkv[:, Hkv * D:2 * Hkv * D]).reshape(N, Hkv, D)
    vb = np.ascontiguousarray(qkv[:, 2 * Hkv * D:]).reshape(N, Hkv, D)
    oracle.reshape_and_cache(layer1, g, kb, vb, slots)
    assert np.array_equal(dev_to_u16(dpool), pool)


def test_reshape_bad_slot_sets_error_and_writes_nothing_for_it():
    rng = np.random.default_rng(102)
    NB, bs, Hkv, D = 4, 16, 2, 128
    g = oracle.Geom(NB, bs, Hkv, D, "bf16")
    pool = random_pool(rng, g)
    key = to_bits(rng.standard_normal((3, Hkv, D)), "bf16")
    slots = np.array([5, NB * bs, -7], np.int64)
    dpool = u16_to_dev(pool, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(dpool, desc_of(NB, bs, Hkv, D, "bf16"), u16_to_dev(key, "bf16"),
                          u16_to_dev(key, "bf16"), torch.from_numpy(slots).cuda(), dev_err=err)
    assert pkv.read_device_errors(err) == pkv.DEVERR_SLOT
    assert oracle.reshape_and_cache(pool, g, key, key, slots) == oracle.ERR_SLOT
    assert np.array_equal(dev_to_u16(dpool), pool)


@pytest.mark.parametrize("layers", [1, 3])
def test_copy_blocks_bit_exact(layers):
    rng = np.random.default_rng(103)
    NB, bs, Hkv, D = 40, 16, 8, 128
    g = oracle.Geom(NB, bs, Hkv, D, "bf16", num_layers=layers)
    pool = random_pool(rng, g)
    ids = rng.permutation(NB)
    pairs = np.stack([ids[:12], ids[12:24]], axis=1)
    dpool = u16_to_dev(pool, "bf16")
    pkv.copy_blocks(dpool, desc_of(NB, bs, Hkv, D, "bf16", num_layers=layers), pairs)
    assert oracle.copy_blocks(pool, g, pairs) == 0
    assert np.array_equal(dev_to_u16(dpool), pool)


def test_copy_blocks_many_pairs_and_padded_layer_stride():
    # more pairs than one launch carries, and layers placed with a gap between them
    rng = np.random.default_rng(104)
    NB, bs, Hkv, D = 3000, 8, 1, 64
    geom = oracle.Geom(NB, bs, Hkv, D, "f16", num_layers=2)
    stride_elems = geom.layer_elems + 64
    g = oracle.Geom(NB, bs, Hkv, D, "f16", num_layers=2, layer_stride=stride_elems)
    pool = rng.integers(0, 1 << 16, size=2 * stride_elems, dtype=np.uint32).astype(np.uint16)
    ids = rng.permutation(NB)
    pairs = np.stack([ids[:1500], ids[1500:]], axis=1)
    dpool = u16_to_dev(pool, "f16")
    pkv.copy_blocks(dpool, desc_of(NB, bs, Hkv, D, "f16", 2, stride_elems * 2), pairs)
    oracle.copy_blocks(pool, g, pairs)
    assert np.array_equal(dev_to_u16(dpool), pool)


def test_swap_out_and_in_bit_exact_round_trip():
    rng = np.random.default_rng(105)
    NB, NH, bs, Hkv, D, L = 64, 16, 16, 8, 128, 2
    gd = oracle.Geom(NB, bs, Hkv, D, "bf16", num_layers=L)
    gh = oracle.Geom(NH, bs, Hkv, D, "bf16", num_layers=L)
    dev = random_pool(rng, gd)
    host_np = np.zeros(gh.layer_elems * L, dtype=np.uint16)
    ddev = u16_to_dev(dev, "bf16")
    dhost = torch.zeros(gh.layer_elems * L, dtype=torch.bfloat16).pin_memory()
    dd, dh = desc_of(NB, bs, Hkv, D, "bf16", L), desc_of(NH, bs, Hkv, D, "bf16", L)
    out_pairs = np.stack([rng.choice(NB, 10, replace=False), rng.choice(NH, 10, replace=False)], axis=1)
    pkv.swap_blocks(dhost, dh, ddev, dd, 0, out_pairs)
    torch.cuda.synchronize()
    oracle.swap_blocks(host_np, gh, dev, gd, out_pairs)
    assert np.array_equal(dhost.view(torch.int16).numpy().view(np.uint16), host_np)
    # clobber the swapped-out device blocks, swap them back in
    saved = dev.copy()
    ddev.view(L, NB, -1)[:, torch.from_numpy(out_pairs[:, 0]).cuda()] = 0
    in_pairs = out_pairs[:, ::-1].copy()
    pkv.swap_blocks(ddev, dd, dhost, dh, 1, in_pairs)
    assert np.array_equal(dev_to_u16(ddev), saved)


def test_swap_requires_pinned_host_memory():
    dd = desc_of(4, 16, 1, 64, "f16")
    dev = torch.zeros(4 * 2 * 16 * 64, dtype=torch.float16, device="cuda")
    host = torch.zeros_like(dev, device="cpu")              # pageable
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.swap_blocks(host, dd, dev, dd, 0, [[0, 1]])
    assert e.value.status == pkv.PA_ERR_INVALID_ARG


def test_cow_worked_example_on_gpu():
    ex = json.load(open(os.path.join(GOLDEN, "cow_worked_example.json")))
    bs = ex["block_size"]
    NB, Hkv, D = 6, 2, 64
    g = oracle.Geom(NB, bs, Hkv, D, "f16")
    rng = np.random.default_rng(106)
    n_prompt = ex["prompt_tokens"]
    pk = to_bits(rng.standard_normal((n_prompt, Hkv, D)), "f16")
    pv = to_bits(rng.standard_normal((n_prompt, Hkv, D)), "f16")
    pool = np.full(g.layer_elems, NAN_BITS["f16"], dtype=np.uint16)
    t = np.arange(n_prompt)
    oracle.reshape_and_cache(pool, g, pk, pv, np.array([0, 1])[t // bs] * bs + t % bs)
    dpool = u16_to_dev(pool, "f16")
    desc = desc_of(NB, bs, Hkv, D, "f16")
    off = ex["expected_new_token_position"]["block_offset"]
    for seq in ex["write_order"]:
        pairs = ex["expected_copy_pairs"][seq]
        last = ex["expected_tables"][seq][-1]
        if pairs:
            pkv.copy_blocks(dpool, desc, pairs)
            oracle.copy_blocks(pool, g, np.array(pairs))
        nk = to_bits(rng.standard_normal((1, Hkv, D)), "f16")
        nv = to_bits(rng.standard_normal((1, Hkv, D)), "f16")
        slot = np.array([last * bs + off], np.int64)
        pkv.reshape_and_cache(dpool, desc, u16_to_dev(nk, "f16"), u16_to_dev(nv, "f16"),
                              torch.from_numpy(slot).cuda())
        oracle.reshape_and_cache(pool, g, nk, nv, slot)
        assert np.array_equal(dev_to_u16(dpool), pool), seq
