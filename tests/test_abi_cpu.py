"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point the header declares, and its host-side logic (sizes, layout, argument
validation) behaves as documented.  No call here reaches a kernel launch."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_168_gb300 import _lib, build as build_mod
from paged_kv_cache_168_gb300._lib import CacheDesc
from paged_helpers import to_bits

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTED) == names


def test_cache_bytes(lib):
    d = CacheDesc(num_blocks=8192 // 16, block_size=16, num_kv_heads=40, head_size=128)
    # one LLaMA-13B layer for an 8192-token request: 2 x 8192 x 40 x 128 x 2 bytes
    assert _lib.cache_bytes(d) == 2 * 8192 * 40 * 128 * 2
    assert _lib.cache_bytes(CacheDesc(10, 16, 2, 96)) == 0          # unsupported head size
    assert _lib.cache_bytes(CacheDesc(10, 1, 2, 128)) == 10 * 2 * 2 * 128 * 2   # token-granular blocks
    assert _lib.cache_bytes(CacheDesc(10, 3, 2, 128)) == 0          # block size must be a power of two <= 32
    assert _lib.cache_bytes(CacheDesc(0, 16, 2, 128)) == 0


@pytest.mark.parametrize("bs,D,dtype", [(1, 128, torch.float16), (4, 64, torch.bfloat16), (8, 64, torch.float16),
                                        (16, 128, torch.bfloat16), (32, 128, torch.float16)])
def test_library_layout_agrees_with_oracle_layout(lib, bs, D, dtype):
    d = CacheDesc(3, bs, 2, D, dtype)
    g = oracle.Geom(3, bs, 2, D)
    for b in range(3):
        for h in range(2):
            for part in range(2):
                for t in range(bs):
                    for dim in range(0, D, 3):
                        assert _lib.cache_element_offset(d, b, h, part, t, dim) == \
                            oracle.cache_offset(g, b, h, part, t, dim)
    assert _lib.cache_element_offset(d, 3, 0, 0, 0, 0) == -1
    assert _lib.cache_element_offset(d, 0, 0, 2, 0, 0) == -1


def test_default_partition_size(lib):
    def ps(num_seqs, num_kv_heads, max_ctx, P=0, bs=16, D=128, kv_int8=False):
        return _lib.decode_partition_size(CacheDesc(100, bs, num_kv_heads, D, kv_int8=kv_int8), num_seqs, max_ctx, P)
    assert ps(8, 8, 131072, P=256) == 256                 # an explicit size is kept
    # tensor-core shapes: the longest partition that still gives >= 912
    # (sequence, kv head, partition) items
    assert ps(64, 32, 4096) == 4096                       # 2048 pairs: one partition each
    assert ps(128, 8, 2304) == 4096                       # 1024 pairs
    assert ps(256, 8, 8192) == 4096                       # capped at 4096 up to 32768 tokens
    assert ps(8, 8, 131072) == 8192                       # 64 pairs x 16 partitions
    assert ps(8, 8, 120000) == 8192                       # 64 x 15 = 960
    assert ps(8, 8, 16384) == 1024                        # 64 x 16 = 1024; 2048 gives 512
    assert ps(8, 8, 32768) == 2048                        # not long: the cap stays 4096
    assert ps(1, 8, 4096) == 512                          # too few items at any size: the shortest
    assert ps(0, 8, 4096) == 512 and ps(64, 8, 0) == 512
    assert ps(256, 8, 8192, bs=1, kv_int8=True) == 4096   # 8-bit caches: tensor cores at any block size
    assert ps(2000, 8, 8192, kv_int8=True) == 512         # beyond 1024 sequences: CUDA-core kernel
    # CUDA-core shapes keep 512 (1024 past 32768 tokens)
    assert ps(64, 32, 4096, bs=1) == 512 and ps(64, 32, 4096, D=64) == 512
    assert ps(8, 8, 131072, bs=4) == 1024
    assert _lib.load().pa_decode_partition_size(None, 64, 4096, 0) == 512


def test_workspace_sizing(lib):
    def wb(S, Hq, Hkv, D, max_ctx, P=0, bs=16):
        return _lib.decode_workspace_bytes(CacheDesc(100, bs, Hkv, D), S, Hq, max_ctx, P)
    assert wb(64, 32, 32, 128, 512, 512) == 0             # one partition: no workspace
    assert wb(64, 32, 32, 128, 4096) == 0                  # the default is one 4096-token partition here
    assert wb(64, 32, 32, 128, 4096, bs=1) == 64 * 32 * 8 * 130 * 4   # CUDA-core kernel: 512
    assert wb(64, 32, 32, 128, 4096, 512) == 64 * 32 * 8 * 130 * 4
    assert wb(8, 64, 8, 128, 131072, 1024) == 8 * 64 * 128 * 130 * 4
    assert wb(8, 64, 8, 128, 131072) == 8 * 64 * 16 * 130 * 4
    assert wb(8, 64, 8, 64, 16384) == 8 * 64 * 32 * 66 * 4
    assert _lib.load().pa_decode_workspace_bytes(None, 8, 64, 16384, 512) == 0
    # sizes that do not fit saturate (a wrapped, small size would pass as enough)
    huge = _lib.decode_workspace_bytes(CacheDesc(100, 16, 65535, 128), 65535, 65535 * 16, 2**31 - 1, 128)
    assert huge == 2**64 - 1


def test_status_strings(lib):
    assert _lib.status_string(0) == "ok"
    assert "workspace" in _lib.status_string(4)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _desc(**kw):
    base = dict(num_blocks=16, block_size=16, num_kv_heads=2, head_size=128, dtype=torch.float16)
    base.update(kw)
    return CacheDesc(**base).c()


def _copy(lib, pairs, desc=None):
    arr = np.ascontiguousarray(np.asarray(pairs, np.int64).reshape(-1, 2))
    return lib.pa_copy_blocks(ctypes.c_void_p(FAKE), ctypes.byref(desc or _desc()),
                              arr.ctypes.data_as(ctypes.c_void_p), arr.shape[0], None)


def test_copy_blocks_rejects_bad_pair_lists(lib):
    assert _copy(lib, [[0, 1], [2, 1]]) == _lib.PA_ERR_INVALID_ARG       # repeated dst
    assert b"repeated" in lib.pa_last_error_message()
    assert _copy(lib, [[0, 1], [1, 2]]) == _lib.PA_ERR_INVALID_ARG       # dst is also a src
    assert _copy(lib, [[0, 16]]) == _lib.PA_ERR_INVALID_ARG              # out of range
    assert _copy(lib, [[-1, 3]]) == _lib.PA_ERR_INVALID_ARG
    assert _copy(lib, [[0, 1]], _desc(head_size=96)) == _lib.PA_ERR_UNSUPPORTED
    assert _copy(lib, [[0, 1]], _desc(block_size=12)) == _lib.PA_ERR_UNSUPPORTED
    assert _copy(lib, np.zeros((0, 2))) == _lib.PA_OK                     # nothing to do


def _decode(lib, desc=None, S=2, Hq=4, max_ctx=100, P=0, ws=0, q=FAKE, scale=0.1, bt_stride=8):
    return lib.pa_decode(ctypes.c_void_p(FAKE), ctypes.c_void_p(q), Hq * 128, ctypes.c_void_p(FAKE),
                         ctypes.byref(desc or _desc()), 0, ctypes.c_void_p(FAKE), bt_stride,
                         ctypes.c_void_p(FAKE), S, Hq, max_ctx, scale, P, None, ws, None, None)


def test_decode_rejects_bad_arguments(lib):
    assert _decode(lib, Hq=3) == _lib.PA_ERR_INVALID_ARG                  # not a multiple of Hkv
    assert _decode(lib, Hq=6) == _lib.PA_ERR_UNSUPPORTED                  # group of 3
    assert _decode(lib, desc=_desc(head_size=80)) == _lib.PA_ERR_UNSUPPORTED
    assert _decode(lib, max_ctx=4096) == _lib.PA_ERR_WORKSPACE_TOO_SMALL
    assert _decode(lib, P=100) == _lib.PA_ERR_INVALID_ARG                 # not a multiple of 128
    assert _decode(lib, q=FAKE + 8) == _lib.PA_ERR_INVALID_ARG            # misaligned q
    assert _decode(lib, scale=0.0) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, scale=float("nan")) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, bt_stride=0) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, S=70000) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, S=0) == _lib.PA_OK                                 # nothing to do


def _decode_static(lib, desc=None, S=2, Hq=4, max_ctx=100, P=0, scale=0.1):
    return lib.pa_decode_static_workspace(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), Hq * 128,
                                          ctypes.c_void_p(FAKE), ctypes.byref(desc or _desc()), 0,
                                          ctypes.c_void_p(FAKE), 8, ctypes.c_void_p(FAKE), S, Hq, max_ctx, scale, P,
                                          None, None)


def test_static_workspace_checks_arguments_before_its_size(lib):
    # a bad argument is reported as such, even where the shapes would also be
    # too large for the library's fixed workspace
    assert _decode_static(lib, P=100) == _lib.PA_ERR_INVALID_ARG
    assert _decode_static(lib, S=4096, Hq=64, desc=_desc(num_kv_heads=8), max_ctx=8192, P=64) == _lib.PA_ERR_INVALID_ARG
    assert b"partition_size" in lib.pa_last_error_message()
    assert _decode_static(lib, Hq=6) == _lib.PA_ERR_UNSUPPORTED
    assert _decode_static(lib, scale=0.0) == _lib.PA_ERR_INVALID_ARG
    # valid arguments, too large a workspace: refused before any launch
    assert _decode_static(lib, S=4096, Hq=64, desc=_desc(num_kv_heads=8), max_ctx=8192, P=128) == \
        _lib.PA_ERR_WORKSPACE_TOO_SMALL
    assert b"PA_STATIC_WORKSPACE_BYTES" in lib.pa_last_error_message()
    assert _decode_static(lib, S=0) == _lib.PA_OK


def test_static_workspace_size_matches_the_header():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    m = re.search(r"#define\s+PA_STATIC_WORKSPACE_BYTES\s+\(([0-9u\s*]+)\)", src)
    assert m, "PA_STATIC_WORKSPACE_BYTES not found in pagedkv.h"
    value = 1
    for f in m.group(1).split("*"):
        value *= int(f.strip().rstrip("u"))
    assert value == _lib.STATIC_WORKSPACE_BYTES


def test_shared_prefix_sizes_and_checks(lib):
    d = CacheDesc(100, 16, 8, 128, torch.bfloat16)
    # beam-shaped: 32 groups x 4 beams, 32/8 heads, contexts up to 2305 tokens: the
    # prefixes are the long items, 32 x 8 x ceil(2305 / 4096) = 256 >= 1.5 x 152
    assert _lib.decode_shared_prefix_partition_size(d, 128, 32, 32, 2305) == 4096
    # 8 groups: 8 x 8 x ceil(2305 / 1024) = 192 < 228 at 1024; 320 at 512
    assert _lib.decode_shared_prefix_partition_size(d, 128, 32, 8, 2305) == 512
    assert _lib.decode_shared_prefix_partition_size(d, 128, 32, 32, 2305, 1024) == 1024
    assert _lib.decode_shared_prefix_partition_size(d, 128, 32, 0, 2305) == _lib.decode_partition_size(d, 128, 2305)
    # workspace: (ceil(ctx / P) + 1) partitions per row, plus three ints per sequence
    want = 128 * 32 * (1 + 1) * 130 * 4 + 3 * 128 * 4
    assert _lib.decode_shared_prefix_workspace_bytes(d, 128, 32, 32, 2305) == -(-want // 16) * 16
    # shapes the dedicated kernel does not serve size as pa_decode does
    d64 = CacheDesc(100, 16, 8, 64, torch.bfloat16)
    assert _lib.decode_shared_prefix_workspace_bytes(d64, 128, 32, 32, 2305, 512) == \
        _lib.decode_workspace_bytes(d64, 128, 32, 2305, 512)
    assert _lib.decode_shared_prefix_workspace_bytes(d, 161, 32, 32, 2305, 512) == \
        _lib.decode_workspace_bytes(d, 161, 32, 2305, 512)                # above 160 sequences
    assert _lib.decode_shared_prefix_workspace_bytes(d, 160, 32, 32, 2305, 512) != \
        _lib.decode_workspace_bytes(d, 160, 32, 2305, 512)

    def call(num_groups=2, gs=FAKE, pl=FAKE, ws=1 << 30, P=256):
        return lib.pa_decode_shared_prefix(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 4 * 128,
                                           ctypes.c_void_p(FAKE), ctypes.byref(_desc()), 0, ctypes.c_void_p(FAKE), 8,
                                           ctypes.c_void_p(FAKE), 4, 4, 100, 0.1, ctypes.c_void_p(gs),
                                           ctypes.c_void_p(pl), num_groups, P, ctypes.c_void_p(FAKE), ws, None, None)
    assert call(num_groups=5) == _lib.PA_ERR_INVALID_ARG                   # more groups than sequences
    assert call(num_groups=-1) == _lib.PA_ERR_INVALID_ARG
    assert call(gs=0) == _lib.PA_ERR_INVALID_ARG                            # NULL group starts
    assert call(pl=FAKE + 2) == _lib.PA_ERR_INVALID_ARG                     # misaligned prefix lengths
    assert call(P=100) == _lib.PA_ERR_INVALID_ARG                           # bad partition size first
    assert call(ws=16) == _lib.PA_ERR_WORKSPACE_TOO_SMALL


def test_reshape_rejects_bad_arguments(lib):
    call = lambda stride, n=4, key=FAKE, layer=0: lib.pa_reshape_and_cache(
        ctypes.c_void_p(FAKE), ctypes.byref(_desc()), layer, ctypes.c_void_p(key), stride,
        ctypes.c_void_p(FAKE), 256, ctypes.c_void_p(FAKE), n, None, None)
    assert call(255) == _lib.PA_ERR_INVALID_ARG          # stride below one token row
    assert call(260) == _lib.PA_ERR_INVALID_ARG          # not a multiple of 8
    assert call(256, key=FAKE + 2) == _lib.PA_ERR_INVALID_ARG
    assert call(256, layer=1) == _lib.PA_ERR_INVALID_ARG
    assert call(256, n=-1) == _lib.PA_ERR_INVALID_ARG
    assert call(256, n=0) == _lib.PA_OK


def test_swap_rejects_mismatched_pools(lib):
    arr = np.array([[0, 1]], np.int64)
    st = lib.pa_swap_blocks(ctypes.c_void_p(FAKE), ctypes.byref(_desc()), ctypes.c_void_p(FAKE),
                            ctypes.byref(_desc(num_kv_heads=4)), 0, arr.ctypes.data_as(ctypes.c_void_p), 1, None)
    assert st == _lib.PA_ERR_INVALID_ARG
    st = lib.pa_swap_blocks(ctypes.c_void_p(FAKE), ctypes.byref(_desc()), ctypes.c_void_p(FAKE),
                            ctypes.byref(_desc()), 2, arr.ctypes.data_as(ctypes.c_void_p), 1, None)
    assert st == _lib.PA_ERR_INVALID_ARG


def test_read_device_errors_rejects_null(lib):
    assert lib.pa_read_device_errors(None, None, 0, None) == _lib.PA_ERR_INVALID_ARG


# ---------------------------------------------------------------- 8-bit cache (host side)

def test_int8_cache_bytes(lib):
    # per block and kv head: K and V codes (2 x bs x 128 bytes) + two fp32 scale areas padded to 16 bytes
    assert _lib.cache_bytes(CacheDesc(10, 16, 2, 128, kv_int8=True)) == 10 * 2 * (2 * 16 * 128 + 2 * 64)
    assert _lib.cache_bytes(CacheDesc(10, 1, 2, 128, kv_int8=True)) == 10 * 2 * (2 * 128 + 2 * 16)
    assert _lib.cache_bytes(CacheDesc(10, 2, 3, 128, kv_int8=True)) == 10 * 3 * (2 * 2 * 128 + 2 * 16)
    assert _lib.cache_bytes(CacheDesc(10, 16, 2, 64, kv_int8=True)) == 0     # 8-bit needs head_size 128
    for bs in (1, 2, 4, 8, 16, 32):
        g = oracle.Geom(5, bs, 3, 128, "bf16")
        assert _lib.cache_bytes(CacheDesc(5, bs, 3, 128, torch.bfloat16, kv_int8=True)) == 5 * oracle.i8_block_bytes(g)


@pytest.mark.parametrize("bs", [1, 2, 8, 16, 32])
def test_int8_offsets_point_at_what_the_oracle_writes(lib, bs):
    # A vector with one non-zero element d quantises to code 127 at d, zeros
    # elsewhere, and scale |x_d| / 127: the library's offsets must find them.
    rng = np.random.default_rng(bs)
    nb, hkv = 3, 2
    g = oracle.Geom(nb, bs, hkv, 128, "f16")
    d = CacheDesc(nb, bs, hkv, 128, torch.float16, kv_int8=True)
    for _ in range(12):
        slot, h, part, dim = int(rng.integers(nb * bs)), int(rng.integers(hkv)), int(rng.integers(2)), \
            int(rng.integers(128))
        pool = np.zeros(nb * oracle.i8_block_bytes(g), np.uint8)
        kv = np.zeros((2, 1, hkv, 128))
        kv[part, 0, h, dim] = 2.5
        assert oracle.reshape_and_cache_i8(pool, g, to_bits(kv[0], "f16"), to_bits(kv[1], "f16"),
                                           np.array([slot])) == 0
        b, t = slot // bs, slot % bs
        off = _lib.cache_element_offset(d, b, h, part, t, dim)
        assert pool.view(np.int8)[off] == 127
        assert int(np.count_nonzero(pool.view(np.int8) == 127)) == 1
        so = _lib.cache_scale_offset(d, b, h, part, t)
        assert so % 4 == 0 and pool[so:so + 4].view(np.float32)[0] == np.float32(2.5) / np.float32(127)
    assert _lib.cache_scale_offset(CacheDesc(nb, bs, hkv, 128), 0, 0, 0, 0) == -1    # 16-bit cache
    assert _lib.cache_scale_offset(d, nb, 0, 0, 0) == -1


def test_int8_decode_limits(lib):
    d8 = _desc(dtype=torch.bfloat16, kv_int8=True)
    assert _decode(lib, desc=d8, Hq=32) == _lib.PA_ERR_UNSUPPORTED        # group 16
    assert _decode(lib, desc=_desc(kv_int8=True, head_size=64)) == _lib.PA_ERR_UNSUPPORTED
    st = lib.pa_decode_window(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 4 * 128, ctypes.c_void_p(FAKE),
                              ctypes.byref(d8), 0, ctypes.c_void_p(FAKE), 8, ctypes.c_void_p(FAKE), 2, 4, 100,
                              0.1, -1, 0, 0, None, 0, None, None)
    assert st == _lib.PA_ERR_INVALID_ARG                                    # windows over 8-bit caches are
    #                                                                         validated like 16-bit ones
    # an 8-bit pool and a 16-bit pool are different geometries for swapping
    arr = np.array([[0, 1]], np.int64)
    st = lib.pa_swap_blocks(ctypes.c_void_p(FAKE), ctypes.byref(_desc()), ctypes.c_void_p(FAKE),
                            ctypes.byref(_desc(kv_int8=True)), 0, arr.ctypes.data_as(ctypes.c_void_p), 1, None)
    assert st == _lib.PA_ERR_INVALID_ARG


def _prefill(lib, desc=None, S=2, Hq=4, max_q=100, q=FAKE, scale=0.1, q_stride=4 * 128):
    return lib.pa_prefill(ctypes.c_void_p(FAKE), ctypes.c_void_p(q), q_stride, ctypes.c_void_p(FAKE),
                          ctypes.byref(desc or _desc()), 0, ctypes.c_void_p(FAKE), 8, ctypes.c_void_p(FAKE),
                          ctypes.c_void_p(FAKE), S, Hq, max_q, scale, None, None)


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, Hq=3) == _lib.PA_ERR_INVALID_ARG                 # not a multiple of Hkv
    assert _prefill(lib, Hq=64) == _lib.PA_ERR_UNSUPPORTED                # group 32
    assert _prefill(lib, desc=_desc(block_size=4)) == _lib.PA_ERR_UNSUPPORTED
    assert _prefill(lib, desc=_desc(kv_int8=True)) == _lib.PA_ERR_UNSUPPORTED
    assert _prefill(lib, q=FAKE + 8) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, q_stride=4 * 128 - 8) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, scale=-1.0) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, max_q=-1) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, S=0) == _lib.PA_OK and _prefill(lib, max_q=0) == _lib.PA_OK    # nothing to do
