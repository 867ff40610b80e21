"""fp64 CPU oracle for paged KV-cache decode -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and the oracle shares no code with it.

The arithmetic lives in ``pagedkv_oracle.c`` (plain C, double precision,
OpenMP over (sequence, head) pairs); this module compiles it with gcc and wraps
it with ctypes.  All 16-bit cache / query data are passed as ``numpy.uint16``
arrays holding raw fp16 or bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

ERR_BLOCK_ID = 1
ERR_SLOT = 2
ERR_CONTEXT = 4

DTYPE_CODES = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Geom(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("layer_stride", ctypes.c_int64),
    ]


@dataclass
class Geom:
    """Cache geometry: num_blocks blocks of block_size token slots, per layer."""
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_size: int
    dtype: str = "f16"
    num_layers: int = 1
    layer_stride: int = 0   # elements between layers; 0 means packed layers

    @property
    def block_elems(self) -> int:
        return self.num_kv_heads * 2 * self.block_size * self.head_size

    @property
    def layer_elems(self) -> int:
        return self.num_blocks * self.block_elems

    def c(self) -> _Geom:
        return _Geom(self.num_blocks, self.block_size, self.num_kv_heads, self.head_size,
                     DTYPE_CODES[self.dtype], self.num_layers,
                     self.layer_stride or self.layer_elems)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    G = ctypes.POINTER(_Geom)
    lib.oracle_elem_to_double.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.oracle_elem_to_double.restype = dbl
    lib.oracle_cache_offset.argtypes = [G, i64, i64, ctypes.c_int, i64, i64]
    lib.oracle_cache_offset.restype = i64
    lib.oracle_reshape_and_cache.argtypes = [P, G, P, i64, P, i64, P, i32]
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    lib.oracle_gather.argtypes = [P, G, P, i32, i32, P, P]
    lib.oracle_gather.restype = ctypes.c_int
    lib.oracle_contiguous_attention.argtypes = [P, P, P, i32, i32, dbl, P]
    lib.oracle_contiguous_attention.restype = None
    lib.oracle_decode.argtypes = [P, P, i64, P, G, P, i32, P, i32, i32, i32, dbl, P, i32, i32]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_decode_window.argtypes = [P, P, i64, P, G, P, i32, P, i32, i32, i32, dbl, i32, i32, P, i32, i32]
    lib.oracle_decode_window.restype = ctypes.c_int
    lib.oracle_window_start.argtypes = [i32, i32, i32, i32]
    lib.oracle_window_start.restype = i32
    lib.oracle_partition_stats.argtypes = [P, P, G, P, i32, i32, dbl, i32, P, P, P]
    lib.oracle_partition_stats.restype = ctypes.c_int
    lib.oracle_merge_partitions.argtypes = [P, P, P, i32, i32, P]
    lib.oracle_merge_partitions.restype = None
    lib.oracle_copy_blocks.argtypes = [P, G, P, i32]
    lib.oracle_copy_blocks.restype = ctypes.c_int
    lib.oracle_swap_blocks.argtypes = [P, G, P, G, P, i32]
    lib.oracle_swap_blocks.restype = ctypes.c_int
    lib.oracle_i8_chunk_bytes.argtypes = [G]
    lib.oracle_i8_chunk_bytes.restype = i64
    lib.oracle_reshape_and_cache_i8.argtypes = [P, G, P, i64, P, i64, P, i32]
    lib.oracle_reshape_and_cache_i8.restype = ctypes.c_int
    lib.oracle_decode_i8.argtypes = [P, P, i64, P, G, P, i32, P, i32, i32, i32, dbl, i32]
    lib.oracle_decode_i8.restype = ctypes.c_int
    lib.oracle_decode_i8_window.argtypes = [P, P, i64, P, G, P, i32, P, i32, i32, i32, dbl, i32, i32, i32]
    lib.oracle_decode_i8_window.restype = ctypes.c_int
    lib.oracle_copy_blocks_bytes.argtypes = [P, i64, i32, i32, i64, P, i32]
    lib.oracle_copy_blocks_bytes.restype = ctypes.c_int
    lib.oracle_prefill.argtypes = [P, P, i64, P, G, P, i32, P, P, i32, i32, dbl, i32]
    lib.oracle_prefill.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a: np.ndarray) -> np.ndarray:
    assert a.dtype == np.uint16, "16-bit data are passed as raw uint16 bits"
    return np.ascontiguousarray(a)


def max_threads() -> int:
    return _load().oracle_max_threads()


def elem_to_double(bits: int, dtype: str) -> float:
    return _load().oracle_elem_to_double(bits, DTYPE_CODES[dtype])


def cache_offset(geom: Geom, block: int, head: int, part: int, t: int, d: int) -> int:
    return _load().oracle_cache_offset(ctypes.byref(geom.c()), block, head, part, t, d)


def reshape_and_cache(layer: np.ndarray, geom: Geom, key: np.ndarray, value: np.ndarray,
                      slot_mapping: np.ndarray) -> int:
    """Write new tokens' K/V (key/value: uint16 [N, Hkv, D]) into ``layer`` in place."""
    key, value = _u16(key), _u16(value)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    n = sm.shape[0]
    row = geom.num_kv_heads * geom.head_size
    return _load().oracle_reshape_and_cache(_ptr(layer), ctypes.byref(geom.c()), _ptr(key), row,
                                            _ptr(value), row, _ptr(sm), n)


def gather(layer: np.ndarray, geom: Geom, table_row: np.ndarray, ctx: int, kv_head: int):
    """Contiguous K, V (float64 [ctx, D]) of one sequence and kv head."""
    tr = np.ascontiguousarray(table_row, dtype=np.int32)
    K = np.zeros((max(ctx, 0), geom.head_size))
    V = np.zeros((max(ctx, 0), geom.head_size))
    err = _load().oracle_gather(_ptr(layer), ctypes.byref(geom.c()), _ptr(tr), ctx, kv_head,
                                _ptr(K), _ptr(V))
    if err:
        raise IndexError("block id out of range in block table")
    return K, V


def contiguous_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.zeros(q.shape[0])
    _load().oracle_contiguous_attention(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.shape[0],
                                        scale, _ptr(out))
    return out


def decode(q: np.ndarray, layer: np.ndarray, geom: Geom, block_tables: np.ndarray,
           context_lens: np.ndarray, scale: float, max_context_len: int | None = None,
           sel: np.ndarray | None = None, nthreads: int = 0, window: int = 0, ring: int = 0):
    """Paged decode attention in fp64.

    q: uint16 [S, Hq, D].  Returns (out float64 [S, Hq, D] or [len(sel), D], error bits).
    sel: optional int32 [n, 2] list of (sequence, query head) pairs to compute.
    window > 0 attends only positions >= ctx - window; ring > 0 reads the table
    row as a ring of that many blocks (logical block j at entry j % ring).
    """
    q = _u16(q)
    S, Hq, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    if max_context_len is None:
        max_context_len = int(cl.max()) if cl.size else 0
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        out = np.zeros((sel.shape[0], D))
        nsel = sel.shape[0]
    else:
        out = np.zeros((S, Hq, D))
        nsel = 0
    err = _load().oracle_decode_window(_ptr(out), _ptr(q), Hq * D, _ptr(layer), ctypes.byref(geom.c()),
                                       _ptr(bt), bt.shape[1], _ptr(cl), S, Hq, max_context_len, scale, window,
                                       ring, _ptr(sel), nsel, nthreads)
    return out, err


def window_start(ctx: int, block_size: int, window: int, ring: int) -> int:
    """First position a (window, ring) decode attends for context length ctx."""
    return _load().oracle_window_start(ctx, block_size, window, ring)


def partition_stats(q_row: np.ndarray, layer: np.ndarray, geom: Geom, table_row: np.ndarray,
                    ctx: int, kv_head: int, scale: float, P: int):
    """Per-partition (m_p, l_p, o_p) of one (sequence, head) for partitions of P tokens."""
    q_row = _u16(q_row)
    tr = np.ascontiguousarray(table_row, dtype=np.int32)
    n_max = max(1, (ctx + P - 1) // P)
    m, l = np.zeros(n_max), np.zeros(n_max)
    o = np.zeros((n_max, geom.head_size))
    n = _load().oracle_partition_stats(_ptr(q_row), _ptr(layer), ctypes.byref(geom.c()), _ptr(tr),
                                       ctx, kv_head, scale, P, _ptr(m), _ptr(l), _ptr(o))
    if n < 0:
        raise IndexError("block id out of range in block table")
    return m[:n], l[:n], o[:n]


def merge_partitions(m: np.ndarray, l: np.ndarray, o: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    D = o.shape[1] if o.ndim == 2 else 0
    out = np.zeros(D)
    _load().oracle_merge_partitions(_ptr(m), _ptr(l), _ptr(o), m.shape[0], D, _ptr(out))
    return out


def copy_blocks(pool: np.ndarray, geom: Geom, pairs: np.ndarray) -> int:
    """Copy whole blocks in place for every (src, dst) pair, all layers."""
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return _load().oracle_copy_blocks(_ptr(pool), ctypes.byref(geom.c()), _ptr(pr), pr.shape[0])


def swap_blocks(dst: np.ndarray, dst_geom: Geom, src: np.ndarray, src_geom: Geom,
                pairs: np.ndarray) -> int:
    """Copy whole blocks src pool -> dst pool for every (src block, dst block) pair."""
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return _load().oracle_swap_blocks(_ptr(dst), ctypes.byref(dst_geom.c()), _ptr(src),
                                      ctypes.byref(src_geom.c()), _ptr(pr), pr.shape[0])


# ---------------------------------------------------------------- 8-bit KV cache
# Geom.dtype names the 16-bit type of q / new K,V / output ("f16" or "bf16");
# the pool holds int8 codes and fp32 scales (uint8 arrays here).

def prefill(q: np.ndarray, layer: np.ndarray, geom: Geom, block_tables: np.ndarray, context_lens: np.ndarray,
            query_start_loc: np.ndarray, scale: float, nthreads: int = 0):
    """Causal prefill / extend over the paged cache: q uint16 [T, Hq, D] packed by
    query_start_loc (int32 [S + 1]); returns (out [T, Hq, D] fp64, error bits)."""
    q, layer = _u16(q), _u16(layer)
    T, Hq, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    assert qsl.shape[0] == cl.shape[0] + 1
    out = np.zeros((T, Hq, D))
    err = _load().oracle_prefill(_ptr(out), _ptr(q), Hq * D, _ptr(layer), ctypes.byref(geom.c()), _ptr(bt),
                                 bt.shape[1], _ptr(cl), _ptr(qsl), cl.shape[0], Hq, scale, nthreads)
    return out, err


def i8_block_bytes(geom: Geom) -> int:
    """Bytes of one block (all kv heads) of an 8-bit cache."""
    return geom.num_kv_heads * _load().oracle_i8_chunk_bytes(ctypes.byref(geom.c()))


def reshape_and_cache_i8(layer: np.ndarray, geom: Geom, key: np.ndarray, value: np.ndarray,
                         slot_mapping: np.ndarray) -> int:
    """Quantise and write new tokens' K/V (uint16 [N, Hkv, D]) into an 8-bit layer (uint8)."""
    assert layer.dtype == np.uint8 and geom.head_size == 128
    key, value = _u16(key), _u16(value)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    row = geom.num_kv_heads * geom.head_size
    return _load().oracle_reshape_and_cache_i8(_ptr(layer), ctypes.byref(geom.c()), _ptr(key), row, _ptr(value),
                                               row, _ptr(sm), sm.shape[0])


def decode_i8(q: np.ndarray, layer: np.ndarray, geom: Geom, block_tables: np.ndarray, context_lens: np.ndarray,
              scale: float, max_context_len: int | None = None, nthreads: int = 0, window: int = 0, ring: int = 0):
    """Paged decode over an 8-bit cache (values = code * scale), in fp64; window /
    ring as for ``decode`` (attended positions window_start(...) .. ctx - 1, block
    j of a ring table at entry j % ring)."""
    assert layer.dtype == np.uint8 and geom.head_size == 128
    q = _u16(q)
    S, Hq, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    if max_context_len is None:
        max_context_len = int(cl.max()) if cl.size else 0
    out = np.zeros((S, Hq, D))
    err = _load().oracle_decode_i8_window(_ptr(out), _ptr(q), Hq * D, _ptr(layer), ctypes.byref(geom.c()), _ptr(bt),
                                          bt.shape[1], _ptr(cl), S, Hq, max_context_len, scale, window, ring,
                                          nthreads)
    return out, err


def copy_blocks_bytes(pool: np.ndarray, block_bytes: int, num_blocks: int, pairs: np.ndarray, num_layers: int = 1,
                      layer_stride: int = 0) -> int:
    """Whole-block copies for any block encoding (pool as uint8)."""
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return _load().oracle_copy_blocks_bytes(_ptr(pool), block_bytes, num_blocks, num_layers,
                                            layer_stride or block_bytes * num_blocks, _ptr(pr), pr.shape[0])
