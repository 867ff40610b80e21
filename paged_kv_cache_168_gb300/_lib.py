"""Thin ctypes binding over libpagedkv.so (argument marshalling only).

Every entry point of ``include/pagedkv.h`` is exposed under the same name
without the ``pa_`` prefix.  Tensors are torch tensors used only as device (or
pinned host) memory; pointers, sizes and the current CUDA stream are passed to
the C ABI, which does all the work in its CUDA kernels.  There is no fallback:
if the library is not built, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")
_lib = None

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_WORKSPACE_TOO_SMALL, PA_ERR_OUT_OF_BLOCKS = range(6)
PA_ALLOC_OK, PA_ALLOC_LATER, PA_ALLOC_NEVER = range(3)
PA_F16, PA_BF16, PA_INT8_F16, PA_INT8_BF16 = 0, 1, 2, 3
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_CONTEXT, DEVERR_TIMEOUT, DEVERR_PREFIX = 1, 2, 4, 8, 16
DTYPE_CODE = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}

EXPORTED = [
    "pa_cache_bytes", "pa_cache_element_offset", "pa_cache_scale_offset", "pa_reshape_and_cache", "pa_decode_workspace_bytes",
    "pa_decode_partition_size", "pa_decode", "pa_decode_window", "pa_decode_window_span", "pa_prefill",
    "pa_decode_static_workspace", "pa_decode_shared_prefix", "pa_decode_shared_prefix_partition_size",
    "pa_decode_shared_prefix_workspace_bytes", "pa_copy_blocks", "pa_swap_blocks", "pa_read_device_errors",
    "pa_status_string", "pa_last_error_message",
    "pa_bm_create", "pa_bm_destroy", "pa_bm_can_allocate", "pa_bm_allocate", "pa_bm_append_slot", "pa_bm_fork",
    "pa_bm_free", "pa_bm_block_table", "pa_bm_swap_out", "pa_bm_swap_in", "pa_bm_num_free_blocks",
    "pa_bm_ref_count", "pa_bm_can_append_slots", "pa_bm_can_swap_in", "pa_bm_can_swap_out",
]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("layer_stride_bytes", ctypes.c_int64),
    ]


@dataclass
class CacheDesc:
    """Geometry of a cache pool (mirrors pa_cache_desc).  dtype is the 16-bit type
    of q / K / V / out; kv_int8 stores the cache as 8-bit codes with fp32 scales."""
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_size: int
    dtype: torch.dtype = torch.float16
    num_layers: int = 1
    layer_stride_bytes: int = 0
    kv_int8: bool = False

    def c(self) -> _Desc:
        return _Desc(self.num_blocks, self.block_size, self.num_kv_heads, self.head_size,
                     DTYPE_CODE[self.dtype] + (2 if self.kv_int8 else 0), self.num_layers,
                     self.layer_stride_bytes)


def load():
    """Load libpagedkv.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is not built; run paged_kv_cache_168_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(_Desc)
    lib.pa_cache_bytes.argtypes = [D]
    lib.pa_cache_bytes.restype = sz
    lib.pa_cache_element_offset.argtypes = [D, i64, i32, i32, i32, i32]
    lib.pa_cache_element_offset.restype = i64
    lib.pa_cache_scale_offset.argtypes = [D, i64, i32, i32, i32]
    lib.pa_cache_scale_offset.restype = i64
    lib.pa_reshape_and_cache.argtypes = [P, D, i32, P, i64, P, i64, P, i32, P, P]
    lib.pa_reshape_and_cache.restype = ctypes.c_int
    lib.pa_decode_workspace_bytes.argtypes = [D, i32, i32, i32, i32]
    lib.pa_decode_workspace_bytes.restype = sz
    lib.pa_decode_partition_size.argtypes = [D, i32, i32, i32]
    lib.pa_decode_partition_size.restype = i32
    lib.pa_decode.argtypes = [P, P, i64, P, D, i32, P, i32, P, i32, i32, i32, ctypes.c_float, i32, P, sz, P, P]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_decode_window.argtypes = [P, P, i64, P, D, i32, P, i32, P, i32, i32, i32, ctypes.c_float, i32, i32, i32,
                                     P, sz, P, P]
    lib.pa_decode_window.restype = ctypes.c_int
    lib.pa_prefill.argtypes = [P, P, i64, P, D, i32, P, i32, P, P, i32, i32, i32, ctypes.c_float, P, P]
    lib.pa_prefill.restype = ctypes.c_int
    lib.pa_decode_window_span.argtypes = [i32, i32, i32, i32]
    lib.pa_decode_window_span.restype = i32
    lib.pa_decode_static_workspace.argtypes = [P, P, i64, P, D, i32, P, i32, P, i32, i32, i32, ctypes.c_float,
                                               i32, P, P]
    lib.pa_decode_static_workspace.restype = ctypes.c_int
    lib.pa_decode_shared_prefix.argtypes = [P, P, i64, P, D, i32, P, i32, P, i32, i32, i32, ctypes.c_float, P, P,
                                            i32, i32, P, sz, P, P]
    lib.pa_decode_shared_prefix.restype = ctypes.c_int
    lib.pa_decode_shared_prefix_partition_size.argtypes = [D, i32, i32, i32, i32, i32]
    lib.pa_decode_shared_prefix_partition_size.restype = i32
    lib.pa_decode_shared_prefix_workspace_bytes.argtypes = [D, i32, i32, i32, i32, i32]
    lib.pa_decode_shared_prefix_workspace_bytes.restype = sz
    lib.pa_copy_blocks.argtypes = [P, D, P, i32, P]
    lib.pa_copy_blocks.restype = ctypes.c_int
    lib.pa_swap_blocks.argtypes = [P, D, P, D, i32, P, i32, P]
    lib.pa_swap_blocks.restype = ctypes.c_int
    lib.pa_read_device_errors.argtypes = [P, P, i32, P]
    lib.pa_read_device_errors.restype = ctypes.c_int
    B = ctypes.c_void_p
    PI64, PI32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    lib.pa_bm_create.argtypes = [i32, i32, i32, ctypes.c_float, i32, i32, ctypes.POINTER(ctypes.c_void_p)]
    lib.pa_bm_create.restype = ctypes.c_int
    lib.pa_bm_destroy.argtypes = [B]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_can_allocate.argtypes = [B, i32]
    lib.pa_bm_can_allocate.restype = i32
    lib.pa_bm_allocate.argtypes = [B, i64, P, i32]
    lib.pa_bm_allocate.restype = ctypes.c_int
    lib.pa_bm_append_slot.argtypes = [B, i64, i32, PI64, PI64, PI64]
    lib.pa_bm_append_slot.restype = ctypes.c_int
    lib.pa_bm_fork.argtypes = [B, i64, i64]
    lib.pa_bm_fork.restype = ctypes.c_int
    lib.pa_bm_free.argtypes = [B, i64]
    lib.pa_bm_free.restype = ctypes.c_int
    lib.pa_bm_block_table.argtypes = [B, i64, P, i32, PI32, PI32]
    lib.pa_bm_block_table.restype = ctypes.c_int
    lib.pa_bm_swap_out.argtypes = [B, P, i32, P, i32, PI32]
    lib.pa_bm_swap_out.restype = ctypes.c_int
    lib.pa_bm_swap_in.argtypes = [B, P, i32, P, i32, PI32]
    lib.pa_bm_swap_in.restype = ctypes.c_int
    lib.pa_bm_num_free_blocks.argtypes = [B, i32]
    lib.pa_bm_num_free_blocks.restype = i32
    lib.pa_bm_ref_count.argtypes = [B, i32, i32]
    lib.pa_bm_ref_count.restype = i32
    lib.pa_bm_can_append_slots.argtypes = [B, i32]
    lib.pa_bm_can_append_slots.restype = i32
    lib.pa_bm_can_swap_in.argtypes = [B, P, i32]
    lib.pa_bm_can_swap_in.restype = i32
    lib.pa_bm_can_swap_out.argtypes = [B, P, i32]
    lib.pa_bm_can_swap_out.restype = i32
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error_message.argtypes = []
    lib.pa_last_error_message.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != PA_OK:
        lib = load()
        raise PagedKVError(status, f"{lib.pa_status_string(status).decode()}: "
                                   f"{lib.pa_last_error_message().decode()}")


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _pairs(pairs) -> np.ndarray:
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    return arr


def cache_bytes(desc: CacheDesc) -> int:
    return load().pa_cache_bytes(ctypes.byref(desc.c()))


def cache_element_offset(desc: CacheDesc, block: int, kv_head: int, part: int, slot: int, dim: int) -> int:
    return load().pa_cache_element_offset(ctypes.byref(desc.c()), block, kv_head, part, slot, dim)


def cache_scale_offset(desc: CacheDesc, block: int, kv_head: int, part: int, slot: int) -> int:
    return load().pa_cache_scale_offset(ctypes.byref(desc.c()), block, kv_head, part, slot)


def reshape_and_cache(kv_cache: torch.Tensor, desc: CacheDesc, key: torch.Tensor, value: torch.Tensor,
                      slot_mapping: torch.Tensor, layer: int = 0, dev_err: torch.Tensor | None = None,
                      stream=None) -> None:
    """pa_reshape_and_cache: key/value [N, Hkv, D] (token stride = stride(0))."""
    n = key.shape[0]
    _check(load().pa_reshape_and_cache(_ptr(kv_cache), ctypes.byref(desc.c()), layer, _ptr(key), key.stride(0),
                                       _ptr(value), value.stride(0), _ptr(slot_mapping), n, _ptr(dev_err),
                                       _stream(stream)))


def decode_partition_size(desc: CacheDesc, num_seqs: int, max_context_len: int, partition_size: int = 0) -> int:
    return load().pa_decode_partition_size(ctypes.byref(desc.c()), num_seqs, max_context_len, partition_size)


def decode_workspace_bytes(desc: CacheDesc, num_seqs: int, num_q_heads: int, max_context_len: int,
                           partition_size: int = 0) -> int:
    return load().pa_decode_workspace_bytes(ctypes.byref(desc.c()), num_seqs, num_q_heads, max_context_len,
                                            partition_size)


def decode(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor, desc: CacheDesc,
           block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int, scale: float,
           workspace: torch.Tensor | None = None, partition_size: int = 0, layer: int = 0,
           dev_err: torch.Tensor | None = None, stream=None) -> None:
    """pa_decode: out/q [S, Hq, D]; block_tables int32 [S, W]; context_lens int32 [S]."""
    S, Hq = q.shape[0], q.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode(_ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), ctypes.byref(desc.c()), layer,
                            _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), S, Hq,
                            max_context_len, scale, partition_size, _ptr(workspace), ws_bytes, _ptr(dev_err),
                            _stream(stream)))


def decode_shared_prefix_partition_size(desc: CacheDesc, num_seqs: int, num_q_heads: int, num_groups: int,
                                        max_context_len: int, partition_size: int = 0) -> int:
    return load().pa_decode_shared_prefix_partition_size(ctypes.byref(desc.c()), num_seqs, num_q_heads, num_groups,
                                                         max_context_len, partition_size)


def decode_shared_prefix_workspace_bytes(desc: CacheDesc, num_seqs: int, num_q_heads: int, num_groups: int,
                                         max_context_len: int, partition_size: int = 0) -> int:
    return load().pa_decode_shared_prefix_workspace_bytes(ctypes.byref(desc.c()), num_seqs, num_q_heads, num_groups,
                                                          max_context_len, partition_size)


def decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor, desc: CacheDesc,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int, scale: float,
                         group_start: torch.Tensor, prefix_lens: torch.Tensor, workspace: torch.Tensor | None = None,
                         partition_size: int = 0, layer: int = 0, dev_err: torch.Tensor | None = None,
                         stream=None) -> None:
    """pa_decode_shared_prefix: pa_decode where groups of consecutive sequences
    (group_start int32 [G + 1]) share their first prefix_lens[g] tokens' blocks."""
    S, Hq = q.shape[0], q.shape[1]
    G = prefix_lens.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode_shared_prefix(_ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), ctypes.byref(desc.c()),
                                          layer, _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), S,
                                          Hq, max_context_len, scale, _ptr(group_start), _ptr(prefix_lens), G,
                                          partition_size, _ptr(workspace), ws_bytes, _ptr(dev_err),
                                          _stream(stream)))


def decode_window(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor, desc: CacheDesc,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int, scale: float,
                  window: int, ring_blocks: int = 0, workspace: torch.Tensor | None = None, partition_size: int = 0,
                  layer: int = 0, dev_err: torch.Tensor | None = None, stream=None) -> None:
    """pa_decode_window: decode over the last `window` positions; ring_blocks > 0
    reads table rows as rings (logical block j at entry j % ring_blocks)."""
    S, Hq = q.shape[0], q.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode_window(_ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), ctypes.byref(desc.c()), layer,
                                   _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), S, Hq,
                                   max_context_len, scale, window, ring_blocks, partition_size, _ptr(workspace),
                                   ws_bytes, _ptr(dev_err), _stream(stream)))


def prefill(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor, desc: CacheDesc,
            block_tables: torch.Tensor, context_lens: torch.Tensor, query_start_loc: torch.Tensor,
            max_query_len: int, scale: float, layer: int = 0, dev_err: torch.Tensor | None = None,
            stream=None) -> None:
    """pa_prefill: out/q [T, Hq, D] packed by query_start_loc (int32 [S + 1]); causal
    over each sequence's cache (its last q_len positions are the queries)."""
    S, Hq = context_lens.shape[0], q.shape[1]
    _check(load().pa_prefill(_ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), ctypes.byref(desc.c()), layer,
                             _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), _ptr(query_start_loc),
                             S, Hq, max_query_len, scale, _ptr(dev_err), _stream(stream)))


def decode_window_span(max_context_len: int, block_size: int, window: int, ring_blocks: int = 0) -> int:
    return load().pa_decode_window_span(max_context_len, block_size, window, ring_blocks)


STATIC_WORKSPACE_BYTES = 32 * 1024 * 1024


def decode_static_workspace(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor, desc: CacheDesc,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                            scale: float, partition_size: int = 0, layer: int = 0,
                            dev_err: torch.Tensor | None = None, stream=None) -> None:
    """pa_decode_static_workspace: pa_decode for callers that cannot allocate device
    memory; the library's own fixed workspace (STATIC_WORKSPACE_BYTES per device)
    replaces the caller's.  Calls that can overlap on the GPU must be serialised."""
    S, Hq = q.shape[0], q.shape[1]
    _check(load().pa_decode_static_workspace(_ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache),
                                             ctypes.byref(desc.c()), layer, _ptr(block_tables),
                                             block_tables.stride(0), _ptr(context_lens), S, Hq, max_context_len,
                                             scale, partition_size, _ptr(dev_err), _stream(stream)))


def copy_blocks(kv_cache: torch.Tensor, desc: CacheDesc, pairs, stream=None) -> None:
    """pa_copy_blocks: pairs = host (src, dst) list / array [n, 2]."""
    arr = _pairs(pairs)
    _check(load().pa_copy_blocks(_ptr(kv_cache), ctypes.byref(desc.c()), arr.ctypes.data_as(ctypes.c_void_p),
                                 arr.shape[0], _stream(stream)))


def swap_blocks(dst_pool: torch.Tensor, dst_desc: CacheDesc, src_pool: torch.Tensor, src_desc: CacheDesc,
                direction: int, pairs, stream=None) -> None:
    """pa_swap_blocks: direction 0 = device -> pinned host, 1 = pinned host -> device."""
    arr = _pairs(pairs)
    _check(load().pa_swap_blocks(_ptr(dst_pool), ctypes.byref(dst_desc.c()), _ptr(src_pool),
                                 ctypes.byref(src_desc.c()), direction, arr.ctypes.data_as(ctypes.c_void_p),
                                 arr.shape[0], _stream(stream)))


def read_device_errors(dev_err: torch.Tensor, clear: bool = True, stream=None) -> int:
    host = ctypes.c_uint32(0)
    _check(load().pa_read_device_errors(_ptr(dev_err), ctypes.byref(host), int(clear), _stream(stream)))
    return host.value


def status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


class BlockManager:
    """Host-side block manager (pa_bm_*): block tables, slots, copy-on-write and
    swap pairs for sequences of token ids."""

    def __init__(self, block_size: int, num_gpu_blocks: int, num_cpu_blocks: int = 0, watermark: float = 0.0,
                 sliding_window: int = 0, prefix_caching: bool = False):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.pa_bm_create(block_size, num_gpu_blocks, num_cpu_blocks, watermark, sliding_window,
                                      int(prefix_caching), ctypes.byref(h)))
        self._h = h
        self.block_size = block_size

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def can_allocate(self, num_tokens: int) -> int:
        return self._lib.pa_bm_can_allocate(self._h, num_tokens)

    def allocate(self, seq_id: int, token_ids) -> None:
        t = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        _check(self._lib.pa_bm_allocate(self._h, seq_id, t.ctypes.data_as(ctypes.c_void_p), t.size))

    def append_slot(self, seq_id: int, token_id: int):
        """Slot of the new token and the copy-on-write pair (src, dst), or None."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pa_bm_append_slot(self._h, seq_id, token_id, ctypes.byref(slot), ctypes.byref(src),
                                           ctypes.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_bm_fork(self._h, parent, child))

    def free(self, seq_id: int) -> None:
        _check(self._lib.pa_bm_free(self._h, seq_id))

    def block_table(self, seq_id: int):
        """(int32 block ids of the sequence, its number of tokens)."""
        nb, nt = ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(nb), ctypes.byref(nt)))
        out = np.zeros(nb.value, dtype=np.int32)
        _check(self._lib.pa_bm_block_table(self._h, seq_id, out.ctypes.data_as(ctypes.c_void_p), out.size,
                                           ctypes.byref(nb), ctypes.byref(nt)))
        return out, nt.value

    def _swap(self, fn, seq_ids):
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ctypes.c_int32()
        _check(fn(self._h, ids.ctypes.data_as(ctypes.c_void_p), ids.size, None, 0, ctypes.byref(n)))
        # counting call changes nothing; the second call performs the move
        pairs = np.zeros((max(n.value, 1), 2), dtype=np.int64)
        _check(fn(self._h, ids.ctypes.data_as(ctypes.c_void_p), ids.size, pairs.ctypes.data_as(ctypes.c_void_p),
                  pairs.shape[0], ctypes.byref(n)))
        return pairs[:n.value]

    def swap_out(self, seq_ids):
        """Move the sequences' blocks to the host pool; (device, host) pairs."""
        return self._swap(self._lib.pa_bm_swap_out, seq_ids)

    def swap_in(self, seq_ids):
        """Move the sequences' blocks back to the device pool; (host, device) pairs."""
        return self._swap(self._lib.pa_bm_swap_in, seq_ids)

    def can_append_slots(self, num_running: int) -> bool:
        return self._lib.pa_bm_can_append_slots(self._h, num_running) == 1

    def _can_swap(self, fn, seq_ids) -> int:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        r = fn(self._h, ids.ctypes.data_as(ctypes.c_void_p), ids.size)
        if r < 0:
            _check(PA_ERR_INVALID_ARG)
        return r

    def can_swap_in(self, seq_ids) -> int:
        """Admission of swap_in (an alloc status: OK, LATER or NEVER)."""
        return self._can_swap(self._lib.pa_bm_can_swap_in, seq_ids)

    def can_swap_out(self, seq_ids) -> bool:
        return self._can_swap(self._lib.pa_bm_can_swap_out, seq_ids) == 1

    def num_free(self, on_host: bool = False) -> int:
        return self._lib.pa_bm_num_free_blocks(self._h, int(on_host))

    def ref_count(self, block: int, on_host: bool = False) -> int:
        return self._lib.pa_bm_ref_count(self._h, int(on_host), block)
