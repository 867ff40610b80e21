"""Helpers for the GPU parity tests: move oracle-built inputs to the device, run
the library through its binding, and compare with the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_168_gb300 as pkv
from paged_kv_cache_168_gb300.build import build

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}

# Attention tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle| elementwise, with
# the GPU output in the query dtype and the oracle in fp64 (max-abs 2e-3 and
# max-rel 1e-2, combined in allclose form because one bf16 rounding of an output
# in [1, 2) is already up to 3.9e-3).
ATOL, RTOL = 2e-3, 1e-2


def ensure_built():
    build()
    pkv.load()


def u16_to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(TORCH_DT[dtype])


def dev_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# Plain bound of the decode target, asserted on its own for fp16 decode outputs
# (fp16's half-ulp is at most 9.8e-4 below |o| = 4, so one output rounding fits
# it): max |gpu - oracle| <= 2e-3 and max |gpu - oracle| / max(|oracle|, 1e-3)
# <= 1e-2.  Prefill is held to the combined bound only: its fp16 PV product takes
# the weights as one fp16 operand (11 significant bits), so an output that
# cancels to below 1e-3 can be off by ~1e-4 -- inside 2e-3 + 1e-2 |o|, not
# inside 1e-2 of a 1e-3 floor.
STRICT_ABS, STRICT_REL, REL_FLOOR = 2e-3, 1e-2, 1e-3

# (what, output dtype, elements, max-abs, max-rel) of every comparison in this
# session; the summary at the end of the run prints them per workload.
ERROR_STATS: list = []


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, what: str = "", strict_fp16: bool = True):
    """Elementwise |gpu - oracle| <= ATOL + RTOL * |oracle|; for fp16 outputs (with
    strict_fp16) also the plain bounds max-abs <= 2e-3 and max-rel <= 1e-2
    (relative error over max(|oracle|, 1e-3)).  Returns (max-abs, max-rel) and
    records them."""
    g = got.detach().to(torch.float64).cpu().numpy().reshape(ref.shape)
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), ref.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {ref.size} elements out of tolerance; worst at {i}: "
                             f"gpu {g[i]!r} oracle {ref[i]!r}")
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err / np.maximum(np.abs(ref), REL_FLOOR)).max()) if err.size else 0.0
    dt = str(got.dtype).replace("torch.", "")
    ERROR_STATS.append((what, dt, int(ref.size), max_abs, max_rel))
    if strict_fp16 and got.dtype == torch.float16:
        assert max_abs <= STRICT_ABS, f"{what}: fp16 max-abs {max_abs:.3e} > {STRICT_ABS}"
        assert max_rel <= STRICT_REL, f"{what}: fp16 max-rel {max_rel:.3e} > {STRICT_REL}"
    return max_abs, max_rel


def desc_of(num_blocks, bs, Hkv, D, dtype, num_layers=1, layer_stride_bytes=0):
    return pkv.CacheDesc(num_blocks, bs, Hkv, D, TORCH_DT[dtype] if isinstance(dtype, str) else dtype,
                         num_layers, layer_stride_bytes)


def run_decode(q, pool, desc, tables, ctx, max_ctx, scale, P=0, dev_err=None):
    S, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    nbytes = pkv.decode_workspace_bytes(desc, S, Hq, max_ctx, P)
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=q.device)
    pkv.decode(out, q, pool, desc, tables, ctx, max_ctx, scale, ws, P, dev_err=dev_err)
    return out


def paged_to_dev(p, device="cuda"):
    """Device copies of an oracle-built ``Paged`` case: q, pool, tables, ctx, desc."""
    q = u16_to_dev(p.q_bits, p.dtype, device)
    pool = u16_to_dev(p.pool, p.dtype, device)
    tables = torch.from_numpy(p.tables).to(device)
    ctx = torch.from_numpy(p.ctx).to(device)
    desc = desc_of(p.num_blocks, p.bs, p.Hkv, p.D, p.dtype)
    return q, pool, tables, ctx, desc
