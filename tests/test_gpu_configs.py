"""Full-size parity on the five workloads, in the launch configuration the
benchmark times (DecodeStep, default partition size).

Cache operations are compared bit for bit on the whole pool, and attention on
every (sequence, query head) output row against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import assert_attention_close, dev_to_u16, ensure_built
from paged_kv_cache_168_gb300.step import DecodeStep
from paged_kv_cache_168_gb300.workloads import as_u16, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


@pytest.mark.parametrize("name", ["tiny", "7b", "8b", "70b", "beam"])
def test_full_size_step_matches_oracle(name):
    w = make_workload(name, device="cuda", nan_unused=True)
    cfg = w.cfg
    g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
    pool = as_u16(w.kv_cache).reshape(-1)                       # pool before the step
    step = DecodeStep(w)
    out = step()
    torch.cuda.synchronize()
    assert pkv.read_device_errors(step.dev_err) == 0

    # oracle: the same step on host copies
    if w.host_blocks:
        gh = oracle.Geom(w.host_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
        host = np.zeros(gh.layer_elems, dtype=np.uint16)
        assert oracle.swap_blocks(host, gh, pool, g, w.swap_out_pairs) == 0
        assert oracle.swap_blocks(pool, g, host, gh, w.swap_in_pairs) == 0
        assert np.array_equal(step.host_pool.view(torch.int16).numpy().view(np.uint16), host)
    if w.copy_pairs.shape[0]:
        assert oracle.copy_blocks(pool, g, w.copy_pairs) == 0
    assert oracle.reshape_and_cache(pool, g, as_u16(w.key), as_u16(w.value), w.slot_mapping_np) == 0
    assert np.array_equal(dev_to_u16(w.kv_cache).reshape(-1), pool)

    ref, err = oracle.decode(as_u16(w.q), pool, g, w.block_tables_np, w.context_lens_np, w.scale,
                             max_context_len=w.max_context_len)
    assert err == 0
    assert_attention_close(out, ref, f"full-size {name}")
    # every output row is finite (NaN-filled unused blocks were never read)
    assert bool(torch.isfinite(out).all())
