"""A whole decode step (swap out / in, copy-on-write, reshape_and_cache, decode)
captured into a CUDA graph replays to the same bytes as eager execution."""
import numpy as np
import pytest
import torch

import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import dev_to_u16, ensure_built
from paged_kv_cache_168_gb300.step import DecodeStep
from paged_kv_cache_168_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


@pytest.mark.parametrize("name", ["beam", "70b"])
def test_captured_step_replays_like_eager(name):
    w = make_workload(name, device="cuda", num_seqs=None if name == "beam" else 2)
    stream = torch.cuda.Stream()
    step = DecodeStep(w, stream=stream)
    with torch.cuda.stream(stream):
        eager = step().clone()           # first call on the device also sets kernel attributes
    torch.cuda.synchronize()
    pool_after = dev_to_u16(w.kv_cache)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    step.out.zero_()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(step.out, eager)
        assert np.array_equal(dev_to_u16(w.kv_cache), pool_after)   # the step is idempotent
    assert pkv.read_device_errors(step.dev_err) == 0
