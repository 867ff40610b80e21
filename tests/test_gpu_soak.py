"""Many decode steps back to back.

A race between the decode kernel's roles -- an mbarrier phase seen twice, a
hand-off that a role overtakes -- may show up in one call of thousands only:
its bounded wait then runs out, PA_DEVERR_TIMEOUT is set and the affected rows
come out as zeros.  These tests run the beam workload's whole step (copy-on-write
copies, swap out / in, reshape_and_cache, the shared-prefix decode) and the 8B
workload's step a few thousand times on one stream, read the error word every
500 steps, and check that the last step's output is the same bytes as the
second step's (every step after the first repeats the same cache writes, so
its output cannot change)."""
import pytest
import torch

import paged_kv_cache_168_gb300 as pkv
from gpu_helpers import ensure_built
from paged_kv_cache_168_gb300.step import DecodeStep
from paged_kv_cache_168_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    ensure_built()


@pytest.mark.parametrize("name,steps", [("beam", 3000), ("8b", 1500)])
def test_steps_back_to_back_keep_the_error_word_clear(name, steps):
    w = make_workload(name, device="cuda")
    stream = torch.cuda.Stream()
    step = DecodeStep(w, stream=stream)
    with torch.cuda.stream(stream):
        step()
        step()
        second = step.out.clone()
        torch.cuda.synchronize()
        assert pkv.read_device_errors(step.dev_err, stream=stream) == 0
        for i in range(steps):
            step()
            if (i + 1) % 500 == 0:
                bits = pkv.read_device_errors(step.dev_err, stream=stream)
                assert bits == 0, f"{name}: device error bits {bits:#x} after {i + 1} more steps"
    torch.cuda.synchronize()
    assert torch.equal(step.out, second), f"{name}: the output changed over {steps} identical steps"
