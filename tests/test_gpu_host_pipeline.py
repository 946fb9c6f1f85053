"""HostPipeline: steps fed from and drained to pinned host memory.

More steps than buffer sets, with different inputs every step: each step's
host output must equal the device path's output for the same inputs, with
graphs and with eager launches, for the contiguous and the routed forms.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
from gpu_util import bf16_dev, bf16_host, f32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


@pytest.mark.parametrize("name,graphs,sets,kw", [("tiny", True, 2, {}), ("tiny", False, 3, {}),
                                                 ("decode", True, 3, {}),
                                                 ("decode", True, 2, {"layout": "routed"})])
def test_pipeline_outputs_equal_device_steps(name, graphs, sets, kw):
    w_ = ms.workload(name)
    n_inputs, n_steps = 4, 9
    inputs = [ms.gen_inputs(ms.workload(name, index=w_.index + 100 + i)) for i in range(n_inputs)]
    ref = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, **kw)
    want = [bf16_host(ref.step(f32_dev(inp["logits"]), bf16_dev(inp["x"]))).copy() for inp in inputs]
    h_in = [(torch.from_numpy(inp["logits"]).pin_memory(),
             torch.from_numpy(inp["x"].view(np.int16)).pin_memory()) for inp in inputs]
    h_out = [torch.empty((w_.S, w_.T, w_.H), dtype=torch.int16).pin_memory() for _ in range(n_steps)]
    pipe = m.HostPipeline(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, sets=sets, graphs=graphs, **kw)
    for i in range(n_steps):
        pipe.submit(*h_in[i % n_inputs], h_out[i])
    pipe.synchronize()
    for i in range(n_steps):
        assert np.array_equal(h_out[i].numpy().view(np.uint16), want[i % n_inputs]), i
    assert all(int(p.dev_status.item()) == 0 for p in pipe.paths)
    pipe.release()


_FIRST_USE = r"""
import sys
import numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import combine_moe_route_06_gb300 as m
import moe_synth as ms
w = ms.workload("tiny", T=600)                  # three chunks: the cluster layout
inp = ms.gen_inputs(w)
h_lg = torch.from_numpy(inp["logits"]).pin_memory()
h_x = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
h_out = torch.empty((w.S, w.T, w.H), dtype=torch.int16).pin_memory()
pipe = m.HostPipeline(w.S, w.T, w.H, w.E, w.k, w.P, sets=2, graphs=True)   # first library use
pipe.submit(h_lg, h_x, h_out)
pipe.synchronize()
ref = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P)
out = ref.step(torch.from_numpy(inp["logits"]).cuda(),
               torch.from_numpy(inp["x"].view(np.int16)).cuda().view(torch.bfloat16))
torch.cuda.synchronize()
assert np.array_equal(h_out.numpy(), out.view(torch.int16).cpu().numpy())
assert m.moe_dispatch_layout_kernels(w.S, w.T, w.k, w.E, w.P) == 1
print("first-use pipeline ok")
"""


def test_pipeline_as_first_library_use():
    """A process whose first use of the library is a graph-capturing pipeline: the library's
    one-time device queries run in the pipeline's eager warm-up step, not inside a capture, and
    the captured steps give the device path's bytes with the one-launch layout."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_USE, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "first-use pipeline ok" in r.stdout
