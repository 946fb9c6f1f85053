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
