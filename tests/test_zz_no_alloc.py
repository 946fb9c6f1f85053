"""moe_dispatch_layout_static: the layout for callers that cannot allocate.

Some callers have no way to allocate device memory at the moment they call
the layout (a plugin whose host engine owns all device memory, plain C code
without an allocator), so this entry point keeps its scratch in an array built
into the library.  Only the layout's two-launch form uses that scratch: the
chunk kernel writes every chunk's partition and expert counts into it and the
fix-up kernel reads them back.  These tests call the entry point through the
C ABI on two such shapes in a row (the second reads the array after the first
one filled it with other counts), assert from the launch trace that the
fix-up kernel ran, and check every output against the CPU oracle and against
moe_dispatch_layout with a caller-provided workspace; sizes beyond the
built-in array are refused.  The file sorts last so that, if it fails, a run
that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle

pytestmark = pytest.mark.gpu

KEYS = ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    return m.load_library()


def _outputs(S, T, k, E, P):
    i32 = dict(dtype=torch.int32, device="cuda")
    return {"expert_counts": torch.full((S, E), -7, **i32),
            "expert_rank": torch.full((S, T, k), -7, **i32),
            "part_counts": torch.full((S, P), -7, **i32),
            "part_offsets": torch.full((S, P + 1), -7, **i32),
            "token_slot": torch.full((S, T, P), -7, **i32),
            "dev_status": torch.zeros((1,), **i32)}


def _static_layout(lib, ids, E, P):
    """One call of the static entry point; returns its outputs and the names of
    the kernels it launched (from the library's launch trace)."""
    S, T, k = ids.shape
    o = _outputs(S, T, k, E, P)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    m.trace_enable(None, 16)
    m.trace_reset()
    try:
        rc = lib.moe_dispatch_layout_static(p(ids), S, T, k, E, P, p(o["expert_counts"]),
                                            p(o["expert_rank"]), p(o["part_counts"]),
                                            p(o["part_offsets"]), p(o["token_slot"]),
                                            p(o["dev_status"]), stream)
        assert rc == m.MOE_OK, lib.moe_last_error_message().decode()
        torch.cuda.synchronize()
        kernels = [name for name, _ in m.trace_records()]
    finally:
        m.trace_disable()
    return {key: t.cpu().numpy() for key, t in o.items()}, kernels


def _workspace_layout(ids, E, P):
    S, T, k = ids.shape
    o = _outputs(S, T, k, E, P)
    ws = torch.empty(m.moe_workspace_bytes(S, T, k, E, P), dtype=torch.uint8, device="cuda")
    m.moe_dispatch_layout(ids, E, P, o["expert_counts"], o["expert_rank"], o["part_counts"],
                          o["part_offsets"], o["token_slot"], ws, o["dev_status"])
    torch.cuda.synchronize()
    return {key: t.cpu().numpy() for key, t in o.items()}


def test_static_layout_uses_its_scratch_twice(lib):
    # two shapes longer than one cluster covers (16 chunks of 1,024 tokens):
    # first the large workload's rows at 20,000 tokens (79 chunks of 256 in one
    # source, E = 64), then 2 sources x 17,000 tokens (67 chunks each, E = 384),
    # whose counts overwrite and then read back the same bytes of the array
    cases = [ms.workload("large", T=20000, index=18), ms.workload("prefill", S=2, T=17000, index=17)]
    for w in cases:
        assert lib.moe_dispatch_layout_kernels(w.S, w.T, w.k, w.E, w.P) == 2, w
        ids_np, _ = oracle.route_topk(ms.gen_logits(w), w.k)
        ids = torch.from_numpy(ids_np).cuda()
        got, kernels = _static_layout(lib, ids, w.E, w.P)
        assert kernels == ["k_layout_local", "k_layout_fix"], (w.name, kernels)
        ref = oracle.dispatch_layout(ids_np, w.E, w.P)
        for key in KEYS:
            assert np.array_equal(got[key], ref[key]), (w.name, key)
        assert int(got["dev_status"][0]) == ref["status"] == 0
        want = _workspace_layout(ids, w.E, w.P)
        for key in KEYS:
            assert np.array_equal(got[key], want[key]), (w.name, key)


def test_static_layout_refuses_sizes_beyond_its_scratch(lib):
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: the call is refused first
    rc = lib.moe_dispatch_layout_static(fake, 8, 40000, 2, 1024, 32, fake, fake, fake, fake,
                                        fake, fake, ctypes.c_void_p(0))
    assert rc == m.MOE_ERR_INVALID_ARG
    assert "scratch" in lib.moe_last_error_message().decode()
