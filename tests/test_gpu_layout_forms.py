"""The dispatch layout's two launch forms on the GPU vs the oracle.

The layout works on 256-token chunks.  With one chunk per source (a decode
step) it is one launch of one CTA per source.  With 2 to 16 chunks per source
(up to 4,096 tokens) it is one launch with a thread-block cluster per source
and a CTA per chunk: the CTAs lay out their chunks in shared memory, meet at the cluster
barrier, exchange counts through distributed shared memory and store final
values.  Sources of up to 16,384 tokens take the same cluster form with chunks
of 1,024 tokens (and threads) where their shared memory fits.  Longer sources
take two launches (chunk-local layout, then a fix-up through the workspace).  Both forms must give the oracle's outputs bit for bit
(a2a-backends section 1.3 and 3.2: slots, counts, offsets; section 1.5: the
expert ranks the receiver's runs are built from), with ragged tails, repeated
and invalid ids, and E smaller than the cluster.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import oracle
from gpu_util import DEV, host, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _ids(S, T, k, E, seed, dups=False, bad=False):
    rng = np.random.default_rng(seed)
    if dups:
        ids = rng.integers(0, E, size=(S, T, k)).astype(np.int32)      # repeats allowed
    else:
        ids = np.argsort(rng.random((S, T, E)), axis=2)[:, :, :k].astype(np.int32)
    if bad:
        ids[rng.random(ids.shape) < 0.01] = -1
        ids[rng.random(ids.shape) < 0.005] = E + 3
    return ids


def _layout(ids, E, P):
    """Runs moe_dispatch_layout; returns its outputs and the kernels it launched."""
    S, T, k = ids.shape
    ws = torch.empty(max(m.moe_workspace_bytes(S, T, k, E, P), 256), dtype=torch.uint8,
                     device=DEV).fill_(0xAB)
    ec = torch.full((S, E), -7, dtype=torch.int32, device=DEV)
    er = torch.full((S, T, k), -7, dtype=torch.int32, device=DEV)
    pc = torch.full((S, P), -7, dtype=torch.int32, device=DEV)
    po = torch.full((S, P + 1), -7, dtype=torch.int32, device=DEV)
    ts = torch.full((S, T, P), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    d_ids = i32_dev(ids)
    torch.cuda.synchronize()
    m.trace_enable("k_layout", 16)
    try:
        m.moe_dispatch_layout(d_ids, E, P, ec, er, pc, po, ts, ws, st)
        torch.cuda.synchronize()
        kernels = [name for name, _ in m.trace_records()]
    finally:
        m.trace_disable()
    out = {"expert_counts": host(ec), "expert_rank": host(er), "part_counts": host(pc),
           "part_offsets": host(po), "token_slot": host(ts), "status": int(st.item())}
    return out, kernels


def _check(ids, E, P, form):
    got, kernels = _layout(ids, E, P)
    want = oracle.dispatch_layout(ids, E, P)
    for key in ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot",
                "status"):
        assert np.array_equal(got[key], want[key]), key
    want_kernels = {"cluster": ["k_layout_cluster"], "one": ["k_layout_local"],
                    "two": ["k_layout_local", "k_layout_fix"]}[form]
    assert kernels == want_kernels, kernels


@pytest.mark.parametrize("S,T,k,E,P", [(1, 64, 6, 384, 8), (4, 256, 8, 64, 4),
                                       (2, 200, 32, 1024, 32)])
def test_one_chunk(S, T, k, E, P):
    """One chunk per source (a decode step): one CTA per source, values final."""
    _check(_ids(S, T, k, E, seed=S * 31 + T), E, P, "one")


@pytest.mark.parametrize("S,T,k,E,P", [
    (1, 257, 6, 384, 8),         # two chunks, ragged
    (1, 4096, 6, 384, 8),        # the prefill shape: a cluster of 16
    (8, 4096, 6, 384, 8),        # one cluster per source
    (3, 601, 8, 64, 4),
    (2, 1000, 32, 1024, 32),     # the largest k, E and P
    (1, 4000, 1, 8, 8),          # fewer experts than CTAs in the cluster
    (1, 3000, 4, 4, 1),          # one partition
])
def test_cluster_form(S, T, k, E, P):
    _check(_ids(S, T, k, E, seed=S * 100003 + T), E, P, "cluster")


def test_cluster_form_repeats_and_bad_ids():
    ids = _ids(2, 4000, 8, 64, seed=11, dups=True, bad=True)
    assert (ids >= 64).any() and (ids < 0).any()
    _check(ids, 64, 8, "cluster")


@pytest.mark.parametrize("S,T,k,E,P", [
    (1, 4097, 6, 384, 8),        # just past 16 chunks of 256: 5 chunks of 1,024, ragged
    (1, 16384, 8, 64, 8),        # the large shape: a cluster of 16 wide chunks
    (2, 9000, 6, 384, 8),        # one cluster per source
    (1, 12000, 8, 64, 16),       # more partitions
    (3, 5000, 4, 4, 1),          # fewer experts than CTAs, one partition
])
def test_wide_cluster_form(S, T, k, E, P):
    _check(_ids(S, T, k, E, seed=S * 7 + T), E, P, "cluster")


def test_wide_cluster_form_repeats_and_bad_ids():
    ids = _ids(1, 9000, 8, 64, seed=12, dups=True, bad=True)
    assert (ids >= 64).any() and (ids < 0).any()
    _check(ids, 64, 8, "cluster")


@pytest.mark.parametrize("S,T,k,E,P", [
    (1, 16385, 6, 384, 8),       # past 16 chunks of 1,024
    (2, 20000, 8, 64, 8),
    (1, 40000, 32, 64, 32),
    (1, 5000, 32, 1024, 32),     # wide chunks would not fit one CTA's shared memory
])
def test_two_launch_form(S, T, k, E, P):
    _check(_ids(S, T, k, E, seed=S * 7 + T), E, P, "two")


def test_two_launch_form_repeats_and_bad_ids():
    ids = _ids(1, 20000, 32, 64, seed=6, dups=True, bad=True)
    _check(ids, 64, 32, "two")
