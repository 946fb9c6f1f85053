"""The synthetic workloads' skew (CPU).

The skewed receiver view biases the router logits by the log of a Zipf(1.2)
expert popularity: the receivers' loads are uneven (a2a-backends page,
section 1.4, records the busiest of 8 GPUs at 1.39 times the mean rows over
the layers of a run and 1.64 times in its worst layer).  With the popularity
ranks equal to the expert ids the hot experts all sit in partition 0;
`skewed_perm` draws the ranks as a seeded permutation, which spreads them over
the partitions, so its busiest receiver carries a small multiple of the mean
load instead of nearly all of it.
"""
import numpy as np

import moe_synth as ms
import oracle


def test_popularity_ranks():
    w = ms.workload("skewed")
    assert np.array_equal(ms.popularity_rank(w), np.arange(w.E))
    wp = ms.workload("skewed_perm")
    r = ms.popularity_rank(wp)
    assert np.array_equal(np.sort(r), np.arange(wp.E))
    assert not np.array_equal(r, np.arange(wp.E))
    for v in (w, wp):
        p = ms.zipf_popularity(v)
        assert abs(p.sum() - 1.0) < 1e-12
        # the most popular expert is the one of rank 0, and p falls with the rank
        assert np.all(np.diff(p[np.argsort(ms.popularity_rank(v))]) < 0)


def test_skewed_logits_are_normals_plus_log_zipf():
    """logit[s,t,e] = z + ln((e + 1)^-1.2 / sum_i (i + 1)^-1.2) at identity ranks."""
    w = ms.workload("skewed")
    lg = ms.gen_logits(w, S=1, T=3)
    z = ms.normals(w.seed_logits, 3 * w.E).reshape(1, 3, w.E)
    e = np.arange(w.E, dtype=np.float64)
    lnp = -1.2 * np.log(e + 1.0) - np.log(np.sum((e + 1.0) ** -1.2))
    assert np.allclose(lg, (z + lnp).astype(np.float32), rtol=0, atol=2e-6)


def _pairs_per_partition(w):
    ids, _ = oracle.route_topk(ms.gen_logits(w), w.k)
    assert ids.shape == (w.S, w.T, w.k) and ids.min() >= 0 and ids.max() < w.E
    return np.bincount((ids // (w.E // w.P)).reshape(-1), minlength=w.P)


def test_receiver_load_of_the_skewed_workloads():
    w = ms.workload("skewed")
    c = _pairs_per_partition(w)
    assert c.sum() == w.S * w.T * w.k
    assert int(np.argmax(c)) == w.recv_part == 0
    assert c.max() / c.mean() > 7.0
    wp = ms.workload("skewed_perm")
    cp = _pairs_per_partition(wp)
    assert cp.sum() == wp.S * wp.T * wp.k
    ratio = cp.max() / cp.mean()
    assert 1.3 < ratio < 3.0, ratio
    # the receiving partition (the most popularity mass) is among the busiest
    assert cp[wp.recv_part] >= 0.9 * cp.max(), (cp, wp.recv_part)
