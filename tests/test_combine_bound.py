"""The combine accuracy bound used by the GPU parity tests, checked on the CPU.

A numpy emulation of an fp32 accumulation (each product and each partial sum
rounded to fp32, then one round to bf16) must stay inside the bound against
the oracle's exact sum; planted mistakes of the kind the bound is there to
catch (a dropped term, a 0.5% weight error, partial sums kept in bf16) must
break it.
"""
import numpy as np

import moe_synth as ms
import oracle
from gpu_util import combine_within_fp32_bound


def _case(seed=11, N=300, k=6, H=64, R=900):
    rng = np.random.default_rng(seed)
    y = ms.bf16_bits_from_f32(rng.standard_normal((R, H)).astype(np.float32))
    pr = rng.integers(0, R, size=(N, k)).astype(np.int32)
    pr[5, 2] = -1
    pr[9, :] = -1                                   # a token with no pair: exact 0
    w = rng.uniform(0.01, 1.0, size=(N, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    return y, pr, w


def _fp32_combine(y, pr, w, drop_last=False, w_scale=1.0, bf16_partials=False):
    N, k = pr.shape
    H = y.shape[1]
    acc = np.zeros((N, H), np.float32)
    yf = ms.f32_from_bf16_bits(y)
    for j in range(k - 1 if drop_last else k):
        valid = pr[:, j] >= 0
        prod = (w[:, j].astype(np.float64)[:, None] * w_scale
                * yf[np.maximum(pr[:, j], 0)].astype(np.float64)).astype(np.float32)
        acc = np.where(valid[:, None], (acc + prod).astype(np.float32), acc)
        if bf16_partials:
            acc = ms.f32_from_bf16_bits(ms.bf16_bits_from_f32(acc))
    return ms.bf16_bits_from_f32(acc)


def test_fp32_accumulation_is_inside_the_bound():
    y, pr, w = _case()
    want = oracle.combine(y, pr[None], w[None])[0]
    ok, excess = combine_within_fp32_bound(_fp32_combine(y, pr, w), want, y, pr, w)
    assert ok, excess
    assert np.all(want[9] == 0)


def test_planted_mistakes_break_the_bound():
    y, pr, w = _case()
    want = oracle.combine(y, pr[None], w[None])[0]
    for kw in ({"drop_last": True}, {"w_scale": 1.005}, {"bf16_partials": True}):
        ok, excess = combine_within_fp32_bound(_fp32_combine(y, pr, w, **kw), want, y, pr, w)
        assert not ok, kw
        assert excess > 0, kw
