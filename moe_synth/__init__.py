"""Seeded synthetic inputs for the MoE token path.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle.  It holds none of the routing arithmetic: it only draws numbers
(router logits, hidden-state rows, stand-in expert scales) and names the
workload shapes.

Generator: a counter-based splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) feeds a Box-Muller transform
(Box and Muller, 1958).  Element i of a stream with seed s is a function of
(s, i) alone, so any slice can be regenerated without drawing the rest.

Workload shapes follow the a2a-backends page (vincentzed.com/writing/a2a-backends):
bf16 rows of 5,120 elements (section 1.1), 384 experts with top-6 spread as 48
per GPU over 8 GPUs (introduction, section 1.1), a prefill batch of 4,096 rows
per GPU and a decode step of 64 (section 1.1).
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "normals", "bf16_bits_from_f32", "popularity_rank",
    "zipf_popularity",
    "f32_from_bf16_bits", "gen_logits", "gen_x", "gen_scales", "gen_inputs",
]

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_SEED_BASE = 0x6D6F6531  # "moe1"
_SEED_RANK = 0x72616E6B00000000  # "rank": popularity permutations, apart from the other streams


def _splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs start..start+n-1 of splitmix64 seeded with `seed`.

    Output i is mix(seed + (i + 1) * gamma); mix is the finaliser of the
    published generator.
    """
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def normals(seed: int, n: int, start: int = 0) -> np.ndarray:
    """n standard normal float64 draws: Box-Muller on pairs of splitmix64 outputs.

    Draw 2m uses outputs 2m (u1) and 2m+1 (u2) and gives r*cos(2*pi*u2);
    draw 2m+1 gives r*sin(2*pi*u2), with r = sqrt(-2 ln u1) and u1 in (0, 1].
    """
    if n == 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + n + 1) // 2
    z = _splitmix64(seed, 2 * p0, 2 * (p1 - p0))
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * (p1 - p0), dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    off = start - 2 * p0
    return out[off:off + n]


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    S sources (emulated sending ranks), T tokens per source, H hidden size,
    E experts, k experts per token, P partitions (emulated expert-parallel
    ranks) holding E/P contiguous experts each.  `zipf_s` > 0 biases expert
    popularity; `recv_part` is the receiving partition of the permute step
    (-1: all partitions).  With `zipf_perm` the popularity ranks are a seeded
    permutation of the experts instead of their ids (popularity_rank).
    """
    name: str
    index: int
    S: int
    T: int
    H: int
    E: int
    k: int
    P: int
    zipf_s: float = 0.0
    recv_part: int = -1
    zipf_perm: bool = False

    @property
    def seed_logits(self) -> int:
        return 2 * (_SEED_BASE + self.index)

    @property
    def seed_x(self) -> int:
        return 2 * (_SEED_BASE + self.index) + 1

    @property
    def seed_rank(self) -> int:
        return _SEED_RANK + self.index


def popularity_rank(w: Workload) -> np.ndarray:
    """Popularity rank of each expert (0 = most popular), int64 [E].

    The experts' ids when `zipf_perm` is off; otherwise expert e's rank is its
    place when E normal draws of stream seed_rank are sorted ascending (stable),
    a seeded permutation.
    """
    if not w.zipf_perm:
        return np.arange(w.E, dtype=np.int64)
    order = np.argsort(normals(w.seed_rank, w.E), kind="stable")
    rank = np.empty(w.E, dtype=np.int64)
    rank[order] = np.arange(w.E, dtype=np.int64)
    return rank


def zipf_popularity(w: Workload) -> np.ndarray:
    """p_e proportional to (rank_e + 1)^-zipf_s, summing to 1, float64 [E]."""
    p = (popularity_rank(w) + 1.0) ** (-w.zipf_s)
    return p / p.sum()


def _busiest_partition(w: Workload) -> Workload:
    """`w` receiving at the partition whose experts hold the most popularity."""
    mass = zipf_popularity(w).reshape(w.P, w.E // w.P).sum(axis=1)
    return dataclasses.replace(w, recv_part=int(np.argmax(mass)))


WORKLOADS = {
    # tiny: 128 tokens, 256-wide rows, 16 experts top-2 over 4 partitions
    "tiny": Workload("tiny", 0, S=1, T=128, H=256, E=16, k=2, P=4),
    # decode step: 64 rows per rank, 5,120-wide, 384 experts top-6 over 8 partitions
    "decode": Workload("decode", 1, S=1, T=64, H=5120, E=384, k=6, P=8),
    # prefill batch: 4,096 rows per rank, same model shape
    "prefill": Workload("prefill", 2, S=1, T=4096, H=5120, E=384, k=6, P=8),
    # receiver view: 8 sources of 4,096 tokens, Zipf(1.2) popularity, partition 0 receives
    "skewed": Workload("skewed", 3, S=8, T=4096, H=5120, E=384, k=6, P=8, zipf_s=1.2, recv_part=0),
    # large batch: 16,384 tokens, 2,048-wide, 64 experts top-8 over 8 partitions
    "large": Workload("large", 4, S=1, T=16384, H=2048, E=64, k=8, P=8),
    # the skewed receiver view with the popularity ranks shuffled over the
    # experts (a seeded permutation): the hot experts spread over the
    # partitions; the busiest one receives
    "skewed_perm": _busiest_partition(
        Workload("skewed_perm", 5, S=8, T=4096, H=5120, E=384, k=6, P=8, zipf_s=1.2,
                 zipf_perm=True)),
}


def workload(name: str, **override) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller T)."""
    return dataclasses.replace(WORKLOADS[name], **override)


def gen_logits(w: Workload, S: int | None = None, T: int | None = None) -> np.ndarray:
    """Router logits, float32 [S, T, E].

    Each logit is N(0, 1).  With zipf_s > 0 the log of a Zipf popularity is
    added, logit[s,t,e] = z + ln p_e with p_e proportional to
    (rank_e + 1)^-zipf_s: with ranks equal to the ids expert 0 is the most
    popular and partition 0 the busiest receiver; with permuted ranks
    (zipf_perm) the hot experts are spread over the partitions.
    """
    S = w.S if S is None else S
    T = w.T if T is None else T
    z = normals(w.seed_logits, S * T * w.E).reshape(S, T, w.E)
    if w.zipf_s > 0:
        z = z + np.log(zipf_popularity(w))[None, None, :]
    return z.astype(np.float32)


def gen_x(w: Workload, S: int | None = None, T: int | None = None, chunk_rows: int = 4096) -> np.ndarray:
    """Hidden-state rows ~N(0, 1) rounded to bfloat16, as uint16 bits [S, T, H]."""
    S = w.S if S is None else S
    T = w.T if T is None else T
    n_rows = S * T
    out = np.empty((n_rows, w.H), dtype=np.uint16)
    for r0 in range(0, n_rows, chunk_rows):
        r1 = min(n_rows, r0 + chunk_rows)
        v = normals(w.seed_x, (r1 - r0) * w.H, start=r0 * w.H).astype(np.float32)
        out[r0:r1] = bf16_bits_from_f32(v).reshape(r1 - r0, w.H)
    return out.reshape(S, T, w.H)


def gen_scales(w: Workload, identity: bool = False) -> np.ndarray:
    """Stand-in expert scales s_e = (e + 1) / E as float32 [E] (all ones if identity)."""
    if identity:
        return np.ones(w.E, dtype=np.float32)
    return (np.arange(1, w.E + 1, dtype=np.float64) / w.E).astype(np.float32)


def gen_inputs(w: Workload, S: int | None = None, T: int | None = None) -> dict:
    """logits, x and stand-in scales for workload `w` (optionally a smaller S or T)."""
    return {"logits": gen_logits(w, S, T), "x": gen_x(w, S, T), "scales": gen_scales(w)}
