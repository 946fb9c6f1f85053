"""Helpers shared by the GPU tests: numpy <-> torch bf16 bits, path runners."""
from __future__ import annotations

import numpy as np
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms

DEV = "cuda"


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(DEV)


def f32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def close_bf16(got_bits: np.ndarray, want_bits: np.ndarray, rel=1e-2, floor=1e-3) -> bool:
    """|got - want| <= rel * max(|want|, floor), elementwise on bf16 values."""
    g = ms.f32_from_bf16_bits(got_bits).astype(np.float64)
    w = ms.f32_from_bf16_bits(want_bits).astype(np.float64)
    return bool(np.all(np.abs(g - w) <= rel * np.maximum(np.abs(w), floor)))


def worst_rel(got_bits, want_bits, floor=1e-3) -> float:
    g = ms.f32_from_bf16_bits(got_bits).astype(np.float64)
    w = ms.f32_from_bf16_bits(want_bits).astype(np.float64)
    return float(np.max(np.abs(g - w) / np.maximum(np.abs(w), floor))) if g.size else 0.0


def run_layout(ids: np.ndarray, E: int, P: int):
    S, T, k = ids.shape
    d_ids = i32_dev(ids)
    ec = torch.full((S, E), -7, dtype=torch.int32, device=DEV)
    er = torch.full((S, T, k), -7, dtype=torch.int32, device=DEV)
    pc = torch.full((S, P), -7, dtype=torch.int32, device=DEV)
    po = torch.full((S, P + 1), -7, dtype=torch.int32, device=DEV)
    ts = torch.full((S, T, P), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(m.moe_workspace_bytes(S, T, k, E, P), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_dispatch_layout(d_ids, E, P, ec, er, pc, po, ts, ws, st)
    torch.cuda.synchronize()
    return {"expert_counts": host(ec), "expert_rank": host(er), "part_counts": host(pc),
            "part_offsets": host(po),
            "token_slot": host(ts), "status": int(st.item())}


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """One unit in the last place of bf16 (8 significant bits) at |v|; the
    smallest normal's unit for |v| below 2^-126 or v == 0."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def combine_within_fp32_bound(got_bits, want_bits, y_bits, pair_row, w, chunk=512):
    """The combine's own accuracy, element by element: the kernel sums k
    products w_j * y_j with fp32 FMAs and rounds once to bf16; the oracle sums
    exactly and rounds once.  A chain of k FMAs is off the exact sum by at most
    k * 2^-24 * sum_j |w_j y_j| (each FMA rounds its result once), and two
    roundings to nearest of sums that close differ by at most that plus one
    bf16 unit.  The test uses k * 2^-23 (twice the first-order bound) plus one
    unit at max(|got|, |want|).  A dropped term, a weight applied twice or a
    sum kept in bf16 breaks it.  Returns (ok, worst excess over the bound).

    got_bits / want_bits: bf16 bits [N, H]; y_bits: bf16 bits of the rows the
    combine read; pair_row [N, k] (-1: skipped); w float32 [N, k]."""
    got = ms.f32_from_bf16_bits(np.asarray(got_bits)).astype(np.float64)
    want = ms.f32_from_bf16_bits(np.asarray(want_bits)).astype(np.float64)
    N, k = pair_row.shape
    worst = -np.inf
    ok = True
    for n0 in range(0, N, chunk):
        n1 = min(N, n0 + chunk)
        pr = pair_row[n0:n1]
        absum = np.zeros((n1 - n0, got.shape[1]), np.float64)
        for j in range(k):
            valid = pr[:, j] >= 0
            if not np.any(valid):
                continue
            rows = ms.f32_from_bf16_bits(y_bits[pr[valid, j]]).astype(np.float64)
            absum[valid] += np.abs(w[n0:n1][valid, j].astype(np.float64))[:, None] * np.abs(rows)
        g, r = got[n0:n1], want[n0:n1]
        bound = k * 2.0 ** -23 * absum + bf16_ulp(np.maximum(np.abs(g), np.abs(r)))
        excess = np.abs(g - r) - bound
        worst = max(worst, float(excess.max()) if excess.size else -np.inf)
        ok = ok and bool(np.all(excess <= 0))
    return ok, worst
