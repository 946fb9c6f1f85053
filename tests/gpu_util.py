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
