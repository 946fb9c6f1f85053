"""CPU oracle for the MoE token path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library (``combine_moe_route_06_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, double precision, loops in
the order the pages state the definitions); this module only compiles it with
gcc and marshals numpy arrays through ctypes.  Status words use bit 1 for an
inconsistent index input, bit 2 for capacity overflow and bit 3 for an expert
id >= E.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BIT_INCONSISTENT = 1 << 1
BIT_CAPACITY = 1 << 2
BIT_BAD_ID = 1 << 3


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc -O2); returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_mutant(n: int, path: str) -> str:
    """Compile the oracle with planted mistake number n (ORC_MUTANT, see moe_oracle.c)
    into `path`; the test suite uses it to show that its pins reject the mistake."""
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORC_MUTANT={int(n)}",
                    "-o", path, _SRC, "-lm"], check=True)
    return path


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MOE_ORACLE_LIB names another build of moe_oracle.c: only the
            # mutant tests set it, to run the pins against a planted mistake
            lib = ctypes.CDLL(os.environ.get("MOE_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_expected_copies.argtypes = [i32, i32, i32]
            lib.oracle_expected_copies.restype = ctypes.c_double
            lib.oracle_route_topk.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_dispatch_layout.argtypes = [P, i32, i64, i32, i32, i32, P, P, P, P, P, P]
            lib.oracle_dispatch_pack.argtypes = [P, i32, i64, i32, i32, P, i64, P, P, P]
            lib.oracle_permute_to_experts.argtypes = [P, P, P, i32, i64, i32, i32, i32, i32,
                                                      i32, i32, i64, i64, P, P, P, P, P]
            lib.oracle_expert_scale.argtypes = [P, P, P, i32, i32, i64, P]
            lib.oracle_permute_masked.argtypes = [P, P, P, i32, i64, i32, i32, i32, i32, i32,
                                                  i64, i64, P, P, P, P, P]
            lib.oracle_combine_stage1.argtypes = [P, P, P, P, P, i32, i64, i32, i32, i32, i32,
                                                  i32, i64, P, P]
            lib.oracle_combine_stage2.argtypes = [P, P, i32, i64, i32, i32, i64, P, P]
            lib.oracle_e4m3_from_double.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_quantize_mxfp8_block.argtypes = [P, P, P]
            lib.oracle_quantize_mxfp8_block.restype = None
            lib.oracle_dispatch_pack_mxfp8.argtypes = [P, i32, i64, i32, i32, P, i64, P, P, P]
            lib.oracle_expert_scale_mxfp8.argtypes = [P, P, P, i32, i32, i64, P]
            lib.oracle_plan_placement.argtypes = [P, i32, i32, i32, P, P, P, P]
            lib.oracle_map_replicas.argtypes = [P, i32, i64, i32, i32, P, P, i32, P]
            lib.oracle_e2m1_from_double.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_from_double.restype = ctypes.c_uint8
            lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_to_double.restype = ctypes.c_double
            lib.oracle_quantize_nvfp4_block.argtypes = [P, ctypes.c_float, P, P]
            lib.oracle_quantize_nvfp4_block.restype = None
            lib.oracle_dispatch_pack_nvfp4.argtypes = [P, i32, i64, i32, i32, ctypes.c_float, P, i64,
                                                       P, P, P]
            lib.oracle_expert_scale_nvfp4.argtypes = [P, P, P, i32, i32, ctypes.c_float, i64, P]
            lib.oracle_dispatch_pack_routed.argtypes = [P, P, P, i32, i64, i32, i32, i32, P, i64,
                                                        P, P, P, P, P]
            lib.oracle_routed_expert_stage1.argtypes = [P, P, P, P, i32, i64, i32, i32, i32, i32,
                                                        i32, P, P, P]
            lib.oracle_combine.argtypes = [P, P, P, i32, i64, i32, i32, P]
            for f in ("oracle_route_topk", "oracle_dispatch_layout", "oracle_dispatch_pack",
                      "oracle_permute_to_experts", "oracle_expert_scale", "oracle_combine",
                      "oracle_permute_masked", "oracle_combine_stage1",
                      "oracle_combine_stage2", "oracle_dispatch_pack_mxfp8",
                      "oracle_expert_scale_mxfp8", "oracle_plan_placement",
                      "oracle_map_replicas", "oracle_dispatch_pack_routed",
                      "oracle_routed_expert_stage1", "oracle_dispatch_pack_nvfp4",
                      "oracle_expert_scale_nvfp4"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


def bf16_to_double(b: int) -> float:
    return _load().oracle_bf16_to_double(int(b))


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def expected_copies(E: int, G: int, k: int) -> float:
    """Mean number of destination GPUs per token under uniform top-k routing."""
    return _load().oracle_expected_copies(E, G, k)


def route_topk(logits: np.ndarray, k: int):
    """logits float32 [..., E] -> (ids int32 [..., k], w float64 [..., k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    E = logits.shape[-1]
    lead = logits.shape[:-1]
    N = int(np.prod(lead)) if lead else 1
    ids = np.empty(lead + (k,), dtype=np.int32)
    w = np.empty(lead + (k,), dtype=np.float64)
    _check(_load().oracle_route_topk(_p(logits), N, E, k, _p(ids), _p(w)), "route_topk")
    return ids, w


def dispatch_layout(ids: np.ndarray, E: int, P: int) -> dict:
    """ids int32 [S, T, k] -> expert_counts, expert_rank, part_counts, part_offsets, token_slot, status."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    S, T, k = ids.shape
    out = {
        "expert_counts": np.empty((S, E), np.int32),
        "expert_rank": np.empty((S, T, k), np.int32),
        "part_counts": np.empty((S, P), np.int32),
        "part_offsets": np.empty((S, P + 1), np.int32),
        "token_slot": np.empty((S, T, P), np.int32),
    }
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_dispatch_layout(_p(ids), S, T, k, E, P, _p(out["expert_counts"]),
                                          _p(out["expert_rank"]), _p(out["part_counts"]), _p(out["part_offsets"]),
                                          _p(out["token_slot"]), _p(st)), "dispatch_layout")
    out["status"] = int(st[0])
    return out


def dispatch_pack(x: np.ndarray, token_slot: np.ndarray, cap_send: int, send: np.ndarray | None = None):
    """x uint16 [S, T, H] (bf16 bits), token_slot [S, T, P] -> (send [S, cap, H], send_src [S, cap], status).

    Rows of `send` that no slot writes keep the contents of the `send` passed
    in (zeros if none is given).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, T, H = x.shape
    P = token_slot.shape[2]
    if send is None:
        send = np.zeros((S, cap_send, H), np.uint16)
    send_src = np.empty((S, cap_send), np.int32)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_dispatch_pack(_p(x), S, T, H, P, _p(token_slot), cap_send, _p(send),
                                        _p(send_src), _p(st)), "dispatch_pack")
    return send, send_src, int(st[0])


def permute_to_experts(send: np.ndarray, token_slot: np.ndarray, ids: np.ndarray, E: int,
                       recv_part: int = -1, align: int = 1, cap_recv: int | None = None,
                       recv: np.ndarray | None = None) -> dict:
    """Receiver permute; returns recv, expert_offsets, pair_row, recv_pair, status.

    Rows of `recv` at or beyond min(expert_offsets[E], cap_recv) keep the
    contents of the `recv` passed in (zeros if none is given).
    """
    send = np.ascontiguousarray(send, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    S, cap_send, H = send.shape
    _, T, P = token_slot.shape
    k = ids.shape[2]
    if cap_recv is None:
        cap_recv = S * T * k + E * (align - 1)
    if recv is None:
        recv = np.zeros((cap_recv, H), np.uint16)
    out = {
        "recv": recv,
        "expert_offsets": np.empty(E + 1, np.int32),
        "pair_row": np.empty((S, T, k), np.int32),
        "recv_pair": np.empty(cap_recv, np.int32),
    }
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_permute_to_experts(
        _p(send), _p(token_slot), _p(ids), S, T, k, E, P, H, recv_part, align, cap_send,
        cap_recv, _p(recv), _p(out["expert_offsets"]), _p(out["pair_row"]),
        _p(out["recv_pair"]), _p(st)), "permute_to_experts")
    out["status"] = int(st[0])
    return out


def permute_masked(send: np.ndarray, token_slot: np.ndarray, ids: np.ndarray, E: int,
                   recv_part: int, block_rows: int, recv: np.ndarray | None = None) -> dict:
    """Masked receive layout: one block of block_rows rows per expert of the receiving set.

    Returns recv [blocks*block_rows, H], masked_counts [blocks], pair_row, recv_pair, status.
    Rows past each block's count keep the contents of the `recv` passed in.
    """
    send = np.ascontiguousarray(send, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    S, cap_send, H = send.shape
    _, T, P = token_slot.shape
    k = ids.shape[2]
    nb = E if recv_part < 0 else E // P
    if recv is None:
        recv = np.zeros((nb * block_rows, H), np.uint16)
    out = {"recv": recv, "masked_counts": np.empty(nb, np.int32),
           "pair_row": np.empty((S, T, k), np.int32),
           "recv_pair": np.empty(nb * block_rows, np.int32)}
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_permute_masked(
        _p(send), _p(token_slot), _p(ids), S, T, k, E, P, H, recv_part, block_rows, cap_send,
        _p(recv), _p(out["masked_counts"]), _p(out["pair_row"]), _p(out["recv_pair"]), _p(st)),
        "permute_masked")
    out["status"] = int(st[0])
    return out


def expert_scale(recv: np.ndarray, expert_offsets: np.ndarray, scale: np.ndarray,
                 y: np.ndarray | None = None) -> np.ndarray:
    """Stand-in expert: y[row] = bf16(recv[row] * scale[expert of row])."""
    recv = np.ascontiguousarray(recv, dtype=np.uint16)
    expert_offsets = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    cap, H = recv.shape
    E = scale.shape[0]
    if y is None:
        y = np.zeros_like(recv)
    _check(_load().oracle_expert_scale(_p(recv), _p(expert_offsets), _p(scale), E, H, cap, _p(y)),
           "expert_scale")
    return y


def combine(y: np.ndarray, pair_row: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[s, t] = bf16(sum_j w[s,t,j] * y[pair_row[s,t,j]]) with a double sum; uint16 [S, T, H]."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    pair_row = np.ascontiguousarray(pair_row, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    S, T, k = pair_row.shape
    H = y.shape[1]
    out = np.empty((S, T, H), np.uint16)
    _check(_load().oracle_combine(_p(y), _p(pair_row), _p(w), S, T, k, H, _p(out)), "combine")
    return out


def combine_stage1(y: np.ndarray, pair_row: np.ndarray, w: np.ndarray, ids: np.ndarray,
                   token_slot: np.ndarray, E: int, cap_send: int, recv_part: int = -1,
                   ret: np.ndarray | None = None):
    """Stage 1 of the split combine: one pre-added bf16 row per (token, partition) slot.

    Returns (ret [S, cap_send, H], status); rows without a slot keep the `ret` passed in.
    """
    y = np.ascontiguousarray(y, dtype=np.uint16)
    pair_row = np.ascontiguousarray(pair_row, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, T, k = pair_row.shape
    P = token_slot.shape[2]
    H = y.shape[1]
    if ret is None:
        ret = np.zeros((S, cap_send, H), np.uint16)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_combine_stage1(_p(y), _p(pair_row), _p(w), _p(ids), _p(token_slot), S, T,
                                         k, E, P, H, recv_part, cap_send, _p(ret), _p(st)),
           "combine_stage1")
    return ret, int(st[0])


def combine_stage2(ret: np.ndarray, token_slot: np.ndarray):
    """Stage 2: out[s, t] = bf16(sum of the token's returned rows), double sum; (out, status)."""
    ret = np.ascontiguousarray(ret, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, cap_send, H = ret.shape
    _, T, P = token_slot.shape
    out = np.empty((S, T, H), np.uint16)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_combine_stage2(_p(ret), _p(token_slot), S, T, P, H, cap_send, _p(out),
                                         _p(st)), "combine_stage2")
    return out, int(st[0])


def e4m3_from_double(v: float) -> int:
    return int(_load().oracle_e4m3_from_double(float(v)))


def e4m3_to_double(b: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(b)))


def quantize_mxfp8(row: np.ndarray):
    """bf16 bits [H] (H % 32 == 0) -> (codes uint8 [H], scales uint8 [H/32])."""
    row = np.ascontiguousarray(row, dtype=np.uint16)
    H = row.shape[0]
    codes = np.empty(H, np.uint8)
    scales = np.empty(H // 32, np.uint8)
    lib = _load()
    for b in range(H // 32):
        lib.oracle_quantize_mxfp8_block(
            ctypes.c_void_p(row.ctypes.data + 64 * b), ctypes.c_void_p(codes.ctypes.data + 32 * b),
            ctypes.c_void_p(scales.ctypes.data + b))
    return codes, scales


def dispatch_pack_mxfp8(x: np.ndarray, token_slot: np.ndarray, cap_send: int,
                        send_q: np.ndarray | None = None):
    """Pack with MXFP8 records -> (send_q uint8 [S, cap, H + H/32], send_src, status).

    A record is the H E4M3 codes followed by the H/32 E8M0 block scales.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, T, H = x.shape
    P = token_slot.shape[2]
    if send_q is None:
        send_q = np.zeros((S, cap_send, H + H // 32), np.uint8)
    send_src = np.empty((S, cap_send), np.int32)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_dispatch_pack_mxfp8(_p(x), S, T, H, P, _p(token_slot), cap_send,
                                              _p(send_q), _p(send_src), _p(st)),
           "dispatch_pack_mxfp8")
    return send_q, send_src, int(st[0])


def expert_scale_mxfp8(recv_q: np.ndarray, expert_offsets: np.ndarray, scale: np.ndarray,
                       y: np.ndarray | None = None) -> np.ndarray:
    """Dequantizing stand-in expert: recv_q uint8 [cap, H + H/32] -> y bf16 bits [cap, H].

    Rows outside every expert run keep the contents of the `y` passed in (zeros if none).
    """
    recv_q = np.ascontiguousarray(recv_q, dtype=np.uint8)
    cap, rb = recv_q.shape
    H = rb * 32 // 33
    assert H + H // 32 == rb
    E = expert_offsets.shape[0] - 1
    if y is None:
        y = np.zeros((cap, H), np.uint16)
    _check(_load().oracle_expert_scale_mxfp8(_p(recv_q), _p(np.ascontiguousarray(expert_offsets, np.int32)),
                                             _p(np.ascontiguousarray(scale, np.float32)), E, H, cap, _p(y)),
           "expert_scale_mxfp8")
    return y


def plan_placement(load: np.ndarray, P: int, R: int) -> dict:
    """Placement by load plus redundant copies of the busiest experts.

    load int64 [E] (pairs per logical expert in a past batch), P partitions, R
    spare slots per partition.  Returns copy_offsets [E+1], copy_slots
    [n_copies] (physical slots, original first), slot_expert [P*(E/P+R)]
    (-1 = empty), part_load [P], Lp = E/P + R and E_phys = P*Lp.
    """
    load = np.ascontiguousarray(load, dtype=np.int64)
    E = load.shape[0]
    Lp = E // P + R
    co = np.empty(E + 1, np.int32)
    cs = np.full(E + P * R, -1, np.int32)
    se = np.empty(P * Lp, np.int32)
    pl = np.empty(P, np.int64)
    _check(_load().oracle_plan_placement(_p(load), E, P, R, _p(co), _p(cs), _p(se), _p(pl)),
           "plan_placement")
    return {"copy_offsets": co, "copy_slots": cs[:co[-1]].copy(), "slot_expert": se,
            "part_load": pl, "Lp": Lp, "E_phys": P * Lp}


def map_replicas(ids: np.ndarray, E: int, copy_offsets: np.ndarray, copy_slots: np.ndarray,
                 E_phys: int) -> np.ndarray:
    """Physical expert of every pair: the r-th pair of e from a source -> copy r mod n_e."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    S, T, k = ids.shape
    phys = np.empty_like(ids)
    _check(_load().oracle_map_replicas(_p(ids), S, T, k, E,
                                       _p(np.ascontiguousarray(copy_offsets, np.int32)),
                                       _p(np.ascontiguousarray(copy_slots, np.int32)), E_phys,
                                       _p(phys)), "map_replicas")
    return phys


def dispatch_pack_routed(x: np.ndarray, ids: np.ndarray, w: np.ndarray, token_slot: np.ndarray,
                         cap_send: int, send: np.ndarray | None = None):
    """Pack with the routing payload -> (send, send_src, send_ids [S,cap,k], send_w [S,cap,k], status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, T, H = x.shape
    k = ids.shape[2]
    P = token_slot.shape[2]
    if send is None:
        send = np.zeros((S, cap_send, H), np.uint16)
    send_src = np.empty((S, cap_send), np.int32)
    send_ids = np.empty((S, cap_send, k), np.int32)
    send_w = np.empty((S, cap_send, k), np.float32)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_dispatch_pack_routed(_p(x), _p(ids), _p(w), S, T, H, k, P, _p(token_slot),
                                               cap_send, _p(send), _p(send_src), _p(send_ids),
                                               _p(send_w), _p(st)), "dispatch_pack_routed")
    return send, send_src, send_ids, send_w, int(st[0])


def routed_expert_stage1(send: np.ndarray, send_ids: np.ndarray, send_w: np.ndarray,
                         part_offsets: np.ndarray, E: int, recv_part: int = -1,
                         scale: np.ndarray | None = None, ret: np.ndarray | None = None):
    """Routed stand-in expert + stage-1 pre-add per row -> (ret [S, cap, H], status).

    Rows outside the receiving partitions' regions keep the `ret` passed in (zeros if none).
    """
    send = np.ascontiguousarray(send, dtype=np.uint16)
    send_ids = np.ascontiguousarray(send_ids, dtype=np.int32)
    send_w = np.ascontiguousarray(send_w, dtype=np.float32)
    part_offsets = np.ascontiguousarray(part_offsets, dtype=np.int32)
    S, cap, H = send.shape
    k = send_ids.shape[2]
    P = part_offsets.shape[1] - 1
    if ret is None:
        ret = np.zeros_like(send)
    sc = None if scale is None else np.ascontiguousarray(scale, dtype=np.float32)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_routed_expert_stage1(_p(send), _p(send_ids), _p(send_w), _p(part_offsets),
                                               S, cap, k, E, P, H, recv_part,
                                               None if sc is None else _p(sc), _p(ret), _p(st)),
           "routed_expert_stage1")
    return ret, int(st[0])


def e2m1_from_double(v: float) -> int:
    return int(_load().oracle_e2m1_from_double(float(v)))


def e2m1_to_double(c: int) -> float:
    return float(_load().oracle_e2m1_to_double(int(c)))


def quantize_nvfp4(row: np.ndarray, g: float = 1.0):
    """bf16 bits [H] (H % 16 == 0), tensor scale g -> (codes uint8 [H/2], two per byte,
    scales uint8 [H/16])."""
    row = np.ascontiguousarray(row, dtype=np.uint16)
    H = row.shape[0]
    codes = np.empty(H // 2, np.uint8)
    scales = np.empty(H // 16, np.uint8)
    lib = _load()
    for b in range(H // 16):
        lib.oracle_quantize_nvfp4_block(
            ctypes.c_void_p(row.ctypes.data + 32 * b), float(g),
            ctypes.c_void_p(codes.ctypes.data + 8 * b),
            ctypes.c_void_p(scales.ctypes.data + b))
    return codes, scales


def dispatch_pack_nvfp4(x: np.ndarray, token_slot: np.ndarray, cap_send: int, g: float = 1.0,
                        send_q: np.ndarray | None = None):
    """Pack with NVFP4 records -> (send_q uint8 [S, cap, H/2 + H/16], send_src, status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    token_slot = np.ascontiguousarray(token_slot, dtype=np.int32)
    S, T, H = x.shape
    P = token_slot.shape[2]
    if send_q is None:
        send_q = np.zeros((S, cap_send, H // 2 + H // 16), np.uint8)
    send_src = np.empty((S, cap_send), np.int32)
    st = np.zeros(1, np.uint32)
    _check(_load().oracle_dispatch_pack_nvfp4(_p(x), S, T, H, P, float(g), _p(token_slot), cap_send,
                                              _p(send_q), _p(send_src), _p(st)),
           "dispatch_pack_nvfp4")
    return send_q, send_src, int(st[0])


def expert_scale_nvfp4(recv_q: np.ndarray, expert_offsets: np.ndarray, scale: np.ndarray,
                       g: float = 1.0, y: np.ndarray | None = None) -> np.ndarray:
    """Dequantizing stand-in expert: recv_q uint8 [cap, H/2 + H/16] -> y bf16 bits [cap, H]."""
    recv_q = np.ascontiguousarray(recv_q, dtype=np.uint8)
    cap, rb = recv_q.shape
    H = rb * 16 // 9
    assert H // 2 + H // 16 == rb
    E = expert_offsets.shape[0] - 1
    if y is None:
        y = np.zeros((cap, H), np.uint16)
    _check(_load().oracle_expert_scale_nvfp4(_p(recv_q), _p(np.ascontiguousarray(expert_offsets, np.int32)),
                                             _p(np.ascontiguousarray(scale, np.float32)), E, H, float(g),
                                             cap, _p(y)),
           "expert_scale_nvfp4")
    return y


def run_path(x: np.ndarray, logits: np.ndarray, E: int, k: int, P: int, scales: np.ndarray | None,
             recv_part: int = -1, align: int = 1) -> dict:
    """The whole path: route -> layout -> pack -> permute -> stand-in expert -> combine.

    `scales` None means the identity expert (combine reads the permuted rows).
    """
    S, T, H = x.shape
    ids, w64 = route_topk(logits, k)
    w = w64.astype(np.float32)
    lay = dispatch_layout(ids, E, P)
    cap_send = T * min(k, P)
    send, send_src, st_pack = dispatch_pack(x, lay["token_slot"], cap_send)
    per = permute_to_experts(send, lay["token_slot"], ids, E, recv_part=recv_part, align=align)
    y = per["recv"] if scales is None else expert_scale(per["recv"], per["expert_offsets"], scales)
    out = combine(y, per["pair_row"], w)
    return {"ids": ids, "w": w64, "layout": lay, "send": send, "send_src": send_src,
            "permute": per, "y": y, "out": out,
            "status": lay["status"] | st_pack | per["status"]}
