"""C ABI checks that need no GPU: the library loads, exports every function that
include/moe_route.h declares, and its host-side validation rejects bad
arguments before anything is enqueued (so these calls never reach CUDA)."""
import ctypes
import os
import re

import pytest

import combine_moe_route_06_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_route.h")


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)) - {"MOE_STATUS_BIT"})


def test_header_declares_the_path():
    names = declared_functions()
    for f in ("moe_route_topk", "moe_dispatch_layout", "moe_dispatch_pack",
              "moe_permute_to_experts", "moe_combine", "moe_workspace_bytes"):
        assert f in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.moe_version() >= 10000
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(2) == b"capacity exceeded"


def test_workspace_bytes(lib):
    assert m.moe_workspace_bytes(1, 4096, 6, 384, 8) > 0
    assert m.moe_workspace_bytes(1, 4096, 6, 384, 8) % 256 == 0
    assert m.moe_workspace_bytes(1, 8192, 6, 384, 8) >= m.moe_workspace_bytes(1, 4096, 6, 384, 8)
    assert m.moe_workspace_bytes(1, 0, 6, 384, 8) > 0
    assert m.moe_workspace_bytes(1, 16, 6, 385, 8) == 0       # E % P != 0
    assert m.moe_workspace_bytes(0, 16, 6, 384, 8) == 0       # S < 1


def test_kernel_count_queries(lib):
    """The permute's form depends only on S*E (the map runs inside the copy while S*E + 2E + 1
    counts fit in 48 KiB); invalid sizes give -1 for both queries without touching a device."""
    assert lib.moe_permute_to_experts_kernels(1, 4096, 6, 384, 8) == 1
    assert lib.moe_permute_to_experts_kernels(8, 4096, 6, 384, 8) == 1
    assert lib.moe_permute_to_experts_kernels(9, 64, 8, 1024, 8) == 1      # 45,060 bytes: fits
    assert lib.moe_permute_to_experts_kernels(10, 64, 8, 1024, 8) == 2     # 49,156 bytes: not
    assert lib.moe_permute_to_experts_kernels(1, 16, 6, 385, 8) == -1     # E % P != 0
    assert lib.moe_permute_to_experts_kernels(0, 16, 6, 384, 8) == -1     # S < 1
    assert lib.moe_dispatch_layout_kernels(1, 16, 33, 384, 8) == -1       # k > 32
    assert lib.moe_dispatch_layout_kernels(1, -1, 6, 384, 8) == -1        # T < 0


FAKE = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced: the calls are rejected first
FAKE_MIS = ctypes.c_void_p((1 << 20) + 2)
NULL = ctypes.c_void_p(0)
ST = ctypes.c_void_p(0)


def _msg(lib):
    return lib.moe_last_error_message().decode()


@pytest.mark.parametrize("args,needle", [
    ((FAKE, 0, 4, 16, 2, FAKE, FAKE, ST), "S=0"),
    ((FAKE, 1, -1, 16, 2, FAKE, FAKE, ST), "T=-1"),
    ((FAKE, 1, 4, 16, 0, FAKE, FAKE, ST), "k=0"),
    ((FAKE, 1, 4, 16, 33, FAKE, FAKE, ST), "k=33"),
    ((FAKE, 1, 4, 2, 3, FAKE, FAKE, ST), "E=2"),
    ((FAKE, 1, 4, 2048, 3, FAKE, FAKE, ST), "E=2048"),
    ((NULL, 1, 4, 16, 2, FAKE, FAKE, ST), "null pointer `logits`"),
    ((FAKE, 1, 4, 16, 2, FAKE_MIS, FAKE, ST), "`topk_ids` is not 4-byte aligned"),
])
def test_route_rejects(lib, args, needle):
    assert lib.moe_route_topk(*args) == m.MOE_ERR_INVALID_ARG
    assert needle in _msg(lib)


def test_layout_rejects(lib):
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    good = [FAKE, 1, 64, 2, 16, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, FAKE, ST]
    bad = list(good)
    bad[5] = 3                                         # E % P != 0
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "multiple of P" in _msg(lib)
    bad = list(good)
    bad[5] = 64
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "P=64" in _msg(lib)
    bad = list(good)
    bad[12] = ws - 1                                   # workspace too small
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "ws_bytes" in _msg(lib)
    bad = list(good)
    bad[11] = ctypes.c_void_p((1 << 20) + 16)          # workspace not 256-byte aligned
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "`ws`" in _msg(lib)
    bad = list(good)
    bad[10] = NULL
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "token_slot" in _msg(lib)
    bad = list(good)
    bad[7] = NULL
    assert lib.moe_dispatch_layout(*bad) == m.MOE_ERR_INVALID_ARG and "expert_rank" in _msg(lib)


def test_pack_rejects(lib):
    good = [FAKE, 1, 64, 256, 4, FAKE, FAKE, 128, FAKE, FAKE, FAKE, ST]
    bad = list(good)
    bad[3] = 100                                       # H not a multiple of 8
    assert lib.moe_dispatch_pack(*bad) == m.MOE_ERR_INVALID_ARG and "H=100" in _msg(lib)
    bad = list(good)
    bad[0] = ctypes.c_void_p((1 << 20) + 8)            # rows must be 16-byte aligned
    assert lib.moe_dispatch_pack(*bad) == m.MOE_ERR_INVALID_ARG and "16-byte" in _msg(lib)
    bad = list(good)
    bad[7] = -1
    assert lib.moe_dispatch_pack(*bad) == m.MOE_ERR_INVALID_ARG and "cap_send" in _msg(lib)


def test_permute_rejects(lib):
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    good = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 2, 16, 4, 256, -1, 1, 128, 128, FAKE, FAKE, FAKE,
            FAKE, FAKE, ws, FAKE, ST]
    for idx, val, needle in ((11, 4, "recv_part"), (11, -2, "recv_part"), (12, 0, "align"),
                             (12, 2048, "align"), (14, -3, "capacities"), (10, 4, "H=4"),
                             (4, NULL, "expert_rank")):
        bad = list(good)
        bad[idx] = val
        assert lib.moe_permute_to_experts(*bad) == m.MOE_ERR_INVALID_ARG, needle
        assert needle in _msg(lib)


def test_combine_and_expert_scale_reject(lib):
    assert lib.moe_combine(FAKE, 64, FAKE, FAKE, 1, 8, 2, 12, FAKE, NULL, ST) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(NULL, 64, FAKE, FAKE, 1, 8, 2, 16, FAKE, NULL, ST) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(FAKE, -1, FAKE, FAKE, 1, 8, 2, 16, FAKE, NULL, ST) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_scale(FAKE, FAKE, FAKE, 0, 16, 4, FAKE, ST) == m.MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    # the product path has no fallback: a missing library is an error, not a CPU path
    monkeypatch.setattr(m._build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(m.MoeLibraryMissing):
        m.load_library()


def _rejects(fn, args, needle):
    assert fn(*args) == m.MOE_ERR_INVALID_ARG, needle
    assert needle in _msg(lib_ := m.load_library()), (_msg(lib_), needle)


def test_next_entry_points_reject(lib):
    # masked permute: block_rows must not be negative
    _rejects(lib.moe_permute_to_experts_masked,
             [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 2, 16, 4, 256, -1, -1, 128, FAKE, FAKE, FAKE, FAKE,
              FAKE, ST], "block_rows")
    # two-stage combine: receiving partition out of range
    _rejects(lib.moe_combine_stage1,
             [FAKE, 64, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 16, 4, 256, 4, 64, FAKE, FAKE, ST], "recv_part")
    _rejects(lib.moe_combine_stage2, [FAKE, FAKE, 1, 8, 4, 256, 7, 64, FAKE, FAKE, ST], "recv_part")
    # quantized packs: widths the records need, and a positive tensor scale
    _rejects(lib.moe_dispatch_pack_mxfp8, [FAKE, 1, 8, 96, 4, FAKE, FAKE, 16, FAKE, FAKE, FAKE, ST],
             "H=96")
    _rejects(lib.moe_expert_scale_mxfp8, [FAKE, FAKE, FAKE, 16, 160, 8, FAKE, ST], "H=160")
    _rejects(lib.moe_dispatch_pack_nvfp4,
             [FAKE, 1, 8, 384, 4, ctypes.c_float(1.0), FAKE, FAKE, 16, FAKE, FAKE, FAKE, ST], "H=384")
    _rejects(lib.moe_dispatch_pack_nvfp4,
             [FAKE, 1, 8, 512, 4, ctypes.c_float(0.0), FAKE, FAKE, 16, FAKE, FAKE, FAKE, ST],
             "global_scale")
    _rejects(lib.moe_expert_scale_nvfp4,
             [FAKE, FAKE, FAKE, 16, 512, ctypes.c_float(-2.0), 8, FAKE, ST], "global_scale")
    # routed payload: k and the receiving partition
    _rejects(lib.moe_dispatch_pack_routed,
             [FAKE, FAKE, FAKE, 1, 8, 256, 33, 4, FAKE, FAKE, 16, FAKE, FAKE, FAKE, FAKE, FAKE, ST], "k=33")
    _rejects(lib.moe_routed_expert_stage1,
             [FAKE, FAKE, FAKE, FAKE, 1, 8, 16, 2, 16, 4, 256, 9, NULL, FAKE, FAKE, ST], "recv_part")
    # layout over a placement: slots per partition and the copy count
    ws = lib.moe_workspace_bytes_mapped(1, 64, 2, 16, 4, 5)
    assert ws > 0 and lib.moe_workspace_bytes_mapped(1, 64, 2, 16, 4, 3) == 0   # Lp < E/P
    good = [FAKE, 1, 64, 2, 16, 4, 5, FAKE, FAKE, 18, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws,
            FAKE, ST]
    bad = list(good)
    bad[6] = 3
    _rejects(lib.moe_dispatch_layout_mapped, bad, "Lp=3")
    bad = list(good)
    bad[9] = 40
    _rejects(lib.moe_dispatch_layout_mapped, bad, "n_copies=40")
    bad = list(good)
    bad[17] = ws - 1
    _rejects(lib.moe_dispatch_layout_mapped, bad, "ws_bytes")


def test_dispatch_rejects(lib):
    """moe_dispatch checks the union of the four calls' arguments on the host."""
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    good = [FAKE, FAKE, 1, 64, 256, 16, 2, 4, -1, 1, 128, 128] + [FAKE] * 13 + [FAKE, ws, FAKE, ST]
    for idx, val, needle in ((4, 100, "H=100"), (8, 4, "recv_part"), (9, 0, "align"),
                             (10, -1, "capacities"), (7, 3, "multiple of P"), (6, 33, "k=33"),
                             (0, NULL, "`logits`"), (1, ctypes.c_void_p((1 << 20) + 8), "`x`"),
                             (19, NULL, "`send`"), (21, NULL, "`recv`"), (26, ws - 1, "ws_bytes"),
                             (25, ctypes.c_void_p((1 << 20) + 16), "`ws`")):
        bad = list(good)
        bad[idx] = val
        _rejects(lib.moe_dispatch, bad, needle)
    assert lib.moe_dispatch_kernels(1, 16, 6, 385, 8) == -1     # E % P != 0
    assert lib.moe_dispatch_kernels(1, -1, 6, 384, 8) == -1     # T < 0


def test_dispatch_quantized_rejects(lib):
    """moe_dispatch_quantized checks its format, the row width the format needs and
    the NVFP4 tensor scale on the host, besides moe_dispatch's arguments."""
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    f = ctypes.c_float
    good = ([FAKE, FAKE, 1, 64, 512, 16, 2, 4, 1, f(1.0), -1, 1, 128, 128] + [FAKE] * 13
            + [FAKE, ws, FAKE, ST])
    for idx, val, needle in ((8, 3, "format"), (4, 256, "multiple of 512"), (7, 3, "multiple of P"),
                             (10, 4, "recv_part"), (0, NULL, "`logits`"), (21, NULL, "`send_q`"),
                             (28, ws - 1, "ws_bytes")):
        bad = list(good)
        bad[idx] = val
        _rejects(lib.moe_dispatch_quantized, bad, needle)
    nv = list(good)
    nv[8] = 2
    nv[4] = 384                                         # NVFP4 needs H % 256 == 0
    _rejects(lib.moe_dispatch_quantized, nv, "multiple of 256")
    nv[4] = 256
    nv[9] = f(0.0)
    _rejects(lib.moe_dispatch_quantized, nv, "global_scale")
    assert lib.moe_dispatch_quantized_kernels(1, 16, 6, 385, 8) == -1


def test_dispatch_pack_permute_rejects(lib):
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    good = [FAKE] * 6 + [1, 64, 2, 16, 4, 256, -1, 1, 128, 128] + [FAKE] * 7 + [ws, FAKE, ST]
    for idx, val, needle in ((11, 100, "H=100"), (12, 4, "recv_part"), (13, 0, "align"),
                             (14, -1, "capacities"), (0, NULL, "`x`"), (16, NULL, "`send`"),
                             (23, ws - 1, "ws_bytes")):
        bad = list(good)
        bad[idx] = val
        _rejects(lib.moe_dispatch_pack_permute, bad, needle)
    assert lib.moe_dispatch_pack_permute_kernels(1, 16, 6, 385, 8) == -1
    assert lib.moe_dispatch_pack_permute_kernels(1, 0, 6, 384, 8) == 2
    assert lib.moe_dispatch_pack_permute_kernels(1, 16, 6, 384, 8) == 1


def test_dispatch_pack_permute_masked_rejects(lib):
    good = [FAKE] * 6 + [1, 64, 2, 16, 4, 256, -1, 64, 128] + [FAKE] * 6 + [FAKE, ST]
    for idx, val, needle in ((11, 100, "H=100"), (12, 4, "recv_part"), (13, -1, "block_rows"),
                             (14, -1, "cap_send"), (0, NULL, "`x`"), (18, NULL, "`masked_counts`")):
        bad = list(good)
        bad[idx] = val
        _rejects(lib.moe_dispatch_pack_permute_masked, bad, needle)
    assert lib.moe_dispatch_pack_permute_masked_kernels(1, 16, 6, 384, 8, 8) == -1   # recv_part
    assert lib.moe_dispatch_pack_permute_masked_kernels(1, 0, 6, 384, 8, -1) == 2
    assert lib.moe_dispatch_pack_permute_masked_kernels(1, 16, 6, 384, 8, -1) == 1
    assert lib.moe_dispatch_pack_permute_masked_kernels(12, 16, 8, 1024, 8, -1) == 3


def test_dispatch_masked_rejects(lib):
    """moe_dispatch_masked checks moe_dispatch's arguments with the masked layout's
    block_rows and masked_counts in place of align, cap_recv and expert_offsets."""
    ws = m.moe_workspace_bytes(1, 64, 2, 16, 4)
    good = [FAKE, FAKE, 1, 64, 256, 16, 2, 4, -1, 64, 128] + [FAKE] * 13 + [FAKE, ws, FAKE, ST]
    for idx, val, needle in ((4, 100, "H=100"), (8, 4, "recv_part"), (9, -1, "block_rows"),
                             (10, -1, "cap_send"), (7, 3, "multiple of P"), (0, NULL, "`logits`"),
                             (18, NULL, "`send`"), (21, NULL, "`masked_counts`"),
                             (25, ws - 1, "ws_bytes")):
        bad = list(good)
        bad[idx] = val
        _rejects(lib.moe_dispatch_masked, bad, needle)
    assert lib.moe_dispatch_masked_kernels(1, 16, 6, 384, 8, 8) == -1      # recv_part
    assert lib.moe_dispatch_masked_kernels(1, 16, 6, 385, 8, -1) == -1     # E % P != 0
    assert lib.moe_dispatch_masked_kernels(1, -1, 6, 384, 8, -1) == -1     # T < 0
