"""The C-ABI library loads on a host without a GPU and exports every declared
symbol; host-side validation rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from mxfp4_mixture_experts_top_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_mxfp4.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTS) == names


def test_abi_version_and_status_strings(lib):
    assert moe.abi_version() == 4
    for s in range(8):
        assert lib.moe_status_string(s)
    assert b"unknown" in lib.moe_status_string(99)


def test_rows_capacity():
    assert moe.rows_capacity(37, 32, 6, 16) == 222 + 32 * 15
    assert moe.rows_capacity(8, 256, 6, 16) == 48 + 48 * 15
    assert moe.rows_capacity(8191, 256, 6, 128) == 49146 + 256 * 127
    assert moe.rows_capacity(0, 256, 6, 16) == 0


def test_packed_and_workspace_sizes():
    d = moe.make_desc(8, 4096, 2048, 256, 6, 16)
    # packed bytes equal the canonical MXFP4 bytes (nibbles + scales), only reordered
    assert moe.packed_bytes(d) == 256 * (2 * 2048 * 4096 // 2 + 2 * 2048 * 4096 // 32
                                         + 4096 * 2048 // 2 + 4096 * 2048 // 32)
    lay = moe.workspace_layout(d)
    R = moe.rows_capacity(8, 256, 6, 16)
    # x and SiLU(gate)*up as 2 MXFP8 terms each, with one scale byte per 32 elements
    assert lay["xq"] >= 256 and lay["xs"] >= lay["xq"] + 2 * R * 4096
    RS = (R + 3) // 4 * 4                      # scale words per term and slab: rows rounded up to 4
    assert lay["hq"] >= lay["xs"] + 2 * RS * 4096 // 32
    assert lay["hs"] >= lay["hq"] + 2 * R * 2048
    assert lay["staging"] >= lay["hs"] + 2 * RS * 2048 // 32
    assert lay["total"] >= lay["staging"] + 48 * 4096 * 4
    assert moe.workspace_bytes(d) == lay["total"]
    assert all(v % 256 == 0 for v in lay.values())


@pytest.mark.parametrize("T,H,I,E,k,bm,code", [
    (8, 4096, 2048, 256, 7, 16, 0),     # valid
    (8, 4096, 2048, 256, 0, 16, 1),     # k < 1
    (8, 4096, 2048, 4, 6, 16, 1),       # k > E
    (-1, 4096, 2048, 256, 6, 16, 1),    # T < 0
    (8, 4000, 2048, 256, 6, 16, 2),     # H not a multiple of 128
    (8, 4096, 2000, 256, 6, 16, 2),     # I not a multiple of 128
    (8, 4096, 2048, 2048, 6, 16, 2),    # E > 1024
    (8, 4096, 2048, 256, 6, 24, 2),     # block_m not supported
])
def test_desc_validation(lib, T, H, I, E, k, bm, code):
    d = moe.make_desc(T, H, I, E, k, bm)
    arr = (ctypes.c_size_t * 7)()
    assert lib.moe_mxfp4_workspace_layout(ctypes.byref(d), ctypes.byref(arr)) == code


@pytest.mark.parametrize("T,H,I,E,k,flags,out,want", [
    # decode: 48 pairs over 256 experts, both GEMMs in one launch: gather, GEMMs, combine
    (8, 4096, 2048, 256, 6, 0, 0, ("tiny", True, False, 3)),
    (8, 4096, 2048, 256, 6, 1, 0, ("tiny", True, True, 2)),        # atomic combine: no combine kernel
    (8, 4096, 2048, 256, 6, 1, 1, ("tiny", True, False, 3)),       # bf16 output keeps the slot-ordered combine
    (8, 4096, 2048, 1024, 6, 0, 0, ("tiny", False, False, 4)),     # more than 512 experts: two GEMM launches
    (1, 384, 512, 8, 1, 0, 0, ("tiny", False, False, 4)),          # H not a multiple of 256
    (2, 512, 256, 8, 2, 0, 0, ("tiny", False, False, 4)),          # I below 512
    (512, 4096, 2048, 256, 6, 1, 0, ("small", False, True, 3)),    # 12 rows per expert
    (2048, 4096, 2048, 256, 6, 1, 0, ("mid", False, False, 5)),    # two-pass gather, no atomics
    (4096, 640, 512, 32, 4, 0, 0, ("large", False, False, 5)),     # H % 256 != 0: 96-row weight tiles
    (8191, 4096, 2048, 256, 6, 0, 0, ("huge", False, False, 5)),   # token-major tiles
])
def test_forward_plan(lib, T, H, I, E, k, flags, out, want):
    """The host-side plan of a forward: tile regime by rows per expert, one or two GEMM launches, the
    atomic combine, and the kernel count (no device work)."""
    d = moe.make_desc(T, H, I, E, k, 16, 0.0, flags, out)
    p = moe.forward_plan(d)
    assert (p["regime"], p["fused_gemms"], p["fast_combine"], p["launches"]) == want
    bad = moe.make_desc(T, H, I, E, k, 24)
    arr = (ctypes.c_int * 4)()
    assert lib.moe_mxfp4_forward_plan(ctypes.byref(bad), ctypes.byref(arr)) == 2
    assert lib.moe_mxfp4_forward_plan(ctypes.byref(d), None) == 1


def test_entry_points_reject_bad_arguments_without_launching(lib):
    n0 = moe.launch_count()
    null = None
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x10008)
    assert lib.moe_route(fake, 4, 8, 9, fake, fake, null, null) == 1           # k > E
    assert lib.moe_route(fake, 4, 2048, 6, fake, fake, null, null) == 2        # E > 1024
    assert lib.moe_route(null, 4, 8, 2, fake, fake, null, null) == 1           # null logits
    assert lib.moe_route(odd, 4, 8, 2, fake, fake, null, null) == 3            # misaligned
    assert lib.moe_route(fake, 0, 8, 2, fake, fake, null, null) == 0           # T == 0: no-op
    assert lib.moe_permute(fake, 4, 8, 2, 24, fake, fake, fake, fake, fake, null, null) == 2
    assert lib.moe_permute(fake, 4, 8, 2, 16, null, fake, fake, fake, fake, null, null) == 1
    d = moe.make_desc(4, 512, 256, 8, 2, 16)
    assert lib.moe_mxfp4_forward(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, fake, 16, null) == 4
    assert lib.moe_mxfp4_forward(ctypes.byref(d), odd, fake, fake, fake, fake, fake, fake, fake, 1 << 40, null) == 3
    assert lib.moe_mxfp4_forward(ctypes.byref(d), null, fake, fake, fake, fake, fake, fake, fake, 1 << 40, null) == 1
    bad_out = moe.make_desc(4, 512, 256, 8, 2, 16, 0.0, 0, 2)         # out_dtype is MOE_OUT_F32 or MOE_OUT_BF16
    assert lib.moe_mxfp4_forward(ctypes.byref(bad_out), fake, fake, fake, fake, fake, fake, fake, fake, 1 << 40,
                                 null) == 1
    bf16_out = moe.make_desc(4, 512, 256, 8, 2, 16, 0.0, 0, moe.OUT_BF16)
    assert lib.moe_mxfp4_forward(ctypes.byref(bf16_out), fake, fake, fake, fake, fake, fake, fake, fake, 16,
                                 null) == 4
    bad_flags = moe.make_desc(4, 512, 256, 8, 2, 16, 0.0, 2)          # only MOE_FLAG_FAST_COMBINE is defined
    assert lib.moe_mxfp4_forward(ctypes.byref(bad_flags), fake, fake, fake, fake, fake, fake, fake, fake, 1 << 40,
                                 null) == 1
    fast = moe.make_desc(4, 512, 256, 8, 2, 16, 0.0, moe.FLAG_FAST_COMBINE)
    assert lib.moe_mxfp4_forward(ctypes.byref(fast), fake, fake, fake, fake, fake, fake, fake, fake, 16, null) == 4
    ws16 = ctypes.c_void_p(0x10010)        # 16-byte aligned, not 256: the forward workspace needs 256
    assert lib.moe_mxfp4_forward(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, ws16, 1 << 40, null) == 3
    assert lib.moe_mxfp4_prepack(ctypes.byref(d), fake, fake, fake, fake, fake, 16, null) == 4
    assert lib.moe_mxfp4_dequant_bf16(ctypes.byref(d), fake, 2, 0, fake, null) == 1
    assert lib.moe_mxfp4_dequant_bf16(ctypes.byref(d), fake, 0, 8, fake, null) == 1
    d0 = moe.make_desc(0, 512, 256, 8, 2, 16)
    assert lib.moe_mxfp4_forward(ctypes.byref(d0), null, null, null, null, null, null, null, null, 0, null) == 0
    assert moe.launch_count() == n0


def test_selftest_bounded_wait_rejects_bad_arguments(lib):
    """Argument checks run on the host before any launch (no GPU needed)."""
    fake = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced: every call below fails its checks
    INVALID = 1
    assert lib.moe_selftest_bounded_wait(0, 0, fake, fake, None) == INVALID                # no limit
    assert lib.moe_selftest_bounded_wait(2_000_000_000, 0, fake, fake, None) == INVALID    # over 1 s
    assert lib.moe_selftest_bounded_wait(1_000_000, 1_000_000, fake, fake, None) == INVALID  # abort not before limit
    assert lib.moe_selftest_bounded_wait(1_000_000, 0, None, fake, None) == INVALID         # null error word


def test_permute_needs_no_workspace_and_cache_clears(lib):
    """moe_permute_workspace_size is 0 for every shape (scratch lives in shared memory);
    moe_clear_cache runs without a device and without launching anything."""
    n0 = moe.launch_count()
    for T, E, k, bm in [(0, 8, 2, 16), (8, 256, 6, 16), (8191, 256, 6, 128), (100000, 1024, 8, 64)]:
        assert moe.permute_workspace_size(T, E, k, bm) == 0
    moe.clear_cache()
    moe.clear_cache()
    assert moe.launch_count() == n0


def test_noalloc_error_reader_rejects_a_null_code_pointer(lib):
    assert lib.moe_mxfp4_noalloc_read_device_error(None, None) == 1
