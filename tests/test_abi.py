"""Host-side checks of the C ABI (no GPU needed).

* libpq.so builds for sm_103a and exports every function include/pq.h declares;
* every precondition is rejected on the host with the documented pq_status
  before anything is launched (these calls never reach the device, so they
  are safe on a machine without a GPU and on a GPU machine alike).
"""
import ctypes
import os
import re

import pytest

from gemm_q8_qdot_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions(headers=None):
    inc = os.path.join(ROOT, "include")
    names = set()
    for h in headers or sorted(f for f in os.listdir(inc) if f.endswith(".h")):
        text = open(os.path.join(inc, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pq_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("pq_quantize_q8_0", "pq_qdot_q8_0", "pq_qdot_q8_0_ex", "pq_quantize_qdot_q8_0",
              "pq_qdot_q8_0_blocksums", "pq_q50_qdot", "pq_q50_blocksums", "pq_check_device", "pq_strerror",
              "pq_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "pq_debug_set_tc_fault" in names and "pq_debug_set_prompt_kernel" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding.EXPORTS) <= set(declared_functions(["pq.h"]))


def test_debug_hooks_reject_bad_values(lib):
    lib.pq_debug_set_prompt_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_tc_fault.argtypes = [ctypes.c_int, ctypes.c_ulonglong]
    assert lib.pq_debug_set_prompt_kernel(2) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_debug_set_prompt_kernel(-1) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_debug_set_tc_fault(-2, 0) == binding.PQ_ERR_INVALID_ARG
    lib.pq_debug_set_small_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_small_split.argtypes = [ctypes.c_int]
    lib.pq_debug_small_kernel_config.argtypes = [ctypes.c_void_p]
    for bad in (2, -1):
        assert lib.pq_debug_set_small_kernel(bad) == binding.PQ_ERR_INVALID_ARG
    for bad in (3, 16, -1):
        assert lib.pq_debug_set_small_split(bad) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_debug_small_kernel_config(None) == binding.PQ_ERR_INVALID_ARG
    # host state only: valid values are accepted without a device
    assert lib.pq_debug_set_small_split(0) == binding.PQ_OK
    cfg = (ctypes.c_int * 4)()
    assert lib.pq_debug_small_kernel_config(cfg) == binding.PQ_OK


def test_version_and_strerror(lib):
    assert lib.pq_version() == 105
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.pq_strerror(code).decode()
    assert "unknown" in lib.pq_strerror(99).decode()


# Fake, never-dereferenced device addresses: a failed check returns before any CUDA call.
P16 = 0x10000000          # 16-byte (and 256-byte) aligned
P8 = 0x10000008           # 8-byte aligned only
P2 = 0x10000002


def qdot(lib, A=P16, AS=P16, W=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0, path=0):
    return lib.pq_qdot_q8_0_ex(A, AS, W, WS, C, M, N, K, layout, path, None)


@pytest.mark.parametrize("K", [0, -32, 16, 33, 100])
def test_bad_k(lib, K):
    assert qdot(lib, K=K) == binding.PQ_ERR_SHAPE
    assert lib.pq_qdot_q8_0(P16, P16, P16, P16, P16, 1, 1, K, None) == binding.PQ_ERR_SHAPE
    assert lib.pq_quantize_q8_0(P16, P16, P16, 1, K, None) == binding.PQ_ERR_SHAPE
    assert lib.pq_qdot_q8_0_blocksums(P16, P16, P16, 1, 1, K, 1, None) == binding.PQ_ERR_SHAPE


def test_negative_and_overflowing_sizes(lib):
    assert qdot(lib, M=-1) == binding.PQ_ERR_SHAPE
    assert qdot(lib, N=-5) == binding.PQ_ERR_SHAPE
    assert qdot(lib, M=1 << 41) == binding.PQ_ERR_SHAPE
    assert qdot(lib, M=1 << 30, N=1 << 30, K=1 << 30) == binding.PQ_ERR_SHAPE
    assert lib.pq_quantize_q8_0(P16, P16, P16, -1, 32, None) == binding.PQ_ERR_SHAPE
    assert lib.pq_quantize_q8_0(P16, P16, P16, 1 << 40, 1 << 30, None) == binding.PQ_ERR_SHAPE


def test_empty_problems_are_noops(lib):
    # M == 0 or N == 0 is valid and launches nothing, even with null pointers
    assert qdot(lib, A=None, AS=None, W=None, WS=None, C=None, M=0) == binding.PQ_OK
    assert qdot(lib, A=None, AS=None, W=None, WS=None, C=None, N=0) == binding.PQ_OK
    assert lib.pq_quantize_q8_0(None, None, None, 0, 32, None) == binding.PQ_OK
    assert lib.pq_qdot_q8_0_blocksums(None, None, None, 0, 4, 64, 1, None) == binding.PQ_OK


@pytest.mark.parametrize("which", ["A", "AS", "W", "WS", "C"])
def test_null_pointers(lib, which):
    assert qdot(lib, **{which: None}) == binding.PQ_ERR_INVALID_ARG


def test_null_quantize_and_sums(lib):
    assert lib.pq_quantize_q8_0(None, P16, P16, 1, 32, None) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_quantize_q8_0(P16, None, P16, 1, 32, None) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_quantize_q8_0(P16, P16, None, 1, 32, None) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_qdot_q8_0_blocksums(P16, P16, None, 1, 1, 32, 1, None) == binding.PQ_ERR_INVALID_ARG


def test_alignment(lib):
    assert qdot(lib, A=P8) == binding.PQ_ERR_ALIGN
    assert qdot(lib, W=P8) == binding.PQ_ERR_ALIGN
    assert qdot(lib, AS=P2) == binding.PQ_ERR_ALIGN
    assert qdot(lib, WS=P2) == binding.PQ_ERR_ALIGN
    assert qdot(lib, C=P2) == binding.PQ_ERR_ALIGN
    assert lib.pq_quantize_q8_0(P8, P16, P16, 1, 32, None) == binding.PQ_ERR_ALIGN
    assert lib.pq_quantize_q8_0(P16, P8, P16, 1, 32, None) == binding.PQ_ERR_ALIGN
    assert lib.pq_quantize_q8_0(P16, P16, P2, 1, 32, None) == binding.PQ_ERR_ALIGN
    assert lib.pq_qdot_q8_0_blocksums(P16, P16, P2, 1, 1, 32, 1, None) == binding.PQ_ERR_ALIGN


def test_unknown_codes(lib):
    assert qdot(lib, path=7) == binding.PQ_ERR_INVALID_ARG
    assert qdot(lib, layout=3) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_qdot_q8_0_blocksums(P16, P16, P16, 1, 1, 32, 9, None) == binding.PQ_ERR_INVALID_ARG


def fused(lib, x=P16, A=None, AS=None, W=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0):
    return lib.pq_quantize_qdot_q8_0(x, A, AS, W, WS, C, M, N, K, layout, None)


def test_fused_entry_checks(lib):
    assert fused(lib, K=48) == binding.PQ_ERR_SHAPE
    assert fused(lib, M=0, x=None, W=None, WS=None, C=None) == binding.PQ_OK
    assert fused(lib, x=None) == binding.PQ_ERR_INVALID_ARG
    assert fused(lib, A=P16, AS=None) == binding.PQ_ERR_INVALID_ARG     # A and AS come together
    assert fused(lib, x=P8) == binding.PQ_ERR_ALIGN
    assert fused(lib, A=P8, AS=P16) == binding.PQ_ERR_ALIGN
    assert fused(lib, layout=5) == binding.PQ_ERR_INVALID_ARG


def q50(lib, A=P16, AS=P16, W5=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0):
    return lib.pq_q50_qdot(A, AS, W5, WS, C, M, N, K, layout, None)


def test_q50_entry_checks(lib):
    assert q50(lib, K=48) == binding.PQ_ERR_SHAPE
    assert q50(lib, M=-1) == binding.PQ_ERR_SHAPE
    assert q50(lib, M=0, A=None, AS=None, W5=None, WS=None, C=None) == binding.PQ_OK
    assert q50(lib, W5=None) == binding.PQ_ERR_INVALID_ARG
    assert q50(lib, layout=2) == binding.PQ_ERR_INVALID_ARG
    assert q50(lib, A=P8) == binding.PQ_ERR_ALIGN
    assert q50(lib, W5=P2) == binding.PQ_ERR_ALIGN
    assert lib.pq_q50_blocksums(P16, P16, None, 1, 1, 32, None) == binding.PQ_ERR_INVALID_ARG
    assert lib.pq_q50_blocksums(P16, P16, P2, 1, 1, 32, None) == binding.PQ_ERR_ALIGN
    assert lib.pq_q50_blocksums(P16, P16, P16, 1, 1, 33, None) == binding.PQ_ERR_SHAPE


def fused_q50(lib, x=P16, A=None, AS=None, W5=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0):
    return lib.pq_quantize_q50_qdot(x, A, AS, W5, WS, C, M, N, K, layout, None)


def test_fused_q50_entry_checks(lib):
    assert fused_q50(lib, K=48) == binding.PQ_ERR_SHAPE
    assert fused_q50(lib, N=-2) == binding.PQ_ERR_SHAPE
    assert fused_q50(lib, M=0, x=None, W5=None, WS=None, C=None) == binding.PQ_OK
    assert fused_q50(lib, x=None) == binding.PQ_ERR_INVALID_ARG
    assert fused_q50(lib, W5=None) == binding.PQ_ERR_INVALID_ARG
    assert fused_q50(lib, A=P16, AS=None) == binding.PQ_ERR_INVALID_ARG  # A and AS come together
    assert fused_q50(lib, x=P8) == binding.PQ_ERR_ALIGN
    assert fused_q50(lib, W5=P2) == binding.PQ_ERR_ALIGN
    assert fused_q50(lib, A=P8, AS=P16) == binding.PQ_ERR_ALIGN
    assert fused_q50(lib, layout=4) == binding.PQ_ERR_INVALID_ARG


def host_step(lib, x=P16, W=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0):
    return lib.pq_quantize_qdot_q8_0_host(x, W, WS, C, M, N, K, layout, None)


def test_host_step_entry_checks(lib):
    assert host_step(lib, K=40) == binding.PQ_ERR_SHAPE
    assert host_step(lib, M=-3) == binding.PQ_ERR_SHAPE
    assert host_step(lib, M=0, x=None, W=None, WS=None, C=None) == binding.PQ_OK
    for which in ("x", "W", "WS", "C"):
        assert host_step(lib, **{which: None}) == binding.PQ_ERR_INVALID_ARG
    assert host_step(lib, W=P8) == binding.PQ_ERR_ALIGN
    assert host_step(lib, WS=P2) == binding.PQ_ERR_ALIGN
    assert host_step(lib, layout=9) == binding.PQ_ERR_INVALID_ARG


def noalloc(lib, x=P16, W=P16, WS=P16, C=P16, M=1, N=1, K=32, layout=0):
    return lib.pq_quantize_qdot_q8_0_noalloc(x, W, WS, C, M, N, K, layout, None)


def test_noalloc_rejects_the_shapes_the_allocating_step_rejects(lib):
    """The allocation-free step takes the allocating step's shape rules: an N beyond the
    size limit, or a product that overflows int64, is PQ_ERR_SHAPE on both, before any
    scratch-size check."""
    for kw in ({"N": 1 << 41}, {"M": 1, "N": 1 << 40, "K": 1 << 30}, {"K": 48}, {"N": -1}):
        assert fused(lib, **kw) == binding.PQ_ERR_SHAPE, kw
        assert noalloc(lib, **kw) == binding.PQ_ERR_SHAPE, kw
    assert noalloc(lib, M=0, x=None, W=None, WS=None, C=None) == binding.PQ_OK
    assert noalloc(lib, M=1 << 20, K=4096) == binding.PQ_ERR_SCRATCH
    assert noalloc(lib, x=None) == binding.PQ_ERR_INVALID_ARG
    assert noalloc(lib, layout=2) == binding.PQ_ERR_INVALID_ARG


def test_stream_reader_entry_checks(lib):
    """pq_debug_stream_read rejects bad arguments before anything is launched."""
    d = lib.pq_debug_stream_read
    assert d(P16, P16, 0, 32, P16, 0, None) == binding.PQ_ERR_INVALID_ARG
    assert d(P16, P16, 4, 40, P16, 0, None) == binding.PQ_ERR_INVALID_ARG
    assert d(P16, P16, 4, 32, P16, 2, None) == binding.PQ_ERR_INVALID_ARG
    assert d(P16 + 16, P16, 4, 32, P16, 0, None) == binding.PQ_ERR_ALIGN  # W must be 32-byte aligned
    assert d(P16, P2, 4, 32, P16, 0, None) == binding.PQ_ERR_ALIGN
