"""Failure detection on the GPU without a fault: a bounded wait is made to run out.

The producer of a pipelined kernel is told (test hook, include/pq_debug.h) to
skip one pipeline stage, so the consumers' waits on that stage never complete.
Every wait is bounded: the kernel must give up within its limit, record the
timeout in the library's status word, drain its work in flight, free its
tensor memory and return.  Covered: the tcgen05 kernels (narrow tiles, and both
prompt-shape kernels with Q8_0 and with Q5_0 weights) and the TMA-fed
warp-level MMA kernel, whose CTAs also wait on one another across their cluster.  The test checks the reported status and that the
context stays usable (a normal launch afterwards gives correct results).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads

pytestmark = pytest.mark.gpu


def _hook(lib, stage, cycles):
    lib.pq_debug_set_tc_fault.argtypes = [ctypes.c_int, ctypes.c_ulonglong]
    lib.pq_debug_set_tc_fault.restype = ctypes.c_int
    assert lib.pq_debug_set_tc_fault(stage, cycles) == 0


def _prompt_kernel(lib, which):
    lib.pq_debug_set_prompt_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_prompt_kernel.restype = ctypes.c_int
    assert lib.pq_debug_set_prompt_kernel(which) == 0


# Every CTA must reach the skipped stage.  The warp-level kernel's stages are 8
# blocks of one CTA's K chunk: K = 8192 gives two or more at any K split for one
# m-tile; four m-tiles fit shared memory only with eight-way splits of K = 4096
# (two stages).
@pytest.mark.parametrize("M,kernel,path,K", [(16, 0, "tc", 2048), (256, 0, "tc", 2048), (256, 1, "tc", 2048),
                                             (16, 0, "mma", 8192), (48, 0, "mma", 4096)],
                         ids=["narrow_tiles", "prompt_first_kernel", "prompt_second_kernel", "tma_fed_mma",
                              "tma_fed_mma_two_groups"])
def test_tc_bounded_wait_gives_up_and_recovers(pq, M, kernel, path, K):
    lib = pq.load()
    _prompt_kernel(lib, kernel)
    path = pq.PATH_TC if path == "tc" else pq.PATH_MMA
    rng = np.random.default_rng(M)
    N = 256
    a = workloads.random_int8(rng, (M, K))
    w = workloads.random_int8(rng, (N, K))
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    A, AS, W, WS = (torch.from_numpy(v).cuda() for v in (a, a_s, w, w_s))
    pq.check_device()  # clean status before
    try:
        _hook(lib, 1, 20_000_000)  # ~10 ms at 2 GHz
        C = torch.full((M, N), 123.0, device="cuda")
        pq.qdot_q8_0_ex(A, AS, W, WS, C, path=path)
        with pytest.raises(pq.PQError) as ei:
            pq.check_device()
        assert ei.value.code == pq.PQ_ERR_TIMEOUT
    finally:
        _hook(lib, -1, 0)
    # the context is still usable and the next launch is correct
    try:
        C = pq.qdot_q8_0_ex(A, AS, W, WS, path=path)
        pq.check_device()
    finally:
        _prompt_kernel(lib, 1)  # the default (include/pq_debug.h)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - out) <= bound)


@pytest.mark.parametrize("kernel", [0, 1], ids=["scale_product_mma", "scales_in_registers"])
def test_q50_prompt_bounded_wait_gives_up_and_recovers(pq, kernel):
    """The same for Q5_0 weights at a prompt shape, on both tensor-core kernels: the producer
    skips one stage, the consumers' bounded waits give up, the status reports the timeout
    and the next call on the same operands is correct."""
    lib = pq.load()
    _prompt_kernel(lib, kernel)
    rng = np.random.default_rng(7)
    M, N, K = 256, 256, 2048
    a = workloads.random_int8(rng, (M, K))
    w5 = rng.integers(0, 256, size=(N, K // 32 * 20), dtype=np.uint8)
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    A, AS, W5, WS = (torch.from_numpy(v).cuda() for v in (a, a_s, w5, w_s))
    pq.check_device()  # clean status before
    try:
        _hook(lib, 1, 20_000_000)  # ~10 ms at 2 GHz
        C = torch.full((M, N), 123.0, device="cuda")
        pq.q50_qdot(A, AS, W5, WS, C)
        with pytest.raises(pq.PQError) as ei:
            pq.check_device()
        assert ei.value.code == pq.PQ_ERR_TIMEOUT
    finally:
        _hook(lib, -1, 0)
    try:
        C = pq.q50_qdot(A, AS, W5, WS)
        pq.check_device()
    finally:
        _prompt_kernel(lib, 1)  # the default (include/pq_debug.h)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, w_s)
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - out) <= bound)
