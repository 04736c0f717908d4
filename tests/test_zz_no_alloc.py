"""The allocation-free decode step (pq_quantize_qdot_q8_0_noalloc) against the
allocating one (pq_quantize_qdot_q8_0 without A / AS, whose quantized rows go
to a workspace the library allocates).

The allocation-free form exists for callers that cannot let the library call
cudaMalloc: work recorded into CUDA graphs, serving loops that must not stall
on the allocator, hosts that own every device allocation.  It keeps its
scratch in a fixed device array that is part of the library, so its results
must match the allocating entry point's, call after call, even though every
call reuses the same array.  This file is collected last so that a run that
stops at its first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _c_abi(pq):
    """The two entry points as raw C functions (device pointers, sizes, stream)."""
    lib = pq.load()
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.pq_quantize_qdot_q8_0_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_quantize_qdot_q8_0_noalloc.restype = i32
    lib.pq_quantize_qdot_q8_0.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.pq_quantize_qdot_q8_0.restype = i32
    return lib


def _bound(x, w, w_s):
    """The parity tolerance of the other tests: 1e-5 * sum_b |t_b| + 1e-6 (from the oracle)."""
    qa, sa = oracle.quantize_q8_0(x)
    return oracle.qdot(qa, sa, w, w_s)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (4, 1000, 4096), (12, 700, 2048), (16, 257, 4096), (24, 300, 1024),
                                   (64, 257, 14336), (128, 300, 1024)])
def test_noalloc_matches_allocating_entry_point(pq, M, N, K):
    lib = _c_abi(pq)
    rng = np.random.default_rng(M * 7 + N + K)
    w = workloads.random_int8(rng, (N, K), -127, 127)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1e-2)
    W = torch.from_numpy(w).to(DEV)
    WS = torch.from_numpy(w_s).to(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row: the second must not see the first's scratch
        x = (rng.standard_normal((M, K)) * (1.0 + 3.0 * call)).astype(np.float32)
        X = torch.from_numpy(x).to(DEV)
        C_ref = torch.empty((M, N), dtype=torch.float32, device=DEV)
        C_new = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        st = lib.pq_quantize_qdot_q8_0(X.data_ptr(), None, None, W.data_ptr(), WS.data_ptr(), C_ref.data_ptr(),
                                       M, N, K, 0, stream)
        assert st == 0, pq.strerror(st)
        st = lib.pq_quantize_qdot_q8_0_noalloc(X.data_ptr(), W.data_ptr(), WS.data_ptr(), C_new.data_ptr(),
                                               M, N, K, 0, stream)
        assert st == 0, pq.strerror(st)
        pq.check_device()
        out, bound = _bound(x, w, w_s)
        c_ref = C_ref.cpu().numpy().astype(np.float64)
        c_new = C_new.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(c_new - c_ref) <= bound), f"call {call}: max diff {np.abs(c_new - c_ref).max()}"
        assert np.all(np.abs(c_new - out) <= bound), f"call {call}: outside the oracle's tolerance"


def test_noalloc_rejects_problems_beyond_its_scratch(pq):
    lib = _c_abi(pq)
    K = 4096
    M = (1 << 20) // (K + K // 8) + 1  # one row more than the 1 MiB array holds
    X = torch.zeros((M, K), dtype=torch.float32, device=DEV)
    W = torch.zeros((8, K), dtype=torch.int8, device=DEV)
    WS = torch.zeros((8, K // 32), dtype=torch.float32, device=DEV)
    C = torch.zeros((M, 8), dtype=torch.float32, device=DEV)
    st = lib.pq_quantize_qdot_q8_0_noalloc(X.data_ptr(), W.data_ptr(), WS.data_ptr(), C.data_ptr(), M, 8, K, 0,
                                           torch.cuda.current_stream().cuda_stream)
    assert st == pq.PQ_ERR_SCRATCH
    assert "scratch" in pq.strerror(st)
    # the largest problem that fits still runs
    M -= 1
    st = lib.pq_quantize_qdot_q8_0_noalloc(X[:M].data_ptr(), W.data_ptr(), WS.data_ptr(), C[:M].data_ptr(), M, 8,
                                           K, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    pq.check_device()
    assert torch.all(C[:M] == 0)
