"""GPU parity of the warp-level tensor-core path (mma.sync m16n8k16, M <= 64).

Same bars as the other paths: outputs within |C - out| <= 1e-5 * sum_b |t_b| +
1e-6 of the CPU oracle element by element, block sums identical.  Shapes cover
one to four 16-row m-tiles, ragged weight-row tiles (N not a multiple of 8 or
64), single-block K, K split over clusters of CTAs (including a short last
split), both weight-scale layouts, graph capture, and the full-size workloads.
The path has two kernels (include/pq_debug.h, pq_debug_set_small_kernel): the
TMA-fed one (the default, wherever it takes the shape) and the register-fed
one; the shape tests run both.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads
from tests.test_gpu_parity import (assert_within_bound, dev, host, quantized_workload, rand_operands,
                                   sampled_check)

pytestmark = pytest.mark.gpu

MMA_SHAPES = [(1, 1, 32), (1, 64, 128), (2, 7, 32), (3, 65, 256), (5, 130, 1056), (8, 64, 4096),
              (15, 200, 384), (16, 128, 96), (17, 257, 512), (31, 100, 2048), (32, 640, 3072),
              (33, 90, 160), (47, 300, 1024), (48, 1100, 4096), (63, 129, 640), (64, 1000, 4096),
              # more row tiles than SMs, ragged last tile, splits of unequal length
              (4, 8, 128), (8, 100, 512), (12, 333, 2048), (16, 1000, 4096), (16, 5000, 1024)]


def set_small_kernel(pq, which):
    lib = pq.load()
    lib.pq_debug_set_small_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_small_kernel.restype = ctypes.c_int
    assert lib.pq_debug_set_small_kernel(which) == 0


@pytest.fixture(params=[1, 0], ids=["tma_fed", "register_fed"])
def small_kernel(pq, request):
    set_small_kernel(pq, request.param)
    yield request.param
    set_small_kernel(pq, 1)


@pytest.mark.parametrize("M,N,K", MMA_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_qdot_mma(pq, small_kernel, M, N, K, layout):
    a, a_s, w, w_s = rand_operands(M * 131 + N * 7 + K + layout, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    C = torch.full((M, N), float("nan"), device="cuda:0")
    pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), C, ws_layout=layout, path=pq.PATH_MMA)
    pq.check_device()
    assert_within_bound(C, out, bound, f"mma M={M} N={N} K={K} layout={layout}")


@pytest.mark.parametrize("M,N,K", [(1, 9, 32), (7, 70, 256), (16, 64, 4096), (40, 130, 1280), (64, 72, 512)])
def test_blocksums_mma_exact(pq, M, N, K):
    """The integer stage alone: identical to the oracle's int64 block sums,
    including blocks at the extreme |S| = 32 * 128 * 128."""
    a, _, w, _ = rand_operands(M * 5 + N + K, M, N, K)
    a[:, :32] = -128
    w[:, :32] = -128
    a[:, 32:64] = 127
    S_ref = oracle.blocksums(a, w)
    S = pq.qdot_q8_0_blocksums(dev(a), dev(w), path=pq.PATH_MMA)
    pq.check_device()
    assert np.array_equal(host(S).astype(np.int64), S_ref)


def test_qdot_mma_extreme_values(pq):
    """Every product at its largest magnitude and scales over a wide range."""
    M, N, K = 20, 72, 1024
    a = np.full((M, K), -128, dtype=np.int8)
    w = np.full((N, K), -128, dtype=np.int8)
    w[1::2] = 127
    rng = np.random.default_rng(3)
    a_s = workloads.random_scales(rng, (M, K // 32), 1e-6, 1e3)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-6, 1e3)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(w_s), path=pq.PATH_MMA)
    pq.check_device()
    assert_within_bound(C, out, bound, "extreme values")


def test_qdot_mma_rejects_more_than_64_rows(pq):
    M, N, K = 65, 16, 64
    a, a_s, w, w_s = rand_operands(1, M, N, K)
    with pytest.raises(pq.PQError) as ei:
        pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(w_s), path=pq.PATH_MMA)
    assert ei.value.code == pq.PQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [12, 24])
def test_qdot_mma_in_a_graph(pq, M):
    """Captured with clusters and programmatic dependent launches, replayed twice."""
    N, K = 500, 2048
    a, a_s, w, w_s = rand_operands(99, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    A, AS, W, WS = dev(a), dev(a_s), dev(w), dev(w_s)
    C = torch.full((M, N), float("nan"), device="cuda:0")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(3):
            pq.qdot_q8_0_ex(A, AS, W, WS, C, path=pq.PATH_MMA)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    pq.check_device()
    assert_within_bound(C, out, bound, "graph")


@pytest.mark.parametrize("name", [n for n in workloads.Q8_WORKLOADS if 1 < workloads.Q8_WORKLOADS[n].M <= 64])
def test_qdot_mma_workload_full(pq, name):
    """The small-batch workloads at full size through this path, sampled columns."""
    x, w, qa, sa, qw, sw = quantized_workload(name)
    M, N = qa.shape[0], qw.shape[0]
    A, AS = pq.quantize_q8_0(dev(x))
    W, WS = pq.quantize_q8_0(dev(w))
    C = pq.qdot_q8_0_ex(A, AS, W, WS, path=pq.PATH_MMA)
    pq.check_device()
    rng = np.random.default_rng(2)
    cols = np.unique(np.concatenate([rng.choice(N, 512, replace=False), [0, N - 1]]))
    sampled_check(C, qa, sa, qw, sw, np.arange(M), cols, name)
    assert torch.isfinite(C).all()


# ------------------------------------------------------------------ fused step, 9..16 rows

@pytest.mark.parametrize("M,N,K", [(9, 300, 1024), (12, 1000, 4096), (16, 129, 96), (14, 700, 14336)])
def test_fused_step_equals_quantizer_then_mma(pq, small_kernel, M, N, K):
    """pq_quantize_qdot_q8_0 at 9..16 rows: with the register-fed kernel one kernel
    that quantizes x itself, with the TMA-fed kernel the quantizer and then qdot_t;
    either way its rows, scales and C are bit-identical to the quantizer followed by
    this path's qdot_t."""
    rng = np.random.default_rng(M * 17 + N + K)
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-4, 4, size=(M, 1)))).astype(np.float32)
    x[1, :64] = 0.0  # two all-zero blocks: d = 0, q = 0
    _, _, w, w_s = rand_operands(N + K, 1, N, K)
    X, W, WS = dev(x), dev(w), dev(w_s)
    A = torch.full((M, K), 77, dtype=torch.int8, device="cuda:0")
    AS = torch.full((M, K // 32), -1.0, dtype=torch.float32, device="cuda:0")
    C = pq.quantize_qdot_q8_0(X, W, WS, A=A, AS=AS)
    A2, AS2 = pq.quantize_q8_0(X)
    C2 = pq.qdot_q8_0_ex(A2, AS2, W, WS, path=pq.PATH_MMA)
    pq.check_device()
    assert torch.equal(A, A2) and torch.equal(AS, AS2)
    assert torch.equal(C, C2)
    qa, sa = oracle.quantize_q8_0(x)
    out, bound = oracle.qdot(qa, sa, w, w_s)
    assert_within_bound(C, out, bound, f"fused mma M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [12, 16])
def test_fused_step_in_a_graph(pq, M):
    """The one-kernel step captured once and replayed on new activations: each replay
    quantizes the rows it finds in x."""
    N, K = 600, 2048
    _, _, w, w_s = rand_operands(5, 1, N, K)
    W, WS = dev(w), dev(w_s)
    X = torch.empty((M, K), dtype=torch.float32, device="cuda:0")
    A = torch.empty((M, K), dtype=torch.int8, device="cuda:0")
    AS = torch.empty((M, K // 32), dtype=torch.float32, device="cuda:0")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda:0")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pq.quantize_qdot_q8_0(X, W, WS, C, A=A, AS=AS)
    rng = np.random.default_rng(M)
    for _ in range(2):
        x = (rng.standard_normal((M, K)) * 3.0).astype(np.float32)
        X.copy_(torch.from_numpy(x))
        g.replay()
        torch.cuda.synchronize()
        pq.check_device()
        qa, sa = oracle.quantize_q8_0(x)
        assert np.array_equal(host(A), qa) and np.array_equal(host(AS).view(np.uint32), sa.view(np.uint32))
        out, bound = oracle.qdot(qa, sa, w, w_s)
        assert_within_bound(C, out, bound, "graph replay")


# ------------------------------------------------------------------ the TMA-fed kernel

@pytest.mark.parametrize("M", [1, 16, 17, 33, 64])
def test_tma_kernel_block_sums_exact(pq, M):
    """Weights widened to 1152 + w with the MMA started at -1152 * sum(a): with unit
    scales and four blocks per row, C is the exact integer sum of four block sums
    (each up to 32 * 128 * 128 in magnitude), equal to the oracle's int64 sums."""
    N, K = 200, 128
    rng = np.random.default_rng(M)
    a = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    w = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    a[0, :32] = -128
    w[:, :32] = -128            # block 0 of row 0: +32 * 2^14
    w[1::2, 32:64] = 127
    a[:, 32:64] = -128          # block 1: -32 * 128 * 127 on odd weight rows
    ones_a = np.ones((M, K // 32), dtype=np.float32)
    ones_w = np.ones((N, K // 32), dtype=np.float32)
    exact = oracle.blocksums(a, w).sum(axis=2)
    for layout in (0, 1):
        ws = ones_w if layout == 0 else np.ascontiguousarray(ones_w.T)
        C = pq.qdot_q8_0_ex(dev(a), dev(ones_a), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_MMA)
        pq.check_device()
        assert np.array_equal(host(C).astype(np.int64), exact), f"layout {layout}"


@pytest.mark.parametrize("M,N,K", [(1, 32, 128), (3, 33, 4224), (16, 11008, 4096), (20, 4100, 14336),
                                   (40, 999, 2560), (64, 4096, 4096), (16, 100, 480)])
@pytest.mark.parametrize("layout", [0, 1])
def test_tma_kernel_chunks_and_passes(pq, M, N, K, layout):
    """K chunks of whole four-block stages with a short last chunk (K = 4224, 2560,
    480), clusters owning ragged tile ranges and several 128-row passes, rows past N
    in the last TMA box (zero-filled), against the oracle on sampled columns."""
    a, a_s, w, w_s = rand_operands(M + N + K + layout, M, N, K)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_MMA)
    pq.check_device()
    rng = np.random.default_rng(K)
    cols = np.unique(np.concatenate([rng.choice(N, min(N, 300), replace=False), np.arange(min(N, 40)),
                                     np.arange(max(0, N - 40), N)]))
    out, bound = oracle.qdot(a, a_s, w[cols], w_s[cols])
    got = host(C)[:, cols].astype(np.float64)
    bad = np.abs(got - out) > bound
    assert not bad.any(), f"{int(bad.sum())} elements out of bound, M={M} N={N} K={K}"


def _split_hooks(pq):
    lib = pq.load()
    lib.pq_debug_set_small_split.argtypes = [ctypes.c_int]
    lib.pq_debug_set_small_split.restype = ctypes.c_int
    lib.pq_debug_small_kernel_config.argtypes = [ctypes.c_void_p]
    lib.pq_debug_small_kernel_config.restype = ctypes.c_int
    return lib


def test_tma_kernel_every_cluster_size(pq):
    """The cost model picks the K split by itself, so parity at the shapes above may
    never see some cluster sizes: force each of 1, 2, 4 and 8 CTAs on shapes whose
    chunks fit, check the launch took it (the last launch's configuration), and
    compare with the oracle.  Every size must be exercised by some shape."""
    lib = _split_hooks(pq)
    shapes = [(16, 1000, 1024), (5, 333, 4096), (20, 777, 2048), (16, 300, 8192), (48, 200, 1024),
              (64, 520, 2048), (1, 64, 512)]
    seen = set()
    try:
        for ks in (1, 2, 4, 8):
            assert lib.pq_debug_set_small_split(ks) == 0
            for M, N, K in shapes:
                a, a_s, w, w_s = rand_operands(ks * 7 + M + N + K, M, N, K)
                cfg = (ctypes.c_int * 4)()
                assert lib.pq_debug_small_kernel_config(cfg) == 0
                before = tuple(cfg)
                for layout in (0, 1):
                    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
                    C = torch.full((M, N), float("nan"), device="cuda:0")
                    pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), C, ws_layout=layout, path=pq.PATH_MMA)
                    pq.check_device()
                    out, bound = oracle.qdot(a, a_s, w, w_s)
                    assert_within_bound(C, out, bound, f"ks={ks} M={M} N={N} K={K} layout={layout}")
                assert lib.pq_debug_small_kernel_config(cfg) == 0
                if tuple(cfg) != before and cfg[0] == ks:
                    seen.add(ks)
    finally:
        lib.pq_debug_set_small_split(0)
    assert seen == {1, 2, 4, 8}, f"cluster sizes exercised: {sorted(seen)}"


@pytest.mark.parametrize("M", [3, 8, 12, 16])
def test_step_sees_weights_written_just_before(pq, M):
    """The one-call step at 9..16 rows lets qdot_t stream its first weight stages
    before its own wait on the quantizer (which lets it in only once every kernel
    before the quantizer has completed); at 2..8 rows the dp4a kernel only prefetches
    into L2 before its wait.  Weights rewritten by a kernel just before each step, on
    the same stream and with no synchronization, must be the ones used."""
    N, K = 2000, 4096
    rng = np.random.default_rng(M)
    x = (rng.standard_normal((M, K)) * 2.0).astype(np.float32)
    X = dev(x)
    W = torch.empty((N, K), dtype=torch.int8, device="cuda:0")
    WS = torch.empty((N, K // 32), dtype=torch.float32, device="cuda:0")
    sets = [rand_operands(100 * M + i, 1, N, K)[2:] for i in range(3)]
    srcs = [(dev(w), dev(ws)) for w, ws in sets]
    qa, sa = oracle.quantize_q8_0(x)
    torch.cuda.synchronize()
    outs = []
    for w_d, ws_d in srcs:
        W.copy_(w_d)        # a kernel on the current stream, right before the step
        WS.copy_(ws_d)
        outs.append(pq.quantize_qdot_q8_0(X, W, WS))
    torch.cuda.synchronize()
    pq.check_device()
    for (w, ws), C in zip(sets, outs):
        out, bound = oracle.qdot(qa, sa, w, ws)
        assert_within_bound(C, out, bound, f"weights rewritten before the step, M={M}")
