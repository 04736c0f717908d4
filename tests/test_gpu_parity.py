"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars: quantized bytes and f32 scales bit-identical; integer block sums
identical; qdot_t outputs within |C - out| <= 1e-5 * sum_b |t_b| + 1e-6 of
the oracle's double result (t_b the per-block terms), element by element.
Inputs are seeded (gemm_q8_qdot_gb300.workloads); every expected value comes
from the oracle, never from the GPU.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads
from tests import golden_io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def assert_bytes_equal(q_gpu, s_gpu, q_ref, s_ref):
    q_gpu, s_gpu = host(q_gpu), host(s_gpu)
    bad = np.nonzero(q_gpu != q_ref)
    assert bad[0].size == 0, f"{bad[0].size} quantized bytes differ, first at {[b[0] for b in bad]}"
    sb = np.nonzero(s_gpu.view(np.uint32) != s_ref.view(np.uint32))
    assert sb[0].size == 0, f"{sb[0].size} scales differ, first at {[b[0] for b in sb]}"


def assert_within_bound(C, out, bound, what=""):
    C = host(C).astype(np.float64) if isinstance(C, torch.Tensor) else C.astype(np.float64)
    err = np.abs(C - out)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu {C[i]!r} oracle {out[i]!r} bound {bound[i]!r}")


def rand_operands(seed, M, N, K, lo=-128, hi=127):
    rng = np.random.default_rng(seed)
    a = workloads.random_int8(rng, (M, K), lo, hi)
    w = workloads.random_int8(rng, (N, K), lo, hi)
    a_s = workloads.random_scales(rng, (M, K // 32), 1e-3, 10.0)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1.0)
    return a, a_s, w, w_s


@functools.lru_cache(maxsize=None)
def quantized_workload(name):
    """Oracle-quantized operands of a workload (the inputs both sides share)."""
    wl = workloads.WORKLOADS[name]
    x = workloads.activations(wl)
    w = workloads.weights(wl)
    qa, sa = oracle.quantize_q8_0(x)
    qw, sw = oracle.quantize_q8_0(w)
    return x, w, qa, sa, qw, sw


# ------------------------------------------------------------------ quantizer

def test_quantize_golden_blocks(pq):
    for name, x, d, q in golden_io.quantize_blocks():
        qg, sg = pq.quantize_q8_0(dev(x[None, :]))
        torch.cuda.synchronize()
        assert host(qg)[0].tolist() == q.tolist(), name
        assert host(sg)[0, 0].view(np.uint32) == np.float32(d).view(np.uint32), name


@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (65, 256), (257, 4096), (5, 14336)])
def test_quantize_random(pq, rows, K):
    rng = np.random.default_rng(rows * 1000 + K)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    x *= np.exp(rng.uniform(-30, 30, size=(rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                                               # zero block
    if K >= 64:
        x[-1, 32:64] = (rng.integers(-126, 126, 32) + 0.5).astype(np.float32)  # ties at d = 1
        x[-1, 32] = 127.0
    q_ref, s_ref = oracle.quantize_q8_0(x)
    qg, sg = pq.quantize_q8_0(dev(x))
    torch.cuda.synchronize()
    assert_bytes_equal(qg, sg, q_ref, s_ref)


def near_tie_rows(rows, K, seed):
    """Blocks built to land x / d on or next to half-integers, at many scales.

    Per block: element 0 is 127 * sc (so amax / 127 is sc up to rounding);
    the others are (n + 0.5) * sc for random n, or that value's float
    neighbour on either side.  Every fourth block is plain random data; two
    blocks have subnormal scales (d subnormal) and one is near FLT_MAX.
    """
    rng = np.random.default_rng(seed)
    x = np.empty((rows, K), dtype=np.float32)
    blocks = x.reshape(-1, 32)
    for b in range(blocks.shape[0]):
        sc = np.float32(1.0) if b % 4 == 0 else np.float32(np.ldexp(1.0 + rng.uniform(0, 1), int(rng.integers(-30, 30))))
        if b % 4 == 3:
            v = (rng.uniform(-127, 127, 32) * sc).astype(np.float32)
        else:
            n = (rng.integers(-127, 127, 32) + 0.5).astype(np.float32)
            v = (n * sc).astype(np.float32)
            side = rng.integers(0, 3, 32)
            v = np.where(side == 1, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(side == 2, np.nextafter(v, np.float32(-np.inf)), v)
        v[0] = np.float32(127.0) * sc
        v = np.clip(v, -np.float32(127.0) * sc, np.float32(127.0) * sc)
        blocks[b] = v
    blocks[1] = (rng.integers(-127, 128, 32) * np.float32(1e-45)).astype(np.float32)   # subnormal x and d
    blocks[2] = (rng.uniform(-1, 1, 32) * np.float32(3e-41)).astype(np.float32)
    blocks[5] = (rng.uniform(-1, 1, 32) * np.float32(3.0e38)).astype(np.float32)       # near FLT_MAX
    return x


@pytest.mark.parametrize("rows,K", [(1, 4096), (1, 14336), (3, 1024), (64, 256), (12, 2048), (16, 512)])
def test_quantize_near_ties(pq, rows, K):
    """The quantizer's rounding against the oracle's IEEE division on near-tie quotients:
    the standalone quantizer and the fused step's quantized rows, bit for bit."""
    x = near_tie_rows(rows, K, rows * 31 + K)
    q_ref, s_ref = oracle.quantize_q8_0(x)
    qg, sg = pq.quantize_q8_0(dev(x))
    torch.cuda.synchronize()
    assert_bytes_equal(qg, sg, q_ref, s_ref)
    w = np.ones((8, K), dtype=np.int8)
    w_s = np.ones((8, K // 32), dtype=np.float32)
    A = torch.empty((rows, K), dtype=torch.int8, device=DEV)
    AS = torch.empty((rows, K // 32), dtype=torch.float32, device=DEV)
    pq.quantize_qdot_q8_0(dev(x), dev(w), dev(w_s), A=A, AS=AS)
    pq.check_device()
    assert_bytes_equal(A, AS, q_ref, s_ref)


@pytest.mark.parametrize("name", list(workloads.Q8_WORKLOADS))
def test_quantize_workload_full(pq, name):
    x, w, qa, sa, qw, sw = quantized_workload(name)
    qg, sg = pq.quantize_q8_0(dev(x))
    assert_bytes_equal(qg, sg, qa, sa)
    qg, sg = pq.quantize_q8_0(dev(w))
    assert_bytes_equal(qg, sg, qw, sw)


def test_quantize_output_bounds(pq):
    """Stores stay inside q [rows, K] and s [rows, K/32]: guard bytes around both."""
    rows, K = 7, 96
    x = np.random.default_rng(1).standard_normal((rows, K)).astype(np.float32)
    qbuf = torch.full((rows * K + 64,), 0x5A, dtype=torch.int8, device=DEV)
    sbuf = torch.full((rows * K // 32 + 16,), 7.25, dtype=torch.float32, device=DEV)
    q = qbuf[16:16 + rows * K].view(rows, K)
    s = sbuf[4:4 + rows * K // 32].view(rows, K // 32)
    pq.quantize_q8_0(dev(x), q, s)
    torch.cuda.synchronize()
    qh, sh = host(qbuf), host(sbuf)
    assert np.all(qh[:16] == 0x5A) and np.all(qh[16 + rows * K:] == 0x5A)
    assert np.all(sh[:4] == 7.25) and np.all(sh[4 + rows * K // 32:] == 7.25)
    q_ref, s_ref = oracle.quantize_q8_0(x)
    assert_bytes_equal(q, s, q_ref, s_ref)


# ------------------------------------------------------------------ qdot, small shapes

SMALL_SHAPES = [(1, 1, 32), (1, 7, 64), (1, 64, 256), (1, 300, 1056), (2, 9, 96), (3, 17, 128),
                (5, 33, 256), (8, 64, 512), (13, 70, 160), (1, 2, 14336)]


@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_qdot_simt_small(pq, M, N, K, layout):
    a, a_s, w, w_s = rand_operands(M * 7 + N * 13 + K, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_SIMT)
    torch.cuda.synchronize()
    assert_within_bound(C, out, bound, f"simt M={M} N={N} K={K} layout={layout}")


@pytest.mark.parametrize("M,N,K", [(1, 5, 32), (2, 9, 96), (4, 33, 256), (5, 64, 1024), (1, 3, 14336)])
def test_blocksums_simt_exact(pq, M, N, K):
    a, _, w, _ = rand_operands(M + N + K, M, N, K)
    a[:, :32] = -128
    w[:, :32] = -128   # block 0: 32 * 16384 = 524288, the largest block sum
    S_ref = oracle.blocksums(a, w)
    S = pq.qdot_q8_0_blocksums(dev(a), dev(w), path=pq.PATH_SIMT)
    torch.cuda.synchronize()
    assert np.array_equal(host(S).astype(np.int64), S_ref)


def test_qdot_16byte_aligned_operands(pq):
    """Bases 16 but not 32 bytes aligned take the two-128-bit-load variant."""
    M, N, K = 3, 40, 256
    a, a_s, w, w_s = rand_operands(99, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    abuf = torch.zeros(M * K + 16, dtype=torch.int8, device=DEV)
    wbuf = torch.zeros(N * K + 16, dtype=torch.int8, device=DEV)
    A = abuf[16:].view(M, K)
    W = wbuf[16:].view(N, K)
    A.copy_(dev(a))
    W.copy_(dev(w))
    assert A.data_ptr() % 32 == 16 and W.data_ptr() % 32 == 16
    C = pq.qdot_q8_0_ex(A, dev(a_s), W, dev(w_s), path=pq.PATH_SIMT)
    torch.cuda.synchronize()
    assert_within_bound(C, out, bound, "16-byte aligned")


def test_qdot_output_guard_and_empty(pq):
    M, N, K = 2, 37, 64
    a, a_s, w, w_s = rand_operands(5, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    cbuf = torch.full((M * N + 64,), -3.5, dtype=torch.float32, device=DEV)
    C = cbuf[32:32 + M * N].view(M, N)
    pq.qdot_q8_0(dev(a), dev(a_s), dev(w), dev(w_s), C)
    torch.cuda.synchronize()
    ch = host(cbuf)
    assert np.all(ch[:32] == -3.5) and np.all(ch[32 + M * N:] == -3.5)
    assert_within_bound(C, out, bound, "guarded")
    # empty problems leave C untouched
    pq.qdot_q8_0(dev(a[:0]), dev(a_s[:0]), dev(w), dev(w_s), C[:0])
    torch.cuda.synchronize()


def test_qdot_extreme_values(pq):
    """All -128 against all -128 (largest block sums) and against +127, scale 0 blocks."""
    M, N, K = 2, 24, 4096
    a = np.full((M, K), -128, np.int8)
    w = np.full((N, K), -128, np.int8)
    w[1::2] = 127
    a_s = np.ones((M, K // 32), np.float32)
    w_s = np.full((N, K // 32), 0.5, np.float32)
    w_s[:, 3] = 0.0
    out, bound = oracle.qdot(a, a_s, w, w_s)
    C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(w_s), path=pq.PATH_SIMT)
    torch.cuda.synchronize()
    assert_within_bound(C, out, bound, "extremes")


# ------------------------------------------------------------------ full-size workloads

def sampled_check(C, qa, sa, qw, sw, rows, cols, what):
    out, bound = oracle.qdot(qa[rows], sa[rows], qw[cols], sw[cols])
    assert_within_bound(host(C)[np.ix_(rows, cols)], out, bound, what)


@pytest.mark.parametrize("name", [n for n in workloads.Q8_WORKLOADS if workloads.Q8_WORKLOADS[n].M <= 8])
def test_qdot_workload_full_simt(pq, name):
    """The decode / small-batch workloads at full size, the launch the benchmark times."""
    x, w, qa, sa, qw, sw = quantized_workload(name)
    M, N = qa.shape[0], qw.shape[0]
    A, AS = pq.quantize_q8_0(dev(x))
    W, WS = pq.quantize_q8_0(dev(w))
    C = pq.qdot_q8_0(A, AS, W, WS)
    torch.cuda.synchronize()
    if M * N * qa.shape[1] <= 2e8:
        out, bound = oracle.qdot(qa, sa, qw, sw)
        assert_within_bound(C, out, bound, name)
    else:
        rng = np.random.default_rng(0)
        cols = np.sort(rng.choice(N, 1024, replace=False))
        sampled_check(C, qa, sa, qw, sw, np.arange(M), cols, name)


# ------------------------------------------------------------------ tensor-core path

TC_SHAPES = [(1, 16, 128), (9, 100, 256), (16, 128, 128), (17, 300, 384), (33, 130, 128), (64, 257, 512),
             (65, 64, 256), (130, 200, 128), (256, 384, 1024), (300, 129, 256),
             # narrow tiles over many scale groups, split along K into units of unequal length
             (5, 2000, 2048), (24, 700, 3072), (48, 1100, 4096),
             # many more output tiles than SMs: every persistent CTA takes several tiles
             # in turn and carries its pipeline phases from one to the next
             (512, 14336, 128), (384, 2048, 1024)]


@pytest.mark.parametrize("M,N,K", TC_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_qdot_tc_small(pq, M, N, K, layout):
    a, a_s, w, w_s = rand_operands(M * 31 + N * 7 + K + layout, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s, omp=True)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    if layout == 1 and N % 4 != 0:
        # the [K/32, N] scale plane is loaded by TMA only when its rows are 16-byte
        # multiples: the tensor-core path declines, the automatic path falls back
        with pytest.raises(pq.PQError) as ei:
            pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_TC)
        assert ei.value.code == pq.PQ_ERR_UNSUPPORTED
        C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_AUTO)
    else:
        C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=pq.PATH_TC)
    pq.check_device()
    assert_within_bound(C, out, bound, f"tc M={M} N={N} K={K} layout={layout}")


DEFAULT_PROMPT_KERNEL = 1  # scales in registers (include/pq_debug.h)


def _set_prompt_kernel(pq, which):
    import ctypes
    lib = pq.load()
    lib.pq_debug_set_prompt_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_prompt_kernel.restype = ctypes.c_int
    assert lib.pq_debug_set_prompt_kernel(which) == 0


PROMPT_SHAPES = [(65, 64, 256), (130, 200, 128), (256, 384, 1024), (300, 129, 256), (384, 2048, 1024),
                 # few output tiles: K split over the CTAs, partial tiles added into C
                 (128, 256, 4096), (200, 64, 2048), (96, 130, 512)]


@pytest.mark.parametrize("which", [0, 1], ids=["scale_product_mma", "scales_in_registers"])
@pytest.mark.parametrize("M,N,K", PROMPT_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_prompt_kernels(pq, which, M, N, K, layout):
    """Both tensor-core kernels of the prompt shapes (M > 64) against the oracle: the one
    with the scale-product MMA and the one applying the scales in registers (the default);
    ragged M and N, both scale layouts, split K."""
    a, a_s, w, w_s = rand_operands(M * 7 + N * 3 + K + layout + 1000 * which, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s, omp=True)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    path = pq.PATH_TC if (layout == 0 or N % 4 == 0) else pq.PATH_AUTO
    try:
        _set_prompt_kernel(pq, which)
        C = pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(ws), ws_layout=layout, path=path)
        pq.check_device()
    finally:
        _set_prompt_kernel(pq, DEFAULT_PROMPT_KERNEL)
    assert_within_bound(C, out, bound, f"kernel {which} M={M} N={N} K={K} layout={layout}")


@pytest.mark.parametrize("which", [0, 1], ids=["scale_product_mma", "scales_in_registers"])
def test_prompt_kernels_at_full_size(pq, which):
    """Both prompt kernels at the benchmark's full size (M = 512, K = 4096, N = 14336) on one
    complete row per 128-row band and one column per 128-column band."""
    name = "prompt_m512_k4096_n14336"
    x, w, qa, sa, qw, sw = quantized_workload(name)
    A, AS = pq.quantize_q8_0(dev(x))
    W, WS = pq.quantize_q8_0(dev(w))
    try:
        _set_prompt_kernel(pq, which)
        C = host(pq.qdot_q8_0(A, AS, W, WS))
        pq.check_device()
    finally:
        _set_prompt_kernel(pq, DEFAULT_PROMPT_KERNEL)
    M, N = qa.shape[0], qw.shape[0]
    rng = np.random.default_rng(3)
    rows = np.array([b + rng.integers(0, min(128, M - b)) for b in range(0, M, 128)])
    cols = np.array([b + rng.integers(0, min(128, N - b)) for b in range(0, N, 128)])
    out, bound = oracle.qdot(qa[rows], sa[rows], qw, sw, omp=True)
    assert_within_bound(C[rows], out, bound, "rows")
    out, bound = oracle.qdot(qa, sa, qw[cols], sw[cols], omp=True)
    assert_within_bound(C[:, cols], out, bound, "columns")


def test_qdot_tc_unaligned_scales_fall_back(pq):
    """Scale planes 4- but not 16-byte aligned: auto path still correct (dp4a kernel)."""
    M, N, K = 40, 96, 256
    a, a_s, w, w_s = rand_operands(17, M, N, K)
    out, bound = oracle.qdot(a, a_s, w, w_s)
    buf = torch.zeros(a_s.size + 1, dtype=torch.float32, device=DEV)
    AS = buf[1:].view(M, K // 32)
    AS.copy_(dev(a_s))
    with pytest.raises(pq.PQError) as ei:
        pq.qdot_q8_0_ex(dev(a), AS, dev(w), dev(w_s), path=pq.PATH_TC)
    assert ei.value.code == pq.PQ_ERR_UNSUPPORTED
    C = pq.qdot_q8_0(dev(a), AS, dev(w), dev(w_s))
    pq.check_device()
    assert_within_bound(C, out, bound, "unaligned scales")


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (20, 70, 256), (64, 128, 128), (100, 140, 256), (128, 256, 512)])
def test_blocksums_tc_exact(pq, M, N, K):
    a, _, w, _ = rand_operands(M + 3 * N + K, M, N, K)
    a[:, :32] = -128
    w[:, :32] = -128
    a[:, 32:64] = 127
    S_ref = oracle.blocksums(a, w)
    S = pq.qdot_q8_0_blocksums(dev(a), dev(w), path=pq.PATH_TC)
    pq.check_device()
    assert np.array_equal(host(S).astype(np.int64), S_ref)


def test_qdot_tc_unsupported_k(pq):
    """The tensor-core path needs K % 128 == 0; the explicit path says so, auto falls back."""
    M, N, K = 20, 40, 96
    a, a_s, w, w_s = rand_operands(4, M, N, K)
    with pytest.raises(pq.PQError) as ei:
        pq.qdot_q8_0_ex(dev(a), dev(a_s), dev(w), dev(w_s), path=pq.PATH_TC)
    assert ei.value.code == pq.PQ_ERR_UNSUPPORTED
    out, bound = oracle.qdot(a, a_s, w, w_s)
    C = pq.qdot_q8_0(dev(a), dev(a_s), dev(w), dev(w_s))
    pq.check_device()
    assert_within_bound(C, out, bound, "auto fallback")


@pytest.mark.parametrize("name", [n for n in workloads.Q8_WORKLOADS if workloads.Q8_WORKLOADS[n].M > 8])
def test_qdot_workload_full_tc(pq, name):
    """Small-batch (M = 16, 64) and prompt (M = 512) workloads at full size, as benchmarked."""
    x, w, qa, sa, qw, sw = quantized_workload(name)
    M, N = qa.shape[0], qw.shape[0]
    A, AS = pq.quantize_q8_0(dev(x))
    W, WS = pq.quantize_q8_0(dev(w))
    C = pq.qdot_q8_0(A, AS, W, WS)
    pq.check_device()
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(M, min(M, 24), replace=False))
    cols = np.sort(np.concatenate([rng.choice(N, 384, replace=False), [0, N - 1]]))
    sampled_check(C, qa, sa, qw, sw, rows, np.unique(cols), name)
    # a property at full size: every row of C is finite
    assert torch.isfinite(C).all()


def test_qdot_prompt_full_rows_and_columns(pq):
    """The prompt GEMM (M = 512, K = 4096, N = 14336) at full size, as benchmarked, on
    complete rows and columns: one row inside every 128-row band (all 14336 columns) and
    one column inside every 128-column band (all 512 rows).  Together they cross every
    128 x 128 output tile, so every unit of work a persistent CTA takes -- first, second
    or third in its turn -- is compared with the oracle, not only a random sample."""
    name = "prompt_m512_k4096_n14336"
    x, w, qa, sa, qw, sw = quantized_workload(name)
    M, N = qa.shape[0], qw.shape[0]
    A, AS = pq.quantize_q8_0(dev(x))
    W, WS = pq.quantize_q8_0(dev(w))
    C = host(pq.qdot_q8_0(A, AS, W, WS))
    pq.check_device()
    rng = np.random.default_rng(2)
    rows = np.array([b + rng.integers(0, min(128, M - b)) for b in range(0, M, 128)])
    cols = np.array([b + rng.integers(0, min(128, N - b)) for b in range(0, N, 128)])
    out, bound = oracle.qdot(qa[rows], sa[rows], qw, sw, omp=True)
    assert_within_bound(C[rows], out, bound, f"{name} rows {rows.tolist()}")
    out, bound = oracle.qdot(qa, sa, qw[cols], sw[cols], omp=True)
    assert_within_bound(C[:, cols], out, bound, f"{name} {cols.size} columns")


# ------------------------------------------------------------------ fused quantize + qdot

FUSED_SHAPES = [(1, 64, 256), (1, 300, 1056), (2, 17, 128), (3, 129, 512), (4, 64, 4096), (7, 33, 96),
                (8, 257, 256), (1, 40, 14336), (1, 4000, 64), (1, 9000, 128), (1, 96, 49152),
                # 9..16 rows: the quantizer and the warp-level MMA path (one split,
                # several splits, a short last split, ragged N, long K)
                (9, 130, 512), (16, 300, 4096), (10, 5, 32), (15, 129, 96), (12, 333, 2048),
                (13, 1000, 4096), (16, 2000, 14336), (11, 64, 1056),
                # one row, more columns than one CTA per SM holds: warps take further columns
                (1, 14336, 4096), (1, 5000, 49152)]


@pytest.mark.parametrize("M,N,K", FUSED_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_qdot_fused(pq, M, N, K, layout):
    rng = np.random.default_rng(M * 101 + N + K + layout)
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, size=(M, 1)))).astype(np.float32)
    _, _, w, w_s = rand_operands(N + K, 1, N, K)
    qa, sa = oracle.quantize_q8_0(x)
    out, bound = oracle.qdot(qa, sa, w, w_s)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    A = torch.full((M, K), 77, dtype=torch.int8, device=DEV)
    AS = torch.full((M, K // 32), -1.0, dtype=torch.float32, device=DEV)
    C = pq.quantize_qdot_q8_0(dev(x), dev(w), dev(ws), A=A, AS=AS, ws_layout=layout)
    pq.check_device()
    assert_bytes_equal(A, AS, qa, sa)
    assert_within_bound(C, out, bound, f"fused M={M} N={N} K={K} layout={layout}")
    # without the optional outputs: same result
    C2 = pq.quantize_qdot_q8_0(dev(x), dev(w), dev(ws), ws_layout=layout)
    pq.check_device()
    assert_within_bound(C2, out, bound, "fused, no A/AS")


def test_stream_reader_checksums(pq):
    """The test-only streaming reader reads every weight row: its per-row checksum (the
    32-bit word sum's low byte plus the sum of the row's scales) matches the host's."""
    rng = np.random.default_rng(4)
    for rows, K in ((4096, 4096), (100, 14336), (33, 128)):
        w = workloads.random_int8(rng, (rows, K))
        ws = workloads.random_scales(rng, (rows, K // 32))
        words = w.view(np.uint32).astype(np.uint64).reshape(rows, -1).sum(axis=1)
        ref = ws.astype(np.float64).sum(axis=1) + (words & 0xff).astype(np.float64)
        for early in (False, True):
            out = host(pq.debug_stream_read(dev(w), dev(ws), early=early))
            torch.cuda.synchronize()
            assert np.allclose(out, ref, rtol=1e-5, atol=1e-3), (rows, K, early)


def test_quantize_qdot_large_m(pq):
    """M > 1 runs the quantizer and qdot_t as two kernels, into A / AS or the workspace."""
    M, N, K = 40, 96, 256
    rng = np.random.default_rng(8)
    x = rng.standard_normal((M, K)).astype(np.float32)
    _, _, w, w_s = rand_operands(3, 1, N, K)
    qa, sa = oracle.quantize_q8_0(x)
    out, bound = oracle.qdot(qa, sa, w, w_s)
    C0 = pq.quantize_qdot_q8_0(dev(x), dev(w), dev(w_s))          # workspace route
    pq.check_device()
    assert_within_bound(C0, out, bound, "two-kernel route, workspace")
    A = torch.empty((M, K), dtype=torch.int8, device=DEV)
    AS = torch.empty((M, K // 32), dtype=torch.float32, device=DEV)
    C = pq.quantize_qdot_q8_0(dev(x), dev(w), dev(w_s), A=A, AS=AS)
    pq.check_device()
    assert_bytes_equal(A, AS, qa, sa)
    assert_within_bound(C, out, bound, "two-kernel route")


@pytest.mark.parametrize("name", [n for n in workloads.Q8_WORKLOADS if workloads.Q8_WORKLOADS[n].M <= 16])
def test_quantize_qdot_workload_full(pq, name):
    """Decode / small-batch workloads at full size through the one-call step."""
    x, w, qa, sa, qw, sw = quantized_workload(name)
    M, N = qa.shape[0], qw.shape[0]
    W, WS = pq.quantize_q8_0(dev(w))
    A = torch.empty(qa.shape, dtype=torch.int8, device=DEV)
    AS = torch.empty(sa.shape, dtype=torch.float32, device=DEV)
    C = pq.quantize_qdot_q8_0(dev(x), W, WS, A=A, AS=AS)
    pq.check_device()
    assert_bytes_equal(A, AS, qa, sa)
    rng = np.random.default_rng(2)
    cols = np.sort(rng.choice(N, min(N, 1024), replace=False))
    sampled_check(C, qa, sa, qw, sw, np.arange(M), cols, name)


# ------------------------------------------------------------------ host-buffer decode step

def _host_path(pq, which):
    import ctypes
    lib = pq.load()
    lib.pq_debug_set_host_path.argtypes = [ctypes.c_int]
    lib.pq_debug_set_host_path.restype = ctypes.c_int
    assert lib.pq_debug_set_host_path(which) == 0


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (1, 9800, 256), (4, 300, 1024), (1, 64, 256), (12, 500, 1024)])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("copies", [False, True], ids=["in_place", "copies"])
def test_quantize_qdot_host_buffers(pq, M, N, K, layout, copies):
    """x and C in page-locked host memory: x copied in, C written in place by the step's
    kernels (the default), or C copied out too (forced by the test hook); the result
    matches the oracle on the quantized rows, and a second call of another size on the
    same stream (workspace regrown) is correct too."""
    _host_path(pq, 1 if copies else 0)
    try:
        _host_buffers_case(pq, M, N, K, layout)
    finally:
        _host_path(pq, 0)


def test_quantize_qdot_pageable_host_buffers(pq):
    """Pageable (not page-locked) host buffers take the copy path: same results."""
    M, N, K = 1, 512, 1024
    rng = np.random.default_rng(77)
    x = rng.standard_normal((M, K)).astype(np.float32)
    _, _, w, w_s = rand_operands(78, 1, N, K)
    qa, sa = oracle.quantize_q8_0(x)
    out, bound = oracle.qdot(qa, sa, w, w_s)
    x_host = torch.from_numpy(x.copy())
    C_host = torch.full((M, N), float("nan"), dtype=torch.float32)
    assert not x_host.is_pinned() and not C_host.is_pinned()
    stream = torch.cuda.Stream()
    pq.quantize_qdot_q8_0_host(x_host, dev(w), dev(w_s), C_host, stream=stream)
    stream.synchronize()
    pq.check_device()
    assert_within_bound(C_host.numpy(), out, bound, "pageable host buffers")


def _host_buffers_case(pq, M, N, K, layout):
    rng = np.random.default_rng(M * 7 + N + K + layout)
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, size=(M, 1)))).astype(np.float32)
    _, _, w, w_s = rand_operands(N + 5 * K, 1, N, K)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    qa, sa = oracle.quantize_q8_0(x)
    out, bound = oracle.qdot(qa, sa, w, w_s)
    x_host = torch.from_numpy(x).pin_memory()
    C_host = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    stream = torch.cuda.Stream()
    W, WS = dev(w), dev(ws)
    torch.cuda.synchronize()
    pq.quantize_qdot_q8_0_host(x_host, W, WS, C_host, ws_layout=layout, stream=stream)
    stream.synchronize()
    pq.check_device()
    assert_within_bound(C_host.numpy(), out, bound, f"host step M={M} N={N} K={K} layout={layout}")
    # twice the rows on the same stream
    x2 = np.concatenate([x, x[::-1] * 0.5]).astype(np.float32)
    qa2, sa2 = oracle.quantize_q8_0(x2)
    out2, bound2 = oracle.qdot(qa2, sa2, w, w_s)
    C2 = torch.empty((2 * M, N), dtype=torch.float32).pin_memory()
    pq.quantize_qdot_q8_0_host(torch.from_numpy(x2).pin_memory(), W, WS, C2, ws_layout=layout, stream=stream)
    stream.synchronize()
    pq.check_device()
    assert_within_bound(C2.numpy(), out2, bound2, "host step, regrown workspace")
