"""GPU parity for Q5_0 weights (q50_qdot_t) against the CPU oracle.

Bars as for Q8_0: integer block sums identical; outputs within
1e-5 * sum_b |t_b| + 1e-6 of the oracle's double result, element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads
from tests import golden_io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def operands(seed, M, N, K):
    rng = np.random.default_rng(seed)
    a = workloads.random_int8(rng, (M, K), -128, 127)
    w5 = rng.integers(0, 256, size=(N, K // 32 * 20), dtype=np.uint8)
    a_s = workloads.random_scales(rng, (M, K // 32), 1e-3, 10.0)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1.0)
    return a, a_s, w5, w_s


def within(C, out, bound, what):
    C = C.cpu().numpy().astype(np.float64)
    err = np.abs(C - out)
    assert np.all(err <= bound), f"{what}: {int((err > bound).sum())} outside, worst {np.max(err / bound):.3g}x"


SHAPES = [(1, 1, 32), (1, 7, 64), (1, 300, 1056), (2, 9, 96), (3, 17, 128), (5, 33, 256), (13, 70, 160),
          (1, 2, 14336), (64, 40, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q50_blocksums_exact(pq, M, N, K):
    a, _, w5, _ = operands(M * 3 + N + K, M, N, K)
    S = pq.q50_blocksums(dev(a), dev(w5))
    pq.check_device()
    assert np.array_equal(S.cpu().numpy().astype(np.int64), oracle.blocksums_q5_0(a, w5))


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_q50_qdot(pq, M, N, K, layout):
    a, a_s, w5, w_s = operands(M * 5 + N * 7 + K + layout, M, N, K)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, ws, ws_layout=layout)
    C = pq.q50_qdot(dev(a), dev(a_s), dev(w5), dev(ws), ws_layout=layout)
    pq.check_device()
    within(C, out, bound, f"q50 M={M} N={N} K={K} layout={layout}")


def test_q50_golden_blocks_on_gpu(pq):
    """The hand-derived blocks as one weight row; a one-hot activation reads each element back."""
    blocks = golden_io.q5_0_blocks()
    K = 32 * len(blocks)
    w5 = np.concatenate([b for _, b, _ in blocks])[None, :]
    values = np.concatenate([v for _, _, v in blocks]).astype(np.int64)
    # activation row e picks element e (a one-hot row per element of the first 64)
    M = 64
    a = np.zeros((M, K), np.int8)
    a[np.arange(M), np.arange(M)] = 1
    S = pq.q50_blocksums(dev(a), dev(w5))
    pq.check_device()
    got = S.cpu().numpy()[:, 0, :].sum(axis=1)
    assert got.tolist() == values[:M].tolist()


def test_q50_weight_base_4_byte_aligned(pq):
    """W5 needs only 4-byte alignment (20-byte blocks): an offset view gives the same result."""
    M, N, K = 2, 37, 256
    a, a_s, w5, w_s = operands(99, M, N, K)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, w_s)
    buf = torch.zeros(w5.size + 64, dtype=torch.uint8, device=DEV)
    view = buf[4:4 + w5.size].view(N, K // 32 * 20)
    view.copy_(dev(w5))
    C = pq.q50_qdot(dev(a), dev(a_s), view, dev(w_s))
    pq.check_device()
    within(C, out, bound, "offset W5")


def test_q50_workload_full(pq):
    """The Q5_0 decode workload at full size: Q8_0-quantized activations, sampled columns."""
    wl = workloads.WORKLOADS["q50_decode_m1_k4096_n4096"]
    x = workloads.activations(wl)
    qa, sa = oracle.quantize_q8_0(x)
    w5, ws = workloads.q50_weights(wl)
    C = pq.q50_qdot(dev(qa), dev(sa), dev(w5), dev(ws))
    pq.check_device()
    cols = np.sort(np.random.default_rng(3).choice(wl.N, 512, replace=False))
    out, bound = oracle.qdot_q5_0(qa, sa, w5[cols], ws[cols])
    within(C[:, torch.from_numpy(cols).to(DEV)], out, bound, "q50 decode full size")
    assert torch.isfinite(C).all()


# ------------------------------------------------------------ tensor-core route (M > 64)

TC_SHAPES = [(65, 64, 128), (130, 300, 512), (256, 129, 1024), (512, 256, 4096), (384, 2048, 1024)]
DEFAULT_PROMPT_KERNEL = 1  # scales in registers (include/pq_debug.h)


def _set_prompt_kernel(pq, which):
    import ctypes
    lib = pq.load()
    lib.pq_debug_set_prompt_kernel.argtypes = [ctypes.c_int]
    lib.pq_debug_set_prompt_kernel.restype = ctypes.c_int
    assert lib.pq_debug_set_prompt_kernel(which) == 0


@pytest.mark.parametrize("which", [0, 1], ids=["scale_product_mma", "scales_in_registers"])
@pytest.mark.parametrize("M,N,K", TC_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_q50_qdot_tensor_cores(pq, M, N, K, layout, which):
    """Prompt shapes take a tensor-core kernel, which decodes the Q5_0 blocks to f16 in
    shared memory: the one applying the scales in registers (the default) or the one with
    the scale-product MMA (ragged N, both scale layouts, split K at the small shapes, many
    tiles per CTA at the last)."""
    a, a_s, w5, w_s = operands(M * 11 + N + K + layout, M, N, K)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, ws, ws_layout=layout)
    try:
        _set_prompt_kernel(pq, which)
        C = pq.q50_qdot(dev(a), dev(a_s), dev(w5), dev(ws), ws_layout=layout)
        pq.check_device()
    finally:
        _set_prompt_kernel(pq, DEFAULT_PROMPT_KERNEL)
    within(C, out, bound, f"q50 tc kernel {which} M={M} N={N} K={K} layout={layout}")


def test_q50_tensor_cores_under_capture(pq):
    """Captured on a stream without a workspace yet: the kernel converts the activations
    itself; the replay is within tolerance."""
    M, N, K = 128, 192, 512
    a, a_s, w5, w_s = operands(5, M, N, K)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, w_s)
    A, AS, W5, WS = dev(a), dev(a_s), dev(w5), dev(w_s)
    C = torch.full((M, N), float("nan"), device=DEV)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pq.q50_qdot(A, AS, W5, WS, C)
    g.replay()
    torch.cuda.synchronize()
    pq.check_device()
    within(C, out, bound, "q50 tc captured")


def test_q50_prompt_unaligned_weights_fall_back(pq):
    """W5 only 4-byte aligned at a prompt shape: the tensor-core kernel declines (TMA wants 16
    bytes) and the dp4a kernel gives the same result."""
    M, N, K = 96, 40, 256
    a, a_s, w5, w_s = operands(123, M, N, K)
    out, bound = oracle.qdot_q5_0(a, a_s, w5, w_s)
    buf = torch.zeros(w5.size + 64, dtype=torch.uint8, device=DEV)
    view = buf[4:4 + w5.size].view(N, K // 32 * 20)
    view.copy_(dev(w5))
    C = pq.q50_qdot(dev(a), dev(a_s), view, dev(w_s))
    pq.check_device()
    within(C, out, bound, "q50 offset W5, prompt shape")


@pytest.mark.parametrize("which", [0, 1], ids=["scale_product_mma", "scales_in_registers"])
def test_q50_prompt_workload_full(pq, which):
    """The Q5_0 prompt workload at full size through both tensor-core kernels: one complete
    row per 128-row band and one complete column per 128-column band, so that every
    128 x 128 output tile (every unit of the persistent CTAs) is checked."""
    wl = workloads.WORKLOADS["q50_prompt_m512_k4096_n14336"]
    x = workloads.activations(wl)
    qa, sa = oracle.quantize_q8_0(x)
    w5, ws = workloads.q50_weights(wl)
    try:
        _set_prompt_kernel(pq, which)
        C = pq.q50_qdot(dev(qa), dev(sa), dev(w5), dev(ws))
        pq.check_device()
    finally:
        _set_prompt_kernel(pq, DEFAULT_PROMPT_KERNEL)
    rng = np.random.default_rng(4)
    rows = np.array([b + rng.integers(0, min(128, wl.M - b)) for b in range(0, wl.M, 128)])
    cols = np.array([b + rng.integers(0, min(128, wl.N - b)) for b in range(0, wl.N, 128)])
    out, bound = oracle.qdot_q5_0(qa[rows], sa[rows], w5, ws, omp=True)
    within(C[torch.from_numpy(rows).to(DEV)], out, bound, "q50 prompt full size, rows")
    out, bound = oracle.qdot_q5_0(qa, sa, w5[cols], ws[cols], omp=True)
    within(C[:, torch.from_numpy(cols).to(DEV)], out, bound, "q50 prompt full size, columns")
    assert torch.isfinite(C).all()


# ------------------------------------------------------------ fused quantize + q50_qdot_t

FUSED_SHAPES = [(1, 1, 32), (1, 300, 1056), (1, 4096, 4096), (1, 40, 14336), (1, 9000, 128), (1, 9800, 256),
                (3, 65, 256), (8, 100, 1024)]


@pytest.mark.parametrize("M,N,K", FUSED_SHAPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_q50_qdot(pq, M, N, K, layout):
    """One call: the quantized rows bit-identical to the oracle's quantizer, the result
    within tolerance of the oracle's q50_qdot_t on those rows (one kernel for M = 1 while
    the grid fits two waves, the quantizer then q50_qdot_t otherwise)."""
    rng = np.random.default_rng(M * 11 + N + K + layout)
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, size=(M, 1)))).astype(np.float32)
    _, _, w5, w_s = operands(N * 3 + K, 1, N, K)
    qa, sa = oracle.quantize_q8_0(x)
    ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
    out, bound = oracle.qdot_q5_0(qa, sa, w5, ws, ws_layout=layout)
    A = torch.full((M, K), 77, dtype=torch.int8, device=DEV)
    AS = torch.full((M, K // 32), -1.0, dtype=torch.float32, device=DEV)
    C = pq.quantize_q50_qdot(dev(x), dev(w5), dev(ws), A=A, AS=AS, ws_layout=layout)
    pq.check_device()
    assert np.array_equal(A.cpu().numpy(), qa)
    assert np.array_equal(AS.cpu().numpy().view(np.uint32), sa.view(np.uint32))
    within(C, out, bound, f"fused q50 M={M} N={N} K={K} layout={layout}")
    C2 = pq.quantize_q50_qdot(dev(x), dev(w5), dev(ws), ws_layout=layout)  # without A / AS
    pq.check_device()
    within(C2, out, bound, "fused q50, no A/AS")
