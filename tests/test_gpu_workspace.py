"""The tensor-core path's per-stream workspace (pre-tiled activations for M > 64).

For prompt-sized M the library converts the activations once per call into a
workspace that belongs to the (device, stream) pair; it must not allocate
while the stream is being captured into a CUDA graph (the kernel then converts
the activations itself), and calls on two streams must not share a workspace.
Every expected value comes from the CPU oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_q8_qdot_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _operands(seed, M, N, K):
    rng = np.random.default_rng(seed)
    a = workloads.random_int8(rng, (M, K), -127, 127)
    w = workloads.random_int8(rng, (N, K), -127, 127)
    a_s = workloads.random_scales(rng, (M, K // 32), 1e-3, 10.0)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1.0)
    return a, a_s, w, w_s


def _check(C, a, a_s, w, w_s, what):
    out, bound = oracle.qdot(a, a_s, w, w_s)
    err = np.abs(C.cpu().numpy().astype(np.float64) - out)
    assert np.all(err <= bound), f"{what}: {int((err > bound).sum())} outside tolerance"


def test_capture_on_a_fresh_stream_then_eager_then_capture(pq):
    """Captured before the stream has a workspace (no allocation allowed), eagerly
    (allocates it), captured again (uses it): all three within tolerance."""
    M, N, K = 192, 256, 1024
    a, a_s, w, w_s = _operands(11, M, N, K)
    A, AS, W, WS = (torch.from_numpy(v).to(DEV) for v in (a, a_s, w, w_s))
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    C1 = torch.full((M, N), float("nan"), device=DEV)
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        pq.qdot_q8_0(A, AS, W, WS, C1)
    g1.replay()
    torch.cuda.synchronize()
    pq.check_device()
    _check(C1, a, a_s, w, w_s, "captured without a workspace")
    with torch.cuda.stream(stream):
        C2 = pq.qdot_q8_0(A, AS, W, WS)
    stream.synchronize()
    pq.check_device()
    _check(C2, a, a_s, w, w_s, "eager (workspace allocated)")
    C3 = torch.full((M, N), float("nan"), device=DEV)
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=stream):
        pq.qdot_q8_0(A, AS, W, WS, C3)
    for _ in range(2):
        g3.replay()
    torch.cuda.synchronize()
    pq.check_device()
    _check(C3, a, a_s, w, w_s, "captured with the workspace")


def test_two_streams_do_not_share_a_workspace(pq):
    """Prompt-shaped calls on two streams, issued alternately without synchronizing
    in between: each stream's results stay those of its own inputs."""
    M, N, K = 256, 384, 2048
    ops = [_operands(20 + i, M, N, K) for i in range(2)]
    dev_ops = [tuple(torch.from_numpy(v).to(DEV) for v in o) for o in ops]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty((M, N), device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(3):
        for i in (0, 1):
            with torch.cuda.stream(streams[i]):
                A, AS, W, WS = dev_ops[i]
                pq.qdot_q8_0(A, AS, W, WS, outs[i])
    torch.cuda.synchronize()
    pq.check_device()
    for i in (0, 1):
        _check(outs[i], *ops[i], f"stream {i}")


@pytest.mark.parametrize("M", [65, 130, 512])
def test_prompt_path_with_and_without_workspace_agree(pq, M):
    """The pre-tiled activations (allocating entry point) and the in-kernel conversion
    (allocation-free entry point) give results within the oracle's tolerance."""
    N, K = 320, 1024
    rng = np.random.default_rng(M)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = workloads.random_int8(rng, (N, K), -127, 127)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1e-2)
    X, W, WS = (torch.from_numpy(v).to(DEV) for v in (x, w, w_s))
    C_a = pq.quantize_qdot_q8_0(X, W, WS)
    C_n = pq.quantize_qdot_q8_0_noalloc(X, W, WS)
    torch.cuda.synchronize()
    pq.check_device()
    qa, sa = oracle.quantize_q8_0(x)
    _check(C_a, qa, sa, w, w_s, "with workspace")
    _check(C_n, qa, sa, w, w_s, "without workspace")
