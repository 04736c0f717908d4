"""The split of qdot_t across ranks (gemm_q8_qdot_gb300.sharded) on CPU: two gloo ranks.

Each rank holds its shard of the weight rows (column split) or of the activation
rows (row split) and computes its part with a local contraction; the gather
assembles the full C.  On GPUs the local contraction is the library's kernel on
the rank's own device memory; here, with no GPU, the test hands the splitter the
oracle as its local contraction, so what is checked is the partitioning, the
padding of unequal shards and the gather.  The gathered C is compared with the
oracle run on the whole problem, element by element, within the qdot_t
tolerance.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from gemm_q8_qdot_gb300 import sharded, workloads  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_qdot(A, AS, W, WS, layout):
    import oracle
    out, _ = oracle.qdot(A.numpy(), AS.numpy(), W.numpy(), WS.numpy(), ws_layout=layout)
    return torch.from_numpy(out.astype(np.float32))


def _oracle_step(x, W, WS, layout):
    import oracle
    qa, sa = oracle.quantize_q8_0(x.numpy())
    return _oracle_qdot(torch.from_numpy(qa), torch.from_numpy(sa), W, WS, layout)


def _problem(M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = workloads.random_int8(rng, (N, K), -127, 127)
    w_s = workloads.random_scales(rng, (N, K // 32), 1e-4, 1e-1)
    return x, w, w_s


def _worker(rank, world, port, cases, q):
    try:
        _run(rank, world, port, cases, q)
    except BaseException as e:  # report instead of leaving the other rank waiting
        q.put((rank, repr(e)))
        raise


def _run(rank, world, port, cases, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=__import__("datetime").timedelta(seconds=60))
    import oracle
    results = []
    for (M, N, K, layout) in cases:
        x, w, w_s = _problem(M, N, K, M * 1000 + N * 10 + K + layout)
        qa, sa = oracle.quantize_q8_0(x)
        W = torch.from_numpy(w)
        WS = torch.from_numpy(w_s if layout == 0 else np.ascontiguousarray(w_s.T))
        Wl, WSl = sharded.shard_weights(W, WS, world, rank, layout)
        col = sharded.ColumnSplit(Wl, WSl, N, world, rank, ws_layout=layout,
                                  local_qdot=_oracle_qdot, local_step=_oracle_step)
        C_col = col.qdot(torch.from_numpy(qa), torch.from_numpy(sa))
        C_step = col.step(torch.from_numpy(x))
        C_local = col.qdot(torch.from_numpy(qa), torch.from_numpy(sa), gather=False)
        row = sharded.RowSplit(W, WS, world, rank, ws_layout=layout, local_qdot=_oracle_qdot)
        C_row = row.qdot(torch.from_numpy(qa), torch.from_numpy(sa))
        results.append((C_col.numpy(), C_step.numpy(), C_local.numpy(), C_row.numpy()))
    dist.destroy_process_group()
    q.put((rank, results))


CASES = [(1, 64, 256, 0),    # even split of the columns, one activation row (decode)
         (5, 37, 96, 0),     # odd N and odd M: unequal shards, padded for the gather
         (3, 9, 128, 1),     # the qmma_t scale layout [K/32, N]
         (1, 1, 32, 0)]      # fewer weight rows than ranks: one rank holds none


def test_split_qdot_matches_the_whole_problem():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, CASES, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, res = q.get(timeout=300)
        assert not isinstance(res, str), f"rank {rank} failed: {res}"
        out[rank] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    for ci, (M, N, K, layout) in enumerate(CASES):
        x, w, w_s = _problem(M, N, K, M * 1000 + N * 10 + K + layout)
        qa, sa = oracle.quantize_q8_0(x)
        ref, bound = oracle.qdot(qa, sa, w, w_s)
        for rank in range(world):
            C_col, C_step, C_local, C_row = out[rank][ci]
            for what, C in (("column split", C_col), ("column-split step", C_step), ("row split", C_row)):
                assert C.shape == (M, N), (what, C.shape)
                err = np.abs(C.astype(np.float64) - ref)
                assert np.all(err <= bound), f"{what} {M}x{N}x{K} rank {rank}: {int((err > bound).sum())} bad"
            lo, hi = sharded.shard_range(N, world, rank)
            assert C_local.shape == (M, hi - lo)
            assert np.all(np.abs(C_local.astype(np.float64) - ref[:, lo:hi]) <= bound[:, lo:hi])


def test_shard_range_covers_every_row_once():
    for n in (0, 1, 2, 7, 4096, 14336, 11008):
        for world in (1, 2, 3, 8):
            spans = [sharded.shard_range(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[r][1] == spans[r + 1][0] for r in range(world - 1))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharded.shard_range(10, 2, 2)
