"""Pins for the CPU oracle: values and properties fixed by the pages and by
mathematics, none of them computed by the oracle itself.

* hand-derived blocks for the quantizer (ties-to-even ``round`` from the spec's
  Elementwise table; the d = amax/127 reading) -- tests/golden/;
* hand-derived qdot_t values from the "Quantized built-ins and formats" Q8_0
  formula -- tests/golden/;
* brute force in exact rational arithmetic on tiny inputs (Python ints and
  fractions.Fraction, independent of the C code);
* a float64 library matmul (torch, CPU) of the dequantized operands, the
  textbook special case of qdot_t;
* closed forms and invariants (scale linearity, transpose symmetry, additivity
  over K, quantizer round-trip bounds).

Each pin is also run against deliberately broken builds of the oracle
(``ORACLE_MUTANT``); every mutant must fail at least one pin.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from gemm_q8_qdot_gb300 import workloads
from tests import golden_io

MUTANTS = {
    1: "round ties away from zero",
    2: "truncate instead of round",
    3: "scale divisor 128",
    5: "a zero-extended instead of sign-extended",
    6: "last K block dropped",
    7: "activation scale row index ignored",
    8: "activation and weight operands swapped",
}


# ---------------------------------------------------------------- quantizer pins

def pin_quantize_golden(mutant=0):
    for name, x, d, q in golden_io.quantize_blocks():
        qo, so = oracle.quantize_q8_0(x[None, :], mutant=mutant)
        assert so[0, 0].view(np.uint32) == np.float32(d).view(np.uint32), (name, so[0, 0], d)
        assert np.array_equal(qo[0], q), (name, qo[0], q)


def pin_quantize_invariants(mutant=0):
    rng = np.random.default_rng(7)
    R, K = 64, 256
    x = rng.standard_normal((R, K)).astype(np.float32)
    x *= np.exp(rng.uniform(-20, 20, size=(R, 1))).astype(np.float32)  # tiny to huge rows
    x[3, 32:64] = 0.0                              # an all-zero block
    x[5, 64:96] = np.float32(3.25)                 # a constant block
    q, s = oracle.quantize_q8_0(x, mutant=mutant)
    xb = x.reshape(R, K // 32, 32).astype(np.float64)
    qb = q.reshape(R, K // 32, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    d = s.astype(np.float64)
    assert np.all(np.abs(qb) <= 127)
    nz = amax > 0
    assert np.all(d[~nz] == 0) and np.all(qb[~nz] == 0)
    # d is amax / 127 rounded once to f32: within half an f32 ulp of the exact quotient
    rel = np.abs(d[nz] * 127.0 - amax[nz]) / amax[nz]
    assert np.all(rel <= 2.0 ** -24 * 1.0001), rel.max()
    # every nonzero block reaches +-127 at its largest element
    assert np.all(np.abs(qb).max(axis=2)[nz] == 127)
    # round-to-nearest of the f32 quotient: |x/d - q| <= 1/2 + (rounding of x/d, at most
    # 2^-24 * |x/d| <= 2^-24 * 128 = 2^-17)
    err = np.abs(xb - qb * d[:, :, None])
    assert np.all(err <= d[:, :, None] * (0.5 + 2.0 ** -17 + 1e-12)), (err / np.maximum(d[:, :, None], 1e-300)).max()
    # the sign of q follows x (q = 0 allowed)
    assert np.all(qb * np.sign(xb) >= 0)


def pin_quantize_requantize(mutant=0):
    """Quantizing the dequantized values q*d again gives back the same bytes."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    q, s = oracle.quantize_q8_0(x, mutant=mutant)
    xd = (q.reshape(16, 4, 32).astype(np.float32) * s[:, :, None]).reshape(16, 128)
    q2, _ = oracle.quantize_q8_0(xd, mutant=mutant)
    assert np.array_equal(q, q2)


# ---------------------------------------------------------------- contraction pins

def pin_qdot_golden(mutant=0):
    for c in golden_io.qdot_cases():
        out, bound = oracle.qdot(c["a"], c["a_scales"], c["w"], c["w_scales"], mutant=mutant)
        for (i, j), v in c["out"].items():
            assert out[i, j] == v, (c["name"], i, j, out[i, j], v)


def _fraction_qdot(a, a_s, w, w_s):
    """Exact value of the qdot_t sum in rationals, by brute force over (i, j, b, k)."""
    M, K = a.shape
    N = w.shape[0]
    KB = K // 32
    res = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            tot = Fraction(0)
            for b in range(KB):
                s = 0
                for k in range(32 * b, 32 * b + 32):
                    s += int(a[i, k]) * int(w[j, k])
                tot += Fraction(float(a_s[i, b])) * Fraction(float(w_s[j, b])) * s
            res[i][j] = tot
    return res


def pin_qdot_bruteforce(mutant=0):
    rng = np.random.default_rng(3)
    for (M, N, K) in [(1, 1, 32), (2, 3, 64), (3, 2, 96), (5, 4, 32), (4, 5, 64)]:
        a = workloads.random_int8(rng, (M, K))
        w = workloads.random_int8(rng, (N, K))
        a[0, 0] = -128
        w[-1, -1] = -128
        a_s = workloads.random_scales(rng, (M, K // 32))
        w_s = workloads.random_scales(rng, (N, K // 32))
        out, bound = oracle.qdot(a, a_s, w, w_s, mutant=mutant)
        exact = _fraction_qdot(a, a_s, w, w_s)
        S = oracle.blocksums(a, w, mutant=mutant)
        for i in range(M):
            for j in range(N):
                # integer block sums, exactly
                for b in range(K // 32):
                    ref = sum(int(a[i, k]) * int(w[j, k]) for k in range(32 * b, 32 * b + 32))
                    assert S[i, j, b] == ref
                assert abs(Fraction(out[i, j]) - exact[i][j]) <= Fraction(1, 10 ** 12) * (abs(exact[i][j]) + 1e-30) + Fraction(1, 10 ** 15)


def pin_qdot_matmul(mutant=0):
    """qdot_t equals the float64 matmul of the dequantized operands (M != N != K)."""
    import torch
    rng = np.random.default_rng(5)
    M, N, K = 6, 9, 128
    a = workloads.random_int8(rng, (M, K))
    w = workloads.random_int8(rng, (N, K))
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    out, bound = oracle.qdot(a, a_s, w, w_s, mutant=mutant)
    ad = torch.from_numpy(a.astype(np.float64)) * torch.from_numpy(np.repeat(a_s.astype(np.float64), 32, axis=1))
    wd = torch.from_numpy(w.astype(np.float64)) * torch.from_numpy(np.repeat(w_s.astype(np.float64), 32, axis=1))
    ref = (ad @ wd.T).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), np.abs(out - ref).max()


def pin_qdot_closed_forms(mutant=0):
    for K in (32, 256, 4096):
        a = np.ones((2, K), np.int8)
        w = np.ones((3, K), np.int8)
        out, _ = oracle.qdot(a, np.full((2, K // 32), 0.5, np.float32), w,
                             np.full((3, K // 32), 0.25, np.float32), mutant=mutant)
        assert np.all(out == K / 8.0)
        a = np.full((1, K), -128, np.int8)
        w = np.full((2, K), -128, np.int8)
        S = oracle.blocksums(a, w, mutant=mutant)
        assert np.all(S == 32 * 128 * 128)


def pin_qdot_invariants(mutant=0):
    rng = np.random.default_rng(9)
    M, N, K = 4, 7, 192
    a = workloads.random_int8(rng, (M, K))
    w = workloads.random_int8(rng, (N, K))
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    out, _ = oracle.qdot(a, a_s, w, w_s, mutant=mutant)
    # linearity in each scale plane (powers of two are exact)
    a_s2 = a_s.copy()
    a_s2[2] *= 2
    out2, _ = oracle.qdot(a, a_s2, w, w_s, mutant=mutant)
    assert np.array_equal(out2[2], 2 * out[2]) and np.array_equal(np.delete(out2, 2, 0), np.delete(out, 2, 0))
    w_s2 = w_s.copy()
    w_s2[4] *= 0.5
    out3, _ = oracle.qdot(a, a_s, w, w_s2, mutant=mutant)
    assert np.array_equal(out3[:, 4], 0.5 * out[:, 4])
    # transpose symmetry: qdot(A, W) = qdot(W, A)^T
    outT, _ = oracle.qdot(w, w_s, a, a_s, mutant=mutant)
    assert np.allclose(outT.T, out, rtol=1e-14, atol=0)
    # additivity over K: the two halves sum to the whole
    h = K // 2
    o1, _ = oracle.qdot(a[:, :h], a_s[:, : h // 32], w[:, :h], w_s[:, : h // 32], mutant=mutant)
    o2, _ = oracle.qdot(a[:, h:], a_s[:, h // 32:], w[:, h:], w_s[:, h // 32:], mutant=mutant)
    assert np.allclose(o1 + o2, out, rtol=1e-13, atol=1e-300)


def pin_qmma_layout(mutant=0):
    """qmma_t's [K/32, N] scale layout gives the same sums as qdot_t's [N, K/32]."""
    rng = np.random.default_rng(13)
    M, N, K = 3, 5, 96
    a = workloads.random_int8(rng, (M, K))
    w = workloads.random_int8(rng, (N, K))
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    o0, _ = oracle.qdot(a, a_s, w, w_s, ws_layout=0, mutant=mutant)
    o1, _ = oracle.qdot(a, a_s, w, np.ascontiguousarray(w_s.T), ws_layout=1, mutant=mutant)
    assert np.array_equal(o0, o1)


def pin_bound(mutant=0):
    """The tolerance is 1e-5 * sum_b |t_b| + 1e-6 with t_b the per-block terms."""
    c = golden_io.qdot_cases()[0]
    out, bound = oracle.qdot(c["a"], c["a_scales"], c["w"], c["w_scales"], mutant=mutant)
    # case "mixed": |t| = (32, 32) and (6, 1024)
    assert bound[0, 0] == pytest.approx(1e-5 * 64 + 1e-6, rel=1e-15)
    assert bound[0, 1] == pytest.approx(1e-5 * 1030 + 1e-6, rel=1e-15)


PINS = [pin_quantize_golden, pin_quantize_invariants, pin_quantize_requantize, pin_qdot_golden,
        pin_qdot_bruteforce, pin_qdot_matmul, pin_qdot_closed_forms, pin_qdot_invariants,
        pin_qmma_layout, pin_bound]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_mutant_is_caught(mutant):
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


def test_oracle_on_workload_shapes():
    """The oracle quantizes the seeded workload inputs with the format's invariants."""
    wl = workloads.WORKLOADS["parity_m1_k256_n64"]
    x = workloads.activations(wl)
    w = workloads.weights(wl)
    qa, sa = oracle.quantize_q8_0(x)
    qw, sw = oracle.quantize_q8_0(w)
    assert qa.shape == (1, 256) and sa.shape == (1, 8) and qw.shape == (64, 256) and sw.shape == (64, 8)
    out, bound = oracle.qdot(qa, sa, qw, sw)
    # dequantized product is close to the f32 product it approximates (Q8_0 error ~ 1%)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.abs(out - ref).max() <= 0.05 * np.abs(ref).max()


def test_threaded_build_gives_the_same_bytes():
    """The OpenMP build of the oracle (loops over rows and output elements shared among the
    host cores, each element computed by the same sequential loop) returns exactly what the
    single-thread build returns: quantized bytes, scales, block sums and qdot_t values."""
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((37, 256)) * np.exp(rng.uniform(-8, 8, (37, 1)))).astype(np.float32)
    q1, s1 = oracle.quantize_q8_0(x)
    q2, s2 = oracle.quantize_q8_0(x, omp=True)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    a, a_s = q1[:5], s1[:5]
    w, w_s = q1[5:], s1[5:]
    assert np.array_equal(oracle.blocksums(a, w), oracle.blocksums(a, w, omp=True))
    for layout in (0, 1):
        ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
        o1, b1 = oracle.qdot(a, a_s, w, ws, ws_layout=layout)
        o2, b2 = oracle.qdot(a, a_s, w, ws, ws_layout=layout, omp=True)
        assert np.array_equal(o1.view(np.uint64), o2.view(np.uint64))
        assert np.array_equal(b1.view(np.uint64), b2.view(np.uint64))
    w5 = rng.integers(0, 256, (32, 256 // 32 * 20), dtype=np.uint8)
    assert np.array_equal(oracle.decode_q5_0(w5, 256), oracle.decode_q5_0(w5, 256, omp=True))
    assert np.array_equal(oracle.blocksums_q5_0(a, w5), oracle.blocksums_q5_0(a, w5, omp=True))
    ws5 = np.abs(workloads.random_scales(rng, (32, 8)))
    o1, _ = oracle.qdot_q5_0(a, a_s, w5, ws5)
    o2, _ = oracle.qdot_q5_0(a, a_s, w5, ws5, omp=True)
    assert np.array_equal(o1.view(np.uint64), o2.view(np.uint64))
