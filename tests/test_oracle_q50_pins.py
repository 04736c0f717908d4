"""Pins for the oracle's Q5_0 weight path (q50_qdot_t), none computed by the oracle itself.

* hand-derived block decodes (tests/golden/q5_0_blocks.txt) from the format on
  the pages ("Phobos Language Spec" section 10, Q5_0 row; "Quantized built-ins
  and formats", built-in table) and the reading of the qh bit order;
* an independent Python decode of random blocks (bit operations on Python
  ints), compared element by element;
* q50_qdot_t against the separately pinned Q8_0 qdot_t applied to the
  Python-decoded weights (the pages define q50_qdot_t as qdot_t against the
  decoded elements q - 16);
* brute-force block sums in Python integers, closed forms, and the qmma_t
  scale layout.

Each pin also runs against deliberately broken builds (qh bit order reversed,
nibble halves swapped, the -16 offset dropped); each must fail at least one pin.
"""
import numpy as np
import pytest

import oracle
from gemm_q8_qdot_gb300 import workloads
from tests import golden_io

MUTANTS = {
    9: "qh bit order reversed",
    10: "nibble halves swapped",
    11: "minus-16 offset dropped",
}


def py_decode_block(blk) -> list[int]:
    """One 20-byte Q5_0 block -> 32 ints, written from the format description."""
    qh = int(blk[0]) | int(blk[1]) << 8 | int(blk[2]) << 16 | int(blk[3]) << 24
    vals = []
    for e in range(32):
        byte = int(blk[4 + e % 16])
        nib = byte & 0xF if e < 16 else byte >> 4
        vals.append((nib | ((qh >> e) & 1) << 4) - 16)
    return vals


def py_decode(w5, K) -> np.ndarray:
    R = w5.shape[0]
    out = np.empty((R, K), np.int8)
    for r in range(R):
        for b in range(K // 32):
            out[r, 32 * b: 32 * b + 32] = py_decode_block(w5[r, 20 * b: 20 * b + 20])
    return out


def random_q50(rng, rows, K) -> np.ndarray:
    return rng.integers(0, 256, size=(rows, K // 32 * 20), dtype=np.uint8)


def pin_q50_golden(mutant=0):
    for name, blk, values in golden_io.q5_0_blocks():
        got = oracle.decode_q5_0(blk[None, :], 32, mutant=mutant)[0]
        assert got.tolist() == values.tolist(), name


def pin_q50_python_decode(mutant=0):
    rng = np.random.default_rng(21)
    w5 = random_q50(rng, 5, 96)
    assert np.array_equal(oracle.decode_q5_0(w5, 96, mutant=mutant), py_decode(w5, 96))


def pin_q50_qdot_reduces_to_q8(mutant=0):
    rng = np.random.default_rng(22)
    for M, N, K, layout in ((1, 3, 32, 0), (3, 4, 96, 0), (2, 5, 128, 1)):
        a = workloads.random_int8(rng, (M, K))
        w5 = random_q50(rng, N, K)
        a_s = workloads.random_scales(rng, (M, K // 32))
        w_s = workloads.random_scales(rng, (N, K // 32))
        ws = w_s if layout == 0 else np.ascontiguousarray(w_s.T)
        out, bound = oracle.qdot_q5_0(a, a_s, w5, ws, ws_layout=layout, mutant=mutant)
        ref, ref_bound = oracle.qdot(a, a_s, py_decode(w5, K), ws, ws_layout=layout)
        assert np.array_equal(out, ref) and np.array_equal(bound, ref_bound)


def pin_q50_blocksums_bruteforce(mutant=0):
    rng = np.random.default_rng(23)
    M, N, K = 2, 3, 64
    a = workloads.random_int8(rng, (M, K), -128, 127)
    w5 = random_q50(rng, N, K)
    S = oracle.blocksums_q5_0(a, w5, mutant=mutant)
    for i in range(M):
        for j in range(N):
            for b in range(K // 32):
                vals = py_decode_block(w5[j, 20 * b: 20 * b + 20])
                assert S[i, j, b] == sum(int(a[i, 32 * b + e]) * vals[e] for e in range(32))


def pin_q50_closed_forms(mutant=0):
    K = 128
    a = np.ones((2, K), np.int8)
    ones = np.full((3, K // 32 * 20), 0xFF, np.uint8)      # every element 15
    zeros = np.zeros((3, K // 32 * 20), np.uint8)          # every element -16
    assert np.all(oracle.blocksums_q5_0(a, ones, mutant=mutant) == 32 * 15)
    assert np.all(oracle.blocksums_q5_0(a, zeros, mutant=mutant) == -32 * 16)
    out, _ = oracle.qdot_q5_0(a, np.full((2, K // 32), 0.5, np.float32), ones,
                              np.full((3, K // 32), 0.25, np.float32), mutant=mutant)
    assert np.all(out == K * 15 * 0.125)


def pin_q50_qmma_layout(mutant=0):
    rng = np.random.default_rng(24)
    M, N, K = 2, 3, 64
    a = workloads.random_int8(rng, (M, K))
    w5 = random_q50(rng, N, K)
    a_s = workloads.random_scales(rng, (M, K // 32))
    w_s = workloads.random_scales(rng, (N, K // 32))
    o0, _ = oracle.qdot_q5_0(a, a_s, w5, w_s, ws_layout=0, mutant=mutant)
    o1, _ = oracle.qdot_q5_0(a, a_s, w5, np.ascontiguousarray(w_s.T), ws_layout=1, mutant=mutant)
    assert np.array_equal(o0, o1)


PINS = [pin_q50_golden, pin_q50_python_decode, pin_q50_qdot_reduces_to_q8, pin_q50_blocksums_bruteforce,
        pin_q50_closed_forms, pin_q50_qmma_layout]


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


def test_golden_reading_of_qh_is_what_the_python_decode_does():
    """The hand-derived fixture and the Python decode agree (both written from the format text)."""
    for name, blk, values in golden_io.q5_0_blocks():
        assert py_decode_block(blk) == values.tolist(), name
