"""Parsers for the hand-derived fixtures under tests/golden/ (test helper)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def quantize_blocks():
    """Yields (name, x f32[32], d f32, q int8[32]) from q8_0_quantize_blocks.txt."""
    out = []
    cur = None
    with open(os.path.join(GOLDEN, "q8_0_quantize_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                cur = {"name": vals[0]}
                out.append(cur)
            elif key == "x":
                x = np.zeros(32, np.float32)
                x[: len(vals)] = np.array([float(v) for v in vals], np.float32)
                cur["x"] = x
            elif key == "d":
                cur["d"] = np.float32(float.fromhex(vals[0]))
            elif key == "q":
                assert len(vals) == 32
                cur["q"] = np.array([int(v) for v in vals], np.int8)
    return [(b["name"], b["x"], b["d"], b["q"]) for b in out]


def qdot_cases():
    """Yields dicts with a, as, w, ws, expected {(i, j): value} from q8_0_qdot_worked.txt."""
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, "q8_0_qdot_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "out": {}}
                cases.append(cur)
            elif key == "shape":
                M, N, K = map(int, vals)
                KB = K // 32
                cur.update(M=M, N=N, K=K, a=np.zeros((M, K), np.int8), w=np.zeros((N, K), np.int8),
                           a_scales=np.zeros((M, KB), np.float32), w_scales=np.zeros((N, KB), np.float32))
            elif key in ("a", "w"):
                r, b, v = int(vals[0]), int(vals[1]), int(vals[2])
                cur[key][r, 32 * b: 32 * b + 32] = v
            elif key in ("as", "ws"):
                r = int(vals[0])
                arr = cur["a_scales" if key == "as" else "w_scales"]
                arr[r, :] = np.array([float(v) for v in vals[1:]], np.float32)
            elif key == "out":
                cur["out"][(int(vals[0]), int(vals[1]))] = float(vals[2])
    return cases


def q5_0_blocks():
    """Yields (name, bytes uint8[20], values int8[32]) from q5_0_blocks.txt."""
    out = []
    cur = None
    with open(os.path.join(GOLDEN, "q5_0_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                cur = {"name": vals[0]}
                out.append(cur)
            elif key == "bytes":
                assert len(vals) == 20
                cur["bytes"] = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "values":
                assert len(vals) == 32
                cur["values"] = np.array([int(v) for v in vals], np.int8)
    return [(b["name"], b["bytes"], b["values"]) for b in out]
