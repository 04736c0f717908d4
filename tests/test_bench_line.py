"""The benchmark's final JSON line on CPU: every workload's figures stay in its last
part, and the line stays short enough to be kept whole by a reader that keeps only the
end of the output."""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gemm_q8_qdot_gb300 import workloads  # noqa: E402

OTHERS = ("prompt_m512_k4096_n14336", "ffn_up_m1_k4096_n14336", "ffn_down_m1_k14336_n4096",
          "smallm_m4_k4096_n11008", "smallm_m16_k4096_n11008", "smallm_m64_k4096_n11008",
          "q50_decode_m1_k4096_n4096", "q50_prompt_m512_k4096_n14336")


def _fake(name):
    wl = workloads.WORKLOADS[name]
    tensor = wl.M > 64
    rl = {"bound": "tensor" if tensor else "hbm", "achieved": 12345.6789, "peak": 6775.6,
          "unit": "TFLOP/s" if tensor else "GB/s", "frac": 0.123456, "traffic": 123456789.0,
          "kernel": "qdot_tc", "peak_source": "measured hbm_gbs", "algorithmic_bytes": 123456789}
    if tensor:
        rl.update(int8_library_tops=155.5, frac_of_int8_library=2.034)
    extra = {} if tensor else {"stream_reader_ms": {"chained": 0.0047612, "early": 0.0040123},
                               "e2e_copies": {"value": 604.123, "unit": "GB/s"}}
    return {**extra, "value": 12345.678, "unit": "TOPS" if tensor else "GB/s", "ms_per_step": 0.1234567,
            "step": "pq_quantize_q8_0 + pq_qdot_q8_0", "roofline": rl, "weight_copies": 15,
            "kernel_ms": {"dominant": 0.12345}, "e2e": {"value": 604.123, "unit": "GB/s",
                                                        "h2d_bytes_per_step": 16384, "d2h_bytes_per_step": 16384}}


def _cpu(name):
    return {"value": 12.34567, "unit": "GB/s", "cores": 144, "kind": "oracle",
            "cpu": "Neoverse-V2 (a long model name string)", "single_thread": 1.23456,
            "sample": f"{name}: x quantized + contracted with the first 4096 of 14336 weight rows, "
                      "1234 steps in 4.0 s on every core; single thread 456 rows, 12 steps in 4.0 s"}


def _line():
    args = argparse.Namespace(workload=bench.HEADLINE, steps=20, warmup=5)
    head = _fake(bench.HEADLINE)
    others = {n: _fake(n) for n in OTHERS}
    cpus = {n: _cpu(n) for n in (bench.HEADLINE,) + OTHERS}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"], "samples": 123}
    return bench.final_line(head, others, cpus, args, 1, clocks)


def test_final_line_holds_every_workload_at_its_end():
    line = _line()
    text = json.dumps(line)
    assert list(line)[-2:] == ["prompt", "workloads"]
    assert set(line["workloads"]) == {"fields", bench.HEADLINE, *OTHERS}
    fields = line["workloads"]["fields"]
    assert fields == ["value", "unit", "ms_per_step", "roofline_frac", "cpu_baseline_value"]
    for n in (bench.HEADLINE,) + OTHERS:
        assert len(line["workloads"][n]) == len(fields)
        assert line["workloads"][n][fields.index("cpu_baseline_value")] == 12.35
    # the prompt GEMM (second half of the metric) and every workload fit in the last
    # 1400 characters of the line, and the whole line stays under 3000 characters
    tail = text[-1400:]
    assert '"prompt": {' in tail and '"workloads": {' in tail
    assert len(text) < 3000, len(text)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks"):
        assert k in line, k
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in line["roofline"] and k in line["prompt"]["roofline"], k
    assert set(line["step_variants"]) == {"reader_chained_ms", "reader_early_ms", "e2e_with_copies"}


def test_compact_keeps_errors_short():
    assert bench.compact({"error": "x" * 500}) == {"error": "x" * 80}
