"""Q8_0 block-scaled contraction (qdot_t) and row quantizer for GB300 (sm_103a).

The compute runs in libpq.so (hand-written CUDA kernels behind the C ABI in
include/pq.h); this package holds the ctypes binding, the build step and the
seeded workload generators.
"""
from .binding import (EXPORTS, PATH_AUTO, PATH_MMA, PATH_SIMT, PATH_TC, PQ_ERR_ALIGN, PQ_ERR_CUDA,
                      PQ_ERR_INVALID_ARG, PQ_ERR_SCRATCH, PQ_ERR_SHAPE, PQ_ERR_TIMEOUT, PQ_ERR_UNSUPPORTED,
                      PQ_OK, debug_stream_read, quantize_qdot_q8_0_host, quantize_qdot_q8_0_noalloc, q50_qdot, quantize_q50_qdot, q50_blocksums,
                      WS_KB_N, WS_N_KB, PQError, check_device, lib_path, load, qdot_q8_0,
                      qdot_q8_0_blocksums, qdot_q8_0_ex, quantize_q8_0, quantize_qdot_q8_0, strerror)

__all__ = ["EXPORTS", "debug_stream_read", "PATH_AUTO", "PATH_SIMT", "PATH_TC", "PATH_MMA", "WS_N_KB", "WS_KB_N", "PQError",
           "PQ_OK", "PQ_ERR_INVALID_ARG", "PQ_ERR_SHAPE", "PQ_ERR_ALIGN", "PQ_ERR_CUDA",
           "PQ_ERR_TIMEOUT", "PQ_ERR_UNSUPPORTED", "PQ_ERR_SCRATCH", "quantize_qdot_q8_0_noalloc",
           "quantize_qdot_q8_0_host", "load", "lib_path", "quantize_q8_0",
           "qdot_q8_0", "qdot_q8_0_ex", "quantize_qdot_q8_0", "qdot_q8_0_blocksums", "q50_qdot", "quantize_q50_qdot",
           "q50_blocksums",
           "check_device", "strerror"]
