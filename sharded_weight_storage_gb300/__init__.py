"""Sharded weight storage ("store sharded, compute full") for NVIDIA GB300.

The compute path is the CUDA library libsws.so (C ABI in include/sws.h); this
package is its ctypes binding plus device-memory plumbing on top of PyTorch.
Importing it loads the library and fails loudly when it has not been built.
"""
from ._lib import (BF16, E4M3, F16, E_ALIGN, E_CUDA, E_INVALID, E_STATE, E_TIMEOUT, E_UNSUPPORTED, E_WORKSPACE, F32,
                   OK, RUN_FUSED, RUN_TIMING, RUN_FIRST_PREFETCHED, W_COLD, SRC_FUSED, SRC_SLOT0, SRC_SLOT1, U8, W_SKIPPED, Ctx, Graph, Plan,
                   SwsError,
                   last_error, lib, plan_create, quantize_x, relayout, workspace_bytes, set_option, silu_mul,
                   OPT_DECODE_KERNEL, DECODE_AUTO, DECODE_MMA, DECODE_TCGEN05, OPT_PREFILL_KERNEL,
                   PREFILL_AUTO, PREFILL_SINGLE, PREFILL_PAIR, OPT_GATHER_ENGINE, GATHER_TMA, GATHER_COPY_ENGINE,
                   GATHER_TMA_SHARED_SM, OPT_HOST_WAIT_MS, OPT_CHECK_BOUNDS, SCALES_IN_T, relayout_scales, linear_noalloc,
                   noalloc_status, test_bounded_wait_noalloc, test_check_relayout,
                   test_settle_plan)

lib()  # load now: no silent fallback when the extension is missing

__all__ = ["Plan", "Ctx", "Graph", "SwsError", "plan_create", "relayout", "workspace_bytes", "quantize_x", "silu_mul", "lib",
           "last_error", "E4M3", "BF16", "F16", "F32", "U8", "SRC_SLOT0", "SRC_SLOT1", "SRC_FUSED", "RUN_FUSED",
           "RUN_TIMING", "RUN_FIRST_PREFETCHED", "W_COLD", "OK", "W_SKIPPED", "E_INVALID", "E_ALIGN", "E_STATE", "E_CUDA", "E_TIMEOUT",
           "E_UNSUPPORTED", "E_WORKSPACE", "set_option", "OPT_DECODE_KERNEL", "DECODE_AUTO",
           "DECODE_MMA", "DECODE_TCGEN05", "OPT_PREFILL_KERNEL", "PREFILL_AUTO", "PREFILL_SINGLE",
           "PREFILL_PAIR", "OPT_GATHER_ENGINE", "GATHER_TMA", "GATHER_COPY_ENGINE", "GATHER_TMA_SHARED_SM",
           "OPT_HOST_WAIT_MS", "OPT_CHECK_BOUNDS", "SCALES_IN_T", "relayout_scales", "linear_noalloc", "noalloc_status",
           "test_bounded_wait_noalloc", "test_check_relayout", "test_settle_plan"]
