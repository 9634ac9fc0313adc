"""ctypes binding of libsws.so: the C ABI of include/sws.h, one Python function
per C call, argument marshalling only. Device pointers and streams are plain
integers (e.g. tensor.data_ptr(), torch.cuda.current_stream().cuda_stream)."""
from __future__ import annotations

import ctypes as C
import os
import warnings
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsws.so")

OK, W_SKIPPED, W_COLD = 0, 1, 2
E_INVALID, E_ALIGN, E_STATE, E_CUDA, E_TIMEOUT, E_UNSUPPORTED, E_WORKSPACE = -1, -2, -3, -4, -5, -6, -7
E4M3, BF16, F32, U8, F16 = 0, 1, 2, 3, 4
SRC_SLOT0, SRC_SLOT1, SRC_FUSED = 0, 1, 2
RUN_FUSED, RUN_TIMING, RUN_FIRST_PREFETCHED = 1, 2, 4
SCALES_IN_T = 1  # plan flag
OPT_DECODE_KERNEL = 1
DECODE_AUTO, DECODE_MMA, DECODE_TCGEN05 = 0, 1, 2
OPT_PREFILL_KERNEL = 2
PREFILL_AUTO, PREFILL_SINGLE, PREFILL_PAIR = 0, 1, 2
OPT_GATHER_ENGINE = 3
GATHER_TMA, GATHER_COPY_ENGINE, GATHER_TMA_SHARED_SM = 0, 1, 2
OPT_HOST_WAIT_MS = 4
OPT_CHECK_BOUNDS = 5

_NAMES = {0: "SWS_OK", 1: "SWS_W_SKIPPED", 2: "SWS_W_COLD", -1: "SWS_E_INVALID", -2: "SWS_E_ALIGN", -3: "SWS_E_STATE",
          -4: "SWS_E_CUDA", -5: "SWS_E_TIMEOUT", -6: "SWS_E_UNSUPPORTED", -7: "SWS_E_WORKSPACE"}


class SwsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class _Entry(C.Structure):
    _fields_ = [("layer", C.c_int32), ("dtype", C.c_int32), ("rows", C.c_int64), ("cols", C.c_int64)]


class _LayerIO(C.Structure):
    _fields_ = [("x", C.POINTER(C.c_void_p)), ("y", C.POINTER(C.c_void_p)), ("m", C.c_int64)]


_lib: Optional[C.CDLL] = None

# (name, restype, argtypes)
_PROTOS = [
    ("sws_plan_create", C.c_int, [C.POINTER(_Entry), C.c_int32, C.c_int32, C.c_uint32, C.POINTER(C.c_void_p)]),
    ("sws_plan_info", C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    ("sws_plan_layer", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                 C.POINTER(C.c_int32)]),
    ("sws_plan_entry", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                 C.POINTER(C.c_int32)]),
    ("sws_plan_scales", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    ("sws_plan_slot_bytes", C.c_int64, [C.c_void_p]),
    ("sws_plan_destroy", None, [C.c_void_p]),
    ("sws_relayout", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_void_p]),
    ("sws_relayout_scales", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                       C.c_void_p]),
    ("sws_workspace_bytes", C.c_int64, [C.c_void_p, C.c_int64]),
    ("sws_ctx_create", C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.c_void_p, C.c_void_p, C.POINTER(C.c_void_p),
                                 C.POINTER(C.c_void_p), C.c_void_p, C.c_int64, C.POINTER(C.c_void_p)]),
    ("sws_ctx_destroy", None, [C.c_void_p]),
    ("sws_gather_to_slot", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]),
    ("sws_linear", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    ("sws_layer_linears", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(_LayerIO), C.c_void_p]),
    ("sws_linear_noalloc", C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int64,
                                     C.c_void_p, C.c_void_p]),
    ("sws_noalloc_status", C.c_int, [C.c_int32, C.POINTER(C.c_int32)]),
    ("sws_run_layers", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(_LayerIO), C.c_uint32, C.c_void_p,
                                 C.c_void_p]),
    ("sws_run_timing", C.c_int, [C.c_void_p, C.POINTER(C.c_float), C.POINTER(C.c_float), C.c_int32]),
    ("sws_graph_capture", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(_LayerIO), C.c_uint32, C.c_void_p,
                                    C.c_void_p, C.POINTER(C.c_void_p)]),
    ("sws_graph_launch", C.c_int, [C.c_void_p, C.c_void_p]),
    ("sws_graph_destroy", None, [C.c_void_p]),
    ("sws_quantize_x", C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    ("sws_silu_mul", C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p]),
    ("sws_prefetch_layer", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]),
    ("sws_test_bounded_wait", C.c_int, [C.c_void_p, C.c_int64, C.c_void_p]),
    ("sws_test_check_relayout", C.c_int, [C.c_void_p, C.c_int32, C.c_int64]),
    ("sws_test_settle_plan", C.c_int, [C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64), C.c_int32,
                                       C.c_int64, C.POINTER(C.c_int32), C.c_int32]),
    ("sws_wait_prefetch", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]),
    ("sws_ctx_status", C.c_int, [C.c_void_p, C.c_int32]),
    ("sws_trace_begin", C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]),
    ("sws_trace_count", C.c_int32, [C.c_void_p]),
    ("sws_set_option", C.c_int, [C.c_int32, C.c_int64]),
    ("sws_last_error", C.c_char_p, []),
    ("sws_version", C.c_int32, []),
]
EXPORTED = [p[0] for p in _PROTOS]


def lib() -> C.CDLL:
    """The loaded library. Raises if libsws.so has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                              "g.build()'); there is no non-CUDA fallback")
        l = C.CDLL(LIB_PATH)
        for name, res, args in _PROTOS:
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def last_error() -> str:
    return lib().sws_last_error().decode(errors="replace")


def check(rc: int, what: str = "") -> int:
    if rc < 0:
        raise SwsError(rc, f"{what}: {last_error()}" if what else last_error())
    if rc == W_SKIPPED:
        warnings.warn(f"{what}: {last_error()}", RuntimeWarning, stacklevel=3)
    return rc


def _ptrs(vals: Sequence[int]):
    arr = (C.c_void_p * max(1, len(vals)))()
    for i, v in enumerate(vals):
        arr[i] = C.c_void_p(int(v) if v else None)
    return arr


class Plan:
    """sws_plan_create / sws_plan_* / sws_plan_destroy."""

    def __init__(self, entries: Sequence[tuple], n_shards: int, flags: int = 0):
        """entries: (layer, dtype, rows, cols) in declaration order."""
        arr = (_Entry * max(1, len(entries)))()
        for i, (layer, dtype, rows, cols) in enumerate(entries):
            arr[i] = _Entry(layer, dtype, rows, cols)
        h = C.c_void_p()
        self.status = check(lib().sws_plan_create(arr, len(entries), n_shards, flags, C.byref(h)), "plan_create")
        self.handle = h
        self.n_entries = len(entries)

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.sws_plan_destroy(self.handle)
            self.handle = None

    def info(self):
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        check(lib().sws_plan_info(self.handle, C.byref(a), C.byref(b), C.byref(c)), "plan_info")
        return a.value, b.value, c.value

    def layer(self, layer: int):
        t, ch, n = C.c_int64(), C.c_int64(), C.c_int32()
        check(lib().sws_plan_layer(self.handle, layer, C.byref(t), C.byref(ch), C.byref(n)), "plan_layer")
        return t.value, ch.value, n.value

    def entry(self, j: int):
        o, nb, sh = C.c_int64(), C.c_int64(), C.c_int32()
        check(lib().sws_plan_entry(self.handle, j, C.byref(o), C.byref(nb), C.byref(sh)), "plan_entry")
        return o.value, nb.value, bool(sh.value)

    def scales(self, j: int):
        """(offset in T, bytes) of entry j's block scales, (-1, 0) when not in T."""
        o, nb = C.c_int64(), C.c_int64()
        check(lib().sws_plan_scales(self.handle, j, C.byref(o), C.byref(nb)), "plan_scales")
        return o.value, nb.value

    @property
    def slot_bytes(self) -> int:
        return lib().sws_plan_slot_bytes(self.handle)


def plan_create(entries, n_shards, flags=0) -> Plan:
    return Plan(entries, n_shards, flags)


def relayout(plan: Plan, layer: int, row_shards: Sequence[int], chunks: Sequence[int], stream: int = 0):
    check(lib().sws_relayout(plan.handle, layer, _ptrs(row_shards), _ptrs(chunks), C.c_void_p(stream or None)),
          "relayout")


def relayout_scales(plan: Plan, layer: int, scales: Sequence[int], chunks: Sequence[int], stream: int = 0):
    """scales[k]: device pointer to the full block scales of the layer's k-th entry (0 if not in T)."""
    check(lib().sws_relayout_scales(plan.handle, layer, _ptrs(scales), _ptrs(chunks), C.c_void_p(stream or None)),
          "relayout_scales")


def workspace_bytes(plan: Plan, max_m: int) -> int:
    v = lib().sws_workspace_bytes(plan.handle, max_m)
    if v < 0:
        raise SwsError(E_INVALID, "workspace_bytes: " + last_error())
    return v


def set_option(option: int, value: int):
    check(lib().sws_set_option(option, value), "set_option")


def linear_noalloc(w: int, scales: int, rows: int, cols: int, x: int, m: int, y: int, stream: int = 0):
    """Decode linear with the library's fixed device scratch (no workspace)."""
    check(lib().sws_linear_noalloc(C.c_void_p(w), C.c_void_p(scales), rows, cols, C.c_void_p(x), m, C.c_void_p(y),
                                   C.c_void_p(stream or None)), "linear_noalloc")


def test_check_relayout(plan: "Plan", layer: int, chunk_bytes: int) -> int:
    """sws_test_check_relayout: the SWS_OPT_CHECK_BOUNDS check of the relayout's
    copy segments against chunks of `chunk_bytes` (host only). Returns the code."""
    return lib().sws_test_check_relayout(plan.handle, layer, chunk_bytes)


def test_settle_plan(rows: Sequence[int], cols: Sequence[int], elem_bytes: int, grid: int) -> list:
    """sws_test_settle_plan: the settle tasks of a tcgen05 decode launch over
    these linears on `grid` CTAs (host only), as tuples (linear, row block,
    rows, first CTA, last CTA, first CTA's partial slot)."""
    n = len(rows)
    cap = 256
    out = (C.c_int32 * (6 * cap))()
    r = (C.c_int64 * n)(*rows)
    c = (C.c_int64 * n)(*cols)
    k = lib().sws_test_settle_plan(n, r, c, elem_bytes, grid, out, cap)
    check(k if k < 0 else 0, "test_settle_plan")
    return [tuple(out[6 * t:6 * t + 6]) for t in range(k)]


def noalloc_status(clear: bool = False) -> int:
    """Status word of linear_noalloc's scratch: 0 or an SWS_E_* code. A host
    wait that ran out, or a CUDA error, raises."""
    v = C.c_int32()
    check(lib().sws_noalloc_status(1 if clear else 0, C.byref(v)), "noalloc_status")
    return v.value


def test_bounded_wait_noalloc(limit_ns: int, stream: int = 0):
    """The bounded-wait check on linear_noalloc's status word."""
    check(lib().sws_test_bounded_wait(None, limit_ns, C.c_void_p(stream or None)), "test_bounded_wait")


def quantize_x(x: int, m: int, k: int, xq: int, ex: int, stream: int = 0):
    check(lib().sws_quantize_x(C.c_void_p(x), m, k, C.c_void_p(xq), C.c_void_p(ex), C.c_void_p(stream or None)),
          "quantize_x")


def silu_mul(gu: int, m: int, f: int, act: int, stream: int = 0):
    """act[m, f] = SiLU(gu[:, :f]) * gu[:, f:] (bf16 in and out, device pointers)."""
    check(lib().sws_silu_mul(C.c_void_p(gu), m, f, C.c_void_p(act), C.c_void_p(stream or None)), "silu_mul")


class Graph:
    """A captured lookahead run (sws_graph_capture); destroy it before its context."""

    def __init__(self, handle: int):
        self.handle = handle

    def launch(self, stream: int = 0):
        check(lib().sws_graph_launch(self.handle, C.c_void_p(stream or None)), "graph_launch")

    def close(self):
        if self.handle:
            lib().sws_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Ctx:
    """sws_ctx_create and the calls that take a context."""

    def __init__(self, plan: Plan, chunks: Sequence[int], slot0: int, slot1: int, scales: Sequence[int],
                 replicated: Optional[Sequence[int]], workspace: int, ws_bytes: int):
        h = C.c_void_p()
        rep = _ptrs(replicated) if replicated is not None else None
        check(lib().sws_ctx_create(plan.handle, _ptrs(chunks), C.c_void_p(slot0 or None), C.c_void_p(slot1 or None),
                                   _ptrs(scales), rep, C.c_void_p(workspace or None), ws_bytes, C.byref(h)),
              "ctx_create")
        self.handle = h
        self.plan = plan  # keeps the plan alive

    def close(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.sws_ctx_destroy(self.handle)
            self.handle = None

    __del__ = close

    def gather_to_slot(self, layer: int, slot: int, stream: int = 0):
        check(lib().sws_gather_to_slot(self.handle, layer, slot, C.c_void_p(stream or None)), "gather_to_slot")

    def linear(self, entry: int, src: int, x: int, m: int, y: int, stream: int = 0):
        check(lib().sws_linear(self.handle, entry, src, C.c_void_p(x), m, C.c_void_p(y), C.c_void_p(stream or None)),
              "linear")

    def layer_linears(self, layer: int, src: int, xs: Sequence[int], ys: Sequence[int], m: int, stream: int = 0):
        xa, ya = _ptrs(xs), _ptrs(ys)
        io = _LayerIO(C.cast(xa, C.POINTER(C.c_void_p)), C.cast(ya, C.POINTER(C.c_void_p)), m)
        check(lib().sws_layer_linears(self.handle, layer, src, C.byref(io), C.c_void_p(stream or None)),
              "layer_linears")

    @staticmethod
    def _io_array(io: Sequence[tuple]):
        n = max(1, len(io))
        arr = (_LayerIO * n)()
        keep = []
        for i, (xs, ys, m) in enumerate(io):
            xa, ya = _ptrs(xs), _ptrs(ys)
            keep += [xa, ya]
            arr[i] = _LayerIO(C.cast(xa, C.POINTER(C.c_void_p)), C.cast(ya, C.POINTER(C.c_void_p)), m)
        return arr, keep

    def run_layers(self, first: int, last: int, io: Sequence[tuple], flags: int, main: int, side: int):
        """io[l - first] = (x_ptrs, y_ptrs, m) for layer l."""
        arr, keep = self._io_array(io)
        check(lib().sws_run_layers(self.handle, first, last, arr, flags, C.c_void_p(main or None),
                                   C.c_void_p(side or None)), "run_layers")

    def graph_capture(self, first: int, last: int, io: Sequence[tuple], flags: int, main: int, side: int) -> "Graph":
        """Records run_layers(first, last, io, flags, main, side) as a CUDA
        graph instantiated with per-node priorities; replay with Graph.launch."""
        arr, keep = self._io_array(io)
        h = C.c_void_p()
        check(lib().sws_graph_capture(self.handle, first, last, arr, flags, C.c_void_p(main or None),
                                      C.c_void_p(side or None), C.byref(h)), "graph_capture")
        return Graph(h.value)

    def prefetch_layer(self, layer: int, slot: int, stream: int = 0):
        """Gathers `layer` into `slot` on `stream` ahead of use (draft-model layer 0)."""
        check(lib().sws_prefetch_layer(self.handle, layer, slot, C.c_void_p(stream or None)), "prefetch_layer")

    def wait_prefetch(self, layer: int, slot: int, stream: int = 0) -> bool:
        """`stream` waits for the prefetch of `layer`; returns True on a cold
        start, when the gather had to run inline on `stream`."""
        return check(lib().sws_wait_prefetch(self.handle, layer, slot, C.c_void_p(stream or None)),
                     "wait_prefetch") == W_COLD

    def test_bounded_wait(self, limit_ns: int, stream: int = 0):
        check(lib().sws_test_bounded_wait(self.handle, limit_ns, C.c_void_p(stream or None)), "test_bounded_wait")

    def run_timing(self, n: int):
        a = (C.c_float * n)()
        b = (C.c_float * n)()
        check(lib().sws_run_timing(self.handle, a, b, n), "run_timing")
        return list(a), list(b)

    def status(self, clear: bool = False) -> int:
        """The context's device status word (0 or an SWS_E_* code). A host wait
        that ran out, or a CUDA error, raises (sws_last_error is set)."""
        rc = lib().sws_ctx_status(self.handle, 1 if clear else 0)
        if rc < 0 and last_error():
            raise SwsError(rc, "ctx_status: " + last_error())
        return rc

    def trace_begin(self, records: int, capacity: int, stream: int = 0):
        check(lib().sws_trace_begin(self.handle, C.c_void_p(records or None), capacity, C.c_void_p(stream or None)),
              "trace_begin")

    def trace_count(self) -> int:
        return lib().sws_trace_count(self.handle)
