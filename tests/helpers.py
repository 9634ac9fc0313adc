"""Shared set-up for the GPU parity tests: the same seeded inputs feed the CUDA
library (through the C ABI) and the CPU oracle."""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np
import torch

import oracle as O
import workloads as WL

# Floating-point bar for linears (output vs the float64 oracle on dequantised
# weights): max |err| <= 1e-2 * max |ref| + 1e-3 and ||err||_F / ||ref||_F <= 5e-3.
ATOL_ABS = 1e-3
ATOL_REL_MAX = 1e-2
REL_FRO = 5e-3


def assert_close(y: np.ndarray, ref: np.ndarray, what: str = ""):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    mref = float(np.max(np.abs(ref))) if ref.size else 0.0
    assert float(err.max(initial=0.0)) <= ATOL_REL_MAX * mref + ATOL_ABS, \
        f"{what}: max err {err.max():.3e} vs bound {ATOL_REL_MAX * mref + ATOL_ABS:.3e}"
    nref = float(np.linalg.norm(ref))
    if nref > 0:
        rel = float(np.linalg.norm(y - ref)) / nref
        assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return WL.bf16_to_f64(WL.bf16_bits(t.detach().cpu()))


@dataclasses.dataclass
class LayerData:
    codes: Dict[int, np.ndarray]   # global entry id -> uint8 [rows, cols]
    scales: Dict[int, np.ndarray]  # global entry id -> float32


def workload_entries(w: WL.Workload, n_layers: int | None = None):
    n_layers = w.n_layers if n_layers is None else n_layers
    return [(l, e.rows, e.cols) for l in range(n_layers) for e in w.entries]


def draw_layers(w: WL.Workload, n_layers: int | None = None) -> List[LayerData]:
    n_layers = w.n_layers if n_layers is None else n_layers
    ne = len(w.entries)
    out = []
    bases = None
    if w.n_layers > 1:
        bases = [WL.base_layer(w, b) for b in range(min(w.n_base, n_layers))]
    for l in range(n_layers):
        lw = WL.layer_weights(w, l, bases)
        out.append(LayerData({l * ne + j: lw.codes[j] for j in range(ne)},
                             {l * ne + j: lw.scales[j] for j in range(ne)}))
    return out


def build_stack(S, entries, n_shards, layers: List[LayerData], max_m=64):
    """Loads every layer through the relayout kernel and creates the context."""
    from sharded_weight_storage_gb300.storage import ShardedStack
    st = ShardedStack([(l, S.E4M3, r, c) for (l, r, c) in entries], n_shards, max_m=max_m)
    for l, ld in enumerate(layers):
        st.load_layer(l, {j: torch.from_numpy(v) for j, v in ld.codes.items()},
                      {j: torch.from_numpy(v) for j, v in ld.scales.items()})
    st.make_ctx()
    return st


def weight_bytes(bits: np.ndarray) -> np.ndarray:
    """16-bit weight bit patterns [rows, cols] -> the weight's bytes [rows, 2 * cols]."""
    return np.ascontiguousarray(bits).view(np.uint8).reshape(bits.shape[0], -1)


def typed_stack(S, shapes, n, weights, scales=None, max_m=64):
    """shapes: (layer, dtype, rows, cols); weights[j]: uint8 bytes [rows, cols * elem];
    scales[j]: block scales or one per-tensor scale of an E4M3 entry."""
    from sharded_weight_storage_gb300.storage import ShardedStack
    st = ShardedStack(shapes, n, max_m=max_m)
    for l in sorted({s[0] for s in shapes}):
        js = [j for j, s in enumerate(shapes) if s[0] == l]
        st.load_layer(l, {j: torch.from_numpy(weights[j]) for j in js},
                      {j: scales[j] for j in js if scales and j in scales})
    st.make_ctx()
    return st


def linear_kinds(st, j, src, x, m):
    """Runs one linear with tracing on; returns y and the kernel ids (trace tag
    bits 48..55) of its linear records."""
    rec = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
    st.ctx.trace_begin(rec.data_ptr(), 4, 0)
    _, _, rows, _ = st.entries[j]
    y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(j, src, x.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    n = st.ctx.trace_count()
    st.ctx.trace_begin(0, 0, 0)
    tags = [int(t) for t in rec.view(4, 4)[:n, 0].tolist()]
    return y, [(t >> 48) & 0xFF for t in tags if (t >> 56) == 2]


def x_f64(x: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> float64 array of its exact values."""
    return WL.bf16_to_f64(WL.bf16_bits(x.cpu()))


def oracle_layer_T(entries, n_shards, layer: int, ld: LayerData):
    plan = O.plan_layout([(l, r, c, 1) for (l, r, c) in entries], n_shards)
    shards = {j: WL.row_shards(q, n_shards) for j, q in ld.codes.items() if plan.sharded[j]}
    chunks = O.relayout(plan, layer, shards)
    return plan, chunks, O.gather(chunks)
