"""Seeded synthetic inputs for the sharded-weight path.

This module only draws numbers: weight codes, block scales and activations with
the shapes and value distributions of the workloads below. It holds none of the
method's arithmetic (no packing, chunking, gathering or linear algebra), so both
the CPU oracle and the CUDA library can consume what it produces.

Recipe (every tensor has its own stream, keyed by (workload, layer, entry, kind)):
  * weights: w ~ N(0, 0.02) drawn in float32; one scale per 128x128 block,
    s = float32(2**u) with u ~ U(-8, -4); codes q = e4m3fn(w / s) using PyTorch's
    float8_e4m3fn cast (round to nearest even). |w/s| stays far below 448.
  * activations: x ~ N(0, 1) drawn in float32 and rounded to bfloat16.
  * stacks of many layers of one shape: a few base layers are drawn as above and
    layer l is base[l % n_base] with every weight row multiplied by an
    independent random sign (+1 / -1) drawn for that layer. For i.i.d. symmetric
    weights a per-row sign flip leaves the joint distribution unchanged, while
    making every layer's bytes distinct.

The workload shapes follow the shared-expert byte counts of the vLLM PR #50656
report ("Functionality and motivation": gate_up 176.2 MB + down 88.1 MB per
layer) and the KDA-layer target list of the weight-sharding blog ("Only shard
truly replicated weights").
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------

KIND_W, KIND_S, KIND_X, KIND_SIGN = 0, 1, 2, 3


@dataclasses.dataclass(frozen=True)
class EntrySpec:
    name: str
    rows: int  # out_features (dim 0, the dimension rows are sharded along)
    cols: int  # in_features


@dataclasses.dataclass(frozen=True)
class Workload:
    key: int
    name: str
    n_shards: int
    entries: Tuple[EntrySpec, ...]
    m_values: Tuple[int, ...]
    n_layers: int = 1
    n_base: int = 1  # distinct base layers for stacks (see module docstring)
    description: str = ""


TINY = Workload(
    key=1, name="tiny_flat_layer", n_shards=4,
    entries=(EntrySpec("W_a", 512, 256), EntrySpec("W_b", 384, 256), EntrySpec("W_c", 256, 512)),
    m_values=(1,),
    description="tiny flat layer, N=4, decode M=1",
)

SHARED_EXPERT = Workload(
    key=2, name="shared_expert_layer", n_shards=16,
    entries=(EntrySpec("gate_up", 24576, 7168), EntrySpec("down", 7168, 12288)),
    m_values=(1, 8, 32, 64),
    description="shared-expert-like layer (gate_up 176.2 MB + down 88.1 MB), N=16, decode",
)

ATTN_KDA = Workload(
    key=3, name="attn_kda_layer", n_shards=16,
    entries=(
        EntrySpec("qkv", 12288, 7168), EntrySpec("f_b", 4096, 7168),
        EntrySpec("o", 7168, 8192), EntrySpec("g", 8192, 7168),
        EntrySpec("latent_up", 7168, 2048), EntrySpec("latent_down", 2048, 7168),
        EntrySpec("shared_gate_up", 8192, 7168), EntrySpec("shared_down", 7168, 4096),
    ),
    m_values=(1, 16, 64),
    description="attention/KDA-like layer of 8 FP8 weights, N=16, decode",
)

STACK92 = Workload(
    key=4, name="decode_stack_92", n_shards=16, entries=SHARED_EXPERT.entries,
    m_values=(32,), n_layers=92, n_base=2,
    description="92-layer decode stack of shared-expert layers, N=16, M=32, lookahead",
)

PREFILL = Workload(
    key=5, name="prefill_kda_8", n_shards=8, entries=ATTN_KDA.entries,
    m_values=(2048, 8192), n_layers=8, n_base=1,
    description="prefill on KDA-layer weights, N=8, 8 layers",
)

WORKLOADS: Dict[int, Workload] = {w.key: w for w in (TINY, SHARED_EXPERT, ATTN_KDA, STACK92, PREFILL)}


def scaled_workload(base: Workload, rows_div: int = 1, cols_div: int = 1, n_layers: int | None = None,
                    name: str | None = None) -> Workload:
    """A smaller workload with the same entry list and shard count (shapes divided)."""
    ents = tuple(EntrySpec(e.name, max(1, e.rows // rows_div), max(1, e.cols // cols_div)) for e in base.entries)
    return dataclasses.replace(base, entries=ents, name=name or (base.name + "_small"),
                               n_layers=base.n_layers if n_layers is None else n_layers)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def rng_for(workload_key: int, layer: int, entry: int, kind: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(0, spawn_key=(workload_key, layer, entry, kind)))


def _to_e4m3_codes(v: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    t = t.clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def draw_weight(workload_key: int, layer: int, entry: int, rows: int, cols: int) -> Tuple[np.ndarray, np.ndarray]:
    """(codes uint8 [rows, cols], scales float32 [ceil(rows/128), ceil(cols/128)])."""
    rb, cb = -(-rows // 128), -(-cols // 128)
    s = np.float32(2.0) ** rng_for(workload_key, layer, entry, KIND_S).uniform(-8.0, -4.0, size=(rb, cb)).astype(np.float32)
    s = s.astype(np.float32)
    w = rng_for(workload_key, layer, entry, KIND_W).standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(0.02)
    for b in range(rb):
        row_scale = np.repeat(s[b], 128)[:cols]
        w[b * 128:(b + 1) * 128] /= row_scale[None, :]
    return _to_e4m3_codes(w), s


def draw_weight_bf16(workload_key: int, layer: int, entry: int, rows: int, cols: int) -> np.ndarray:
    """bf16 weight [rows, cols] as uint16 bit patterns, w ~ N(0, 0.02) rounded
    to bf16 (the unquantised weight variant)."""
    import torch
    w = rng_for(workload_key, layer, entry, KIND_W).standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(0.02)
    return torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw_weight_f16(workload_key: int, layer: int, entry: int, rows: int, cols: int) -> np.ndarray:
    """f16 weight [rows, cols] as uint16 bit patterns, w ~ N(0, 0.02) rounded
    to IEEE binary16 (the unquantised weight variant stored as FP16)."""
    w = rng_for(workload_key, layer, entry, KIND_W).standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(0.02)
    return w.astype(np.float16).view(np.uint16)


def draw_row_signs(workload_key: int, layer: int, entry: int, rows: int) -> np.ndarray:
    """Per-row sign-bit mask (0x00 or 0x80) for layer `layer` of a stack."""
    bits = rng_for(workload_key, layer, entry, KIND_SIGN).integers(0, 2, size=rows, dtype=np.uint8)
    return (bits * np.uint8(0x80)).astype(np.uint8)


def draw_x(workload_key: int, entry: int, m: int, k: int):
    """bf16 activations [m, k] (torch CPU tensor), x ~ N(0, 1) rounded to bf16."""
    import torch
    x = rng_for(workload_key, 0, entry, KIND_X).standard_normal((m, k), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def bf16_bits(x) -> np.ndarray:
    import torch
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class LayerWeights:
    codes: List[np.ndarray]   # per entry, uint8 [rows, cols]
    scales: List[np.ndarray]  # per entry, float32 block scales


def base_layer(workload: Workload, base: int) -> LayerWeights:
    codes, scales = [], []
    for j, e in enumerate(workload.entries):
        q, s = draw_weight(workload.key, base, j, e.rows, e.cols)
        codes.append(q)
        scales.append(s)
    return LayerWeights(codes, scales)


def layer_weights(workload: Workload, layer: int, bases: Sequence[LayerWeights] | None = None) -> LayerWeights:
    """Weights of one layer. Single-layer workloads draw directly; stacks derive
    layer `layer` from base[layer % n_base] with per-row sign flips."""
    if workload.n_layers == 1:
        return base_layer(workload, 0)
    if bases is None:
        bases = [base_layer(workload, layer % workload.n_base)]
        b = bases[0]
    else:
        b = bases[layer % workload.n_base]
    codes = []
    for j, e in enumerate(workload.entries):
        signs = draw_row_signs(workload.key, layer, j, e.rows)
        codes.append(b.codes[j] ^ signs[:, None])
    return LayerWeights(codes, [s for s in b.scales])


def row_shards(codes: np.ndarray, n: int) -> List[np.ndarray]:
    """The loader's convention: shard r holds rows [r*rows/n, (r+1)*rows/n)."""
    rows = codes.shape[0]
    assert rows % n == 0
    k = rows // n
    return [np.ascontiguousarray(codes[r * k:(r + 1) * k]) for r in range(n)]


def apply_row_signs(codes, signs):
    """Layer codes of a stack: base codes with each row's sign bit flipped where
    signs[row] == 0x80. Works on numpy arrays and torch tensors alike."""
    return codes ^ signs[:, None]
