"""Plain, slow CPU oracle for the 'store sharded, compute full' weight path.

TEST INFRASTRUCTURE. Only tests/, the package smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA
library and imports nothing from it. Every function is written from the text of
the pages it cites, in float64 where the path computes in floating point.

Sources (page title, section):
  [WS]  Weight sharding blog (zdszero.github.io/weight_sharding.html)
        - "核心抽象：存储分片，计算不分片" (core abstraction: W split along dim 0)
        - "一层一次 AllGather：flat layout" (flat layout steps 1-4, chunk boundaries)
        - "提前一层：lookahead 与 ping-pong slot" (lookahead, slots A/B, gate event)
        - "代价：通信量与显存账" (per-rank traffic, resident memory)
        - "SGLang 中的实现" (planner loop: reset / pre_dispatch / maybe_dispatch /
          update_done_event)
        - "只 shard 真正 replicated 的权重" (rows not divisible by N: warn and skip)
        - "加载：行 shard 先行，finalize 再重排" (row-shard loading, per-weight
          temporary AllGather then copy of the rank's byte window)
        - "CUDA graph 与 draft 模型" (wait at most once)
  [OCP] OCP 8-bit floating point specification, E4M3 encoding (bias 7, no
        infinities, S.1111.111 is NaN, largest finite 448).
  [PR]  vLLM PR #50656 report, "功能与动机" (shared-expert byte counts).

Readings taken where the pages are silent (each also listed in the design notes):
  * pad bytes are 0x00; the 16*N tail padding sits at the end of T;
  * an entry's 16-byte rule is applied to its size, so every offset is 16-aligned;
  * row shard r of an [out, in] weight holds rows [r*out/N, (r+1)*out/N);
  * Y = X W^T with W [out, in]; block scale s[o // 128, i // 128] multiplies the
    decoded code; partial edge blocks use ceil(./128) indexing;
  * BF16 weights: the same linear with W decoded from bfloat16 patterns and
    no scales; FP16 weights: W from binary16 patterns and x rounded to f16 (the
    f16 tensor-core operand); ModelOpt FP8: one float32 scale for the whole weight;
  * prefill activations: per (row, 128-column group) scale e = 2^k with k the
    smallest integer such that amax <= 448 * 2^k (amax = 0 gives e = 1), and
    codes xq = e4m3_rne(x / e), ties to even, saturating to +-448.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# E4M3 (OCP E4M3FN) from its definition [OCP]
# ---------------------------------------------------------------------------


def e4m3_code_value(code: int) -> float:
    """Value of one 8-bit E4M3FN code: sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([e4m3_code_value(c) for c in range(256)], dtype=np.float64)
# the 127 finite non-negative values, codes 0x00 .. 0x7E, ascending
_E4M3_POS = E4M3_TABLE[:0x7F].copy()
E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3FN code to each float64 value, ties to the even code,
    magnitudes above 448 saturate to 448. The sign bit follows the sign of the
    input (so -0.0 and negative values that round to zero give 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    i = np.searchsorted(_E4M3_POS, a, side="left")  # first index with POS[i] >= a
    i = np.clip(i, 1, 0x7E)
    lo = _E4M3_POS[i - 1]
    hi = _E4M3_POS[i]
    d_lo = a - lo
    d_hi = hi - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 0))
    idx = np.where(take_hi, i, i - 1).astype(np.uint8)
    return idx | (np.signbit(v).astype(np.uint8) << np.uint8(7))


# ---------------------------------------------------------------------------
# flat layout [WS "一层一次 AllGather：flat layout"]
# ---------------------------------------------------------------------------


def roundup(x: int, m: int) -> int:
    return ((x + m - 1) // m) * m


@dataclasses.dataclass
class LayerLayout:
    layer: int
    entries: List[int]          # global entry indices packed into T, in order
    offsets: Dict[int, int]     # entry -> o_j
    sizes: Dict[int, int]       # entry -> s_j (bytes)
    total: int                  # |T|
    chunk: int                  # C = |T| / N
    # scales inside T (optional layout): entry -> offset / bytes of its block-scale tensor
    scale_offsets: Dict[int, int] = dataclasses.field(default_factory=dict)
    scale_sizes: Dict[int, int] = dataclasses.field(default_factory=dict)


@dataclasses.dataclass
class Plan:
    n_shards: int
    rows: List[int]
    cols: List[int]
    elem_bytes: List[int]
    layer_of: List[int]
    sharded: List[bool]
    layers: Dict[int, LayerLayout]

    @property
    def slot_bytes(self) -> int:
        return max([ly.total for ly in self.layers.values()], default=0)


def scale_grid(rows: int, cols: int) -> Tuple[int, int]:
    """Shape of a weight's block-scale tensor: one float32 per 128 x 128 block."""
    return -(-rows // 128), -(-cols // 128)


def plan_layout(entries: Sequence[Tuple], n_shards: int, scales_in_t: bool = False) -> Plan:
    """entries: (layer, rows, cols, elem_bytes) or (layer, rows, cols,
    elem_bytes, block_scaled) in declaration order.

    An entry is stored sharded when its rows divide by N; otherwise it stays
    replicated and is left out of T ([WS "只 shard 真正 replicated 的权重"]).
    The sharded entries of a layer are concatenated in declaration order, each
    padded to a 16-byte multiple, and T is padded to a multiple of 16*N; the
    chunk size is C = |T| / N ([WS "flat layout" steps 1-2]).

    scales_in_t (a layout the pages do not use - they keep scales replicated,
    outside T): each sharded block-scaled entry is followed by its float32
    block-scale tensor as an entry of its own, padded to 16 bytes like any
    entry."""
    if n_shards < 1:
        raise ValueError("N must be >= 1")
    layer_of = [e[0] for e in entries]
    rows = [e[1] for e in entries]
    cols = [e[2] for e in entries]
    eb = [e[3] for e in entries]
    scaled = [bool(e[4]) if len(e) > 4 else False for e in entries]
    sharded = [r % n_shards == 0 for r in rows]
    layers: Dict[int, LayerLayout] = {}
    for j, e in enumerate(entries):
        layer, r, c, b = e[:4]
        ly = layers.setdefault(layer, LayerLayout(layer, [], {}, {}, 0, 0))
        if not sharded[j]:
            continue
        s = r * c * b
        ly.offsets[j] = ly.total
        ly.sizes[j] = s
        ly.entries.append(j)
        ly.total += roundup(s, 16)  # each entry padded to 16 B
        if scales_in_t and scaled[j]:
            gr, gc = scale_grid(r, c)
            ly.scale_offsets[j] = ly.total
            ly.scale_sizes[j] = 4 * gr * gc
            ly.total += roundup(4 * gr * gc, 16)
    for ly in layers.values():
        ly.total = roundup(ly.total, 16 * n_shards)  # total padded to 16*N
        ly.chunk = ly.total // n_shards
    return Plan(n_shards, rows, cols, eb, layer_of, sharded, layers)


def pack(plan: Plan, layer: int, weight_bytes: Dict[int, np.ndarray],
         scales: Dict[int, np.ndarray] | None = None) -> np.ndarray:
    """T: the layer's entries in order at their offsets, zero padding
    ([WS "flat layout" step 1]); with scales in T, each scale tensor's float32
    bytes at its own offset."""
    ly = plan.layers[layer]
    t = np.zeros(ly.total, dtype=np.uint8)
    for j in ly.entries:
        b = np.ascontiguousarray(weight_bytes[j]).view(np.uint8).reshape(-1)
        assert b.size == ly.sizes[j]
        t[ly.offsets[j]:ly.offsets[j] + ly.sizes[j]] = b
    for j, o in ly.scale_offsets.items():
        b = np.ascontiguousarray(np.asarray(scales[j], dtype=np.float32)).view(np.uint8).reshape(-1)
        assert b.size == ly.scale_sizes[j]
        t[o:o + b.size] = b
    return t


def split_chunks(plan: Plan, layer: int, t: np.ndarray) -> List[np.ndarray]:
    """T_i = T[iC:(i+1)C] ([WS "flat layout" step 2])."""
    ly = plan.layers[layer]
    c = ly.chunk
    return [t[i * c:(i + 1) * c].copy() for i in range(plan.n_shards)]


def gather(chunks: Sequence[np.ndarray]) -> np.ndarray:
    """all_gather_into_tensor: every rank ends with the concatenation of all
    chunks in rank order ([WS "flat layout" step 3])."""
    return np.concatenate([np.asarray(c, dtype=np.uint8).reshape(-1) for c in chunks]) if len(chunks) else np.zeros(0, np.uint8)


def view(plan: Plan, layer: int, t: np.ndarray, j: int) -> np.ndarray:
    """W_j = view(T[o_j : o_j + s_j]) as [rows, cols] ([WS "flat layout" step 4])."""
    ly = plan.layers[layer]
    o, s = ly.offsets[j], ly.sizes[j]
    return t[o:o + s].reshape(plan.rows[j], plan.cols[j] * plan.elem_bytes[j])


def scales_view(plan: Plan, layer: int, t: np.ndarray, j: int) -> np.ndarray:
    """Entry j's block scales read from T (scales-in-T layout): the float32
    tensor [ceil(rows/128), ceil(cols/128)] at its offset."""
    ly = plan.layers[layer]
    o, s = ly.scale_offsets[j], ly.scale_sizes[j]
    return t[o:o + s].copy().view(np.float32).reshape(scale_grid(plan.rows[j], plan.cols[j]))


def relayout(plan: Plan, layer: int, shards: Dict[int, Sequence[np.ndarray]],
             scales: Dict[int, np.ndarray] | None = None) -> List[np.ndarray]:
    """Row shards -> flat chunks, as the finalize step does it: for each weight,
    a temporary AllGather of its N row shards restores the full weight, and each
    rank copies out the bytes that fall into its window [rank*C, (rank+1)*C) of T;
    everything else in the window stays zero
    ([WS "加载：行 shard 先行，finalize 再重排" step 2]). With scales in T, every
    rank holds each full scale tensor (replicated, like the block-FP8 variant
    that keeps full shapes until finalize) and copies out its window the same way."""
    ly = plan.layers[layer]
    n, c = plan.n_shards, ly.chunk
    chunks = [np.zeros(c, dtype=np.uint8) for _ in range(n)]

    def copy_window(full, lo, hi):
        for rank in range(n):
            w_lo, w_hi = rank * c, (rank + 1) * c
            a, b = max(lo, w_lo), min(hi, w_hi)
            if a < b:
                chunks[rank][a - w_lo:b - w_lo] = full[a - lo:b - lo]

    for j in ly.entries:
        full = gather([np.ascontiguousarray(x).view(np.uint8).reshape(-1) for x in shards[j]])
        copy_window(full, ly.offsets[j], ly.offsets[j] + ly.sizes[j])
    for j, o in ly.scale_offsets.items():
        full = np.ascontiguousarray(np.asarray(scales[j], dtype=np.float32)).view(np.uint8).reshape(-1)
        copy_window(full, o, o + ly.scale_sizes[j])
    return chunks


def chunk_map(plan: Plan, layer: int, g: int) -> Tuple[int, int]:
    """Byte g of T lives in chunk g // C at offset g % C."""
    c = plan.layers[layer].chunk
    return g // c, g % c


# ---------------------------------------------------------------------------
# cost model [WS "代价：通信量与显存账"]
# ---------------------------------------------------------------------------


def gather_bytes_received(plan: Plan, layer: int, rank: int) -> int:
    """Bytes a rank must receive to hold the full T: every chunk but its own."""
    ly = plan.layers[layer]
    return sum(ly.chunk for i in range(plan.n_shards) if i != rank)


def resident_bytes_per_rank(plan: Plan) -> int:
    """One chunk of every layer plus two full-layer slots."""
    return sum(ly.chunk for ly in plan.layers.values()) + 2 * plan.slot_bytes


# ---------------------------------------------------------------------------
# linears [WS "核心抽象"]: the GEMM sees the full W; Y = X W^T
# ---------------------------------------------------------------------------


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[o, i] = e4m3(q[o, i]) * s[o // 128, i // 128] in float64."""
    rows, cols = codes.shape
    s = np.asarray(scales, dtype=np.float64)
    s_full = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:rows, :cols]
    return e4m3_decode(codes) * s_full


def linear(x: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y = X W^T in float64 with W the dequantized weight."""
    return np.asarray(x, dtype=np.float64) @ dequant(codes, scales).T


def dequant_at(codes: np.ndarray, scales: np.ndarray, rows=None, cols=None) -> np.ndarray:
    """The sub-matrix W[rows][:, cols] of the dequantized weight, computed for
    the selected rows and columns only: element (o, i) is
    e4m3(q[o, i]) * s[o // 128, i // 128] in float64 (None selects all)."""
    r = np.arange(codes.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    c = np.arange(codes.shape[1]) if cols is None else np.asarray(cols, dtype=np.int64)
    s = np.asarray(scales, dtype=np.float64)[np.ix_(r // 128, c // 128)]
    return e4m3_decode(np.asarray(codes)[np.ix_(r, c)]) * s


def linear_rows(x: np.ndarray, codes: np.ndarray, scales: np.ndarray, rows) -> np.ndarray:
    """Y[:, rows] of Y = X W^T: the outputs of the selected weight rows, from
    those rows alone (for checking samples of full-size outputs)."""
    return np.asarray(x, dtype=np.float64) @ dequant_at(codes, scales, rows=rows).T


# Weight variants ([WS "加载：行 shard 先行，finalize 再重排", "量化变体"]): BF16
# weights go through the same flat layout; ModelOpt FP8 keeps its per-tensor
# scale replicated, outside T.


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """Value of each 16-bit bfloat16 pattern in float64: sign bit, 8 exponent
    bits (bias 127), 7 fraction bits; exponent 0 is subnormal (f * 2^-133),
    exponent 255 is infinity (f = 0) or NaN."""
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    f = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + f / 128.0, (e - 127).astype(np.int64))
    sub = np.ldexp(f, -133)
    v = np.where(e == 0, sub, normal)
    v = np.where(e == 255, np.where(f == 0, np.inf, np.nan), v)
    return sign * v


def linear_bf16(x: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Y = X W^T in float64 with W [out, in] given as bfloat16 bit patterns."""
    return np.asarray(x, dtype=np.float64) @ bf16_decode(w_bits).T


def f16_decode(bits: np.ndarray) -> np.ndarray:
    """Value of each 16-bit IEEE binary16 pattern in float64: sign bit, 5
    exponent bits (bias 15), 10 fraction bits; exponent 0 is subnormal
    (f * 2^-24), exponent 31 is infinity (f = 0) or NaN."""
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    sub = np.ldexp(f, -24)
    v = np.where(e == 0, sub, normal)
    v = np.where(e == 31, np.where(f == 0, np.inf, np.nan), v)
    return sign * v


def f16_round(v: np.ndarray) -> np.ndarray:
    """Nearest binary16 value of each float64 (11 significant bits, subnormal
    spacing 2^-24), ties to the even significand; beyond the largest finite
    value (65504) the result is infinity."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    fin = np.isfinite(v) & (v != 0)
    f, p = np.frexp(np.abs(v[fin]))
    p = np.maximum(p, -13)                     # below 2^-14 the spacing stays 2^-24
    scaled = np.ldexp(np.abs(v[fin]), 11 - p)  # significand in [1024, 2048)
    r = np.floor(scaled)
    frac = scaled - r
    r = r + ((frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1)))
    mag = np.ldexp(r, p - 11)
    mag = np.where(mag > 65504.0, np.inf, mag)
    out[fin] = np.sign(v[fin]) * mag
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    return out


def linear_f16(x: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Y = X W^T in float64 with W [out, in] given as binary16 patterns; the
    activations enter the f16 tensor-core operand, so they are rounded to f16
    first (exact for bf16 values with |x| in [2^-14, 65504])."""
    return f16_round(np.asarray(x, dtype=np.float64)) @ f16_decode(w_bits).T


def linear_per_tensor(x: np.ndarray, codes: np.ndarray, scale: float) -> np.ndarray:
    """Y = X W^T with W[o, i] = e4m3(q[o, i]) * s, one scale for the whole
    weight (ModelOpt FP8), in float64."""
    return np.asarray(x, dtype=np.float64) @ (e4m3_decode(codes) * float(np.float32(scale))).T


# Shared-expert chain (the second workload shape): gate_up -> SiLU(gate) * up
# -> down, with bf16 tensors between the steps.


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value of each float64 (8 significant bits), ties to the
    even significand; results beyond the largest finite bf16 become infinity."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    fin = np.isfinite(v) & (v != 0)
    f, p = np.frexp(np.abs(v[fin]))          # |v| = f * 2^p, f in [0.5, 1)
    p = np.maximum(p, -125)                  # below 2^-126 the spacing stays 2^-133
    scaled = np.ldexp(np.abs(v[fin]), 8 - p)  # the significand as a number in [128, 256)
    r = np.floor(scaled)
    frac = scaled - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1))
    r = r + up
    mag = np.ldexp(r, p - 8)
    mag = np.where(mag > (2 - 2.0 ** -7) * 2.0 ** 127, np.inf, mag)
    out[fin] = np.sign(v[fin]) * mag
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    return out


def silu_mul(gu: np.ndarray) -> np.ndarray:
    """act[m, j] = silu(g[m, j]) * u[m, j] with gu = [g | u] ([m, 2F], the gate
    half first) and silu(g) = g / (1 + e^-g), in float64."""
    gu = np.asarray(gu, dtype=np.float64)
    f = gu.shape[1] // 2
    g, u = gu[:, :f], gu[:, f:]
    return g / (1.0 + np.exp(-g)) * u


def quantize_x(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Prefill activation quantiser: for each row and each 128-column group,
    e = 2^k with k the smallest integer such that amax <= 448 * 2^k (e = 1 when
    the group is all zeros), and xq = e4m3_rne(x / e). Returns (xq uint8 [M, K],
    e float32 [M, ceil(K / 128)])."""
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    g = -(-k // 128)
    xq = np.zeros((m, k), dtype=np.uint8)
    e = np.ones((m, g), dtype=np.float64)
    for gi in range(g):
        blk = x[:, gi * 128:(gi + 1) * 128]
        amax = np.max(np.abs(blk), axis=1) if blk.shape[1] else np.zeros(m)
        # amax = f * 2^p with f in [0.5, 1). 448 = 0.875 * 2^9.
        f, p = np.frexp(amax)
        kk = np.where(f <= 0.875, p - 9, p - 8)
        kk = np.where(amax == 0.0, 0, kk)
        e[:, gi] = np.ldexp(1.0, kk)
        xq[:, gi * 128:(gi + 1) * 128] = e4m3_encode_rne(blk / e[:, gi:gi + 1])
    return xq, e.astype(np.float32)


def dequant_x(xq: np.ndarray, e: np.ndarray) -> np.ndarray:
    m, k = xq.shape
    e_full = np.repeat(np.asarray(e, dtype=np.float64), 128, axis=1)[:, :k]
    return e4m3_decode(xq) * e_full


# ---------------------------------------------------------------------------
# schedule model [WS "提前一层：lookahead 与 ping-pong slot", "SGLang 中的实现"]
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Op:
    stream: str        # "main" or "side"
    kind: str          # "wait_call_start", "gather", "record_ready", "wait_done",
                       # "wait_ready", "compute", "record_done"
    layer: int
    slot: int


def slot_of(layer: int, first: int) -> int:
    """Slots A/B are used by layers in turn."""
    return (layer - first) % 2


def schedule(first: int, last: int) -> List[Op]:
    """Issue order of the planner loop: pre_dispatch(first) gathers the first
    layer; each step issues the gather of layer l+1 on the side stream, gated on
    done(l-1) because it overwrites the slot layer l-1 used; the layer waits on
    its ready event once, computes on its slot and records done(l)."""
    ops: List[Op] = []
    if last < first:
        return ops
    ops.append(Op("side", "wait_call_start", first, -1))
    ops.append(Op("side", "gather", first, slot_of(first, first)))
    ops.append(Op("side", "record_ready", first, slot_of(first, first)))
    for layer in range(first, last + 1):
        nxt = layer + 1
        if nxt <= last:
            if layer - 1 >= first:
                ops.append(Op("side", "wait_done", layer - 1, slot_of(layer - 1, first)))
            ops.append(Op("side", "gather", nxt, slot_of(nxt, first)))
            ops.append(Op("side", "record_ready", nxt, slot_of(nxt, first)))
        ops.append(Op("main", "wait_ready", layer, slot_of(layer, first)))
        ops.append(Op("main", "compute", layer, slot_of(layer, first)))
        ops.append(Op("main", "record_done", layer, slot_of(layer, first)))
    return ops


def happens_before(first: int, last: int) -> List[Tuple[Tuple[str, int], Tuple[str, int]]]:
    """Edges the schedule guarantees between device work:
    (("compute", l-1) -> ("gather", l+1)) and (("gather", l) -> ("compute", l))."""
    edges = []
    for layer in range(first, last + 1):
        edges.append((("gather", layer), ("compute", layer)))
        if layer - 2 >= first:
            edges.append((("compute", layer - 2), ("gather", layer)))
    return edges


def max_live_layers(first: int, last: int) -> int:
    """Replays the issue order and counts layers whose full weights are held
    (gathered and not yet done) at once; the slot rule keeps it at two."""
    live, peak = set(), 0
    for op in schedule(first, last):
        if op.kind == "gather":
            live.add(op.layer)
        elif op.kind == "record_done":
            live.discard(op.layer)
        peak = max(peak, len(live))
    return peak
