"""Pins of the CPU oracle against facts that do not come from the oracle itself:
format definitions checked against a library cast, hand-derived layout numbers,
byte counts printed by the pages, exact rational arithmetic and invariants."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from conftest import GOLDEN

# ---------------------------------------------------------------------------
# E4M3 decode / encode
# ---------------------------------------------------------------------------


def test_e4m3_table_matches_torch_cast_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.E4M3_TABLE
    nan_ref, nan_ours = np.isnan(ref), np.isnan(ours)
    assert np.array_equal(nan_ref, nan_ours)
    assert np.array_equal(ref[~nan_ref], ours[~nan_ours])
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(ours[~nan_ours]))


def test_e4m3_closed_forms():
    assert O.E4M3_TABLE[0x7E] == 448.0
    assert O.E4M3_TABLE[0x01] == 2.0 ** -9
    assert O.E4M3_TABLE[0x07] == 7 * 2.0 ** -9
    assert O.E4M3_TABLE[0x08] == 2.0 ** -6
    assert O.E4M3_TABLE[0x38] == 1.0
    assert O.E4M3_TABLE[0xB8] == -1.0
    assert math.isnan(O.E4M3_TABLE[0x7F]) and math.isnan(O.E4M3_TABLE[0xFF])
    assert O.E4M3_TABLE[0x80] == 0.0 and np.signbit(O.E4M3_TABLE[0x80])
    # 126 distinct positive finite values, strictly increasing with the code
    pos = O.E4M3_TABLE[1:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_e4m3_encode_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode_rne(O.e4m3_decode(codes)), codes)


def test_e4m3_encode_midpoints_go_to_even_code():
    pos = O.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2.0
    got = O.e4m3_encode_rne(mids)
    lo = np.arange(0, 0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    assert np.array_equal(O.e4m3_encode_rne(-mids), (want | 0x80).astype(np.uint8))


def test_e4m3_encode_matches_torch_cast_random():
    rng = np.random.default_rng(123)
    mag = 2.0 ** rng.uniform(-14, np.log2(448.0), size=200_000)
    v = mag * rng.choice([-1.0, 1.0], size=mag.size)
    v = v.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode_rne(v), ref)


def test_e4m3_encode_saturates():
    assert O.e4m3_encode_rne(np.array([1e6, -1e6, 448.0, 465.0]))[:].tolist() == [0x7E, 0xFE, 0x7E, 0x7E]


# ---------------------------------------------------------------------------
# flat layout
# ---------------------------------------------------------------------------


def _read_offsets_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "layout_offsets.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, ents, total, chunk = [p.strip() for p in line.split("|")]
            name, n = head.split()
            offs = dict((kv.split("=")[0], int(kv.split("=")[1])) for kv in ents.split())
            rows[name] = (int(n), offs, int(total), int(chunk))
    return rows


def _plan_for(w: WL.Workload, n=None):
    return O.plan_layout([(0, e.rows, e.cols, 1) for e in w.entries], n or w.n_shards)


@pytest.mark.parametrize("wname", ["tiny_flat_layer", "shared_expert_layer", "attn_kda_layer", "prefill_kda_8"])
def test_layout_matches_hand_derived_offsets(wname):
    gold = _read_offsets_golden()[wname]
    w = [x for x in WL.WORKLOADS.values() if x.name == wname][0]
    n, offs, total, chunk = gold
    assert n == w.n_shards
    p = _plan_for(w)
    ly = p.layers[0]
    for j, e in enumerate(w.entries):
        assert ly.offsets[j] == offs[e.name]
    assert ly.total == total and ly.chunk == chunk


def test_shared_expert_sizes_match_printed_byte_counts():
    vals = {}
    with open(os.path.join(GOLDEN, "pages_byte_counts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, v, unit, dec = line.split()
                vals[name] = (float(v), unit, int(dec))
    p = _plan_for(WL.SHARED_EXPERT)
    ly = p.layers[0]

    def fmt(nbytes, unit, dec):
        div = 1e6 if unit == "MB" else 2.0 ** 30
        return round(nbytes / div, dec)

    assert fmt(ly.sizes[0], "MB", 1) == vals["shared_gate_up"][0]
    assert fmt(ly.sizes[1], "MB", 1) == vals["shared_down"][0]
    assert fmt(ly.total, "MB", 1) == vals["shared_layer"][0]
    assert fmt(92 * ly.total, "GiB", 1) == vals["shared_92_layers"][0]


def test_worked_example_rank1_holds_tail_of_a_and_head_of_b():
    p = _plan_for(WL.TINY)
    ly = p.layers[0]
    c = ly.chunk
    want = []
    with open(os.path.join(GOLDEN, "flat_layout_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                r, name, a, b = line.split()
                want.append((int(r), name, int(a), int(b)))
    names = [e.name for e in WL.TINY.entries]
    rank = 1
    got = []
    for j in ly.entries:
        lo, hi = ly.offsets[j], ly.offsets[j] + ly.sizes[j]
        a, b = max(lo, rank * c), min(hi, (rank + 1) * c)
        if a < b:
            rowb = p.cols[j]
            got.append((rank, names[j], (a - lo) // rowb, (b - lo) // rowb - 1))
    assert got == want


def _rand_shapes(rng, n_entries, n):
    ents = []
    for _ in range(n_entries):
        rows = int(rng.integers(1, 9)) * n if rng.random() < 0.8 else int(rng.integers(1, 40))
        cols = int(rng.integers(1, 70))
        ents.append((0, rows, cols, int(rng.choice([1, 1, 2, 4]))))
    return ents


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 16])
def test_layout_invariants_random_shapes(n):
    rng = np.random.default_rng(n)
    for trial in range(20):
        ents = _rand_shapes(rng, int(rng.integers(1, 7)), n)
        p = O.plan_layout(ents, n)
        ly = p.layers[0]
        assert ly.total % (16 * n) == 0 and ly.chunk * n == ly.total
        data = {j: rng.integers(0, 256, size=ly.sizes[j], dtype=np.uint8) for j in ly.entries}
        t = O.pack(p, 0, data)
        for j in ly.entries:
            assert ly.offsets[j] % 16 == 0
            assert np.array_equal(O.view(p, 0, t, j).reshape(-1), data[j])
        # bytes outside every entry are zero
        covered = np.zeros(ly.total, bool)
        for j in ly.entries:
            covered[ly.offsets[j]:ly.offsets[j] + ly.sizes[j]] = True
        assert not t[~covered].any()
        ch = O.split_chunks(p, 0, t)
        assert len(ch) == n and all(x.size == ly.chunk for x in ch)
        assert np.array_equal(O.gather(ch), t)
        # replicated entries are exactly those whose rows do not divide by N
        for j, (_, rows, _, _) in enumerate(ents):
            assert (j in ly.entries) == (rows % n == 0)


def test_chunk_size_depends_only_on_total_and_n():
    # Two layouts with different weight boundaries but the same |T|.
    a = O.plan_layout([(0, 16, 64, 1), (0, 16, 192, 1)], 4)
    b = O.plan_layout([(0, 16, 128, 1), (0, 16, 128, 1)], 4)
    assert a.layers[0].total == b.layers[0].total
    assert a.layers[0].chunk == b.layers[0].chunk
    assert a.layers[0].offsets[1] != b.layers[0].offsets[1]


def test_chunks_straddle_weights_in_kda_layer():
    p = _plan_for(WL.ATTN_KDA)
    ly = p.layers[0]
    c = ly.chunk
    straddling = []
    for i in range(p.n_shards):
        inside = [j for j in ly.entries if ly.offsets[j] < (i + 1) * c and ly.offsets[j] + ly.sizes[j] > i * c]
        if len(inside) > 1:
            straddling.append(i)
    assert 5 in straddling  # f_b's tail and o's head share chunk 5
    # boundaries 4, 8 and 12 fall exactly on entry starts
    starts = set(ly.offsets.values())
    assert {4 * c, 8 * c, 12 * c} <= starts


# ---------------------------------------------------------------------------
# relayout: per-weight row shards -> flat chunks
# ---------------------------------------------------------------------------


def _relayout_by_byte_formula(p, shards, n):
    """Independent formulation: chunk byte b of rank i is T byte g = i*C + b; in
    entry j at local byte u = g - o_j it comes from row shard u // (s_j/N) at
    offset u % (s_j/N); every other byte is zero."""
    ly = p.layers[0]
    c = ly.chunk
    out = [np.zeros(c, np.uint8) for _ in range(n)]
    for i in range(n):
        for b in range(c):
            g = i * c + b
            for j in ly.entries:
                u = g - ly.offsets[j]
                if 0 <= u < ly.sizes[j]:
                    per = ly.sizes[j] // n
                    out[i][b] = shards[j][u // per].reshape(-1)[u % per]
    return out


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7])
def test_relayout_matches_byte_formula(n):
    rng = np.random.default_rng(100 + n)
    for trial in range(4):
        ents = [(0, int(rng.integers(1, 5)) * n, int(rng.integers(1, 40)), 1) for _ in range(int(rng.integers(1, 5)))]
        p = O.plan_layout(ents, n)
        ly = p.layers[0]
        full = {j: rng.integers(0, 256, size=(ents[j][1], ents[j][2]), dtype=np.uint8) for j in ly.entries}
        shards = {j: WL.row_shards(full[j], n) for j in ly.entries}
        got = O.relayout(p, 0, shards)
        want = _relayout_by_byte_formula(p, shards, n)
        for a, b in zip(got, want):
            assert np.array_equal(a, b)
        # and it agrees with packing the full weights and slicing T
        t = O.pack(p, 0, full)
        for a, b in zip(got, O.split_chunks(p, 0, t)):
            assert np.array_equal(a, b)


def test_relayout_n1_is_identity_of_pack():
    ents = [(0, 3, 5, 1), (0, 2, 16, 1)]
    p = O.plan_layout(ents, 1)
    rng = np.random.default_rng(7)
    full = {j: rng.integers(0, 256, size=(r, c), dtype=np.uint8) for j, (_, r, c, _) in enumerate(ents)}
    ch = O.relayout(p, 0, {j: [full[j]] for j in full})
    assert len(ch) == 1 and np.array_equal(ch[0], O.pack(p, 0, full))


# ---------------------------------------------------------------------------
# cost model
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("wname", ["tiny_flat_layer", "shared_expert_layer", "attn_kda_layer"])
def test_per_rank_traffic_is_n_minus_1_over_n_of_s(wname):
    w = [x for x in WL.WORKLOADS.values() if x.name == wname][0]
    p = _plan_for(w)
    s = p.layers[0].total
    n = p.n_shards
    for rank in range(n):
        got = O.gather_bytes_received(p, 0, rank)
        assert Fraction(got) == Fraction(n - 1, n) * s


def test_resident_memory_formula_92_layer_stack():
    w = WL.STACK92
    ents = [(layer, e.rows, e.cols, 1) for layer in range(w.n_layers) for e in w.entries]
    p = O.plan_layout(ents, w.n_shards)
    r = sum(ly.total for ly in p.layers.values())
    assert r == 24_310_185_984
    assert Fraction(O.resident_bytes_per_rank(p)) == Fraction(r, w.n_shards) + 2 * p.slot_bytes
    assert p.slot_bytes == 264_241_152


# ---------------------------------------------------------------------------
# linear
# ---------------------------------------------------------------------------


def _bf16_values(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    return WL.bf16_to_f64(WL.bf16_bits(x))


def test_linear_matches_exact_rational_dot_products():
    rng = np.random.default_rng(5)
    for (m, out, inn) in [(1, 3, 5), (2, 130, 7), (4, 5, 200), (3, 2, 256)]:
        q = rng.integers(0, 256, size=(out, inn), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x11  # no NaN codes
        s = (2.0 ** rng.uniform(-8, -4, size=(-(-out // 128), -(-inn // 128)))).astype(np.float32)
        x = _bf16_values(rng, (m, inn))
        y = O.linear(x, q, s)
        for a in range(m):
            for o in range(out):
                exact = sum(Fraction(float(x[a, i])) * Fraction(float(O.E4M3_TABLE[q[o, i]]))
                            * Fraction(float(s[o // 128, i // 128])) for i in range(inn))
                assert abs(Fraction(float(y[a, o])) - exact) <= Fraction(1, 10**12) * (1 + abs(exact))


def test_linear_one_hot_selects_dequantized_column():
    rng = np.random.default_rng(9)
    q = rng.integers(0, 0x7E, size=(200, 300), dtype=np.uint8)
    s = (2.0 ** rng.uniform(-8, -4, size=(2, 3))).astype(np.float32)
    for i in [0, 127, 128, 299]:
        x = np.zeros((1, 300))
        x[0, i] = 1.0
        y = O.linear(x, q, s)[0]
        col = np.array([O.E4M3_TABLE[q[o, i]] * float(s[o // 128, i // 128]) for o in range(200)])
        assert np.array_equal(y, col)


def test_linear_zero_scales_give_zero():
    rng = np.random.default_rng(10)
    q = rng.integers(0, 0x7E, size=(64, 256), dtype=np.uint8)
    x = _bf16_values(rng, (3, 256))
    assert not O.linear(x, q, np.zeros((1, 2), np.float32)).any()


def test_linear_transposition_and_block_index_are_pinned():
    # A scale that differs between the two 128-blocks of a row catches a swapped
    # block index; a non-square weight catches a transposed operand.
    q = np.full((130, 256), 0x38, np.uint8)  # all ones
    s = np.array([[1.0, 2.0], [4.0, 8.0]], np.float32)
    x = np.ones((1, 256))
    y = O.linear(x, q, s)[0]
    assert y[0] == 128 * 1.0 + 128 * 2.0 and y[129] == 128 * 4.0 + 128 * 8.0


# ---------------------------------------------------------------------------
# weight variants: BF16 weights, per-tensor FP8 scale
# ---------------------------------------------------------------------------


def test_bf16_decode_closed_forms():
    # 1.0, -2.0, 0.5, largest finite, smallest normal, smallest subnormal, zeros
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,
             0x0080: 2.0 ** -126, 0x0001: 2.0 ** -133, 0x0000: 0.0, 0x8000: -0.0, 0x4049: 3.140625}
    for bits, want in cases.items():
        got = O.bf16_decode(np.array([bits]))[0]
        assert got == want and np.signbit(got) == np.signbit(want), hex(bits)
    assert np.isinf(O.bf16_decode(np.array([0x7F80]))[0]) and np.isnan(O.bf16_decode(np.array([0x7FC0]))[0])


def test_bf16_decode_matches_torch_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.int64)
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    o = O.bf16_decode(bits)
    same = (o == t) | (np.isnan(o) & np.isnan(t))
    assert same.all()


def _rand_bf16_bits(rng, shape):
    v = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * 0.05).to(torch.bfloat16)
    return v.view(torch.int16).numpy().astype(np.uint16)


def test_linear_bf16_matches_exact_rational_dot_products():
    rng = np.random.default_rng(31)
    for (m, out, inn) in [(1, 3, 5), (2, 17, 64), (3, 5, 130)]:
        w = _rand_bf16_bits(rng, (out, inn))
        x = _bf16_values(rng, (m, inn))
        y = O.linear_bf16(x, w)
        wv = O.bf16_decode(w)
        for a in range(m):
            for o in range(out):
                exact = sum(Fraction(float(x[a, i])) * Fraction(float(wv[o, i])) for i in range(inn))
                assert abs(Fraction(float(y[a, o])) - exact) <= Fraction(1, 10**12) * (1 + abs(exact))


def test_linear_bf16_one_hot_and_transposition():
    rng = np.random.default_rng(32)
    w = _rand_bf16_bits(rng, (40, 24))  # non-square: a transposed operand fails
    for i in (0, 7, 23):
        x = np.zeros((1, 24))
        x[0, i] = 1.0
        assert np.array_equal(O.linear_bf16(x, w)[0], O.bf16_decode(w[:, i]))


def test_f16_decode_closed_forms_and_every_pattern():
    cases = {0x3C00: 1.0, 0xC000: -2.0, 0x3800: 0.5, 0x7BFF: 65504.0, 0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24,
             0x0000: 0.0, 0x3555: 0.333251953125}
    for bits, want in cases.items():
        assert O.f16_decode(np.array([bits]))[0] == want, hex(bits)
    assert np.isinf(O.f16_decode(np.array([0x7C00]))[0]) and np.isnan(O.f16_decode(np.array([0x7E00]))[0])
    bits = np.arange(1 << 16, dtype=np.int64)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    o = O.f16_decode(bits)
    assert ((o == ref) | (np.isnan(o) & np.isnan(ref))).all()


def test_f16_round_closed_forms_and_numpy():
    cases = {1 + 2.0 ** -11: 1.0, 1 + 3 * 2.0 ** -11: 1 + 2.0 ** -9, 1 + 2.0 ** -11 + 2.0 ** -30: 1 + 2.0 ** -10,
             2.0 ** -25: 0.0, 3 * 2.0 ** -26: 2.0 ** -24, 65519.0: 65504.0, 0.0: 0.0}
    for v, want in cases.items():
        assert O.f16_round(np.array([v]))[0] == want, v
    assert np.isinf(O.f16_round(np.array([65520.0]))[0])
    rng = np.random.default_rng(43)
    v = rng.standard_normal(50000) * 10.0 ** rng.integers(-9, 5, 50000)
    assert np.array_equal(O.f16_round(v), v.astype(np.float16).astype(np.float64))


def test_linear_f16_exact_rational_and_one_hot():
    rng = np.random.default_rng(44)
    w = (rng.standard_normal((7, 40)) * 0.05).astype(np.float16).view(np.uint16)
    x = _bf16_values(rng, (3, 40))
    y = O.linear_f16(x, w)
    wv, xv = O.f16_decode(w), O.f16_round(x)
    for a in range(3):
        for o in range(7):
            exact = sum(Fraction(float(xv[a, i])) * Fraction(float(wv[o, i])) for i in range(40))
            assert abs(Fraction(float(y[a, o])) - exact) <= Fraction(1, 10**12) * (1 + abs(exact))
    e = np.zeros((1, 40))
    e[0, 9] = 1.0
    assert np.array_equal(O.linear_f16(e, w)[0], O.f16_decode(w[:, 9]))


def test_linear_per_tensor_is_block_linear_with_a_constant_grid():
    rng = np.random.default_rng(33)
    q = rng.integers(0, 0x7E, size=(300, 260), dtype=np.uint8)
    x = _bf16_values(rng, (4, 260))
    s = np.float32(0.0371)
    grid = np.full((3, 3), s, np.float32)
    assert np.array_equal(O.linear_per_tensor(x, q, s), O.linear(x, q, grid))
    # and it scales linearly in s (powers of two are exact)
    assert np.array_equal(O.linear_per_tensor(x, q, 0.25), 0.25 * O.linear_per_tensor(x, q, 1.0))


# ---------------------------------------------------------------------------
# shared-expert chain: bf16 rounding, SiLU * up
# ---------------------------------------------------------------------------


def test_bf16_round_closed_forms():
    cases = {1.0: 1.0, 1 + 2.0 ** -8: 1.0, 1 + 3 * 2.0 ** -8: 1 + 2.0 ** -6, 1 + 2.0 ** -8 + 2.0 ** -30: 1 + 2.0 ** -7,
             -(1 + 2.0 ** -7 + 2.0 ** -8): -(1 + 2.0 ** -6), 2.0 ** -133: 2.0 ** -133, 2.0 ** -135: 0.0,
             3 * 2.0 ** -135: 2.0 ** -133, 0.0: 0.0, 3.39e38: (2 - 2.0 ** -7) * 2.0 ** 127}
    for v, want in cases.items():
        assert O.bf16_round(np.array([v]))[0] == want, v
    assert np.isinf(O.bf16_round(np.array([3.4e38 * 1.01]))[0])


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(41)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(2000) * 1e-39]).astype(np.float32)
    t = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(v.astype(np.float64)), t)


def test_silu_mul_closed_forms_and_half_order():
    ln3 = np.log(3.0)
    gu = np.array([[0.0, ln3, -ln3, 40.0, -40.0, 2.0, 2.0, 2.0, 2.0, 1.5]])  # g | u, F = 5
    a = O.silu_mul(gu)[0]
    assert a[0] == 0.0                                   # silu(0) = 0 whatever u is
    assert abs(a[1] - 0.75 * ln3 * 2.0) < 1e-15          # sigmoid(ln 3) = 3/4
    assert abs(a[2] - (-0.25 * ln3) * 2.0) < 1e-15       # sigmoid(-ln 3) = 1/4
    assert abs(a[3] - 40.0 * 2.0) < 1e-12                # silu(x) -> x
    assert abs(a[4]) < 1e-15                             # silu(-x) -> 0
    # swapping the halves (silu on the up half) would give silu(2) * 0 = 0 for column 0
    assert O.silu_mul(np.array([[1.0, 0.0]]))[0, 0] == 0.0 and O.silu_mul(np.array([[0.0, 1.0]]))[0, 0] == 0.0
    assert abs(O.silu_mul(np.array([[1.0, 1.0]]))[0, 0] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16


# ---------------------------------------------------------------------------
# prefill activation quantiser
# ---------------------------------------------------------------------------


def _k_exact(amax: float) -> int:
    """Smallest integer k with amax <= 448 * 2^k, by exact rational search."""
    if amax == 0:
        return 0
    a = Fraction(amax)
    k = 0
    while a > 448 * Fraction(2) ** k:
        k += 1
    while a <= 448 * Fraction(2) ** (k - 1):
        k -= 1
    return k


def test_quantizer_scale_exponent_matches_rational_search():
    rng = np.random.default_rng(11)
    x = _bf16_values(rng, (64, 300)) * (2.0 ** rng.integers(-20, 20, size=(64, 1)))
    x[3] = 0.0
    x[4, :5] = 448.0
    x[4, 5:] = 0.0
    x[5] = 0.0
    x[5, 0] = 450.0  # next bf16 above 448
    xq, e = O.quantize_x(x)
    for m in range(x.shape[0]):
        for g in range(e.shape[1]):
            amax = float(np.max(np.abs(x[m, g * 128:(g + 1) * 128])))
            assert e[m, g] == 2.0 ** _k_exact(amax)
    assert e[3, 0] == 1.0 and e[4, 0] == 1.0 and e[5, 0] == 2.0


def test_quantizer_codes_match_library_cast():
    rng = np.random.default_rng(12)
    x = _bf16_values(rng, (32, 512)) * 3.0
    xq, e = O.quantize_x(x)
    e_full = np.repeat(e.astype(np.float64), 128, axis=1)[:, :512]
    ref = torch.from_numpy((x / e_full).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(xq, ref)
    assert np.all(np.abs(x / e_full) <= 448.0)


def test_quantizer_is_invariant_under_doubling():
    rng = np.random.default_rng(13)
    x = _bf16_values(rng, (8, 384))
    xq1, e1 = O.quantize_x(x)
    xq2, e2 = O.quantize_x(2.0 * x)
    assert np.array_equal(xq1, xq2) and np.array_equal(2 * e1, e2)


def test_quantizer_ragged_group_and_error_bound():
    rng = np.random.default_rng(14)
    x = _bf16_values(rng, (4, 200))
    xq, e = O.quantize_x(x)
    assert e.shape == (4, 2)
    xd = O.dequant_x(xq, e)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normal codes, and
    # absolute error <= half the subnormal step 2^-10 * e below them.
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(e.astype(np.float64), 128, axis=1)[:, :200] * 2.0 ** -10)
    assert np.all(np.abs(xd - x) <= bound)


# ---------------------------------------------------------------------------
# schedule model
# ---------------------------------------------------------------------------


def test_schedule_slots_alternate_and_first_layer_predispatched():
    ops = O.schedule(3, 8)
    gathers = [op for op in ops if op.kind == "gather"]
    assert [g.layer for g in gathers] == list(range(3, 9))
    assert [g.slot for g in gathers] == [0, 1, 0, 1, 0, 1]
    assert ops[1].kind == "gather" and ops[1].layer == 3  # before any compute
    waits = [op for op in ops if op.kind == "wait_ready"]
    assert [w.layer for w in waits] == list(range(3, 9))  # once per layer


def test_schedule_gates_each_gather_on_the_slot_previous_user():
    ops = O.schedule(0, 9)
    for i, op in enumerate(ops):
        if op.kind == "gather" and op.layer >= 2:
            prev = ops[i - 1]
            assert prev.kind == "wait_done" and prev.layer == op.layer - 2 and prev.slot == op.slot
    assert O.max_live_layers(0, 9) == 2
    assert O.max_live_layers(5, 5) == 1
    assert O.schedule(4, 3) == []


# ---------------------------------------------------------------------------
# layouts with non-zero padding, the chunk map, the lookahead's edges
# (hand-typed goldens), each with planted mistakes that must fail them
# ---------------------------------------------------------------------------


def read_padding_golden():
    """Cases of tests/golden/layout_padding.txt: name -> (N, [(entry name, rows,
    cols, elem, offset or -1)], |T|, C)."""
    cases = {}
    with open(os.path.join(GOLDEN, "layout_padding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, ents, total, chunk = [p.strip() for p in line.split("|")]
            name, n = head.split()
            rows = []
            for tok in ents.split():
                nm, rest = tok.split(":")
                shape, off = rest.split("=")
                r, c, e = (int(v) for v in shape.split(","))
                rows.append((nm, r, c, e, int(off)))
            cases[name] = (int(n), rows, int(total), int(chunk))
    return cases


def _layout_matches_padding_golden(plan_fn) -> bool:
    for n, ents, total, chunk in read_padding_golden().values():
        p = plan_fn([(0, r, c, e) for (_, r, c, e, _) in ents], n)
        ly = p.layers[0]
        if (ly.total, ly.chunk) != (total, chunk):
            return False
        for j, (_, _, _, _, off) in enumerate(ents):
            if off < 0:
                if p.sharded[j] or j in ly.offsets:
                    return False
            elif ly.offsets.get(j) != off:
                return False
    return True


def test_layout_with_padding_matches_hand_derived_golden():
    assert _layout_matches_padding_golden(O.plan_layout)


def _mutant_plan(entry_pad, tail_pad):
    """plan_layout with its two padding rules replaced: a planted mistake."""
    def plan(entries, n):
        p = O.plan_layout(entries, n)
        for ly in p.layers.values():
            off = 0
            for j in ly.entries:
                ly.offsets[j] = off
                off += entry_pad(ly.sizes[j], n)
            ly.total = tail_pad(off, n)
            ly.chunk = ly.total // n
        return p
    return plan


@pytest.mark.parametrize("entry_pad,tail_pad", [
    (lambda s, n: O.roundup(s, 16), lambda t, n: O.roundup(t, 16 * n)),      # the rule itself
    (lambda s, n: O.roundup(s, 32), lambda t, n: O.roundup(t, 16 * n)),      # entries over-padded
    (lambda s, n: O.roundup(s, 16 * n), lambda t, n: O.roundup(t, 16 * n)),  # each entry to 16N
    (lambda s, n: O.roundup(s, 16), lambda t, n: O.roundup(t, 16)),          # no 16N tail rule
    (lambda s, n: s, lambda t, n: O.roundup(t, 16 * n)),                     # no 16-byte entry rule
], ids=["rule", "entry32", "entry16N", "tail16", "entry1"])
def test_padding_golden_catches_planted_padding_mistakes(entry_pad, tail_pad, request):
    ok = _layout_matches_padding_golden(_mutant_plan(entry_pad, tail_pad))
    assert ok == (request.node.callspec.id == "rule")


def test_padded_layouts_pack_chunk_and_relayout():
    rng = np.random.default_rng(31)
    for n, ents, total, chunk in read_padding_golden().values():
        p = O.plan_layout([(0, r, c, e) for (_, r, c, e, _) in ents], n)
        ly = p.layers[0]
        data = {j: rng.integers(1, 256, size=(ents[j][1], ents[j][2] * ents[j][3]), dtype=np.uint8)
                for j in ly.entries}
        t = O.pack(p, 0, data)
        assert t.size == total
        pad = np.ones(total, bool)
        for j in ly.entries:
            pad[ly.offsets[j]:ly.offsets[j] + ly.sizes[j]] = False
            assert np.array_equal(O.view(p, 0, t, j), data[j])
        # the padding bytes (per entry and at the tail) are the only zeros
        assert pad.sum() == total - sum(ly.sizes.values()) > 0
        assert not t[pad].any() and t[~pad].all()
        ch = O.split_chunks(p, 0, t)
        assert [c.size for c in ch] == [chunk] * n and np.array_equal(O.gather(ch), t)
        shards = {j: WL.row_shards(data[j], n) for j in ly.entries}
        assert all(np.array_equal(a, b) for a, b in zip(O.relayout(p, 0, shards), ch))


def test_chunk_map_matches_hand_derived_points():
    n, ents, _, _ = read_padding_golden()["pad_n7"]
    layouts = {"tiny_flat_layer": _plan_for(WL.TINY),
               "pad_n7": O.plan_layout([(0, r, c, e) for (_, r, c, e, _) in ents], n)}
    seen = 0
    with open(os.path.join(GOLDEN, "chunk_map_points.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, g, ci, off = line.split()
                assert O.chunk_map(layouts[name], 0, int(g)) == (int(ci), int(off)), line
                seen += 1
    assert seen == 8


def test_chunk_map_finds_every_byte_of_t_in_its_chunk():
    # step 2's byte rule: rank i holds T[i*C, (i+1)*C), so byte g is byte g % C of chunk g // C
    rng = np.random.default_rng(32)
    plans = [O.plan_layout([(0, r, c, e) for (_, r, c, e, _) in ents], n)
             for n, ents, _, _ in read_padding_golden().values()]
    plans.append(_plan_for(WL.TINY))
    for p in plans:
        ly = p.layers[0]
        t = rng.integers(0, 256, size=ly.total, dtype=np.uint8)
        chunks = [t[i * ly.chunk:(i + 1) * ly.chunk] for i in range(p.n_shards)]
        hit = np.zeros((p.n_shards, ly.chunk), bool)
        for g in range(0, ly.total, max(1, ly.total // 4099)):
            ci, off = O.chunk_map(p, 0, g)
            assert 0 <= ci < p.n_shards and 0 <= off < ly.chunk
            assert chunks[ci][off] == t[g]
            assert not hit[ci, off]
            hit[ci, off] = True


def read_edges_golden():
    cases = []
    with open(os.path.join(GOLDEN, "lookahead_edges.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, edges = [p.strip() for p in line.split("|")]
            first, last = (int(v) for v in head.split())
            cases.append((first, last, set(edges.split())))
    return cases


def _edge_names(edges):
    short = {"gather": "g", "compute": "c"}
    return {f"{short[a[0]]}{a[1]}<{short[b[0]]}{b[1]}" for a, b in edges}


def _edges_match_golden(fn) -> bool:
    return all(_edge_names(fn(first, last)) == want for first, last, want in read_edges_golden())


def test_happens_before_matches_hand_listed_edges():
    assert _edges_match_golden(O.happens_before)


def test_edges_golden_catches_planted_schedule_mistakes():
    def no_slot_reuse(first, last):  # the gate on done(l-2) dropped
        return [e for e in O.happens_before(first, last) if e[0][0] != "compute"]

    def gate_one_back(first, last):  # gated on done(l-1) instead of done(l-2)
        out = [e for e in O.happens_before(first, last) if e[0][0] != "compute"]
        return out + [(("compute", l - 1), ("gather", l)) for l in range(first + 1, last + 1)]

    def gate_from_first(first, last):  # the slot-reuse gate also on the second layer
        return O.happens_before(first, last) + [(("compute", first - 1), ("gather", first + 1))] \
            if last > first else O.happens_before(first, last)

    for bad in (no_slot_reuse, gate_one_back, gate_from_first):
        assert not _edges_match_golden(bad), bad.__name__


def test_happens_before_follows_from_the_issue_order():
    """Every listed edge is implied by the schedule's issue order: program
    order on each stream plus record -> wait pairs of the same event."""
    for first, last, _ in read_edges_golden():
        ops = O.schedule(first, last)
        succ = {i: set() for i in range(len(ops))}
        prev_on = {}
        for i, op in enumerate(ops):
            if op.stream in prev_on:
                succ[prev_on[op.stream]].add(i)
            prev_on[op.stream] = i
        for i, a in enumerate(ops):
            for k, b in enumerate(ops):
                if a.layer == b.layer and (a.kind, b.kind) in (("record_ready", "wait_ready"),
                                                               ("record_done", "wait_done")):
                    succ[i].add(k)

        def reach(i):
            seen, todo = set(), [i]
            while todo:
                for k in succ[todo.pop()]:
                    if k not in seen:
                        seen.add(k)
                        todo.append(k)
            return seen

        idx = {(op.kind, op.layer): i for i, op in enumerate(ops) if op.kind in ("gather", "compute")}
        for a, b in O.happens_before(first, last):
            assert idx[b] in reach(idx[a]), (first, last, a, b)
        # the lookahead itself: gather(l + 1) is not ordered after compute(l),
        # so the two may overlap
        for l in range(first, last):
            assert idx[("gather", l + 1)] not in reach(idx[("compute", l)])


def test_dequant_at_and_linear_rows_select_from_the_definition():
    rng = np.random.default_rng(33)
    rows, cols = 300, 200  # partial 128-blocks in both directions
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x41
    sc = (2.0 ** rng.uniform(-8, -4, size=(3, 2))).astype(np.float32)
    rsel, csel = [0, 5, 127, 128, 299], [0, 127, 128, 199]
    got = O.dequant_at(q, sc, rsel, csel)
    for a, o in enumerate(rsel):  # element by element from the definition
        for b, i in enumerate(csel):
            assert got[a, b] == O.e4m3_code_value(int(q[o, i])) * float(sc[o // 128, i // 128])
    assert np.array_equal(O.dequant_at(q, sc), O.dequant(q, sc))
    x = _bf16_values(rng, (3, cols))
    np.testing.assert_allclose(O.linear_rows(x, q, sc, rsel), O.linear(x, q, sc)[:, rsel], rtol=1e-12, atol=0)
    onehot = np.zeros((1, cols))
    onehot[0, 130] = 1.0
    assert np.array_equal(O.linear_rows(onehot, q, sc, rsel)[0], O.dequant_at(q, sc, rsel, [130])[:, 0])


# ---------------------------------------------------------------------------
# block scales inside T (optional layout), hand-typed golden
# ---------------------------------------------------------------------------


def read_scales_golden():
    """Cases of tests/golden/layout_scales_in_t.txt: name -> (N, [(entry name,
    rows, cols, elem, block_scaled, offset, scale offset)], |T|, C)."""
    cases = {}
    with open(os.path.join(GOLDEN, "layout_scales_in_t.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, ents, total, chunk = [p.strip() for p in line.split("|")]
            name, n = head.split()
            rows = []
            for tok in ents.split():
                nm, rest = tok.split(":")
                shape, offs = rest.split("=")
                r, c, e, s = (int(v) for v in shape.split(","))
                o, so = (int(v) for v in offs.split("/"))
                rows.append((nm, r, c, e, bool(s), o, so))
            cases[name] = (int(n), rows, int(total), int(chunk))
    return cases


def _scales_layout_matches_golden(plan_fn) -> bool:
    for n, ents, total, chunk in read_scales_golden().values():
        p = plan_fn([(0, r, c, e, s) for (_, r, c, e, s, _, _) in ents], n)
        ly = p.layers[0]
        if (ly.total, ly.chunk) != (total, chunk):
            return False
        for j, (_, r, c, _, _, off, soff) in enumerate(ents):
            if ly.offsets.get(j, -1) != off or ly.scale_offsets.get(j, -1) != soff:
                return False
            if soff >= 0 and ly.scale_sizes[j] != 4 * (-(-r // 128)) * (-(-c // 128)):
                return False
    return True


def test_scales_in_t_layout_matches_hand_derived_golden():
    assert _scales_layout_matches_golden(lambda e, n: O.plan_layout(e, n, scales_in_t=True))
    # without the flag the same entries give the plain layout: no scale entries
    n, ents, _, _ = read_scales_golden()["scales_tiny"]
    assert O.plan_layout([(0, r, c, e, s) for (_, r, c, e, s, _, _) in ents], n).layers[0].total == 360448


def _mutant_scales_plan(kind):
    """plan_layout with the scales placed by a planted wrong rule."""
    def plan(entries, n):
        p = O.plan_layout(entries, n, scales_in_t=True)
        ly = p.layers[0]
        off = 0
        grids = {j: 4 * (-(-entries[j][1] // 128)) * (-(-entries[j][2] // 128)) for j in ly.scale_offsets}
        tail = []
        for j in ly.entries:
            if kind == "before" and j in grids:  # scales ahead of their weight
                ly.scale_offsets[j] = off
                off += O.roundup(grids[j], 16)
            ly.offsets[j] = off
            off += O.roundup(ly.sizes[j], 16)
            if kind in ("unpadded", "rule") and j in grids:
                ly.scale_offsets[j] = off
                off += grids[j] if kind == "unpadded" else O.roundup(grids[j], 16)
            if kind == "at_end" and j in grids:
                tail.append(j)
        for j in tail:  # all scales after all weights
            ly.scale_offsets[j] = off
            off += O.roundup(grids[j], 16)
        ly.total = O.roundup(off, 16 * n)
        ly.chunk = ly.total // n
        return p
    return plan


@pytest.mark.parametrize("kind", ["rule", "before", "unpadded", "at_end"])
def test_scales_golden_catches_planted_placement_mistakes(kind):
    assert _scales_layout_matches_golden(_mutant_scales_plan(kind)) == (kind == "rule")


def test_scales_in_t_pack_view_and_relayout():
    rng = np.random.default_rng(34)
    for n, ents, total, chunk in read_scales_golden().values():
        p = O.plan_layout([(0, r, c, e, s) for (_, r, c, e, s, _, _) in ents], n, scales_in_t=True)
        ly = p.layers[0]
        data = {j: rng.integers(1, 256, size=(ents[j][1], ents[j][2] * ents[j][3]), dtype=np.uint8)
                for j in ly.entries}
        scales = {j: (2.0 ** rng.uniform(-8, -4, size=O.scale_grid(ents[j][1], ents[j][2]))).astype(np.float32)
                  for j in range(len(ents)) if ents[j][4]}
        t = O.pack(p, 0, data, scales)
        assert t.size == total
        for j in ly.entries:
            assert np.array_equal(O.view(p, 0, t, j), data[j])
        for j in ly.scale_offsets:
            assert np.array_equal(O.scales_view(p, 0, t, j), scales[j])
            # the float32 bytes as they are in memory
            o = ly.scale_offsets[j]
            assert t[o:o + 4].tobytes() == scales[j].reshape(-1)[:1].tobytes()
        ch = O.split_chunks(p, 0, t)
        assert [c.size for c in ch] == [chunk] * n
        shards = {j: WL.row_shards(data[j], n) for j in ly.entries}
        got = O.relayout(p, 0, shards, scales)
        assert all(np.array_equal(a, b) for a, b in zip(got, ch))
