"""FP16 weights, the other unquantised 16-bit format of the blog's variants
list (section "加载：行 shard 先行，finalize 再重排"): IEEE binary16 weights go
through the same flat layout, without scales. The tensor cores take both
operands of one MMA in one format, so the bf16 activations are rounded to f16
first (on the decode path inside the kernels, at prefill sizes by a conversion
kernel into the workspace); the oracle's linear_f16 does the same rounding.
Checked on decode (m <= 64, slot and chunk-map reads) and prefill sizes, with
the kernel that ran read from the trace tag."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, linear_kinds, typed_stack, weight_bytes, x_f64

pytestmark = pytest.mark.gpu

KERNEL_MMA, KERNEL_MMA_FUSED, KERNEL_TC, KERNEL_TC_FUSED, KERNEL_PREFILL = 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


# N = 4. Entry 0 (333 rows) is replicated (333 % 4 != 0); chunk boundaries fall
# inside rows of entries 1 and 2; cols 208 leaves a partial 64-K slab.
SHAPES = [(0, 4, 333, 208), (0, 4, 1000, 1040), (0, 4, 256, 64), (0, 4, 512, 208)]


@pytest.fixture(scope="module")
def f16_stack(S):
    assert S.F16 == 4
    bits = [WL.draw_weight_f16(81, 0, j, r, c) for j, (_, _, r, c) in enumerate(SHAPES)]
    st = typed_stack(S, SHAPES, 4, [weight_bytes(b) for b in bits], max_m=1000)
    st.ctx.gather_to_slot(0, 0, 0)
    return st, bits


@pytest.fixture(params=["tcgen05", "mma"])
def decode_kernel(S, request):
    """The default (tcgen05 kind::f16) or the mma.sync decode kernel on views."""
    S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_AUTO if request.param == "tcgen05" else S.DECODE_MMA)
    yield KERNEL_TC if request.param == "tcgen05" else KERNEL_MMA
    S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_AUTO)


def _bf16_of(v):
    """float64 values -> the bits of their nearest-even bf16 (through float32,
    exact for f16 values: they have 11 significant bits)."""
    return WL.bf16_bits(torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16))


@pytest.mark.parametrize("m", [1, 8, 17, 40, 64])
def test_f16_decode_matches_oracle(S, f16_stack, decode_kernel, m):
    st, bits = f16_stack
    for j, (_, _, r, c) in enumerate(SHAPES):
        x = WL.draw_x(82, j, m, c).cuda()
        y, kinds = linear_kinds(st, j, S.SRC_SLOT0, x, m)
        assert kinds == [decode_kernel]
        assert_close(bf16_tensor_to_f64(y), O.linear_f16(x_f64(x), bits[j]), f"entry {j} m {m}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m", [1, 33])
def test_f16_decode_through_the_chunk_map(S, f16_stack, m):
    st, bits = f16_stack
    for j in (1, 2, 3):  # sharded entries
        _, _, r, c = SHAPES[j]
        x = WL.draw_x(83, j, m, c).cuda()
        y, kinds = linear_kinds(st, j, S.SRC_FUSED, x, m)
        assert kinds == [KERNEL_TC_FUSED]
        assert_close(bf16_tensor_to_f64(y), O.linear_f16(x_f64(x), bits[j]), f"entry {j} m {m} (fused)")


def test_f16_straddling_rows_one_hot(S, f16_stack):
    # Rows that a chunk boundary splits are computed by the settle kernel from
    # the chunks: with one-hot x they give the f16 weight, rounded once to bf16.
    st, bits = f16_stack
    plan = O.plan_layout([(l, r, c, 2) for (l, _, r, c) in SHAPES], 4)
    lay = plan.layers[0]
    straddling = []
    for j, (_, _, r, c) in enumerate(SHAPES):
        if not plan.sharded[j]:
            continue
        o = lay.offsets[j]
        for i in range(1, 4):
            b = i * lay.chunk
            if o < b < o + r * c * 2 and (b - o) % (2 * c):
                straddling.append((j, (b - o) // (2 * c)))
    assert straddling
    rng = np.random.default_rng(6)
    m = 8
    for j, row in straddling:
        _, _, r, c = SHAPES[j]
        cols = rng.integers(0, c, size=m)
        xo = torch.zeros((m, c), dtype=torch.bfloat16)
        xo[np.arange(m), torch.from_numpy(cols)] = 1.0
        y, kinds = linear_kinds(st, j, S.SRC_FUSED, xo.cuda(), m)
        assert kinds == [KERNEL_TC_FUSED]
        want = _bf16_of(O.f16_decode(bits[j][row, cols]))
        assert np.array_equal(WL.bf16_bits(y[:, row].cpu()), want), f"entry {j} row {row}"


@pytest.mark.parametrize("m", [3, 40, 200])
def test_f16_one_hot_gives_the_weight_rounded_to_bf16(S, f16_stack, decode_kernel, m):
    # x = e_i picks column i of W: one product, exact in fp32, then rounded to
    # bf16 (f16 has 3 more significand bits than bf16).
    st, bits = f16_stack
    rng = np.random.default_rng(m + 1)
    for j in (1, 3):
        _, _, r, c = SHAPES[j]
        cols = rng.integers(0, c, size=m)
        xo = torch.zeros((m, c), dtype=torch.bfloat16)
        xo[np.arange(m), torch.from_numpy(cols)] = 1.0
        y, kinds = linear_kinds(st, j, S.SRC_SLOT0, xo.cuda(), m)
        assert kinds == [decode_kernel if m <= 64 else KERNEL_PREFILL]
        want = _bf16_of(O.f16_decode(bits[j][:, cols].T))
        assert np.array_equal(WL.bf16_bits(y.cpu()), want), f"entry {j}"


def test_f16_activation_rounding_is_applied(S, f16_stack, decode_kernel):
    # bf16 activations below the f16 normal range (2^-14) lose significand
    # bits in f16 (spacing 2^-24). With x in [2^-28, 2^-21) the f16 rounding
    # moves Y by about 19 percent, so a result that skipped it (or rounded
    # differently) misses the oracle's f16-rounded Y by far more than the
    # relative bar; the absolute term of the usual bar would hide that at
    # these magnitudes, so the check here is relative only.
    st, bits = f16_stack
    j = 2  # 256 x 64
    _, _, r, c = SHAPES[j]
    for m in (5, 100):
        rng = np.random.default_rng(m)
        xf = (rng.uniform(1, 2, size=(m, c)) * 2.0 ** rng.integers(-28, -22, size=(m, c))).astype(np.float32)
        x = torch.from_numpy(xf).to(torch.bfloat16)
        y, _ = linear_kinds(st, j, S.SRC_SLOT0, x.cuda(), m)
        xd = x_f64(x)
        ref = O.linear_f16(xd, bits[j])
        unrounded = xd @ O.f16_decode(bits[j]).T
        got = bf16_tensor_to_f64(y)
        rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel(unrounded, ref) > 5e-2  # the rounding matters here
        assert rel(got, ref) <= 5e-3, f"m {m}: rel err {rel(got, ref):.3e}"
        assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max(), f"m {m}"


@pytest.mark.parametrize("m", [65, 300, 1000])
def test_f16_prefill_matches_oracle(S, f16_stack, m):
    st, bits = f16_stack
    for j, (_, _, r, c) in enumerate(SHAPES):
        x = WL.draw_x(84, j, m, c).cuda()
        y, kinds = linear_kinds(st, j, S.SRC_SLOT0, x, m)
        assert kinds == [KERNEL_PREFILL]
        assert_close(bf16_tensor_to_f64(y), O.linear_f16(x_f64(x), bits[j]), f"entry {j} m {m}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m", [8, 200])
def test_layer_with_all_three_weight_types(S, m):
    # One layer with E4M3, BF16 and F16 linears: the grouped decode launches
    # (one per weight type) and the prefill layer (side-stream quantiser for
    # E4M3, side-stream f16 rounding for F16, neither for BF16).
    shapes = [(0, S.E4M3, 512, 256), (0, S.F16, 256, 512), (0, S.BF16, 384, 128), (0, S.F16, 384, 384),
              (0, S.E4M3, 256, 384)]
    weights, scales, ref_w = {}, {}, {}
    for j, (_, dt, r, c) in enumerate(shapes):
        if dt == S.E4M3:
            q, sc = WL.draw_weight(85, 0, j, r, c)
            weights[j], scales[j] = q, torch.from_numpy(sc)
            ref_w[j] = (q, sc)
        elif dt == S.BF16:
            b = WL.draw_weight_bf16(85, 0, j, r, c)
            weights[j], ref_w[j] = weight_bytes(b), b
        else:
            b = WL.draw_weight_f16(85, 0, j, r, c)
            weights[j], ref_w[j] = weight_bytes(b), b
    st = typed_stack(S, shapes, 4, weights, scales, max_m=max(m, 64))
    st.ctx.gather_to_slot(0, 1, 0)
    xs = [WL.draw_x(86, j, m, c).cuda() for j, (_, _, r, c) in enumerate(shapes)]
    ys = [torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda") for (_, _, r, c) in shapes]
    st.ctx.layer_linears(0, S.SRC_SLOT1, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
    torch.cuda.synchronize()
    for j, (_, dt, r, c) in enumerate(shapes):
        xf = x_f64(xs[j])
        if dt == S.E4M3:
            if m > 64:
                xq, ex = O.quantize_x(xf)
                ref = O.dequant_x(xq, ex) @ O.dequant(*ref_w[j]).T
            else:
                ref = O.linear(xf, *ref_w[j])
        elif dt == S.BF16:
            ref = O.linear_bf16(xf, ref_w[j])
        else:
            ref = O.linear_f16(xf, ref_w[j])
        assert_close(bf16_tensor_to_f64(ys[j]), ref, f"entry {j} m {m}")
    assert st.ctx.status() == 0


def test_f16_run_layers(S):
    shapes = [(l, S.F16, r, c) for l in range(3) for (r, c) in ((512, 256), (256, 512))]
    bits = [WL.draw_weight_f16(87, l, j, r, c) for j, (l, _, r, c) in enumerate(shapes)]
    st = typed_stack(S, shapes, 4, [weight_bytes(b) for b in bits])
    m = 8
    xs = {j: WL.draw_x(88, j, m, c).cuda() for j, (_, _, r, c) in enumerate(shapes)}
    ys = {j: torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda")
          for j, (_, _, r, c) in enumerate(shapes)}
    io = [([xs[j].data_ptr() for j in st.layer_entries(l)], [ys[j].data_ptr() for j in st.layer_entries(l)], m)
          for l in range(3)]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    for flags in (0, S.RUN_FUSED):
        st.ctx.run_layers(0, 2, io, flags, main.cuda_stream, side.cuda_stream)
        main.synchronize()
        for j in ys:
            assert_close(bf16_tensor_to_f64(ys[j]), O.linear_f16(x_f64(xs[j]), bits[j]), f"entry {j} flags {flags}")
    assert st.ctx.status() == 0


def test_f16_shared_expert_full_size_sampled(S):
    # The shared-expert layer at full size with f16 weights (528 MB, N = 16):
    # decode at M = 32 from the slot and through the chunk map, and prefill at
    # m = 2048, on 40 sampled output rows (all tokens) against the oracle.
    w = WL.SHARED_EXPERT
    shapes = [(0, S.F16, e.rows, e.cols) for e in w.entries]
    bits = [WL.draw_weight_f16(89, 0, j, e.rows, e.cols) for j, e in enumerate(w.entries)]
    st = typed_stack(S, shapes, w.n_shards, [weight_bytes(b) for b in bits], max_m=2048)
    st.ctx.gather_to_slot(0, 0, 0)
    rng = np.random.default_rng(90)
    for j, e in enumerate(w.entries):
        rows = np.unique(np.concatenate([[0, e.rows - 1], rng.choice(e.rows, size=38, replace=False)]))
        wsel = bits[j][rows]
        for m, src, kind in ((32, S.SRC_SLOT0, KERNEL_TC), (32, S.SRC_FUSED, KERNEL_TC_FUSED),
                             (2048, S.SRC_SLOT0, KERNEL_PREFILL)):
            x = WL.draw_x(91, j, m, e.cols).cuda()
            y, kinds = linear_kinds(st, j, src, x, m)
            assert kinds == [kind]
            want = O.linear_f16(x_f64(x), wsel)
            assert_close(bf16_tensor_to_f64(y)[:, rows], want, f"{e.name} m {m} src {src}")
    assert st.ctx.status() == 0
