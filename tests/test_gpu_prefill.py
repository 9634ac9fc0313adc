"""Prefill linears (m > 64): the activation quantiser and the tcgen05
block-scaled FP8 GEMM against the CPU oracle. The oracle quantises the same
bf16 activations with its own quantiser (bit-exact with the GPU one, see
test_gpu_parity.test_quantize_x_bit_exact) and computes
Y = dequant(xq, ex) @ dequant(W)^T in float64; the GPU output must meet the
floating-point bar of helpers.assert_close. The error against the unquantised
bf16 activations is printed, not gated."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import LayerData, assert_close, bf16_tensor_to_f64, build_stack, draw_layers, workload_entries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _ref_quantised(x_bf16, codes, scales, rows=None):
    xf = WL.bf16_to_f64(WL.bf16_bits(x_bf16))
    xq, ex = O.quantize_x(xf)
    xd = O.dequant_x(xq, ex)
    if rows is not None:
        xd = xd[rows]
    return xd @ O.dequant(codes, scales).T, xf


def _rand_layer(rng, shapes):
    codes, scales = {}, {}
    for j, (_, r, c) in enumerate(shapes):
        q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3B  # no NaN codes
        codes[j] = q
        scales[j] = (2.0 ** rng.uniform(-8, -4, size=(-(-r // 128), -(-c // 128)))).astype(np.float32)
    return LayerData(codes, scales)


KERNEL_PREFILL, KERNEL_PREFILL_PAIR = 5, 6


@pytest.fixture(params=["single", "pair"])
def kernel(S, request):
    """Forces one prefill kernel for the test, then restores the default."""
    S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_SINGLE if request.param == "single" else S.PREFILL_PAIR)
    yield KERNEL_PREFILL if request.param == "single" else KERNEL_PREFILL_PAIR
    S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_AUTO)


def _linear_traced(st, j, src, x, m):
    """Runs one linear with tracing on; returns y and the kernel id of its record."""
    rec = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
    st.ctx.trace_begin(rec.data_ptr(), 4, 0)
    _, _, rows, _ = st.entries[j]
    y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(j, src, x.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    n = st.ctx.trace_count()
    st.ctx.trace_begin(0, 0, 0)
    tags = [int(t) for t in rec.view(4, 4)[:n, 0].tolist()]
    return y, [(t >> 48) & 0xFF for t in tags if (t >> 48) & 0xFF in (KERNEL_PREFILL, KERNEL_PREFILL_PAIR)]


@pytest.mark.parametrize("m", [65, 128, 300, 1000])
def test_prefill_ragged_tiles(S, kernel, m):
    # rows not multiples of the 256-row weight tile (nor of 128), several K
    # slabs; with the pair kernel, m = 65 and 128 leave the second CTA's
    # activation rows, and rows = 256 its weight rows, entirely past the edge.
    shapes = [(0, 4 * 64, 128), (0, 4 * 97, 512), (0, 4 * 250, 1152)]
    rng = np.random.default_rng(40 + m)
    ld = _rand_layer(rng, shapes)
    st = build_stack(S, shapes, 4, [ld], max_m=m)
    st.ctx.gather_to_slot(0, 0, 0)
    for j, (_, r, c) in enumerate(shapes):
        x = WL.draw_x(60, j, m, c)
        y, kerns = _linear_traced(st, j, S.SRC_SLOT0, x.cuda(), m)
        assert kerns == [kernel]
        ref, _ = _ref_quantised(x, ld.codes[j], ld.scales[j])
        assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} m {m}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m", [300, 1000])
def test_prefill_pair_and_single_agree_bitwise(S, m):
    # Both kernels add the same per-slab MMA results in the same slab order.
    shapes = [(0, 4 * 97, 512), (0, 4 * 250, 1152)]
    rng = np.random.default_rng(70 + m)
    ld = _rand_layer(rng, shapes)
    st = build_stack(S, shapes, 4, [ld], max_m=m)
    st.ctx.gather_to_slot(0, 0, 0)
    try:
        for j, (_, r, c) in enumerate(shapes):
            x = WL.draw_x(61, j, m, c).cuda()
            S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_SINGLE)
            y1, k1 = _linear_traced(st, j, S.SRC_SLOT0, x, m)
            S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_PAIR)
            y2, k2 = _linear_traced(st, j, S.SRC_SLOT0, x, m)
            assert (k1, k2) == ([KERNEL_PREFILL], [KERNEL_PREFILL_PAIR])
            assert torch.equal(y1, y2), f"entry {j}: max diff {(y1.float() - y2.float()).abs().max().item()}"
    finally:
        S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_AUTO)
    assert st.ctx.status() == 0


def test_prefill_special_cases(S, kernel):
    rng = np.random.default_rng(3)
    r, c, m = 384, 256, 200
    q = rng.integers(0, 0x7E, size=(r, c), dtype=np.uint8)
    sc = (2.0 ** rng.uniform(-8, -4, size=(3, 2))).astype(np.float32)
    ld = LayerData({0: q, 1: q.copy()}, {0: sc, 1: np.zeros_like(sc)})
    st = build_stack(S, [(0, r, c), (0, r, c)], 4, [ld], max_m=m)
    st.ctx.gather_to_slot(0, 1, 0)
    # zero weight scales give exactly zero; all-zero activations give zero
    x = WL.draw_x(61, 0, m, c).cuda()
    y = torch.full((m, r), 7.0, dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(1, S.SRC_SLOT1, x.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    assert not y.float().abs().max().item()
    xz = torch.zeros((m, c), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(0, S.SRC_SLOT1, xz.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    assert not y.float().abs().max().item()
    # one-hot rows: x = 1 at column i gives the dequantised column exactly
    # (ex = 2^-8 makes the code of 1.0 exact), rounded once to bf16
    xo = torch.zeros((m, c), dtype=torch.bfloat16)
    cols = rng.integers(0, c, size=m)
    xo[np.arange(m), torch.from_numpy(cols)] = 1.0
    st.ctx.linear(0, S.SRC_SLOT1, xo.cuda().data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    want = O.dequant_at(q, sc, cols=cols).T
    got = bf16_tensor_to_f64(y)
    assert np.array_equal(got, WL.bf16_to_f64(WL.bf16_bits(torch.from_numpy(want).float().to(torch.bfloat16))))


def test_prefill_kda_layer_small(S):
    w = WL.scaled_workload(WL.ATTN_KDA, rows_div=8, cols_div=8, name="kda_div8")
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, 8, layers, max_m=512)
    st.ctx.gather_to_slot(0, 0, 0)
    m = 512
    xs = [WL.draw_x(w.key, j, m, c) for j, (_, r, c) in enumerate(ents)]
    ys = [torch.empty((m, r), dtype=torch.bfloat16, device="cuda") for (_, r, c) in ents]
    xd = [x.cuda() for x in xs]
    st.ctx.layer_linears(0, S.SRC_SLOT0, [x.data_ptr() for x in xd], [y.data_ptr() for y in ys], m, 0)
    torch.cuda.synchronize()
    for j in range(len(ents)):
        ref, xf = _ref_quantised(xs[j], layers[0].codes[j], layers[0].scales[j])
        got = bf16_tensor_to_f64(ys[j])
        assert_close(got, ref, f"entry {j}")
        exact = xf @ O.dequant(layers[0].codes[j], layers[0].scales[j]).T
        rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
        print(f"entry {j}: relative error vs bf16-exact oracle {rel:.3e}")


@pytest.mark.parametrize("m", [2048, 8192])
def test_prefill_full_size_sampled_rows(S, kernel, m):
    # The prefill workload's weights (KDA-like layer, N = 8), full sizes, at
    # both token counts the benchmark times; the oracle computes 192 sampled
    # token rows (and the first and last) of every linear.
    w = WL.PREFILL
    ents = workload_entries(w, 1)
    layers = draw_layers(WL.scaled_workload(w, n_layers=1), 1)
    st = build_stack(S, ents, w.n_shards, layers, max_m=m)
    st.ctx.gather_to_slot(0, 1, 0)
    rng = np.random.default_rng(m)
    for j, (_, r, c) in enumerate(ents):
        x = WL.draw_x(w.key, j, m, c)
        y = torch.empty((m, r), dtype=torch.bfloat16, device="cuda")
        st.ctx.linear(j, S.SRC_SLOT1, x.cuda().data_ptr(), m, y.data_ptr(), 0)
        torch.cuda.synchronize()
        sel = np.unique(np.concatenate([[0, m - 1], rng.choice(m, size=192, replace=False)]))
        ref, _ = _ref_quantised(x, layers[0].codes[j], layers[0].scales[j], rows=sel)
        assert_close(bf16_tensor_to_f64(y)[sel], ref, f"entry {j} (sampled rows)")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m", [1000, 2048])
def test_layer_equals_linears_alone_bit_for_bit(S, m):
    # A prefill layer of the workload's full-size linears (layer_linears: the
    # next linear's activations quantised on the side stream while the
    # previous GEMM runs, two buffers used in turn) against each linear run
    # alone: the quantiser is exact and the GEMM deterministic, so every
    # output must be equal; m = 1000 ends rows in a partial tile. Sampled rows
    # must meet the oracle.
    w = WL.PREFILL
    ents = workload_entries(w, 1)
    layers = draw_layers(WL.scaled_workload(w, n_layers=1), 1)
    st = build_stack(S, ents, w.n_shards, layers, max_m=m)
    st.ctx.gather_to_slot(0, 0, 0)
    xs = [WL.draw_x(w.key, j, m, c) for j, (_, r, c) in enumerate(ents)]
    xd = [x.cuda() for x in xs]
    ys = [torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda") for (_, r, c) in ents]
    rng = np.random.default_rng(77 + m)
    sel = np.unique(np.concatenate([[0, m - 1], rng.choice(m, size=24, replace=False)]))
    for rep in range(2):  # twice: the second call reuses buffers the first one wrote
        st.ctx.layer_linears(0, S.SRC_SLOT0, [x.data_ptr() for x in xd], [y.data_ptr() for y in ys], m, 0)
        torch.cuda.synchronize()
        assert st.ctx.status() == 0
        for j, (_, r, c) in enumerate(ents):
            alone = torch.empty((m, r), dtype=torch.bfloat16, device="cuda")
            st.ctx.linear(j, S.SRC_SLOT0, xd[j].data_ptr(), m, alone.data_ptr(), 0)
            torch.cuda.synchronize()
            assert torch.equal(ys[j].view(torch.int16), alone.view(torch.int16)), f"rep {rep} entry {j}"
    for j, (_, r, c) in enumerate(ents):
        ref, _ = _ref_quantised(xs[j], layers[0].codes[j], layers[0].scales[j], rows=sel)
        assert_close(bf16_tensor_to_f64(ys[j])[sel], ref, f"entry {j} (sampled rows)")
    assert st.ctx.status() == 0
