"""Block scales inside T (plan flag SWS_SCALES_IN_T): each sharded E4M3
weight's fp32 block-scale tensor is an entry of T right after the weight. The
relayout (sws_relayout + sws_relayout_scales) and the gather against the
oracle's chunks and T byte for byte; decode linears reading the scales from the
slot and through the chunk map, prefill linears from the slot, and the
lookahead run, against the oracle. The caller's own copies of those scales are
overwritten with NaN once the context exists, so a kernel that read them
instead of T would fail. Includes a layout whose chunk boundary falls inside a
scale tensor, a replicated E4M3 entry (its scales stay outside T) and a BF16
entry (no scales)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, x_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _weights(rng, shapes):
    """shapes: (layer, dtype, rows, cols) -> codes (bytes) and block scales (E4M3 only)."""
    codes, scales = {}, {}
    for j, (_, dt, r, c) in enumerate(shapes):
        if dt == 0:  # E4M3
            q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
            q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes
            codes[j] = q
            scales[j] = (2.0 ** rng.uniform(-8, -4, size=O.scale_grid(r, c))).astype(np.float32)
        else:  # BF16
            codes[j] = WL.draw_weight_bf16(31, 0, j, r, c).view(np.uint8).reshape(r, -1)
    return codes, scales


def _build(S, shapes, n, codes, scales, max_m=64):
    from sharded_weight_storage_gb300.storage import ShardedStack
    st = ShardedStack(shapes, n, max_m=max_m, flags=S.SCALES_IN_T)
    for l in sorted({s[0] for s in shapes}):
        js = [j for j, s in enumerate(shapes) if s[0] == l]
        st.load_layer(l, {j: torch.from_numpy(codes[j]) for j in js},
                      {j: torch.from_numpy(scales[j]) for j in js if j in scales})
    st.make_ctx()
    for j in range(len(shapes)):  # the caller's copies of scales that live in T are never read again
        if st.scale_info[j][0] >= 0:
            st.scales[j].fill_(float("nan"))
    torch.cuda.synchronize()
    return st


def _oracle(shapes, n, codes, scales):
    eb = {0: 1, 1: 2}
    return O.plan_layout([(l, r, c, eb[dt], dt == 0) for (l, dt, r, c) in shapes], n, scales_in_t=True)


def _ref(shapes, j, x, codes, scales):
    _, dt, r, c = shapes[j]
    if dt == 0:
        return O.linear(x_f64(x), codes[j], scales[j])
    return O.linear_bf16(x_f64(x), codes[j].view(np.uint16).reshape(r, c))


# a chunk boundary 256 bytes into W_a's 512-byte scale tensor (N = 2)
STRADDLE = ([(0, 0, 1024, 2048), (0, 0, 32, 65472)], 2)
# the tiny workload's shapes, plus a replicated E4M3 entry (rows % 4 != 0) and a BF16 entry
MIXED = ([(0, 0, 512, 256), (0, 0, 384, 256), (0, 0, 130, 256), (0, 1, 256, 512), (0, 0, 256, 512)], 4)


def test_straddle_layout_really_straddles():
    shapes, n = STRADDLE
    p = _oracle(shapes, n, None, None)
    ly = p.layers[0]
    o, s = ly.scale_offsets[0], ly.scale_sizes[0]
    assert o < ly.chunk < o + s and ly.chunk - o == 256


@pytest.mark.parametrize("case", [STRADDLE, MIXED], ids=["straddle", "mixed"])
def test_relayout_and_gather_with_scales_in_t(S, case):
    shapes, n = case
    rng = np.random.default_rng(41)
    codes, scales = _weights(rng, shapes)
    st = _build(S, shapes, n, codes, scales)
    p = _oracle(shapes, n, codes, scales)
    ly = p.layers[0]
    shards = {j: WL.row_shards(codes[j], n) for j in ly.entries}
    want = O.relayout(p, 0, shards, scales)
    for i in range(n):
        assert np.array_equal(st.chunks[0][i].cpu().numpy(), want[i]), f"chunk {i}"
    assert np.array_equal(O.gather(want), O.pack(p, 0, codes, scales))
    st.ctx.gather_to_slot(0, 1, 0)
    torch.cuda.synchronize()
    assert np.array_equal(st.slots[1][:ly.total].cpu().numpy(), O.pack(p, 0, codes, scales))
    for j in ly.scale_offsets:
        assert np.array_equal(st.slot_scales(1, j).cpu().numpy(), scales[j])
    for j, (_, dt, r, c) in enumerate(shapes):
        assert st.scale_info[j] == (ly.scale_offsets.get(j, -1), ly.scale_sizes.get(j, 0))


@pytest.mark.parametrize("case", [STRADDLE, MIXED], ids=["straddle", "mixed"])
@pytest.mark.parametrize("m", [1, 8, 33, 64])
def test_decode_reads_scales_from_t(S, case, m):
    shapes, n = case
    rng = np.random.default_rng(42)
    codes, scales = _weights(rng, shapes)
    st = _build(S, shapes, n, codes, scales)
    st.ctx.gather_to_slot(0, 0, 0)
    for j, (_, dt, r, c) in enumerate(shapes):
        x = WL.draw_x(43, j, m, c)
        ref = _ref(shapes, j, x, codes, scales)
        for src in (S.SRC_SLOT0, S.SRC_FUSED):
            y = torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda")
            st.ctx.linear(j, src, x.cuda().data_ptr(), m, y.data_ptr(), 0)
            torch.cuda.synchronize()
            assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} src {src} m {m}")
    # the whole layer at once (grouped launches; the chunk-map group stages the scales once)
    xs = [WL.draw_x(44, j, m, c).cuda() for j, (_, _, _, c) in enumerate(shapes)]
    for src in (S.SRC_SLOT0, S.SRC_FUSED):
        ys = [torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda") for (_, _, r, _) in shapes]
        st.ctx.layer_linears(0, src, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
        torch.cuda.synchronize()
        for j in range(len(shapes)):
            assert_close(bf16_tensor_to_f64(ys[j]), _ref(shapes, j, xs[j].cpu(), codes, scales),
                         f"layer_linears entry {j} src {src} m {m}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m", [130, 300])
def test_prefill_reads_scales_from_t(S, m):
    shapes = [(0, 0, 512, 1024), (0, 0, 384, 768), (0, 1, 256, 512), (0, 0, 130, 256)]
    n = 4
    rng = np.random.default_rng(45)
    codes, scales = _weights(rng, shapes)
    st = _build(S, shapes, n, codes, scales, max_m=m)
    st.ctx.gather_to_slot(0, 1, 0)
    for j, (_, dt, r, c) in enumerate(shapes):
        x = WL.draw_x(46, j, m, c)
        y = torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda")
        st.ctx.linear(j, S.SRC_SLOT1, x.cuda().data_ptr(), m, y.data_ptr(), 0)
        torch.cuda.synchronize()
        if dt == 0:  # the oracle on the same quantised activations
            ref = O.dequant_x(*O.quantize_x(x_f64(x))) @ O.dequant(codes[j], scales[j]).T
        else:
            ref = _ref(shapes, j, x, codes, scales)
        assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} m {m}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("m,flags", [(8, 0), (8, 1), (130, 0)], ids=["decode", "decode_fused", "prefill"])
def test_lookahead_run_with_scales_in_t(S, m, flags):
    shapes = [(l, 0, r, c) for l in range(3) for (r, c) in ((512, 1024), (256, 768))]
    n = 4
    rng = np.random.default_rng(47)
    codes, scales = _weights(rng, shapes)
    st = _build(S, shapes, n, codes, scales, max_m=m)
    xs = {j: WL.draw_x(48, j, m, c) for j, (_, _, _, c) in enumerate(shapes)}
    xd = {j: x.cuda() for j, x in xs.items()}
    ys = {j: torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda")
          for j, (_, _, r, _) in enumerate(shapes)}
    io = [([xd[j].data_ptr() for j in st.layer_entries(l)], [ys[j].data_ptr() for j in st.layer_entries(l)], m)
          for l in range(3)]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, 2, io, S.RUN_FUSED if flags else 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    for j in range(len(shapes)):
        if m > 64:
            ref = O.dequant_x(*O.quantize_x(x_f64(xs[j]))) @ O.dequant(codes[j], scales[j]).T
        else:
            ref = _ref(shapes, j, xs[j], codes, scales)
        assert_close(bf16_tensor_to_f64(ys[j]), ref, f"entry {j}")
    assert st.ctx.status() == 0


def test_shared_expert_layer_full_size_with_scales_in_t(S):
    # the decode workload's layer (N = 16) with its scales in T: every sampled
    # output row of both linears at the benchmark's m = 32, from the slot and
    # through the chunk map
    w = WL.SHARED_EXPERT
    lw = WL.layer_weights(w, 0)
    shapes = [(0, 0, e.rows, e.cols) for e in w.entries]
    codes = {j: lw.codes[j] for j in range(2)}
    scales = {j: lw.scales[j] for j in range(2)}
    st = _build(S, shapes, w.n_shards, codes, scales)
    p = _oracle(shapes, w.n_shards, None, None)
    assert st.layout[0][0] == p.layers[0].total == 264241152 + 43008 + 21504
    st.ctx.gather_to_slot(0, 0, 0)
    rng = np.random.default_rng(49)
    m = 32
    for j, (_, _, r, c) in enumerate(shapes):
        x = WL.draw_x(w.key, j, m, c)
        sel = np.unique(np.concatenate([[0, r - 1], rng.choice(r, size=512, replace=False)]))
        ref = O.linear_rows(x_f64(x), codes[j], scales[j], sel)
        for src in (S.SRC_SLOT0, S.SRC_FUSED):
            y = torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda")
            st.ctx.linear(j, src, x.cuda().data_ptr(), m, y.data_ptr(), 0)
            torch.cuda.synchronize()
            assert_close(bf16_tensor_to_f64(y)[:, sel], ref, f"{w.entries[j].name} src {src}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("case", [STRADDLE, MIXED], ids=["straddle", "mixed"])
def test_bounds_self_check_passes_every_copy_of_the_path(S, case):
    # SWS_OPT_CHECK_BOUNDS on for the relayout, the scale relayout, the
    # gathers and the chunk-map scale staging: every segment the library
    # builds stays inside its buffers, so all calls go through, and the
    # results are the oracle's.
    shapes, n = case
    rng = np.random.default_rng(91)
    codes, scales = _weights(rng, shapes)
    S.set_option(S.OPT_CHECK_BOUNDS, 1)
    try:
        st = _build(S, shapes, n, codes, scales)
        for slot in (0, 1):
            st.ctx.gather_to_slot(0, slot, 0)
        torch.cuda.synchronize()
        plan = _oracle(shapes, n, codes, scales)
        t = O.pack(plan, 0, {j: codes[j] for j in range(len(shapes))}, scales=scales)
        for slot in (0, 1):
            assert np.array_equal(st.slots[slot][:t.size].cpu().numpy(), t)
        m = 8
        for j in range(len(shapes)):
            x = WL.draw_x(92, j, m, shapes[j][3]).cuda()
            for src in (S.SRC_SLOT0, S.SRC_FUSED):
                y = torch.empty((m, shapes[j][2]), dtype=torch.bfloat16, device="cuda")
                st.ctx.linear(j, src, x.data_ptr(), m, y.data_ptr(), 0)
                torch.cuda.synchronize()
                assert_close(bf16_tensor_to_f64(y), _ref(shapes, j, x, codes, scales), f"entry {j} src {src}")
        assert st.ctx.status() == 0
    finally:
        S.set_option(S.OPT_CHECK_BOUNDS, 0)
