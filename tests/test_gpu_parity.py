"""GPU parity: the CUDA library (called through the C ABI) against the CPU
oracle on the same seeded inputs. Layout, relayout and gather are bit-exact;
linears meet the floating-point bar in helpers.assert_close."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import (assert_close, bf16_tensor_to_f64, build_stack, draw_layers, oracle_layer_T,
                     workload_entries)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _slot_bytes(st, slot, n):
    return st.slots[slot][:n].cpu().numpy()


# ---------------------------------------------------------------------------
# relayout and gather: bit-exact
# ---------------------------------------------------------------------------

SMALL_KDA = WL.scaled_workload(WL.ATTN_KDA, rows_div=16, cols_div=16, name="kda_div16")


@pytest.mark.parametrize("w", [WL.TINY, SMALL_KDA, WL.SHARED_EXPERT, WL.ATTN_KDA], ids=lambda w: w.name)
def test_relayout_and_gather_bit_exact(S, w):
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    plan, chunks, T = oracle_layer_T(ents, w.n_shards, 0, layers[0])
    for i in range(w.n_shards):
        assert np.array_equal(st.chunks[0][i].cpu().numpy(), chunks[i]), f"chunk {i}"
    canary = 0xA5
    for slot in (0, 1):
        st.slots[slot].fill_(canary)
        st.ctx.gather_to_slot(0, slot, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        got = st.slots[slot].cpu().numpy()
        assert np.array_equal(got[:T.size], T)
        assert np.all(got[T.size:] == canary)  # nothing written past |T|
    assert st.ctx.status() == 0


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 16])
def test_relayout_and_gather_random_odd_shapes(S, n):
    rng = np.random.default_rng(300 + n)
    for trial in range(3):
        ents, codes = [], {}
        for j in range(int(rng.integers(1, 6))):
            rows = int(rng.integers(1, 7)) * n if rng.random() < 0.8 else int(rng.integers(1, 30))
            cols = int(rng.integers(1, 300))
            ents.append((0, rows, cols))
            codes[j] = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
        scales = {j: np.ones((-(-r // 128), -(-c // 128)), np.float32) for j, (_, r, c) in enumerate(ents)}
        from helpers import LayerData
        ld = LayerData(codes, scales)
        with _nowarn():
            st = build_stack(S, ents, n, [ld])
        plan, chunks, T = oracle_layer_T(ents, n, 0, ld)
        if T.size == 0:
            continue
        for i in range(n):
            assert np.array_equal(st.chunks[0][i].cpu().numpy(), chunks[i])
        st.slots[1].fill_(0x5A)
        st.ctx.gather_to_slot(0, 1, 0)
        torch.cuda.synchronize()
        got = st.slots[1].cpu().numpy()
        assert np.array_equal(got[:T.size], T)
        assert np.all(got[T.size:] == 0x5A)


class _nowarn:
    def __enter__(self):
        import warnings
        self.c = warnings.catch_warnings()
        self.c.__enter__()
        warnings.simplefilter("ignore")

    def __exit__(self, *a):
        self.c.__exit__(*a)


def test_gather_into_both_slots_of_a_large_layer_with_many_tiles(S):
    # 40 MB over N = 16 chunks of 2.5 MB: many TMA tiles per CTA and a ragged
    # last tile in every chunk (C is not a multiple of the 32 KB tile).
    ents = [(0, 4096, 5120), (0, 2048, 10240 - 16)]
    rng = np.random.default_rng(1)
    from helpers import LayerData
    ld = LayerData({0: rng.integers(0, 256, (4096, 5120), dtype=np.uint8),
                    1: rng.integers(0, 256, (2048, 10224), dtype=np.uint8)},
                   {0: np.ones((32, 40), np.float32), 1: np.ones((16, 80), np.float32)})
    st = build_stack(S, ents, 16, [ld])
    plan, chunks, T = oracle_layer_T(ents, 16, 0, ld)
    assert plan.layers[0].chunk % (32 * 1024) != 0
    for slot in (0, 1):
        st.ctx.gather_to_slot(0, slot, 0)
    torch.cuda.synchronize()
    for slot in (0, 1):
        assert np.array_equal(st.slots[slot][:T.size].cpu().numpy(), T)


# ---------------------------------------------------------------------------
# decode linears (m <= 64)
# ---------------------------------------------------------------------------


def _run_linear(st, j, src, x, m):
    layer, _, rows, cols = st.entries[j]
    y = torch.empty((m, rows), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(j, src, x.data_ptr(), m, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return y


def _check_linear_full(st, ld, j, src, m, key):
    layer, _, rows, cols = st.entries[j]
    x = WL.draw_x(key, j, m, cols)
    y = _run_linear(st, j, src, x.cuda(), m)
    ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x)), ld.codes[j], ld.scales[j])
    assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} src {src} m {m}")


def _check_linear_sampled(st, ld, j, src, m, key, n_rows=384, seed=0):
    """Sampled output rows (n_rows of them, plus the first and last), or every
    row when n_rows is None, computed by the oracle 4096 rows at a time."""
    layer, _, rows, cols = st.entries[j]
    x = WL.draw_x(key, j, m, cols)
    y = bf16_tensor_to_f64(_run_linear(st, j, src, x.cuda(), m))
    xf = WL.bf16_to_f64(WL.bf16_bits(x))
    if n_rows is None:
        for r0 in range(0, rows, 4096):
            sel = np.arange(r0, min(rows, r0 + 4096))
            assert_close(y[:, sel], O.linear_rows(xf, ld.codes[j], ld.scales[j], sel),
                         f"entry {j} src {src} m {m} rows {r0}..{sel[-1]}")
        return
    rng = np.random.default_rng(seed + j)
    sel = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, size=min(n_rows, rows), replace=False)]))
    ref = O.linear_rows(xf, ld.codes[j], ld.scales[j], sel)
    assert_close(y[:, sel], ref, f"entry {j} src {src} m {m} (sampled rows)")


@pytest.mark.parametrize("w", [WL.TINY, SMALL_KDA], ids=lambda w: w.name)
@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 32, 33, 64])
def test_decode_linear_full_output(S, w, m):
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    for slot in (0, 1):
        st.ctx.gather_to_slot(0, slot, 0)
    for j in range(len(ents)):
        for src in (S.SRC_SLOT0, S.SRC_SLOT1, S.SRC_FUSED):
            _check_linear_full(st, layers[0], j, src, m, w.key)


@pytest.mark.parametrize("w,ms", [(WL.SHARED_EXPERT, (1, 8, 32, 64)), (WL.ATTN_KDA, (1, 16, 64))],
                         ids=["shared_expert", "attn_kda"])
def test_decode_linear_full_size_sampled_rows(S, w, ms):
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    st.ctx.gather_to_slot(0, 0, 0)
    for m in ms:
        for j in range(len(ents)):
            # the benchmark's decode size (m = 32 on the shared-expert layer): every output row
            every = w is WL.SHARED_EXPERT and m == 32
            _check_linear_sampled(st, layers[0], j, S.SRC_SLOT0, m, w.key, n_rows=None if every else 384)
            if m in (1, 32, 64):
                _check_linear_sampled(st, layers[0], j, S.SRC_FUSED, m, w.key, seed=7,
                                      n_rows=None if every else 384)


def test_decode_ragged_shapes(S):
    # rows not a multiple of the CTA row block, cols not a multiple of 128,
    # chunk boundaries inside rows.
    rng = np.random.default_rng(5)
    from helpers import LayerData
    shapes = [(0, 6 * 4 * 7, 16 * 37), (0, 4 * 101, 16 * 9), (0, 4 * 3, 16), (0, 4 * 300, 16 * 200)]
    codes, scales = {}, {}
    for j, (_, r, c) in enumerate(shapes):
        q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C  # no NaN codes
        codes[j] = q
        scales[j] = (2.0 ** rng.uniform(-8, -4, size=(-(-r // 128), -(-c // 128)))).astype(np.float32)
    ld = LayerData(codes, scales)
    st = build_stack(S, shapes, 4, [ld])
    st.ctx.gather_to_slot(0, 1, 0)
    for j in range(len(shapes)):
        for m in (1, 5, 13, 40, 64):
            for src in (S.SRC_SLOT1, S.SRC_FUSED):
                _check_linear_full(st, ld, j, src, m, 99)


def test_decode_special_cases(S):
    from helpers import LayerData
    rng = np.random.default_rng(8)
    r, c = 512, 384
    q = rng.integers(0, 0x7E, size=(r, c), dtype=np.uint8)
    sc = (2.0 ** rng.uniform(-8, -4, size=(4, 3))).astype(np.float32)
    zs = np.zeros_like(sc)
    ld = LayerData({0: q, 1: q.copy()}, {0: sc, 1: zs})
    st = build_stack(S, [(0, r, c), (0, r, c)], 4, [ld])
    st.ctx.gather_to_slot(0, 0, 0)
    # zero scales give exactly zero
    x = WL.draw_x(1, 0, 4, c).cuda()
    y = _run_linear(st, 1, S.SRC_SLOT0, x, 4)
    assert not y.float().abs().max().item()
    # one-hot x selects a dequantised column; every product is exact, so the
    # bf16 output is the rounded column
    for i in (0, 127, 128, 383):
        xo = torch.zeros((1, c), dtype=torch.bfloat16)
        xo[0, i] = 1.0
        y = _run_linear(st, 0, S.SRC_SLOT0, xo.cuda(), 1)
        col = O.dequant_at(q, sc, cols=[i])[:, 0]
        want = torch.from_numpy(col).float().to(torch.bfloat16)
        assert torch.equal(y[0].cpu(), want)
    # m = 0 is a no-op
    st.ctx.linear(0, S.SRC_SLOT0, x.data_ptr(), 0, x.data_ptr(), 0)


def test_linear_refuses_a_slot_holding_another_layer(S):
    from helpers import LayerData
    rng = np.random.default_rng(9)
    ents = [(0, 64, 128), (1, 64, 128)]
    lds = [LayerData({0: rng.integers(0, 0x7E, (64, 128), dtype=np.uint8)}, {0: np.ones((1, 1), np.float32)}),
           LayerData({1: rng.integers(0, 0x7E, (64, 128), dtype=np.uint8)}, {1: np.ones((1, 1), np.float32)})]
    st = build_stack(S, ents, 4, lds)
    st.ctx.gather_to_slot(1, 0, 0)
    x = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SwsError) as ei:
        st.ctx.linear(0, S.SRC_SLOT0, x.data_ptr(), 1, y.data_ptr(), 0)
    assert ei.value.code == S.E_STATE
    with pytest.raises(S.SwsError) as ei:
        st.ctx.linear(1, S.SRC_SLOT1, x.data_ptr(), 1, y.data_ptr(), 0)
    assert ei.value.code == S.E_STATE
    st.ctx.linear(1, S.SRC_SLOT0, x.data_ptr(), 1, y.data_ptr(), 0)
    with pytest.raises(S.SwsError) as ei:
        st.ctx.linear(1, S.SRC_SLOT0, x.data_ptr() + 2, 1, y.data_ptr(), 0)
    assert ei.value.code == S.E_ALIGN


# ---------------------------------------------------------------------------
# prefill activation quantiser: bit-exact
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("m,k", [(1, 128), (7, 400), (300, 2048), (2048, 7168)])
def test_quantize_x_bit_exact(S, m, k):
    x = WL.draw_x(50, 0, m, k)
    xs = x.float()
    scale = torch.from_numpy(2.0 ** np.random.default_rng(m).integers(-30, 30, size=(m, 1))).float()
    x = (xs * scale).to(torch.bfloat16)
    x[0, : min(k, 128)] = 0.0
    if m > 2:
        x[1, 5] = 448.0
        x[2, :] = torch.tensor(1e-38).to(torch.bfloat16)
    xd = x.cuda()
    g = -(-k // 128)
    xq = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    ex = torch.empty((m, g), dtype=torch.float32, device="cuda")
    S.quantize_x(xd.data_ptr(), m, k, xq.data_ptr(), ex.data_ptr(), 0)
    torch.cuda.synchronize()
    rq, re = O.quantize_x(WL.bf16_to_f64(WL.bf16_bits(x)))
    assert np.array_equal(ex.cpu().numpy(), re)
    assert np.array_equal(xq.cpu().numpy(), rq)


# ---------------------------------------------------------------------------
# grouped layer linears (one launch per layer and source path)
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("m", [1, 9, 33, 64])
def test_layer_linears_grouped_kda(S, m):
    w = SMALL_KDA
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    st.ctx.gather_to_slot(0, 1, 0)
    xs = [WL.draw_x(w.key, j, m, c).cuda() for j, (_, r, c) in enumerate(ents)]
    for src in (S.SRC_SLOT1, S.SRC_FUSED):
        ys = [torch.full((m, r), float("nan"), dtype=torch.bfloat16, device="cuda") for (_, r, c) in ents]
        st.ctx.layer_linears(0, src, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
        torch.cuda.synchronize()
        for j in range(len(ents)):
            ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[0].codes[j], layers[0].scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), ref, f"entry {j} src {src} m {m}")


def test_layer_linears_ten_entries_with_replicated(S):
    # 10 entries (two launches of the views group), two of them replicated
    # (rows % N != 0) and therefore read from their own buffers even on the
    # fused source.
    from helpers import LayerData
    rng = np.random.default_rng(21)
    shapes = [(0, 4 * (8 + 13 * j) if j not in (3, 7) else 4 * (8 + 13 * j) + 1, 16 * (3 + 5 * j)) for j in range(10)]
    codes, scales = {}, {}
    for j, (_, r, c) in enumerate(shapes):
        q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C
        codes[j] = q
        scales[j] = (2.0 ** rng.uniform(-8, -4, size=(-(-r // 128), -(-c // 128)))).astype(np.float32)
    with _nowarn():
        st = build_stack(S, shapes, 4, [LayerData(codes, scales)])
    assert [st.entry_info[j][2] for j in range(10)] == [j not in (3, 7) for j in range(10)]
    st.ctx.gather_to_slot(0, 0, 0)
    m = 12
    xs = [WL.draw_x(31, j, m, c).cuda() for j, (_, r, c) in enumerate(shapes)]
    for src in (S.SRC_SLOT0, S.SRC_FUSED):
        ys = [torch.empty((m, r), dtype=torch.bfloat16, device="cuda") for (_, r, c) in shapes]
        st.ctx.layer_linears(0, src, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
        torch.cuda.synchronize()
        for j in range(10):
            ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), codes[j], scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), ref, f"entry {j} src {src}")


# ---------------------------------------------------------------------------
# both decode kernels (warp-level mma.sync and tcgen05) on the same checks
# ---------------------------------------------------------------------------


@pytest.fixture(params=["mma", "tcgen05"])
def decode_kernel(S, request):
    S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_MMA if request.param == "mma" else S.DECODE_TCGEN05)
    yield request.param
    S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_AUTO)


@pytest.mark.parametrize("m", [1, 5, 16, 17, 31, 33, 48, 64])
def test_decode_kernels_full_output(S, decode_kernel, m):
    w = SMALL_KDA
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    st.ctx.gather_to_slot(0, 0, 0)
    xs = [WL.draw_x(w.key, j, m, c).cuda() for j, (_, r, c) in enumerate(ents)]
    for j in range(len(ents)):
        y = _run_linear(st, j, S.SRC_SLOT0, xs[j], m)
        ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[0].codes[j], layers[0].scales[j])
        assert_close(bf16_tensor_to_f64(y), ref, f"{decode_kernel} entry {j} m {m}")
    ys = [torch.empty((m, r), dtype=torch.bfloat16, device="cuda") for (_, r, c) in ents]
    st.ctx.layer_linears(0, S.SRC_SLOT0, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
    torch.cuda.synchronize()
    for j in range(len(ents)):
        ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[0].codes[j], layers[0].scales[j])
        assert_close(bf16_tensor_to_f64(ys[j]), ref, f"{decode_kernel} grouped entry {j} m {m}")
    assert st.ctx.status() == 0


def test_decode_kernels_ragged_and_special(S, decode_kernel):
    rng = np.random.default_rng(77)
    shapes = [(0, 4 * 101, 16 * 9), (0, 4 * 3, 16), (0, 4 * 300, 16 * 200), (0, 4 * 64, 16 * 24)]
    codes, scales = {}, {}
    for j, (_, r, c) in enumerate(shapes):
        q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C
        codes[j] = q
        scales[j] = (2.0 ** rng.uniform(-8, -4, size=(-(-r // 128), -(-c // 128)))).astype(np.float32)
    scales[3][:] = 0.0  # an all-zero-scale weight gives exactly zero
    from helpers import LayerData
    ld = LayerData(codes, scales)
    st = build_stack(S, shapes, 4, [ld])
    st.ctx.gather_to_slot(0, 1, 0)
    for m in (1, 7, 20, 64):
        for j in range(len(shapes)):
            _check_linear_full(st, ld, j, S.SRC_SLOT1, m, 98)
    x = WL.draw_x(1, 0, 40, shapes[3][2]).cuda()
    y = _run_linear(st, 3, S.SRC_SLOT1, x, 40)
    assert not y.float().abs().max().item()
    # one-hot rows select dequantised columns. The tcgen05 kernel scales each
    # slab's exact result once, so its output is the column rounded once to
    # fp32 and then to bf16; the mma.sync kernel re-bases its accumulator when
    # the block scale changes (a few fp32 roundings) and meets the tolerance.
    _, r, c = shapes[2]
    for m in (1, 20, 64):
        cols = rng.integers(0, c, size=m)
        xo = torch.zeros((m, c), dtype=torch.bfloat16)
        xo[np.arange(m), torch.from_numpy(cols)] = 1.0
        y = _run_linear(st, 2, S.SRC_SLOT1, xo.cuda(), m)
        want = O.dequant_at(codes[2], scales[2], cols=cols).T
        if decode_kernel == "tcgen05":
            assert torch.equal(y.cpu(), torch.from_numpy(want).float().to(torch.bfloat16)), f"m {m}"
        else:
            assert_close(bf16_tensor_to_f64(y), want, f"{decode_kernel} one-hot m {m}")


def test_decode_kernels_full_size_sampled(S, decode_kernel):
    w = WL.SHARED_EXPERT
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    st.ctx.gather_to_slot(0, 0, 0)
    for m in (8, 32, 64):
        for j in range(len(ents)):
            _check_linear_sampled(st, layers[0], j, S.SRC_SLOT0, m, w.key, seed=3)
