"""Chunk-map (fused) decode linears on the tcgen05 path: the weight bytes are
read from the N chunks through per-chunk tensor maps, rows that a chunk
boundary splits are computed by the settle kernel, and no slot is touched.
Checked against the CPU oracle on layers whose chunk boundaries fall inside
rows, with the kernel that ran read from the trace tag (bits 48..55)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import LayerData, assert_close, bf16_tensor_to_f64, build_stack, draw_layers, workload_entries

pytestmark = pytest.mark.gpu

KERNEL_MMA_FUSED, KERNEL_TC, KERNEL_TC_FUSED = 2, 3, 4


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _linear_traced(S, st, j, src, x, m):
    rec = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
    st.ctx.trace_begin(rec.data_ptr(), 4, 0)
    _, _, rows, cols = st.entries[j]
    y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(j, src, x.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    n = st.ctx.trace_count()
    st.ctx.trace_begin(0, 0, 0)
    tag = int(rec[0].item()) if n else 0
    return y, (tag >> 48) & 0xFF


def _straddling_rows(entries, n_shards):
    """(entry, row) pairs that a chunk boundary splits, from the oracle's plan."""
    plan = O.plan_layout([(l, r, c, 1) for (l, r, c) in entries], n_shards)
    lay = plan.layers[0]
    out = []
    for j, (_, rows, cols) in enumerate(entries):
        o = lay.offsets[j]
        for i in range(1, n_shards):
            b = i * lay.chunk
            if o < b < o + rows * cols and (b - o) % cols:
                out.append((j, (b - o) // cols))
    return out


def _random_layer(rng, shapes):
    codes, scales = {}, {}
    for j, (_, r, c) in enumerate(shapes):
        q = rng.integers(0, 256, size=(r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C  # no NaN codes
        codes[j] = q
        scales[j] = (2.0 ** rng.uniform(-8, -4, size=(-(-r // 128), -(-c // 128)))).astype(np.float32)
    return LayerData(codes, scales)


# N = 4: C = 1,084,544 B; boundaries split entry 0 at rows 1210 and 2420 and
# entry 1 at row 646; a 256-row block is at most 230 KB, so two chunks at most.
SHAPES = [(0, 4 * 700, 16 * 56), (0, 4 * 333, 16 * 72), (0, 4 * 512, 16 * 9)]


@pytest.mark.parametrize("m", [1, 16, 17, 40, 64])
def test_fused_tc_matches_oracle_with_straddling_rows(S, m):
    rng = np.random.default_rng(500 + m)
    ld = _random_layer(rng, SHAPES)
    st = build_stack(S, SHAPES, 4, [ld])
    assert len(_straddling_rows(SHAPES, 4)) == 3
    for j, (_, r, c) in enumerate(SHAPES):
        x = WL.draw_x(77, j, m, c)
        y, kern = _linear_traced(S, st, j, S.SRC_FUSED, x.cuda(), m)
        assert kern == KERNEL_TC_FUSED
        ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x)), ld.codes[j], ld.scales[j])
        assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} m {m}")
    assert st.ctx.status() == 0


def test_fused_tc_straddling_rows_one_hot(S):
    # One-hot activations pick one weight column: a straddling row's output is
    # the dequantised weight, rounded to fp32 and then to bf16, exactly.
    rng = np.random.default_rng(9)
    ld = _random_layer(rng, SHAPES)
    st = build_stack(S, SHAPES, 4, [ld])
    for j, row in _straddling_rows(SHAPES, 4):
        _, r, c = SHAPES[j]
        m = 8
        cols = rng.integers(0, c, size=m)
        xo = torch.zeros((m, c), dtype=torch.bfloat16)
        xo[np.arange(m), torch.from_numpy(cols)] = 1.0
        y, kern = _linear_traced(S, st, j, S.SRC_FUSED, xo.cuda(), m)
        assert kern == KERNEL_TC_FUSED
        want = O.dequant_at(ld.codes[j], ld.scales[j], [row], cols)[0]
        got = y[:, row].cpu()
        assert torch.equal(got, torch.from_numpy(want).float().to(torch.bfloat16)), f"entry {j} row {row}"


def test_fused_tc_kda_layer_matches_oracle_and_slot(S):
    # The chunk-map launch splits each linear into per-chunk segments (its own
    # split-K partition), so it agrees with the slot launch within rounding.
    w = WL.scaled_workload(WL.ATTN_KDA, rows_div=16, cols_div=16, name="kda_div16")
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    st.ctx.gather_to_slot(0, 0, 0)
    for m in (1, 32):
        for j, (_, r, c) in enumerate(ents):
            x = WL.draw_x(w.key, j, m, c).cuda()
            yf, kf = _linear_traced(S, st, j, S.SRC_FUSED, x, m)
            ys, ks = _linear_traced(S, st, j, S.SRC_SLOT0, x, m)
            assert (kf, ks) == (KERNEL_TC_FUSED, KERNEL_TC)
            ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x.cpu())), layers[0].codes[j], layers[0].scales[j])
            assert_close(bf16_tensor_to_f64(yf), ref, f"entry {j} m {m} (fused)")
            assert_close(bf16_tensor_to_f64(yf), bf16_tensor_to_f64(ys), f"entry {j} m {m} (fused vs slot)")


def test_fused_segments_beyond_the_table_use_the_mma_kernel(S):
    # N = 64 chunks of 1 KB over one 1024 x 64 linear: 64 segments, more than
    # one launch's table holds, so the mma.sync kernel reads the chunk map.
    shapes = [(0, 1024, 64)]
    rng = np.random.default_rng(21)
    ld = _random_layer(rng, shapes)
    st = build_stack(S, shapes, 64, [ld])
    for m in (1, 20):
        x = WL.draw_x(5, 0, m, 64)
        y, kern = _linear_traced(S, st, 0, S.SRC_FUSED, x.cuda(), m)
        assert kern == KERNEL_MMA_FUSED
        ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x)), ld.codes[0], ld.scales[0])
        assert_close(bf16_tensor_to_f64(y), ref, f"m {m}")


def test_fused_tc_many_small_chunks(S):
    # 256-row blocks spanning three and more chunks (C = 64,512 B, rows of
    # 448 B): every unit still reads one chunk.
    w = WL.scaled_workload(WL.STACK92, rows_div=16, cols_div=16, n_layers=1, name="stack1_div16")
    ents = workload_entries(w, 1)
    layers = draw_layers(w, 1)
    st = build_stack(S, ents, w.n_shards, layers)
    for m in (8, 33):
        for j, (_, r, c) in enumerate(ents):
            x = WL.draw_x(w.key, j, m, c)
            y, kern = _linear_traced(S, st, j, S.SRC_FUSED, x.cuda(), m)
            assert kern == KERNEL_TC_FUSED
            ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x)), layers[0].codes[j], layers[0].scales[j])
            assert_close(bf16_tensor_to_f64(y), ref, f"entry {j} m {m}")
