"""The prefill workload at full size: the lookahead run (sws_run_layers) over
all eight KDA-like layers (N = 8) at both token counts the benchmark times,
m = 2048 and 8192, with the gather of layer l+1 overlapping layer l's FP8
prefill GEMMs (weight-sharding blog, section "提前一层：lookahead 与
ping-pong slot"). Every linear of every layer is checked against the oracle on
sampled token rows and sampled weight rows (the oracle quantises the sampled
token rows - its per-row rule makes that exact - and dequantises the sampled
weight rows only), and every layer's gather against the concatenation of its
chunks. Layers are the workload's base layer with per-row sign flips, built on
the device the way the benchmark builds them; the oracle derives the sampled
rows from the same base and signs on the host."""
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


@pytest.fixture(scope="module")
def stack(S):
    from sharded_weight_storage_gb300.storage import ShardedStack
    w = WL.PREFILL
    n, ne, L = w.n_shards, len(w.entries), w.n_layers
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * (1 << 30):
        pytest.skip("needs about 25 GB of free device memory")
    base = WL.base_layer(w, 0)
    base_dev = [torch.from_numpy(c).cuda() for c in base.codes]
    base_sc = [torch.from_numpy(s).cuda() for s in base.scales]
    st = ShardedStack([(l, S.E4M3, e.rows, e.cols) for l in range(L) for e in w.entries], n, max_m=max(w.m_values))
    for l in range(L):
        codes, scales = {}, {}
        for j, e in enumerate(w.entries):
            signs = torch.from_numpy(WL.draw_row_signs(w.key, l, j, e.rows)).cuda()
            codes[l * ne + j] = WL.apply_row_signs(base_dev[j], signs)
            scales[l * ne + j] = base_sc[j]
        st.load_layer(l, codes, scales)
    del base_dev, codes
    st.make_ctx()
    yield st, base
    st.ctx.close()
    del st
    torch.cuda.empty_cache()


@pytest.mark.parametrize("m", [2048, 8192])
def test_prefill_lookahead_over_eight_full_size_layers(S, stack, m):
    st, base = stack
    w = WL.PREFILL
    ne, L = len(w.entries), w.n_layers
    # one activation per linear, shared by the layers (the pages chain no
    # activations between linears); one output buffer per linear and layer
    xs = [WL.draw_x(w.key, j, m, e.cols) for j, e in enumerate(w.entries)]
    xd = [x.cuda() for x in xs]
    ys = [[torch.full((m, e.rows), float("nan"), dtype=torch.bfloat16, device="cuda") for e in w.entries]
          for _ in range(L)]
    io = [([x.data_ptr() for x in xd], [y.data_ptr() for y in ys[l]], m) for l in range(L)]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, L - 1, io, 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    assert st.ctx.status() == 0
    rng = np.random.default_rng(5000 + m)
    tok = np.unique(np.concatenate([[0, m - 1], rng.choice(m, size=30, replace=False)]))
    # the oracle's quantised activations of the sampled token rows (per-row rule)
    xdq = [O.dequant_x(*O.quantize_x(x_f64(x)[tok])) for x in xs]
    for l in range(L):
        for j, e in enumerate(w.entries):
            rows = np.unique(np.concatenate([[0, e.rows - 1], rng.choice(e.rows, size=190, replace=False)]))
            codes = base.codes[j] ^ WL.draw_row_signs(w.key, l, j, e.rows)[:, None]
            want = O.linear_rows(xdq[j], codes, base.scales[j], rows)
            got = bf16_tensor_to_f64(ys[l][j][torch.from_numpy(tok).cuda()])[:, rows]
            assert_close(got, want, f"m {m} layer {l} {e.name}")
    # every layer's gather is the concatenation of its chunks, byte for byte
    for l in range(L):
        st.ctx.gather_to_slot(l, l & 1, 0)
        torch.cuda.synchronize()
        t = torch.cat([c for c in st.chunks[l]])
        assert torch.equal(st.slots[l & 1][:t.numel()], t), f"layer {l}"
    assert st.ctx.status() == 0
