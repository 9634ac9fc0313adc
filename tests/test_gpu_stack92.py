"""The 92-layer decode stack at full size (about 24 GB of resident chunks,
N = 16, M = 32): the lookahead run (sws_run_layers) over all 92 layers, its
outputs for layers 0, 1, 45 and 91 on sampled weight rows against the
oracle, and every layer's gather against the concatenation of its chunks
(the gather is a byte copy, so this holds at any size). Layers are the
workload's two base layers with per-row sign flips, built on the device the
way the benchmark builds them; the oracle derives the sampled rows from the
same bases and signs on the host."""
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


def test_stack92_lookahead_full_size(S):
    from sharded_weight_storage_gb300.storage import ShardedStack
    w = WL.STACK92
    n, ne, L, m = w.n_shards, len(w.entries), w.n_layers, 32
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * (1 << 30):
        pytest.skip("needs about 30 GB of free device memory")
    bases = [WL.base_layer(w, b) for b in range(w.n_base)]
    base_dev = [[torch.from_numpy(c).cuda() for c in b.codes] for b in bases]
    base_sc = [[torch.from_numpy(s).cuda() for s in b.scales] for b in bases]
    ents = [(l, S.E4M3, e.rows, e.cols) for l in range(L) for e in w.entries]
    st = ShardedStack(ents, n, max_m=64)
    for l in range(L):
        b = l % w.n_base
        codes, scales = {}, {}
        for j, e in enumerate(w.entries):
            signs = torch.from_numpy(WL.draw_row_signs(w.key, l, j, e.rows)).cuda()
            codes[l * ne + j] = WL.apply_row_signs(base_dev[b][j], signs)
            scales[l * ne + j] = base_sc[b][j]
        st.load_layer(l, codes, scales)
    del base_dev, codes
    st.make_ctx()
    checked = (0, 1, 45, 91)
    xs = [WL.draw_x(w.key, j, m, e.cols).cuda() for j, e in enumerate(w.entries)]
    scratch = [torch.empty((m, e.rows), dtype=torch.bfloat16, device="cuda") for e in w.entries]
    ys = {l: [torch.full((m, e.rows), float("nan"), dtype=torch.bfloat16, device="cuda") for e in w.entries]
          for l in checked}
    io = [([x.data_ptr() for x in xs], [y.data_ptr() for y in ys.get(l, scratch)], m) for l in range(L)]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, L - 1, io, 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    assert st.ctx.status() == 0
    rng = np.random.default_rng(92)
    for l in checked:
        base = bases[l % w.n_base]
        for j, e in enumerate(w.entries):
            rows = np.unique(np.concatenate([[0, e.rows - 1], rng.choice(e.rows, size=38, replace=False)]))
            # layer l's codes: the base layer's with each row's sign bit flipped by its draw
            codes = base.codes[j] ^ WL.draw_row_signs(w.key, l, j, e.rows)[:, None]
            want = O.linear_rows(x_f64(xs[j]), codes, base.scales[j], rows)
            assert_close(bf16_tensor_to_f64(ys[l][j])[:, rows], want, f"layer {l} {e.name}")
    # every layer's slot is the concatenation of its chunks, byte for byte
    for l in range(L):
        st.ctx.gather_to_slot(l, l & 1, 0)
        torch.cuda.synchronize()
        t = torch.cat([c for c in st.chunks[l]])
        assert torch.equal(st.slots[l & 1][:t.numel()], t), f"layer {l}"
    assert st.ctx.status() == 0
