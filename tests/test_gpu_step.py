"""Decode steps back to back on one stream: each step gathers a layer into
slot 0 and runs that layer's decode linears from it, two layers alternating,
with no host synchronisation in between. The decode GEMM lets the kernels
after it launch once every CTA has read all its weights, so the next step's
gather overwrites the slot while the GEMM's last CTAs and the settle grid
still run; every step's outputs must still be its own layer's: bit for bit
the outputs of the same linears run alone, and within the tolerance of the
oracle on sampled rows."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, build_stack, draw_layers, workload_entries

pytestmark = pytest.mark.gpu

W = WL.STACK92  # shared-expert layers (gate_up [24576, 7168], down [7168, 12288]), N = 16


@pytest.fixture(scope="module")
def stack(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ents = workload_entries(W, 2)
    layers = draw_layers(W, 2)  # two base layers: different weights
    st = build_stack(swslib, ents, W.n_shards, layers)
    return swslib, st, layers


@pytest.mark.parametrize("m", [1, 32, 64])
def test_back_to_back_steps_share_one_slot(stack, m):
    S, st, layers = stack
    ne = len(W.entries)
    xs = [WL.draw_x(W.key, j, m, e.cols) for j, e in enumerate(W.entries)]
    xd = [x.cuda() for x in xs]
    s = torch.cuda.current_stream().cuda_stream

    def outputs():
        return [torch.full((m, e.rows), float("nan"), dtype=torch.bfloat16, device="cuda") for e in W.entries]

    # each layer's linears alone, the slot gathered and the device idle before and after
    alone = []
    for l in range(2):
        ys = outputs()
        st.ctx.gather_to_slot(l, 0, s)
        torch.cuda.synchronize()
        st.ctx.layer_linears(l, S.SRC_SLOT0, [x.data_ptr() for x in xd], [y.data_ptr() for y in ys], m, s)
        torch.cuda.synchronize()
        alone.append([y.cpu() for y in ys])
    steps = 8
    ys = [outputs() for _ in range(steps)]
    for k in range(steps):
        l = k % 2
        st.ctx.gather_to_slot(l, 0, s)
        st.ctx.layer_linears(l, S.SRC_SLOT0, [x.data_ptr() for x in xd], [y.data_ptr() for y in ys[k]], m, s)
    torch.cuda.synchronize()
    assert st.ctx.status() == 0
    for k in range(steps):
        for j in range(ne):
            assert torch.equal(ys[k][j].cpu().view(torch.int16), alone[k % 2][j].view(torch.int16)), \
                f"step {k} entry {j} m {m}: differs from the same linears run alone"
    rng = np.random.default_rng(100 + m)
    for j, e in enumerate(W.entries):
        xf = WL.bf16_to_f64(WL.bf16_bits(xs[j]))
        sel = np.unique(np.concatenate([[0, e.rows - 1], rng.choice(e.rows, 256, replace=False)]))
        for l in range(2):
            ref = O.linear_rows(xf, layers[l].codes[l * ne + j], layers[l].scales[l * ne + j], sel)
            assert_close(bf16_tensor_to_f64(alone[l][j])[:, sel], ref, f"layer {l} entry {j} m {m}")
