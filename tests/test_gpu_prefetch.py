"""Draft-model first-layer prefetch (blog section "CUDA graph 与 draft 模型"): the
draft model's layer 0 is gathered early on a dedicated stream and its first
run waits for that gather once; without a prefetch (cold start) the gather
runs inline. Outputs of the target and draft contexts against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, build_stack, draw_layers, workload_entries

pytestmark = pytest.mark.gpu

TARGET = WL.scaled_workload(WL.STACK92, rows_div=16, cols_div=16, n_layers=3, name="target3_div16")
DRAFT = WL.scaled_workload(WL.STACK92, rows_div=16, cols_div=16, n_layers=2, name="draft2_div16")


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


@pytest.fixture(scope="module")
def stacks(S):
    out = {}
    for name, w, key in (("target", TARGET, 0), ("draft", DRAFT, 1)):
        ents = workload_entries(w)
        layers = draw_layers(WL.scaled_workload(w, name=f"{w.name}_k{key}"), w.n_layers)
        out[name] = (build_stack(S, ents, w.n_shards, layers), layers)
    return out


def _io(st, n_layers, m, key):
    xs, ys, io = {}, {}, []
    for l in range(n_layers):
        js = st.layer_entries(l)
        xl = [WL.draw_x(key, j, m, st.entries[j][3]).cuda() for j in js]
        yl = [torch.full((m, st.entries[j][2]), float("nan"), dtype=torch.bfloat16, device="cuda") for j in js]
        for j, a, b in zip(js, xl, yl):
            xs[j], ys[j] = a, b
        io.append(([a.data_ptr() for a in xl], [b.data_ptr() for b in yl], m))
    return xs, ys, io


def _check(st, layers, xs, ys, what):
    for j, y in ys.items():
        l = st.entries[j][0]
        want = O.linear(bf16_tensor_to_f64(xs[j].cpu()), layers[l].codes[j], layers[l].scales[j])
        assert_close(bf16_tensor_to_f64(y), want, f"{what} entry {j}")


def test_prefetched_draft_layer_overlaps_target_and_matches_oracle(S, stacks):
    (tst, tl), (dst, dl) = stacks["target"], stacks["draft"]
    m = 8
    txs, tys, tio = _io(tst, 3, m, 11)
    dxs, dys, dio = _io(dst, 2, m, 12)
    main, side, dside, pre = (torch.cuda.Stream() for _ in range(4))
    for step in range(3):  # the prefetch waits for the previous step's reader of the slot
        for y in list(tys.values()) + list(dys.values()):
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        dst.ctx.prefetch_layer(0, 0, pre.cuda_stream)  # dedicated stream, issued first
        tst.ctx.run_layers(0, 2, tio, 0, main.cuda_stream, side.cuda_stream)
        dst.ctx.run_layers(0, 1, dio, S.RUN_FIRST_PREFETCHED, main.cuda_stream, dside.cuda_stream)
        main.synchronize()
        _check(tst, tl, txs, tys, f"target step {step}")
        _check(dst, dl, dxs, dys, f"draft step {step}")
    assert tst.ctx.status() == 0 and dst.ctx.status() == 0


def test_cold_start_gathers_inline(S, stacks):
    dst, dl = stacks["draft"]
    m = 4
    dxs, dys, dio = _io(dst, 2, m, 13)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    dst.ctx.gather_to_slot(1, 0, main.cuda_stream)  # slot 0 holds layer 1, nothing prefetched
    dst.ctx.run_layers(0, 1, dio, S.RUN_FIRST_PREFETCHED, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    _check(dst, dl, dxs, dys, "cold run")
    # wait_prefetch reports the cold start and leaves the layer in the slot
    assert dst.ctx.wait_prefetch(1, 0, main.cuda_stream) is True
    j = dst.layer_entries(1)[0]
    y = torch.empty((m, dst.entries[j][2]), dtype=torch.bfloat16, device="cuda")
    dst.ctx.linear(j, S.SRC_SLOT0, dxs[j].data_ptr(), m, y.data_ptr(), main.cuda_stream)
    main.synchronize()
    assert torch.equal(y, dys[j])


def test_a_later_gather_invalidates_the_prefetch(S, stacks):
    dst, dl = stacks["draft"]
    m = 4
    dxs, dys, dio = _io(dst, 2, m, 14)
    s = torch.cuda.Stream()
    dst.ctx.prefetch_layer(0, 0, s.cuda_stream)
    assert dst.ctx.wait_prefetch(0, 0, s.cuda_stream) is False  # hit, consumed
    assert dst.ctx.wait_prefetch(0, 0, s.cuda_stream) is True   # nothing pending any more
    dst.ctx.prefetch_layer(0, 0, s.cuda_stream)
    dst.ctx.gather_to_slot(1, 0, s.cuda_stream)                  # overwrites slot 0
    assert dst.ctx.wait_prefetch(0, 0, s.cuda_stream) is True    # so layer 0 is gathered again
    for j in dst.layer_entries(0):
        y = torch.empty((m, dst.entries[j][2]), dtype=torch.bfloat16, device="cuda")
        dst.ctx.linear(j, S.SRC_SLOT0, dxs[j].data_ptr(), m, y.data_ptr(), s.cuda_stream)
        s.synchronize()
        want = O.linear(bf16_tensor_to_f64(dxs[j].cpu()), dl[0].codes[j], dl[0].scales[j])
        assert_close(bf16_tensor_to_f64(y), want, f"entry {j}")


def test_prefetch_flag_needs_the_slot_path(S, stacks):
    dst, _ = stacks["draft"]
    _, _, dio = _io(dst, 2, 2, 15)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    with pytest.raises(S.SwsError) as ei:
        dst.ctx.run_layers(0, 1, dio, S.RUN_FIRST_PREFETCHED | S.RUN_FUSED, main.cuda_stream, side.cuda_stream)
    assert ei.value.code == S.E_INVALID
    with pytest.raises(S.SwsError):
        dst.ctx.prefetch_layer(5, 0, main.cuda_stream)
    with pytest.raises(S.SwsError):
        dst.ctx.prefetch_layer(0, 2, main.cuda_stream)
