"""Lookahead scheduler on the GPU: per-layer outputs against the oracle, the
happens-before edges of the oracle's schedule model checked on device
timestamps, at most two layers resident, and the fused (no-slot) mode."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, build_stack, draw_layers, workload_entries

pytestmark = pytest.mark.gpu

STACK = WL.scaled_workload(WL.STACK92, rows_div=16, cols_div=16, n_layers=7, name="stack7_div16")


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


@pytest.fixture(scope="module")
def stack(S):
    ents = workload_entries(STACK)
    layers = draw_layers(STACK)
    st = build_stack(S, ents, STACK.n_shards, layers)
    return st, layers


def _io(st, first, last, m, key=STACK.key):
    xs, ys, io = {}, {}, []
    for l in range(first, last + 1):
        js = st.layer_entries(l)
        xl = [WL.draw_x(key, j, m, st.entries[j][3]).cuda() for j in js]
        yl = [torch.full((m, st.entries[j][2]), float("nan"), dtype=torch.bfloat16, device="cuda") for j in js]
        for j, a, b in zip(js, xl, yl):
            xs[j], ys[j] = a, b
        io.append(([a.data_ptr() for a in xl], [b.data_ptr() for b in yl], m))
    return xs, ys, io


def _records(rec, n):
    r = rec[: 4 * n].view(n, 4).cpu().numpy().astype(np.uint64)
    out = []
    for tag, t0, t1, _ in r:
        kind, layer = int(tag) >> 56, (int(tag) >> 32) & 0xFFFF
        out.append((kind, layer, int(t0), int(t1)))
    return out


@pytest.mark.parametrize("first,last", [(0, 6), (1, 5), (2, 2), (3, 4)])
def test_run_layers_outputs_and_ordering(S, stack, first, last):
    st, layers = stack
    m = 8
    xs, ys, io = _io(st, first, last, m)
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    rec = torch.zeros(4 * 256, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    st.ctx.trace_begin(rec.data_ptr(), 256, main.cuda_stream)
    st.ctx.run_layers(first, last, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    n_rec = st.ctx.trace_count()
    st.ctx.trace_begin(0, 0, 0)
    exposed, layer_ms = st.ctx.run_timing(last - first + 1)
    assert all(v >= 0 for v in exposed + layer_ms)
    assert st.ctx.status() == 0
    # outputs
    for l in range(first, last + 1):
        for j in st.layer_entries(l):
            x = xs[j].cpu()
            ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(x)), layers[l].codes[j], layers[l].scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), ref, f"layer {l} entry {j}")
    # ordering on device timestamps
    recs = _records(rec, n_rec)
    gathers = {l: (t0, t1) for k, l, t0, t1 in recs if k == 1}
    lin = {}
    for k, l, t0, t1 in recs:
        if k == 2:
            a, b = lin.get(l, (t0, t1))
            lin[l] = (min(a, t0), max(b, t1))
    assert sorted(gathers) == list(range(first, last + 1))
    # exactly one gather per layer (the pages' one all-gather per layer)
    assert sum(1 for k, _, _, _ in recs if k == 1) == last - first + 1
    assert sorted(lin) == list(range(first, last + 1))
    for (kb, lb), (ka, la) in O.happens_before(first, last):
        before = gathers[lb] if kb == "gather" else lin[lb]
        after = gathers[la] if ka == "gather" else lin[la]
        assert after[0] >= before[1], f"{kb}({lb}) must end before {ka}({la}) starts"
    # at most two layers hold full weights at any time
    events = []
    for l in range(first, last + 1):
        events += [(gathers[l][0], 1), (lin[l][1], -1)]
    live = peak = 0
    for _, d in sorted(events, key=lambda e: (e[0], e[1])):
        live += d
        peak = max(peak, live)
    assert peak <= O.max_live_layers(first, last) <= 2


def test_fused_mode_matches_slot_mode_bitwise(S, stack):
    # With one kernel (mma.sync) and one split-K partition, reading the weight
    # bytes from the chunks instead of the slot gives identical bits.
    st, layers = stack
    m = 32
    xs, ys, io = _io(st, 0, 6, m)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_MMA)
    try:
        st.ctx.run_layers(0, 6, io, 0, main.cuda_stream, side.cuda_stream)
        main.synchronize()
        ref = {j: y.clone() for j, y in ys.items()}
        for y in ys.values():
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        st.ctx.run_layers(0, 6, io, S.RUN_FUSED, main.cuda_stream, side.cuda_stream)
        main.synchronize()
    finally:
        S.set_option(S.OPT_DECODE_KERNEL, S.DECODE_AUTO)
    for j in ys:
        assert torch.equal(ys[j], ref[j]), f"entry {j}"


def test_fused_mode_matches_slot_mode_default_kernels(S, stack):
    # The default (tcgen05) launches: the chunk-map one splits each linear into
    # per-chunk segments, so the two agree within rounding, and both meet the
    # oracle's bar.
    st, layers = stack
    m = 32
    xs, ys, io = _io(st, 0, 6, m)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, 6, io, 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    ref = {j: y.clone() for j, y in ys.items()}
    st.ctx.run_layers(0, 6, io, S.RUN_FUSED, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    for j in ys:
        assert_close(bf16_tensor_to_f64(ys[j]), bf16_tensor_to_f64(ref[j]), f"entry {j} fused vs slot")
        l = st.entries[j][0]
        want = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[l].codes[j], layers[l].scales[j])
        assert_close(bf16_tensor_to_f64(ys[j]), want, f"entry {j} fused vs oracle")


def test_run_layers_repeated_calls_reuse_slots(S, stack):
    st, layers = stack
    m = 1
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    for first, last in [(0, 3), (4, 6), (0, 6), (5, 6)]:
        xs, ys, io = _io(st, first, last, m)
        st.ctx.run_layers(first, last, io, 0, main.cuda_stream, side.cuda_stream)
        main.synchronize()
        for l in range(first, last + 1):
            for j in st.layer_entries(l):
                ref = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[l].codes[j], layers[l].scales[j])
                assert_close(bf16_tensor_to_f64(ys[j]), ref, f"({first},{last}) layer {l} entry {j}")


def test_run_layers_rejects_bad_ranges(S, stack):
    st, _ = stack
    with pytest.raises(S.SwsError):
        st.ctx.run_layers(0, 7, [([], [], 1)] * 8, 0, 0, torch.cuda.Stream().cuda_stream)
    with pytest.raises(S.SwsError):
        s = torch.cuda.Stream().cuda_stream
        st.ctx.run_layers(0, 0, [([0, 0], [0, 0], 1)], 0, s, s)


@pytest.mark.parametrize("m", [8, 40])
def test_run_layers_captures_into_a_cuda_graph(S, stack, m):
    # The lookahead schedule (gathers on the side stream, event waits, the
    # programmatic dependent launches of the decode linears) records into one
    # CUDA graph; replaying it gives the eager run's bits, and replays with new
    # activations in the same buffers give their results.
    st, layers = stack
    xs, ys, io = _io(st, 0, 6, m)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, 6, io, 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    ref = {j: y.clone() for j, y in ys.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        with pytest.raises(S.SwsError):  # timing events cannot be captured
            st.ctx.run_layers(0, 6, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
        st.ctx.run_layers(0, 6, io, 0, main.cuda_stream, side.cuda_stream)
    for y in ys.values():
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for j in ys:
        assert torch.equal(ys[j], ref[j]), f"entry {j}: graph replay differs from the eager run"
    for x in xs.values():  # new inputs, same buffers
        x.copy_(torch.flip(x, dims=[1]))
    g.replay()
    torch.cuda.synchronize()
    for l in range(0, 7):
        for j in st.layer_entries(l):
            want = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[l].codes[j], layers[l].scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), want, f"replay 2, layer {l} entry {j}")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("flags", [0, "fused"])
def test_library_graph_keeps_the_eager_results(S, stack, flags):
    # sws_graph_capture records the same run (instantiated with per-node
    # priorities): a launch gives the eager run's bits, a second launch on new
    # activations in the same buffers gives their results; bad arguments are
    # refused before anything is captured.
    st, layers = stack
    fl = S.RUN_FUSED if flags == "fused" else 0
    m = 8
    xs, ys, io = _io(st, 0, 6, m)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, 6, io, fl, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    ref = {j: y.clone() for j, y in ys.items()}
    for bad in (S.RUN_TIMING, S.RUN_FIRST_PREFETCHED):
        with pytest.raises(S.SwsError) as ei:
            st.ctx.graph_capture(0, 6, io, bad, main.cuda_stream, side.cuda_stream)
        assert ei.value.code == S.E_INVALID
    with pytest.raises(S.SwsError) as ei:  # the legacy default stream cannot capture
        st.ctx.graph_capture(0, 6, io, fl, 0, side.cuda_stream)
    assert ei.value.code == S.E_INVALID
    with pytest.raises(S.SwsError):  # a bad range is refused, and main is left usable
        st.ctx.graph_capture(0, 9, io, fl, main.cuda_stream, side.cuda_stream)
    g = st.ctx.graph_capture(0, 6, io, fl, main.cuda_stream, side.cuda_stream)
    try:
        for y in ys.values():
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        g.launch(main.cuda_stream)
        main.synchronize()
        for j in ys:
            assert torch.equal(ys[j], ref[j]), f"entry {j}: graph launch differs from the eager run"
        for x in xs.values():  # new inputs, same buffers
            x.copy_(torch.flip(x, dims=[1]))
        torch.cuda.synchronize()
        g.launch(main.cuda_stream)
        main.synchronize()
        for l in range(0, 7):
            for j in st.layer_entries(l):
                want = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[l].codes[j], layers[l].scales[j])
                assert_close(bf16_tensor_to_f64(ys[j]), want, f"launch 2, layer {l} entry {j}")
    finally:
        g.close()
    if not fl:  # after a capture the slots' layers are unknown to the host: an eager slot read is refused
        j0 = st.layer_entries(6)[0]
        with pytest.raises(S.SwsError) as ei:
            st.ctx.linear(j0, S.SRC_SLOT0, xs[j0].data_ptr(), m, ys[j0].data_ptr(), 0)
        assert ei.value.code == S.E_STATE
    st.ctx.run_layers(0, 6, io, fl, main.cuda_stream, side.cuda_stream)  # eager still works afterwards
    main.synchronize()
    assert st.ctx.status() == 0


def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(S, stack):
    # Failure detection without a fault: a kernel waits (the library's bounded
    # wait) on a barrier nothing arrives at, gives up after 2 ms and records
    # SWS_E_TIMEOUT; the host reads it and the next launches run normally.
    st, layers = stack
    assert st.ctx.status(clear=True) == 0
    st.ctx.test_bounded_wait(2_000_000)
    assert st.ctx.status(clear=True) == S.E_TIMEOUT
    assert st.ctx.status() == 0
    m = 4
    xs, ys, io = _io(st, 2, 2, m)
    st.ctx.gather_to_slot(2, 0, 0)
    for j in st.layer_entries(2):
        st.ctx.linear(j, S.SRC_SLOT0, xs[j].data_ptr(), m, ys[j].data_ptr(), 0)
    torch.cuda.synchronize()
    for j in st.layer_entries(2):
        want = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[2].codes[j], layers[2].scales[j])
        assert_close(bf16_tensor_to_f64(ys[j]), want, f"entry {j} after the timeout")
    assert st.ctx.status() == 0


def test_host_waits_give_up_at_their_deadline(S, stack):
    # A kernel that stands for 100 ms (the bounded wait, on a barrier nothing
    # arrives at) is queued ahead of the work a host wait needs. With a 10 ms
    # host limit, sws_run_timing and sws_ctx_status return SWS_E_TIMEOUT saying
    # that the host wait ran out; once the kernel has returned both succeed and
    # the run's outputs match the oracle.
    st, layers = stack
    assert st.ctx.status(clear=True) == 0
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    m = 4
    xs, ys, io = _io(st, 1, 2, m)
    try:
        S.set_option(S.OPT_HOST_WAIT_MS, 10)
        st.ctx.test_bounded_wait(100_000_000, main.cuda_stream)
        st.ctx.run_layers(1, 2, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
        with pytest.raises(S.SwsError) as ei:
            st.ctx.run_timing(2)
        assert ei.value.code == S.E_TIMEOUT and "host wait" in str(ei.value)
        with pytest.raises(S.SwsError) as ei:
            st.ctx.status()
        assert ei.value.code == S.E_TIMEOUT and "host wait" in str(ei.value)
    finally:
        S.set_option(S.OPT_HOST_WAIT_MS, 10000)
    exposed, layer_ms = st.ctx.run_timing(2)
    assert all(t > 0 for t in layer_ms) and exposed[0] >= 0
    assert st.ctx.status(clear=True) == S.E_TIMEOUT  # the bounded wait's own record
    assert st.ctx.status() == 0
    main.synchronize()
    for l in (1, 2):
        for j in st.layer_entries(l):
            want = O.linear(WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu())), layers[l].codes[j], layers[l].scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), want, f"layer {l} entry {j}")


def test_prefill_layers_record_into_a_cuda_graph(S):
    # m > 64: each layer's linears quantise their activations on the
    # context's own stream, forked from and joined into `main`; that fork and
    # join record into the graph as well.
    w = WL.scaled_workload(WL.ATTN_KDA, rows_div=8, cols_div=8, n_layers=2, name="kda2_div8")
    ents = workload_entries(w)
    layers = draw_layers(w)
    m = 130
    st = build_stack(S, ents, w.n_shards, layers, max_m=m)
    xs, ys, io = _io(st, 0, 1, m, key=w.key)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    st.ctx.run_layers(0, 1, io, 0, main.cuda_stream, side.cuda_stream)
    main.synchronize()
    ref = {j: y.clone() for j, y in ys.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        st.ctx.run_layers(0, 1, io, 0, main.cuda_stream, side.cuda_stream)
    for y in ys.values():
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for j in ys:
        assert torch.equal(ys[j], ref[j]), f"entry {j}: graph replay differs from the eager run"
    for l in range(2):
        for j in st.layer_entries(l):
            xf = WL.bf16_to_f64(WL.bf16_bits(xs[j].cpu()))
            xq, ex = O.quantize_x(xf)
            want = O.dequant_x(xq, ex) @ O.dequant(layers[l].codes[j], layers[l].scales[j]).T
            assert_close(bf16_tensor_to_f64(ys[j]), want, f"layer {l} entry {j}")
    assert st.ctx.status() == 0
