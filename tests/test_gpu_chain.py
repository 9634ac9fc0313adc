"""The shared-expert chain (gate_up -> SiLU(gate) * up -> down, bf16 tensors in
between) and the copy-engine gather, against the CPU oracle. Each stage of the
chain is checked on the GPU's own input to that stage, and the whole chain
against the oracle's chain with bf16 rounding at the same two boundaries."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, bf16_tensor_to_f64, build_stack, draw_layers, oracle_layer_T, workload_entries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _bf16_gu(rng, m, f, scale=2.0):
    return torch.from_numpy((rng.standard_normal((m, 2 * f)) * scale).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("m,f", [(1, 8), (33, 1000), (300, 12288), (7, 24)])
def test_silu_mul_matches_oracle(S, m, f):
    rng = np.random.default_rng(m * 7 + f)
    gu = _bf16_gu(rng, m, f)
    gu[0, 0] = 0.0  # silu(0) * u = 0 exactly
    act = torch.full((m, f), float("nan"), dtype=torch.bfloat16, device="cuda")
    S.silu_mul(gu.cuda().data_ptr(), m, f, act.data_ptr())
    torch.cuda.synchronize()
    ref = O.silu_mul(bf16_tensor_to_f64(gu))
    got = bf16_tensor_to_f64(act)
    # fp32 arithmetic then one rounding to bf16: within one bf16 spacing of the
    # exact value, and equal to its correctly rounded value almost everywhere
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -133)
    assert np.mean(got == O.bf16_round(ref)) > 0.99
    assert got[0, 0] == 0.0


def test_silu_mul_extremes(S):
    vals = torch.tensor([[-100.0, -20.0, 0.0, 20.0, 100.0, 1e-30, -1e-30, 3.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0]],
                        dtype=torch.bfloat16)  # g: 8 values, u: 8 ones
    act = torch.empty((1, 8), dtype=torch.bfloat16, device="cuda")
    S.silu_mul(vals.cuda().data_ptr(), 1, 8, act.data_ptr())
    torch.cuda.synchronize()
    got = bf16_tensor_to_f64(act)[0]
    ref = O.silu_mul(bf16_tensor_to_f64(vals))[0]
    assert got[2] == 0.0 and abs(got[0]) < 1e-40 and got[4] == O.bf16_round(np.array([100.0]))[0]
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -133)


SE = WL.scaled_workload(WL.SHARED_EXPERT, rows_div=8, cols_div=8, name="shared_expert_div8")


@pytest.mark.parametrize("m", [1, 32, 200])
@pytest.mark.parametrize("src_name", ["slot", "fused"])
def test_shared_expert_chain(S, m, src_name):
    if src_name == "fused" and m > 64:
        pytest.skip("chunk-map reads are for decode sizes")
    ents = workload_entries(SE, 1)
    (_, r_gu, c_gu), (_, r_dn, c_dn) = ents
    f = r_gu // 2
    assert c_dn == f
    layers = draw_layers(SE, 1)
    st = build_stack(S, ents, SE.n_shards, layers, max_m=max(m, 64))
    st.ctx.gather_to_slot(0, 0, 0)
    src = S.SRC_SLOT0 if src_name == "slot" else S.SRC_FUSED
    x = WL.draw_x(SE.key, 0, m, c_gu).cuda()
    gu = torch.empty((m, r_gu), dtype=torch.bfloat16, device="cuda")
    act = torch.empty((m, f), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((m, r_dn), dtype=torch.bfloat16, device="cuda")
    st.ctx.linear(0, src, x.data_ptr(), m, gu.data_ptr(), 0)
    S.silu_mul(gu.data_ptr(), m, f, act.data_ptr(), 0)
    st.ctx.linear(1, src, act.data_ptr(), m, y.data_ptr(), 0)
    torch.cuda.synchronize()
    lay = layers[0]

    def lin(xf, j):
        if m > 64:
            xq, ex = O.quantize_x(xf)
            return O.dequant_x(xq, ex) @ O.dequant(lay.codes[j], lay.scales[j]).T
        return O.linear(xf, lay.codes[j], lay.scales[j])

    xf = bf16_tensor_to_f64(x)
    # stage by stage, each on the GPU's own input
    assert_close(bf16_tensor_to_f64(gu), lin(xf, 0), "gate_up")
    a_ref = O.silu_mul(bf16_tensor_to_f64(gu))
    assert np.all(np.abs(bf16_tensor_to_f64(act) - a_ref) <= 2.0 ** -7 * np.abs(a_ref) + 2.0 ** -133)
    assert_close(bf16_tensor_to_f64(y), lin(bf16_tensor_to_f64(act), 1), "down")
    # the whole chain against the oracle's chain
    chain = lin(O.bf16_round(O.silu_mul(O.bf16_round(lin(xf, 0)))), 1)
    assert_close(bf16_tensor_to_f64(y), chain, "chain")
    assert st.ctx.status() == 0


@pytest.mark.parametrize("wname", ["kda_div8", "tiny"])
@pytest.mark.parametrize("engine", ["copy_engine", "tma_shared_sm"])
def test_other_gather_engines_match_oracle_and_kernel(S, engine, wname):
    # The copy-engine gather and the shared-SM TMA kernel (one 48 KB CTA per
    # SM, 16 KB tiles: a different tile split of the same chunks) against the
    # oracle's T and the default kernel, byte for byte. kda_div8's chunks are
    # 21 whole 16 KB tiles (10.5 of the default's 32 KB); the tiny layer's
    # 90,112-byte chunks end in a partial tile for both shapes.
    eng = S.GATHER_COPY_ENGINE if engine == "copy_engine" else S.GATHER_TMA_SHARED_SM
    w = WL.scaled_workload(WL.ATTN_KDA, rows_div=8, cols_div=8, name="kda_div8") if wname == "kda_div8" \
        else WL.scaled_workload(WL.TINY, n_layers=2)
    ents = workload_entries(w, 2)
    layers = draw_layers(w, 2)
    st = build_stack(S, ents, w.n_shards, layers)
    try:
        for l in range(2):
            _, _, t_ref = oracle_layer_T(ents, w.n_shards, l, layers[l])
            S.set_option(S.OPT_GATHER_ENGINE, eng)
            st.slots[1].fill_(0xAB)
            st.ctx.gather_to_slot(l, 1, 0)
            torch.cuda.synchronize()
            ce = st.slots[1][:t_ref.size].cpu().numpy()
            S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)
            st.slots[0].fill_(0xCD)
            st.ctx.gather_to_slot(l, 0, 0)
            torch.cuda.synchronize()
            tma = st.slots[0][:t_ref.size].cpu().numpy()
            assert np.array_equal(ce, t_ref) and np.array_equal(tma, t_ref), f"layer {l}"
    finally:
        S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)


@pytest.mark.parametrize("engine", ["copy_engine", "tma_shared_sm"])
def test_run_layers_with_other_gather_engines(S, engine):
    w = WL.scaled_workload(WL.STACK92, rows_div=16, cols_div=16, n_layers=5, name="stack5_div16")
    ents = workload_entries(w)
    layers = draw_layers(w)
    st = build_stack(S, ents, w.n_shards, layers)
    m = 8
    xs, ys, io = {}, {}, []
    for l in range(5):
        js = st.layer_entries(l)
        xl = [WL.draw_x(w.key, j, m, st.entries[j][3]).cuda() for j in js]
        yl = [torch.full((m, st.entries[j][2]), float("nan"), dtype=torch.bfloat16, device="cuda") for j in js]
        for j, a, b in zip(js, xl, yl):
            xs[j], ys[j] = a, b
        io.append(([a.data_ptr() for a in xl], [b.data_ptr() for b in yl], m))
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    eng = S.GATHER_COPY_ENGINE if engine == "copy_engine" else S.GATHER_TMA_SHARED_SM
    try:
        S.set_option(S.OPT_GATHER_ENGINE, eng)
        st.ctx.run_layers(0, 4, io, 0, main.cuda_stream, side.cuda_stream)
        main.synchronize()
        if engine == "tma_shared_sm":
            # captured and replayed: the same outputs, bit for bit
            first = {j: y.clone() for j, y in ys.items()}
            for y in ys.values():
                y.fill_(float("nan"))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                st.ctx.run_layers(0, 4, io, 0, main.cuda_stream, side.cuda_stream)
            with torch.cuda.stream(main):
                g.replay()
            main.synchronize()
            for j in ys:
                assert torch.equal(ys[j], first[j]), f"entry {j}: graph replay differs"
    finally:
        S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)
    for l in range(5):
        for j in st.layer_entries(l):
            want = O.linear(bf16_tensor_to_f64(xs[j].cpu()), layers[l].codes[j], layers[l].scales[j])
            assert_close(bf16_tensor_to_f64(ys[j]), want, f"layer {l} entry {j}")
    assert st.ctx.status() == 0
