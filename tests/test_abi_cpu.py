"""The C ABI without a GPU: every symbol the header declares is exported, the
planner agrees with the oracle, and bad arguments give the documented codes."""
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as WL
from conftest import ROOT


def _header_functions():
    src = open(os.path.join(ROOT, "include", "sws.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sws_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(swslib):
    lib = swslib.lib()
    names = _header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    from sharded_weight_storage_gb300 import _lib
    assert sorted(_lib.EXPORTED) == names


def test_version(swslib):
    assert swslib.lib().sws_version() >= 100


def _compare_plan(S, ents, n):
    plan = S.Plan([(l, S.E4M3 if eb == 1 else {2: S.BF16, 4: S.F32}[eb], r, c) for (l, r, c, eb) in ents], n)
    ref = O.plan_layout(ents, n)
    n_layers, n_shards, n_entries = plan.info()
    assert n_shards == n and n_entries == len(ents)
    assert n_layers == (max(e[0] for e in ents) + 1 if ents else 0)
    for l in range(n_layers):
        total, chunk, ne = plan.layer(l)
        ly = ref.layers.get(l)
        if ly is None:
            assert total == 0 and chunk == 0 and ne == 0
            continue
        assert (total, chunk) == (ly.total, ly.chunk)
        assert ne == sum(1 for e in ents if e[0] == l)
    for j in range(len(ents)):
        off, nb, sh = plan.entry(j)
        assert sh == ref.sharded[j]
        assert nb == ents[j][1] * ents[j][2] * ents[j][3]
        if sh:
            assert off == ref.layers[ents[j][0]].offsets[j]
        else:
            assert off == -1
    assert plan.slot_bytes == ref.slot_bytes


@pytest.mark.parametrize("w", [WL.TINY, WL.SHARED_EXPERT, WL.ATTN_KDA, WL.PREFILL], ids=lambda w: w.name)
def test_planner_matches_oracle_on_workloads(swslib, w):
    _compare_plan(swslib, [(0, e.rows, e.cols, 1) for e in w.entries], w.n_shards)


def test_planner_matches_hand_derived_padded_layouts(swslib):
    # tests/golden/layout_padding.txt: per-entry and tail padding both non-zero,
    # replicated entries left out of T
    from test_oracle_pins import read_padding_golden
    S = swslib
    dt = {1: S.E4M3, 2: S.BF16, 4: S.F32}
    for n, ents, total, chunk in read_padding_golden().values():
        with pytest.warns(RuntimeWarning):
            plan = S.Plan([(0, dt[e], r, c) for (_, r, c, e, _) in ents], n)
        assert plan.layer(0) == (total, chunk, len(ents))
        assert plan.slot_bytes == total
        for j, (_, r, c, e, off) in enumerate(ents):
            assert plan.entry(j) == (off, r * c * e, off >= 0)
        _compare_plan(S, [(0, r, c, e) for (_, r, c, e, _) in ents], n)


def test_planner_with_scales_in_t_matches_hand_derived_layouts(swslib):
    # tests/golden/layout_scales_in_t.txt: every sharded E4M3 entry followed by
    # its block-scale tensor, 16-byte padded; replicated and non-E4M3 entries
    # have none
    from test_oracle_pins import read_scales_golden
    S = swslib
    for n, ents, total, chunk in read_scales_golden().values():
        dts = [S.E4M3 if s else {1: S.U8, 2: S.BF16, 4: S.F32}[e] for (_, _, _, e, s, _, _) in ents]
        import warnings
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            plan = S.Plan([(0, dt, r, c) for dt, (_, r, c, _, _, _, _) in zip(dts, ents)], n, S.SCALES_IN_T)
        assert plan.layer(0) == (total, chunk, len(ents))
        for j, (_, r, c, e, s, off, soff) in enumerate(ents):
            assert plan.entry(j)[0] == off
            assert plan.scales(j) == ((soff, 4 * (-(-r // 128)) * (-(-c // 128))) if soff >= 0 else (-1, 0))
        plain = S.Plan([(0, dt, r, c) for dt, (_, r, c, _, _, _, _) in zip(dts, ents)], n) \
            if all(r % n == 0 for (_, r, _, _, _, _, _) in ents) else None
        if plain is not None:
            assert all(plain.scales(j) == (-1, 0) for j in range(len(ents)))


@pytest.mark.parametrize("n", [1, 3, 8, 16])
def test_planner_with_scales_in_t_matches_oracle_random(swslib, n):
    S = swslib
    rng = np.random.default_rng(2000 + n)
    import warnings
    for _ in range(25):
        ents = []
        for _ in range(int(rng.integers(1, 9))):
            rows = int(rng.integers(0, 6)) * n * 64 if rng.random() < 0.75 else int(rng.integers(1, 500))
            dt = int(rng.choice([S.E4M3, S.E4M3, S.BF16, S.F32]))
            ents.append((int(rng.integers(0, 3)), dt, rows, int(rng.integers(0, 700))))
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            plan = S.Plan(ents, n, S.SCALES_IN_T)
        eb = {S.E4M3: 1, S.BF16: 2, S.F32: 4}
        ref = O.plan_layout([(l, r, c, eb[dt], dt == S.E4M3) for (l, dt, r, c) in ents], n, scales_in_t=True)
        for l in range(plan.info()[0]):
            ly = ref.layers.get(l)
            assert plan.layer(l)[:2] == ((ly.total, ly.chunk) if ly else (0, 0))
        for j, (l, dt, r, c) in enumerate(ents):
            ly = ref.layers[l]
            assert plan.entry(j)[0] == ly.offsets.get(j, -1)
            assert plan.scales(j) == (ly.scale_offsets.get(j, -1), ly.scale_sizes.get(j, 0))
        assert plan.slot_bytes == ref.slot_bytes


def test_relayout_scales_validates_before_any_launch(swslib):
    S = swslib
    plan = S.Plan([(0, S.E4M3, 8, 16)], 4, S.SCALES_IN_T)
    assert plan.scales(0) == (128, 4)
    assert plan.layer(0) == (192, 48, 1)
    with pytest.raises(S.SwsError) as ei:
        S.relayout_scales(plan, 0, [0], [16, 32, 48, 64])
    assert ei.value.code == S.E_INVALID  # the entry's scales are missing
    with pytest.raises(S.SwsError) as ei:
        S.relayout_scales(plan, 0, [4096], [17, 32, 48, 64])
    assert ei.value.code == S.E_ALIGN
    S.relayout_scales(S.Plan([(0, S.E4M3, 8, 16)], 4), 0, [4096], [16, 32, 48, 64])  # no flag: nothing to do


def test_workspace_grows_by_the_scale_staging_area(swslib):
    S = swslib
    ents = [(0, S.E4M3, 1024, 4096), (0, S.E4M3, 512, 1024), (1, S.E4M3, 256, 256)]
    a = S.workspace_bytes(S.Plan(ents, 4), 64)
    b = S.workspace_bytes(S.Plan(ents, 4, S.SCALES_IN_T), 64)
    # the larger layer's scales, each padded to 16 B: 8*32*4 = 1024 and 4*8*4 = 128, rounded to 256
    assert b - a == 1280


def test_planner_matches_oracle_on_92_layer_stack(swslib):
    w = WL.STACK92
    _compare_plan(swslib, [(l, e.rows, e.cols, 1) for l in range(w.n_layers) for e in w.entries], w.n_shards)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 16, 256])
def test_planner_matches_oracle_random(swslib, n):
    rng = np.random.default_rng(1000 + n)
    import warnings
    for _ in range(25):
        ents = []
        for _ in range(int(rng.integers(1, 9))):
            rows = int(rng.integers(0, 6)) * n if rng.random() < 0.75 else int(rng.integers(1, 50))
            ents.append((int(rng.integers(0, 4)), rows, int(rng.integers(0, 90)), int(rng.choice([1, 2, 4]))))
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            _compare_plan(swslib, ents, n)


def test_skipped_entries_warn_and_stay_out_of_T(swslib):
    S = swslib
    with pytest.warns(RuntimeWarning):
        plan = S.Plan([(0, S.E4M3, 6, 16), (0, S.E4M3, 8, 16)], 4)
    assert plan.status == S.W_SKIPPED
    assert plan.entry(0) == (-1, 96, False)
    assert plan.entry(1) == (0, 128, True)
    assert plan.layer(0) == (128, 32, 2)


@pytest.mark.parametrize("bad", [
    dict(n=0), dict(n=257), dict(rows=-1), dict(cols=-5), dict(dtype=9), dict(layer=-1), dict(flags=2),
])
def test_plan_create_rejects_bad_arguments(swslib, bad):
    S = swslib
    n = bad.get("n", 4)
    ent = (bad.get("layer", 0), bad.get("dtype", S.E4M3), bad.get("rows", 8), bad.get("cols", 16))
    with pytest.raises(S.SwsError) as ei:
        S.Plan([ent], n, bad.get("flags", 0))
    assert ei.value.code == S.E_INVALID


def test_empty_plan_and_empty_layers(swslib):
    S = swslib
    plan = S.Plan([], 4)
    assert plan.info() == (0, 4, 0) and plan.slot_bytes == 0
    plan = S.Plan([(2, S.E4M3, 4, 16)], 4)
    assert plan.layer(0) == (0, 0, 0) and plan.layer(1) == (0, 0, 0)
    assert plan.layer(2) == (64, 16, 1)
    with pytest.raises(S.SwsError):
        plan.layer(3)
    with pytest.raises(S.SwsError):
        plan.entry(1)


def test_workspace_bytes_grows_with_prefill_m(swslib):
    S = swslib
    plan = S.Plan([(0, S.E4M3, 256, 512)], 4)
    a, b, c = S.workspace_bytes(plan, 1), S.workspace_bytes(plan, 64), S.workspace_bytes(plan, 4096)
    assert 0 < a <= b < c
    assert c - b >= 4096 * 512 + 4096 * 4 * 4


def test_workspace_bytes_per_weight_type(swslib):
    # prefill activations in the workspace: E4M3 the quantiser's codes and
    # scales, F16 x rounded to f16 (2 bytes each), BF16 none (x is used as is);
    # two buffers of the largest.
    S = swslib
    m, cols = 4096, 512
    base = {}
    for dt in (S.E4M3, S.BF16, S.F16):
        plan = S.Plan([(0, dt, 256, cols)], 4)
        base[dt] = (S.workspace_bytes(plan, 64), S.workspace_bytes(plan, m))
    assert base[S.BF16][1] == base[S.BF16][0]
    assert base[S.F16][1] - base[S.F16][0] == 2 * (2 * m * cols)
    assert base[S.E4M3][1] - base[S.E4M3][0] == 2 * (m * cols + m * (cols // 128) * 4)
    plan = S.Plan([(0, S.F16, 256, 24)], 4)  # elements of 2 bytes in the layout
    assert plan.entry(0)[1] == 256 * 24 * 2


def test_relayout_validates_before_any_launch(swslib):
    S = swslib
    plan = S.Plan([(0, S.E4M3, 8, 16)], 4)
    with pytest.raises(S.SwsError) as ei:
        S.relayout(plan, 0, [16] * 4, [0, 0, 0, 0])
    assert ei.value.code == S.E_INVALID
    with pytest.raises(S.SwsError) as ei:
        S.relayout(plan, 0, [16] * 4, [17, 32, 48, 64])
    assert ei.value.code == S.E_ALIGN
    with pytest.raises(S.SwsError):
        S.relayout(plan, 1, [16] * 4, [16, 32, 48, 64])


def test_silu_mul_validates_before_any_launch(swslib):
    S = swslib
    S.silu_mul(0, 0, 16, 0)  # m = 0: nothing to do, no device touched
    with pytest.raises(S.SwsError) as ei:
        S.silu_mul(4096, 2, 12, 8192)
    assert ei.value.code == S.E_UNSUPPORTED  # f % 8 != 0
    with pytest.raises(S.SwsError) as ei:
        S.silu_mul(4096, -1, 16, 8192)
    assert ei.value.code == S.E_INVALID
    with pytest.raises(S.SwsError) as ei:
        S.silu_mul(4097, 2, 16, 8192)
    assert ei.value.code == S.E_ALIGN


def test_graph_calls_validate_before_any_cuda_call(swslib):
    import ctypes as C
    L = swslib.lib()
    out = C.c_void_p(123)
    assert L.sws_graph_capture(None, 0, 0, None, 0, None, None, C.byref(out)) == swslib.E_INVALID
    assert out.value is None  # *out is cleared on error
    assert L.sws_graph_capture(None, 0, 0, None, 0, None, None, None) == swslib.E_INVALID
    assert L.sws_graph_launch(None, None) == swslib.E_INVALID
    L.sws_graph_destroy(None)  # a no-op


def test_options_reject_unknown_values(swslib):
    S = swslib
    for opt, bad in ((S.OPT_DECODE_KERNEL, 3), (S.OPT_PREFILL_KERNEL, 3), (S.OPT_GATHER_ENGINE, 3), (99, 0)):
        with pytest.raises(S.SwsError) as ei:
            S.set_option(opt, bad)
        assert ei.value.code == S.E_INVALID
    S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)
    S.set_option(S.OPT_PREFILL_KERNEL, S.PREFILL_AUTO)


def test_linear_noalloc_refuses_bad_sizes_before_any_device_call(swslib):
    # Limits of the fixed scratch and the argument checks run on the host
    # before the device is touched, so they are checkable without a GPU
    # (the pointers below are never dereferenced).
    import ctypes as C
    S = swslib
    L = S.lib()

    def call(rows, cols, m, x=4096, w=4096, sc=8192, y=12288):
        return L.sws_linear_noalloc(C.c_void_p(w), C.c_void_p(sc), rows, cols, C.c_void_p(x), m, C.c_void_p(y), None)

    assert call(4096 * 512 + 1, 16, 16) == S.E_INVALID  # 4097 row blocks of 512 rows (m <= 16)
    assert "exceeds the limit of 2097152 rows" in S.last_error()
    assert call(4096 * 256 + 1, 16, 17) == S.E_INVALID  # 4097 row blocks of 256 rows (m > 16)
    assert "exceeds the limit of 1048576 rows" in S.last_error()
    assert call(256, 16, 65) == S.E_INVALID and "m=65" in S.last_error()
    assert call(256, 16, -1) == S.E_INVALID
    assert call(-1, 16, 4) == S.E_INVALID
    assert call(256, 24, 4) == S.E_UNSUPPORTED  # cols % 16 != 0
    assert call(256, 16, 4, x=4097) == S.E_ALIGN
    assert call(256, 16, 4, w=4104) == S.E_ALIGN
    assert call(256, 16, 4, x=0) == S.E_INVALID
    assert call(0, 16, 4) == S.OK and call(256, 16, 0) == S.OK  # nothing to do


def test_host_wait_option_range(swslib):
    S = swslib
    for bad in (0, -5, 3_600_001):
        with pytest.raises(S.SwsError) as ei:
            S.set_option(S.OPT_HOST_WAIT_MS, bad)
        assert ei.value.code == S.E_INVALID
    S.set_option(S.OPT_HOST_WAIT_MS, 10000)
    assert S.lib().sws_noalloc_status(0, None) == S.E_INVALID


def test_bounds_self_check_of_relayout_segments(swslib):
    # SWS_OPT_CHECK_BOUNDS, host only: every copy segment of the relayout lies
    # inside its row shard and its chunk of C bytes; checked against chunks
    # 16 bytes too short (a planted mistake in the chunk size) it is refused,
    # and against longer ones it passes.
    from test_oracle_pins import read_padding_golden
    import warnings
    S = swslib
    dt = {1: S.E4M3, 2: S.BF16, 4: S.F32}
    plans = []
    for n, ents, total, chunk in read_padding_golden().values():
        plans.append(([(0, dt[e], r, c) for (_, r, c, e, _) in ents], n))
    rng = np.random.default_rng(77)
    for n in (1, 2, 3, 7, 16):
        for _ in range(6):
            ents = []
            for _ in range(int(rng.integers(1, 7))):
                rows = int(rng.integers(1, 5)) * n if rng.random() < 0.8 else int(rng.integers(1, 40))
                ents.append((int(rng.integers(0, 3)), dt[int(rng.choice([1, 2, 4]))], rows, int(rng.integers(1, 90))))
            plans.append((ents, n))
    checked = 0
    for ents, n in plans:
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            plan = S.Plan(ents, n)
        for l in range(plan.info()[0]):
            total, chunk, _ = plan.layer(l)
            assert S.test_check_relayout(plan, l, chunk) == S.OK
            assert S.test_check_relayout(plan, l, chunk + 16) == S.OK
            if total > 0:
                assert S.test_check_relayout(plan, l, chunk - 16) == S.E_INVALID
                assert "outside its buffer" in S.last_error()
                checked += 1
    assert checked >= 20
    for bad in (2, -1):
        with pytest.raises(S.SwsError) as ei:
            S.set_option(S.OPT_CHECK_BOUNDS, bad)
        assert ei.value.code == S.E_INVALID
    S.set_option(S.OPT_CHECK_BOUNDS, 1)
    S.set_option(S.OPT_CHECK_BOUNDS, 0)


def _settle_tasks_by_definition(rows, cols, elem, G):
    """The split-K bookkeeping of a decode launch, from its definition: units
    are (linear, 256-row block, K slab) in order, CTA c takes units
    [c*U//G, (c+1)*U//G), and every row block that more than one CTA works on
    needs one settle task: its first and last CTA, its rows, and where the
    first CTA left its partial sums (its first run's slot 2c when its range
    starts inside that row block, else its last run's, 2c+1)."""
    units = []
    for i, (r, c) in enumerate(zip(rows, cols)):
        slabs = -(-c * elem // 128)
        for rbl in range(-(-r // 256)):
            units += [(i, rbl)] * slabs
    U = len(units)
    start = [c * U // G for c in range(G + 1)]
    owner = [c for c in range(G) for _ in range(start[c], start[c + 1])]
    ctas = {}
    for u, key in enumerate(units):
        ctas.setdefault(key, set()).add(owner[u])
    tasks = []
    for key in dict.fromkeys(units):  # row blocks in unit order
        cs = sorted(ctas[key])
        if len(cs) > 1:
            i, rbl = key
            cf, cl = cs[0], cs[-1]
            tasks.append((i, rbl, min(256, rows[i] - 256 * rbl), cf, cl, 2 * cf + (0 if units[start[cf]] == key else 1)))
    return tasks, U


def test_decode_settle_tasks_match_the_partition(swslib):
    # Host logic of the tcgen05 decode launch: the settle tasks its planner
    # derives with closed-form unit arithmetic, against the tasks read off the
    # partition unit by unit - the decode workloads' layers on one CTA per SM,
    # and random groups (ragged row blocks, 1 to 8 linears, E4M3 and 16-bit
    # weights) on every grid from 1 CTA to one per unit.
    S = swslib
    cases = []
    for w in (WL.SHARED_EXPERT, WL.ATTN_KDA):
        rows = [e.rows for e in w.entries]
        cols = [e.cols for e in w.entries]
        for elem in (1, 2):
            for G in (1, 2, 151, 152, 256):
                cases.append((rows, cols, elem, G))
    rng = np.random.default_rng(2024)
    for _ in range(60):
        n = int(rng.integers(1, 9))
        rows = [int(rng.integers(1, 1400)) for _ in range(n)]
        cols = [16 * int(rng.integers(1, 80)) for _ in range(n)]
        elem = int(rng.choice([1, 2]))
        U = sum(-(-r // 256) * -(-c * elem // 128) for r, c in zip(rows, cols))
        for G in sorted({1, min(U, 256), int(rng.integers(1, min(U, 256) + 1))}):
            cases.append((rows, cols, elem, G))
    n_tasks = 0
    for rows, cols, elem, G in cases:
        want, U = _settle_tasks_by_definition(rows, cols, elem, G)
        got = S.test_settle_plan(rows, cols, elem, G)
        assert got == want, (rows, cols, elem, G)
        n_tasks += len(got)
    assert n_tasks > 500
    # refusals: no linear, more than 8, cols not a multiple of 16, grid outside [1, min(U, 256)]
    with pytest.raises(S.SwsError):
        S.test_settle_plan([], [], 1, 1)
    with pytest.raises(S.SwsError):
        S.test_settle_plan([256] * 9, [128] * 9, 1, 1)
    with pytest.raises(S.SwsError):
        S.test_settle_plan([256], [120], 1, 1)
    with pytest.raises(S.SwsError):
        S.test_settle_plan([256], [256], 1, 3)  # 2 units
    with pytest.raises(S.SwsError):
        S.test_settle_plan([256], [256], 1, 0)
