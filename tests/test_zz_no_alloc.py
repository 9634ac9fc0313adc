"""sws_linear_noalloc: the decode linear for callers that cannot allocate
device memory or hand the library a workspace - for example an inference
engine whose KV-cache pool already holds all the memory left free after the
weights were loaded, so that an allocation in the middle of a decode step
would fail or stall the GPU. Called through the C ABI on two calls in a row
(the second runs on scratch the first left behind) and checked against the
CPU oracle and against the workspace-based sws_linear; also at its row limit,
and its status word is exercised with a wait that runs out. This file is
collected last so that a failure here comes after every other test ran."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import LayerData, assert_close, bf16_tensor_to_f64, build_stack, x_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return swslib


def _codes(rng, rows, cols):
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    return q


def _call(S, w, sc, rows, cols, x, m, y, stream):
    return S.lib().sws_linear_noalloc(C.c_void_p(w), C.c_void_p(sc), rows, cols, C.c_void_p(x), m, C.c_void_p(y),
                                      C.c_void_p(stream))


def test_noalloc_decode_matches_oracle_and_workspace_linear_on_consecutive_calls(S):
    rng = np.random.default_rng(2024)
    rows, cols, n = 2048, 7168, 16  # many K slabs: split-K partial sums go through the scratch
    q = _codes(rng, rows, cols)
    sc = (2.0 ** rng.uniform(-8, -4, size=(rows // 128, cols // 128))).astype(np.float32)
    st = build_stack(S, [(0, rows, cols)], n, [LayerData({0: q}, {0: sc})])
    st.ctx.gather_to_slot(0, 0, 0)
    off, _, _ = st.entry_info[0]
    w_ptr = st.slots[0].data_ptr() + off
    stream = torch.cuda.current_stream().cuda_stream
    for call, m in enumerate((64, 5, 32)):
        x = WL.draw_x(77, call, m, cols)
        xd = x.cuda()
        y_ws = torch.empty((m, rows), dtype=torch.bfloat16, device="cuda")
        st.ctx.linear(0, S.SRC_SLOT0, xd.data_ptr(), m, y_ws.data_ptr(), stream)
        y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _call(S, w_ptr, st.scales[0].data_ptr(), rows, cols, xd.data_ptr(), m, y.data_ptr(), stream)
        assert rc == 0, S.last_error()
        torch.cuda.synchronize()
        assert_close(bf16_tensor_to_f64(y), O.linear(x_f64(x), q, sc), f"call {call} (m={m}) against the oracle")
        assert_close(bf16_tensor_to_f64(y), bf16_tensor_to_f64(y_ws), f"call {call} (m={m}) against sws_linear")
    assert S.noalloc_status() == 0


def test_noalloc_at_its_row_limit(S):
    # 4096 row blocks of 256 rows for 16 < m <= 64: 1,048,576 rows (one 16-column K slab)
    rng = np.random.default_rng(2025)
    rows, cols, m = 4096 * 256, 16, 40
    q = _codes(rng, rows, cols)
    sc = (2.0 ** rng.uniform(-8, -4, size=(rows // 128, 1))).astype(np.float32)
    w = torch.from_numpy(q).cuda()
    s = torch.from_numpy(sc).cuda()
    x = WL.draw_x(78, 0, m, cols)
    xd = x.cuda()
    y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert _call(S, w.data_ptr(), s.data_ptr(), rows, cols, xd.data_ptr(), m, y.data_ptr(), stream) == 0, \
        S.last_error()
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([[0, 255, 256, rows - 1], rng.choice(rows, size=4000, replace=False)]))
    got = bf16_tensor_to_f64(y)
    assert np.all(np.isfinite(got))
    assert_close(got[:, sel], O.linear_rows(x_f64(x), q, sc, sel), "row limit, sampled rows")
    # one row block more is refused before any launch
    assert _call(S, w.data_ptr(), s.data_ptr(), rows + 1, cols, xd.data_ptr(), m, y.data_ptr(), stream) == S.E_INVALID
    assert "exceeds the limit" in S.last_error()
    assert S.noalloc_status() == 0


def test_noalloc_status_word_reports_a_wait_that_ran_out(S):
    # The library's bounded wait, pointed at the status word of the fixed
    # scratch, gives up after 2 ms on a barrier nothing arrives at and records
    # SWS_E_TIMEOUT there; the host reads and clears it, and the next call
    # runs normally.
    assert S.noalloc_status(clear=True) == 0
    S.test_bounded_wait_noalloc(2_000_000)
    assert S.noalloc_status() == S.E_TIMEOUT  # sticky until cleared
    assert S.noalloc_status(clear=True) == S.E_TIMEOUT
    assert S.noalloc_status() == 0
    rng = np.random.default_rng(2026)
    rows, cols, m = 512, 1024, 8
    q = _codes(rng, rows, cols)
    sc = (2.0 ** rng.uniform(-8, -4, size=(rows // 128, cols // 128))).astype(np.float32)
    w, s = torch.from_numpy(q).cuda(), torch.from_numpy(sc).cuda()
    x = WL.draw_x(79, 0, m, cols)
    xd = x.cuda()
    y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    S.linear_noalloc(w.data_ptr(), s.data_ptr(), rows, cols, xd.data_ptr(), m, y.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_close(bf16_tensor_to_f64(y), O.linear(x_f64(x), q, sc), "after the timeout")
    assert S.noalloc_status() == 0
