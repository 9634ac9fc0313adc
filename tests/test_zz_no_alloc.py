"""sws_linear_noalloc: the decode linear for callers that cannot allocate
device memory or pass a workspace (for example an engine whose KV-cache pool
already holds all free memory). Called through the C ABI and checked against
the workspace-based sws_linear on the same inputs, twice in a row, since the
second call runs on scratch left over from the first."""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as WL
from helpers import LayerData, assert_close, bf16_tensor_to_f64, build_stack

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_linear_on_consecutive_calls(swslib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    S = swslib
    lib = S.lib()
    rng = np.random.default_rng(2024)
    rows, cols, n = 2048, 7168, 16  # many K slabs: split-K partial sums go through the scratch
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    sc = (2.0 ** rng.uniform(-8, -4, size=(rows // 128, cols // 128))).astype(np.float32)
    st = build_stack(S, [(0, rows, cols)], n, [LayerData({0: q}, {0: sc})])
    st.ctx.gather_to_slot(0, 0, 0)
    off, _, _ = st.entry_info[0]
    w_ptr = st.slots[0].data_ptr() + off
    stream = torch.cuda.current_stream().cuda_stream
    for call, m in enumerate((64, 5)):
        x = WL.draw_x(77, call, m, cols).cuda()
        y_ref = torch.empty((m, rows), dtype=torch.bfloat16, device="cuda")
        st.ctx.linear(0, S.SRC_SLOT0, x.data_ptr(), m, y_ref.data_ptr(), stream)
        y = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.sws_linear_noalloc(C.c_void_p(w_ptr), C.c_void_p(st.scales[0].data_ptr()), rows, cols,
                                    C.c_void_p(x.data_ptr()), m, C.c_void_p(y.data_ptr()), C.c_void_p(stream))
        assert rc == 0, S.last_error()
        torch.cuda.synchronize()
        assert_close(bf16_tensor_to_f64(y), bf16_tensor_to_f64(y_ref), f"call {call} (m={m})")
    # sizes beyond the limits are refused before any launch
    rc = lib.sws_linear_noalloc(C.c_void_p(w_ptr), C.c_void_p(st.scales[0].data_ptr()), rows, cols,
                                C.c_void_p(x.data_ptr()), 65, C.c_void_p(y.data_ptr()), C.c_void_p(stream))
    assert rc == S.E_INVALID and "m=65" in S.last_error()
