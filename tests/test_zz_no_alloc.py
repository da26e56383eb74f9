"""The batch-1 entry point that allocates no device memory.

Callers that cannot call cudaMalloc when they need a forward (inside CUDA
graph capture, under a runtime that owns all device memory, in a serving loop
that must avoid cudaMalloc's implicit synchronisation) use
muse_lmhead_forward_b1_noalloc, whose scratch lives in a fixed array in the
library's device memory.  This checks, through the C-ABI, that two calls in a
row give the same logits and argmax as the handle-based entry point (within the
parity tolerance of the other GPU tests), and that unsupported widths are
rejected before anything is launched.  The file is named to be collected last.
"""
import numpy as np
import pytest

import q5k_synth as synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def lib():
    import torch
    import q5_lm_head_gb300 as mlh
    from q5_lm_head_gb300 import _build
    _build.build()
    mlh.load_library()
    torch.cuda.set_device(0)
    return mlh


def test_noalloc_matches_handle_forward_twice(lib):
    import torch
    mlh = lib
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    hidden2 = np.ascontiguousarray(hidden[:, ::-1] * 1.5)
    dev = torch.device("cuda", 0)
    w_d = torch.from_numpy(wq).to(dev)
    g_d = torch.from_numpy(gamma).to(dev)
    stream = torch.cuda.current_stream().cuda_stream
    for h in (hidden, hidden2):
        h_d = torch.from_numpy(np.ascontiguousarray(h)).to(dev)
        with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
            ref_l, ref_a = head.forward(h_d, w_d, g_d, synth.RMS_EPS, wl.scale, wl.cap)
        for _ in range(2):   # two calls in a row share (and must re-arm) the scratch
            out_l = torch.full((1, wl.n_rows), float("nan"), device=dev)
            out_a = torch.full((1,), -1, dtype=torch.int32, device=dev)
            st = mlh.muse_lmhead_forward_b1_noalloc(0, h_d.data_ptr(), g_d.data_ptr(), synth.RMS_EPS,
                                                    w_d.data_ptr(), wl.n_rows, wl.k, wl.scale, wl.cap,
                                                    out_l.data_ptr(), out_a.data_ptr(), stream)
            assert st == 0, mlh.muse_lmhead_status_string(st)
            torch.cuda.synchronize()
            assert torch.isfinite(out_l).all()
            assert float((out_l - ref_l).abs().max()) <= TOL
            assert int(out_a[0]) == int(ref_a[0])


def test_noalloc_rejects_unsupported_width_without_launching(lib):
    import torch
    mlh = lib
    k = 512
    w_d = torch.zeros(8 * (k // 256) * 176, dtype=torch.uint8, device="cuda")
    h_d = torch.ones(k, device="cuda")
    out = torch.full((8,), 3.0, device="cuda")
    st = mlh.muse_lmhead_forward_b1_noalloc(0, h_d.data_ptr(), None, 1e-5, w_d.data_ptr(), 8, k, 1.0, 0.0,
                                            out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == -2
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
