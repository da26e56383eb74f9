"""The batch-1 entry point that allocates no device memory.

Some callers cannot call cudaMalloc when they need a forward: runtimes that
reserve all device memory up front through their own allocator and refuse
later allocations, and serving loops that must not risk the implicit device
synchronisation of cudaMalloc/cudaFree.  They use
muse_lmhead_forward_b1_noalloc, whose scratch lives in a fixed array in the
library's device memory.  Through the C-ABI this checks, on two calls in a row
per input (the calls share, and must re-arm, that scratch), every logit
against the f64 oracle within the tolerance of the other GPU parity tests, the
argmax where the oracle's top-2 gap decides it, and that the status word reads
0 after each call; at both widths the fused kernel takes (6,656 with norm, cap
and argmax; 4,096 with none of them).  Unsupported widths are rejected before
anything is launched.  The file is named to be collected last.
"""
import numpy as np
import pytest

import oracle
import q5k_synth as synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
GAP = 4e-3


@pytest.fixture(scope="module")
def lib():
    import torch
    import q5_lm_head_gb300 as mlh
    from q5_lm_head_gb300 import _build
    _build.build()
    mlh.load_library()
    torch.cuda.set_device(0)
    return mlh


def _check(got_l, got_a, ref, what):
    err = np.abs(got_l.astype(np.float64) - ref)
    assert np.all(np.isfinite(got_l)), what
    assert err.max() <= TOL, f"{what}: max|err| {err.max():.3g}"
    if got_a is not None:
        a = int(got_a[0])
        assert a == int(np.argmax(got_l[0])), f"{what}: argmax {a} is not the first max of the logits"
        if oracle.top2_gap(ref)[0] > GAP:
            assert a == int(oracle.argmax_first(ref)[0]), what


@pytest.mark.parametrize("name", ["tiny", "attn_o"])
def test_noalloc_matches_oracle_twice(lib, name):
    import torch
    mlh = lib
    wl = synth.WORKLOADS[name]
    hidden, gamma, wq = synth.inputs_for(wl)
    hidden2 = np.ascontiguousarray(hidden[:, ::-1] * 1.5)
    dev = torch.device("cuda", 0)
    w_d = torch.from_numpy(wq).to(dev)
    g_d = None if gamma is None else torch.from_numpy(gamma).to(dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert mlh.muse_lmhead_noalloc_device_status(0, stream) == 0   # nothing left over from earlier tests
    for h in (hidden, hidden2):
        ref = oracle.lmhead(h, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS)
        h_d = torch.from_numpy(np.ascontiguousarray(h)).to(dev)
        for call in range(2):
            out_l = torch.full((1, wl.n_rows), float("nan"), device=dev)
            out_a = torch.full((1,), -1, dtype=torch.int32, device=dev) if wl.argmax else None
            st = mlh.muse_lmhead_forward_b1_noalloc(
                0, h_d.data_ptr(), None if g_d is None else g_d.data_ptr(), synth.RMS_EPS, w_d.data_ptr(),
                wl.n_rows, wl.k, wl.scale, wl.cap, out_l.data_ptr(), None if out_a is None else out_a.data_ptr(),
                stream)
            assert st == 0, mlh.muse_lmhead_status_string(st)
            assert mlh.muse_lmhead_noalloc_device_status(0, stream) == 0
            _check(out_l.cpu().numpy(), None if out_a is None else out_a.cpu().numpy(), ref,
                   f"{name} call {call}")


def test_noalloc_rejects_unsupported_width_without_launching(lib):
    import torch
    mlh = lib
    k = 512
    w_d = torch.zeros(8 * (k // 256) * 176, dtype=torch.uint8, device="cuda")
    h_d = torch.ones(k, device="cuda")
    out = torch.full((8,), 3.0, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = mlh.muse_lmhead_forward_b1_noalloc(0, h_d.data_ptr(), None, 1e-5, w_d.data_ptr(), 8, k, 1.0, 0.0,
                                            out.data_ptr(), None, stream)
    assert st == -2
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    assert mlh.muse_lmhead_noalloc_device_status(0, stream) == 0
