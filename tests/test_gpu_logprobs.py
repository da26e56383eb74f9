"""GPU parity of muse_lmhead_forward_logprobs: log-softmax over the capped
logits ("Chapter 20 — Final norm, LM head, and the soft cap", §20.7), against
the f64 oracle (oracle.log_softmax of oracle.lmhead).

Bar: |gpu - oracle| <= 2e-3 for every logprob and for the normaliser lse; the
argmax as for the logits; logprobs + lse give back the forward's logits.
Covers the fused batch-1 path (normaliser from the kernel's epilogue), the
tensor-core path and the generic path (a separate pass over the logits).
"""
import numpy as np
import pytest

import oracle
import q5k_synth as synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
GAP = 4e-3


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    import q5_lm_head_gb300 as mlh
    from q5_lm_head_gb300 import _build
    _build.build()
    mlh.load_library()
    torch.cuda.set_device(0)
    return torch


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _case(torch, hidden, gamma, wq, n_rows, k, scale, cap, path=None):
    import q5_lm_head_gb300 as mlh
    b = hidden.shape[0]
    with mlh.LMHead(n_rows, k, max_batch=b, device=0) as head:
        if path is not None:
            assert head.path_name(b) == path
        h, w = _dev(torch, hidden), _dev(torch, wq)
        g = None if gamma is None else _dev(torch, gamma)
        lp, lse, am = head.forward_logprobs(h, w, g, synth.RMS_EPS, scale, cap, True)
        logits, am2 = head.forward(h, w, g, synth.RMS_EPS, scale, cap, True)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        lp, lse, am = lp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy()
        logits, am2 = logits.cpu().numpy(), am2.cpu().numpy()
    ref_logits = oracle.lmhead(hidden, gamma, wq, scale, cap, synth.RMS_EPS)
    ref_lp, ref_lse = oracle.log_softmax(ref_logits)
    assert np.all(np.isfinite(lp)) and np.all(np.isfinite(lse))
    err = np.abs(lp.astype(np.float64) - ref_lp)
    assert err.max() <= TOL, f"logprobs: max|err|={err.max():.3g}"
    assert np.abs(lse.astype(np.float64) - ref_lse).max() <= TOL
    # same argmax as the logits' forward, and logprobs + lse = logits
    assert np.array_equal(am, am2)
    assert np.abs((lp + lse[:, None]) - logits).max() <= 1e-4 * max(1.0, float(np.abs(lse).max()))
    gap = oracle.top2_gap(ref_logits)
    want = oracle.argmax_first(ref_logits)
    for r in range(b):
        if gap[r] > GAP:
            assert am[r] == want[r]
    return err.max()


def test_logprobs_batch1_fused(torch_cuda):
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    _case(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, "gemv_b1")


def test_logprobs_full_lm_head_batch1(torch_cuda):
    wl = synth.WORKLOADS["lmhead_b1"]          # rows 0, 777, 200001 saturate the cap
    hidden, gamma, wq = synth.inputs_for(wl)
    _case(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, "gemv_b1")


@pytest.mark.parametrize("b", [2, 8, 32])      # 32 slots: round-robin tiles
def test_logprobs_tensor_core_path(torch_cuda, b):
    n, k = 20000, 6656
    rng = np.random.default_rng(b)
    hidden = (rng.standard_normal((b, k)) * rng.uniform(0.5, 4.0, (b, 1))).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)
    wq = synth.q5k_matrix(n, k, synth.stream_key(3, f"W:lp{b}"), boost_rows=(5,), boost=50.0)
    _case(torch_cuda, hidden, gamma, wq, n, k, synth.LOGIT_SCALE, synth.SOFTCAP, "gemm_tc")


@pytest.mark.parametrize("n,k,b,cap", [(3000, 768, 3, 20.0), (777, 4096, 1, 0.0), (5000, 1024, 1, 20.0)])
def test_logprobs_generic_and_other_shapes(torch_cuda, n, k, b, cap):
    rng = np.random.default_rng(n + k + b)
    hidden = rng.standard_normal((b, k)).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)
    wq = synth.q5k_matrix(n, k, synth.stream_key(4, f"W:lpg{n}:{k}:{b}"))
    _case(torch_cuda, hidden, gamma, wq, n, k, synth.LOGIT_SCALE if cap > 0 else 1.0, cap)


def test_logprobs_repeat_calls_are_deterministic(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
        h, g, w = _dev(torch, hidden), _dev(torch, gamma), _dev(torch, wq)
        a = [t.clone() for t in head.forward_logprobs(h, w, g)]
        b = [t.clone() for t in head.forward_logprobs(h, w, g)]
        torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
