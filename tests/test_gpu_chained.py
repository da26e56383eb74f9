"""Forwards launched back to back on one stream, with nothing between them.

The batch-1 kernel and the tensor-core path's prep kernel are programmatic
dependent launches: a forward's CTAs may start while the previous forward in
the stream is still finishing, and every thread waits for that grid before it
touches memory.  This checks the ordering that has to hold: three forwards on
different hidden rows enqueued back to back, the first two writing the same
logits and argmax buffers (the second's values must be the ones left there)
and the third its own; every result against the f64 oracle, on the batch-1,
split-K, tensor-core (8 and 16 batch slots) and logprobs paths, and with a
batch-1 and a batch-4 forward of one handle alternating.
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


def _check(got, am, ref, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert err.max() <= TOL, f"{what}: max|err| {err.max():.3g}"
    if am is not None:
        for b in range(ref.shape[0]):
            assert am[b] == int(np.argmax(got[b])), f"{what}: row {b}"
            if oracle.top2_gap(ref[b:b + 1])[0] > GAP:
                assert am[b] == int(oracle.argmax_first(ref[b:b + 1])[0]), f"{what}: row {b}"


def _inputs(n, k, b, seeds):
    wq = synth.q5k_matrix(n, k, synth.stream_key(n + k, "W:chained"), boost_rows=(n // 3,), boost=30.0)
    gamma = synth.normal_f64(k, synth.stream_key(k, "G:chained"), 1.0, 0.1).astype(np.float32)
    hs = [(synth.normal_f64(b * k, synth.stream_key(s, f"H:chained{k}")) * (1.0 + s)).astype(np.float32)
          .reshape(b, k) for s in seeds]
    return wq, gamma, hs


@pytest.mark.parametrize("n,k,b,path", [(5000, 6656, 1, "gemv_b1"), (2000, 13312, 1, "gemv_b1_split"),
                                        (3000, 6656, 4, "gemm_tc"), (3000, 6656, 12, "gemm_tc")])
def test_back_to_back_forwards(torch_cuda, n, k, b, path):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wq, gamma, hs = _inputs(n, k, b, (1, 2, 3))
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        h_d = [_dev(torch, h) for h in hs]
        shared_l = torch.full((b, n), float("nan"), device="cuda")
        shared_a = torch.full((b,), -1, dtype=torch.int32, device="cuda")
        own_l = torch.full((b, n), float("nan"), device="cuda")
        own_a = torch.full((b,), -1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        head.forward(h_d[0], w_d, g_d, logits=shared_l, argmax=shared_a)
        head.forward(h_d[1], w_d, g_d, logits=shared_l, argmax=shared_a)
        head.forward(h_d[2], w_d, g_d, logits=own_l, argmax=own_a)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        for h, (l, a), what in ((hs[1], (shared_l, shared_a), "second into the shared buffers"),
                                (hs[2], (own_l, own_a), "third")):
            ref = oracle.lmhead(h, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
            _check(l.cpu().numpy(), a.cpu().numpy(), ref, f"{path}: {what}")


def test_back_to_back_alternating_batches(torch_cuda):
    """Batch 1 (the batch-1 kernel) and batch 4 (the tensor-core path) of one
    handle, alternating on one stream without a synchronisation."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 4000, 6656
    wq, gamma, hs4 = _inputs(n, k, 4, (5, 6))
    _, _, hs1 = _inputs(n, k, 1, (7, 8))
    with mlh.LMHead(n, k, max_batch=4, device=0) as head:
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        outs = []
        for h in (hs1[0], hs4[0], hs1[1], hs4[1]):
            outs.append(head.forward(_dev(torch, h), w_d, g_d))
        torch.cuda.synchronize()
        assert head.device_status() == 0
        for h, (l, a) in zip((hs1[0], hs4[0], hs1[1], hs4[1]), outs):
            ref = oracle.lmhead(h, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
            _check(l.cpu().numpy(), a.cpu().numpy(), ref, f"batch {h.shape[0]}")


def test_back_to_back_logprobs(torch_cuda):
    """The batch-1 logprobs forward (its normaliser kernels follow it as
    programmatic dependents) twice in a row, then a plain forward."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 6000, 6656
    wq, gamma, hs = _inputs(n, k, 1, (9, 10, 11))
    with mlh.LMHead(n, k, max_batch=1, device=0) as head:
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        lp1 = head.forward_logprobs(_dev(torch, hs[0]), w_d, g_d)
        lp2 = head.forward_logprobs(_dev(torch, hs[1]), w_d, g_d)
        l3, a3 = head.forward(_dev(torch, hs[2]), w_d, g_d)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        for h, lp in ((hs[0], lp1), (hs[1], lp2)):
            ref = oracle.lmhead(h, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
            ref_lp, _ = oracle.log_softmax(ref)
            got = lp[0].cpu().numpy()
            assert np.abs(got.astype(np.float64) - ref_lp).max() <= TOL
        ref = oracle.lmhead(hs[2], gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
        _check(l3.cpu().numpy(), a3.cpu().numpy(), ref, "plain after logprobs")
