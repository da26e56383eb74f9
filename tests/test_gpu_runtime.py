"""GPU runtime behaviour around the forward: capture into CUDA graphs, the
bounded-wait failure path, and the DFlash verify batch.

* A forward captured into a CUDA graph (batch-1 kernel, tensor-core path with
  its programmatic dependent launch, generic path, logprobs) replays to the
  same bits as the eager call, twice in a row (the argmax workspace and the
  shared-tile counters of the tensor-core path re-arm).
* Failure detection without a GPU fault: a self-test kernel waits on an
  mbarrier that nothing arrives on; the bounded wait gives up, the status word
  records it, the kernel returns, and the context keeps working.
* The DFlash verify batch: the drafter proposes 16 tokens per step, so the
  target model's output stage runs at batch 16 with a per-position argmax
  ("Chapter 9 — The Muse Glimmer architecture", §9.12); parity with the oracle
  on the full head.
"""
import time

import numpy as np
import pytest

import oracle
import q5k_synth as synth

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("n,k,b,path", [(2048, 6656, 1, "gemv_b1"), (3000, 6656, 4, "gemm_tc"),
                                        (20000, 6656, 8, "gemm_tc"),    # tiles shared by two CTAs
                                        (500, 768, 2, "gemv_generic"),
                                        (1000, 13312, 1, "gemv_b1_split")])   # chunk partials via the counters
def test_forward_replayed_from_a_cuda_graph_matches_eager(torch_cuda, n, k, b, path):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    rng = np.random.default_rng(n + b)
    hidden = _dev(torch, rng.standard_normal((b, k)).astype(np.float32))
    gamma = _dev(torch, (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32))
    w = _dev(torch, synth.q5k_matrix(n, k, synth.stream_key(2, f"W:graph{n}")))
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
        ref_l, ref_a = head.forward(hidden, w, gamma)
        logits = torch.empty_like(ref_l)
        amax = torch.empty_like(ref_a)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())      # a handle's workspace serves one stream at a time
        with torch.cuda.stream(s):                      # one-time set-up happens before the capture
            head.forward(hidden, w, gamma, logits=logits, argmax=amax, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            head.forward(hidden, w, gamma, logits=logits, argmax=amax, stream=s)
        for _ in range(2):
            logits.zero_()
            amax.fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(logits, ref_l) and torch.equal(amax, ref_a)
        assert head.device_status() == 0


def test_logprobs_replayed_from_a_cuda_graph(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    h, g_, w = _dev(torch, hidden), _dev(torch, gamma), _dev(torch, wq)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
        ref = [t.clone() for t in head.forward_logprobs(h, w, g_)]
        lp, lse, am = torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2])
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())      # a handle's workspace serves one stream at a time
        with torch.cuda.stream(s):
            head.forward_logprobs(h, w, g_, logprobs=lp, lse=lse, argmax=am, stream=s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            head.forward_logprobs(h, w, g_, logprobs=lp, lse=lse, argmax=am, stream=s)
        lp.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for x, y in zip((lp, lse, am), ref):
            assert torch.equal(x, y)


def test_grouped_forward_replayed_from_a_cuda_graph(torch_cuda):
    """The Q/K/V/gate group captured once and replayed: the segment table is a
    kernel argument, so every replay writes the same four outputs, bit for bit
    the eager call's."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    g = synth.GROUPS["attn_qkvg"]
    hidden, gamma, ws = synth.group_inputs(g)
    with mlh.LMHead(1, g.k, max_batch=1, device=0) as head:
        h, gm = _dev(torch, hidden), _dev(torch, gamma)
        wd = [_dev(torch, w) for w in ws]
        ref = head.forward_group(h, [(w, n, sc, cp, None) for w, (_, n, _, sc, cp) in zip(wd, g.segments)], gm)
        outs = [torch.empty_like(r) for r in ref]
        segs = [(w, n, sc, cp, o) for w, (_, n, _, sc, cp), o in zip(wd, g.segments, outs)]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())      # a handle's workspace serves one stream at a time
        with torch.cuda.stream(s):
            head.forward_group(h, segs, gm, stream=s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            head.forward_group(h, segs, gm, stream=s)
        for _ in range(2):
            for o in outs:
                o.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert all(torch.equal(o, r) for o, r in zip(outs, ref))
        assert head.device_status() == 0


def test_bounded_wait_gives_up_and_reports_without_a_fault(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
        assert head.device_status() == 0
        t0 = time.perf_counter()
        assert mlh.muse_lmhead_selftest_wait_timeout(head.handle) == 0
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 10.0                  # the wait is bounded
        assert head.device_status() & mlh.STATUS_WAIT_TIMEOUT
        # the context is intact: clear the word, run a forward, check it against the oracle
        assert mlh.muse_lmhead_clear_device_status(head.handle) == 0
        torch.cuda.synchronize()
        assert head.device_status() == 0
        logits, amax = head.forward(_dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma))
        torch.cuda.synchronize()
        assert head.device_status() == 0
    ref = oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS)
    assert np.abs(logits.cpu().numpy() - ref).max() <= 2e-3


def test_cleared_status_then_tensor_core_forward(torch_cuda):
    """The same failure path on a handle with the tensor-core workspace: after
    the self-test and the clear (which also re-arms the shared-tile counters), a
    batch-4 forward over more tiles than SMs (tiles shared by two CTAs) matches
    the oracle and records no fault."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k, b = 20000, 6656, 4
    wq = synth.q5k_matrix(n, k, synth.stream_key(12, "W:clear"))
    hidden = synth.normal_f64(b * k, synth.stream_key(12, "H:clear")).astype(np.float32).reshape(b, k)
    gamma = synth.normal_f64(k, synth.stream_key(12, "G:clear"), 1.0, 0.1).astype(np.float32)
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == "gemm_tc"
        assert mlh.muse_lmhead_selftest_wait_timeout(head.handle) == 0
        torch.cuda.synchronize()
        assert head.device_status() & mlh.STATUS_WAIT_TIMEOUT
        assert mlh.muse_lmhead_clear_device_status(head.handle) == 0
        torch.cuda.synchronize()
        assert head.device_status() == 0
        logits, amax = head.forward(_dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma))
        torch.cuda.synchronize()
        assert head.device_status() == 0
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
    assert np.abs(logits.cpu().numpy() - ref).max() <= 2e-3
    want, gap, got = oracle.argmax_first(ref), oracle.top2_gap(ref), amax.cpu().numpy()
    assert all(int(got[i]) == int(want[i]) for i in range(b) if gap[i] > 4e-3)


def test_dflash_verify_batch16(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["dflash_verify_b16"]
    hidden, gamma, wq = synth.inputs_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=16, device=0) as head:
        assert head.path_name(16) == "gemm_tc"
        logits, amax = head.forward(_dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma))
        torch.cuda.synchronize()
        assert head.device_status() == 0
        logits, amax = logits.cpu().numpy(), amax.cpu().numpy()
    ref = oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS)
    assert np.abs(logits - ref).max() <= 2e-3
    gap, want = oracle.top2_gap(ref), oracle.argmax_first(ref)
    for b in range(16):
        assert amax[b] == int(np.argmax(logits[b]))
        if gap[b] > 4e-3:
            assert amax[b] == want[b]
