"""GPU parity of Q4_K weights (144-byte blocks: ggml's block_q4_K, the FFN
bulk's format and the 756.5 MB alternative head of "Chapter 20 — Final norm,
LM head, and the soft cap" §20.7) against the f64 oracle's own Q4_K parser.

Same bar as Q5_K: |gpu - oracle| <= 2e-3 on every logit, argmax equal where
the oracle's top-2 gap exceeds 4e-3.  Covers the fused batch-1 kernel (K =
6,656 and 4,096), the tensor-core kernel (batches 2..32, an even number of
blocks per row), the generic kernel (the other shapes), the logprobs forward
and the grouped batch-1 call.
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


def _check(got, am, ref):
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= TOL, f"max|err|={err.max():.3g}"
    if am is not None:
        gap, want = oracle.top2_gap(ref), oracle.argmax_first(ref)
        for b in range(ref.shape[0]):
            assert am[b] == int(np.argmax(got[b]))
            if gap[b] > GAP:
                assert am[b] == want[b]


def _run(torch, hidden, gamma, wq, n, k, scale, cap, path=None, want_argmax=True):
    import q5_lm_head_gb300 as mlh
    b = hidden.shape[0]
    with mlh.LMHead(n, k, max_batch=b, device=0, fmt="q4_k") as head:
        if path is not None:
            assert head.path_name(b) == path
        out = head.forward(_dev(torch, hidden), _dev(torch, wq), None if gamma is None else _dev(torch, gamma),
                           synth.RMS_EPS, scale, cap, want_argmax)
        torch.cuda.synchronize()
        assert head.device_status() == 0
    if want_argmax:
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy(), None


def test_q4k_full_head_batch1(torch_cuda):
    wl = synth.WORKLOADS["lmhead_q4k_b1"]
    hidden, gamma, wq = synth.inputs_for(wl)
    assert wq.shape == (wl.n_rows, 26 * 144)
    got, am = _run(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, "gemv_b1")
    _check(got, am, oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS, fmt="q4_k"))


def test_q4k_full_head_batch8(torch_cuda):
    wl = synth.WORKLOADS["lmhead_q4k_b8"]        # same weights as the batch-1 head, rows scaled by U(0.5, 4)
    hidden, gamma, wq = synth.inputs_for(wl)
    got, am = _run(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, "gemm_tc")
    ref = oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS, fmt="q4_k")
    _check(got, am, ref)
    for r in synth.BOOSTED_ROWS:                 # past the cap's knee
        assert np.abs(ref[:, r]).max() > 19.0 and np.abs(got[:, r]).max() <= 20.0


@pytest.mark.parametrize("n,k,b,norm,cap,path", [
    (777, 4096, 1, True, 20.0, "gemv_b1"),      # fused kernel, K = 4,096
    (25, 6656, 1, False, 0.0, "gemv_b1"),       # fewer rows than one stage per CTA
    (3001, 6656, 3, True, 20.0, "gemm_tc"),     # ragged last 128-row tile
    (129, 6656, 2, False, 0.0, "gemm_tc"),      # one row past a tile, cap off
    (5000, 4096, 16, True, 20.0, "gemm_tc"),
    (1000, 512, 32, True, 20.0, "gemm_tc"),     # two blocks per row, 32 batch rows
    (500, 512, 1, True, 20.0, "gemm_tc"),       # batch 1 at a K with no fused build
    (300, 768, 1, True, 20.0, "gemv_generic"),  # batch 1, odd number of blocks per row
    (64, 768, 8, False, 0.0, "gemv_generic"),   # odd number of blocks per row
])
def test_q4k_shapes(torch_cuda, n, k, b, norm, cap, path):
    rng = np.random.default_rng(n * 7 + k + b)
    hidden = rng.standard_normal((b, k)).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32) if norm else None
    wq = synth.q5k_matrix(n, k, synth.stream_key(9, f"W:q4:{n}:{k}"), boost_rows=(n // 2,), boost=50.0,
                          fmt="q4_k")
    scale = synth.LOGIT_SCALE if cap > 0 else 1.0
    got, am = _run(torch_cuda, hidden, gamma, wq, n, k, scale, cap, path)
    _check(got, am, oracle.lmhead(hidden, gamma, wq, scale, cap, synth.RMS_EPS, fmt="q4_k"))


@pytest.mark.parametrize("b", [1, 4])
def test_q4k_logprobs(torch_cuda, b):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 30000, 6656
    rng = np.random.default_rng(5 + b)
    hidden = rng.standard_normal((b, k)).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)
    wq = synth.q5k_matrix(n, k, synth.stream_key(10, "W:q4lp"), fmt="q4_k")
    with mlh.LMHead(n, k, max_batch=b, device=0, fmt="q4_k") as head:
        assert head.path_name(b) == ("gemv_b1" if b == 1 else "gemm_tc")
        lp, lse, am = head.forward_logprobs(_dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma))
        torch.cuda.synchronize()
        lp, lse = lp.cpu().numpy(), lse.cpu().numpy()
    ref_lp, ref_lse = oracle.log_softmax(oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP,
                                                       synth.RMS_EPS, fmt="q4_k"))
    assert np.abs(lp - ref_lp).max() <= TOL and np.abs(lse - ref_lse).max() <= TOL


def test_q4k_handle_rejects_q5k_sized_weights(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 64, 6656
    w5 = _dev(torch, synth.q5k_matrix(n, k, synth.stream_key(0, "W:q4-wrong")))
    with mlh.LMHead(n, k, max_batch=1, device=0, fmt="q4_k") as head:
        with pytest.raises(ValueError):
            head.forward(torch.zeros((1, k), device="cuda"), w5)
        with pytest.raises(ValueError):
            head.forward_group(torch.zeros((k,), device="cuda"), [(w5, n, 1.0, 0.0, None)])


@pytest.mark.parametrize("k,shapes", [
    (6656, ((4096, 1.0, 0.0), (4096, 1.0, 0.0), (256, 1.0, 0.0), (256, synth.LOGIT_SCALE, synth.SOFTCAP))),
    (4096, ((6656, 1.0, 0.0), (300, 1.0, 0.0))),
])
def test_q4k_grouped_call(torch_cuda, k, shapes):
    """The grouped batch-1 call on Q4_K matrices (the attention group's shapes
    at K = 6,656; two matrices at K = 4,096), against the oracle per matrix."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    rng = np.random.default_rng(k)
    hidden = rng.standard_normal(k).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)
    mats = [synth.q5k_matrix(n, k, synth.stream_key(13 + i, f"W:q4grp{k}"), fmt="q4_k")
            for i, (n, _, _) in enumerate(shapes)]
    with mlh.LMHead(max(n for n, _, _ in shapes), k, max_batch=1, device=0, fmt="q4_k") as head:
        outs = head.forward_group(_dev(torch, hidden), [(_dev(torch, w), n, sc, cp, None)
                                                        for w, (n, sc, cp) in zip(mats, shapes)],
                                  _dev(torch, gamma), synth.RMS_EPS)
        torch.cuda.synchronize()
        assert head.device_status() == 0
    for out, w, (n, sc, cp) in zip(outs, mats, shapes):
        ref = oracle.lmhead(hidden.reshape(1, k), gamma, w, sc, cp, synth.RMS_EPS, fmt="q4_k")[0]
        assert np.abs(out.cpu().numpy().astype(np.float64) - ref).max() <= TOL


@pytest.mark.parametrize("name,path", [("ffn_up_q4k", "gemv_b1"), ("ffn_down_q4k", "gemv_b1_split")])
def test_q4k_ffn_shapes(torch_cuda, name, path):
    """One block's FFN shapes in Q4_K at batch 1: gate/up [6656 -> 19968] on the
    fused kernel, down [19968 -> 6656] (78 blocks per row: three chunks of the
    6,656-column build) on the fused kernel split along K."""
    wl = synth.WORKLOADS[name]
    hidden, gamma, wq = synth.inputs_for(wl)
    got, _ = _run(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, path, want_argmax=False)
    _check(got, None, oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS, fmt="q4_k"))
