"""GPU parity of the batch-1 kernel split along K (path "gemv_b1_split").

A K of S chunks of a built width (S x 6,656 or S x 4,096 columns, S = 2..16)
runs the fused batch-1 kernel with each CTA on one column chunk; the S chunk
partials of every 12-row tile meet in the workspace and the last CTA to arrive
adds them in chunk order, then applies the final norm's result, scale, soft
cap and argmax ("Chapter 20 — Final norm, LM head, and the soft cap": §20.1
the computation, §20.3 the block format).  The RMS factor of the final norm
covers the whole row, all chunks.

A Q4_K matrix of at most three chunks whose rows, shared evenly over the SMs,
give every CTA at most eight 12-row tiles runs the chunks inside each CTA
instead (the K loop): a CTA streams all chunks of its own rows, one after the
other, and adds the chunk sums of a row in chunk order in registers.

Bar as everywhere: |gpu - oracle| <= 2e-3 on every logit (after the cap, raw
with it off); the argmax equal to the oracle's where its top-2 gap exceeds
4e-3.  Also: logprobs, repeated forwards bit for bit (whichever CTA finishes a
tile), the counters' re-arming after a recorded fault, and the path choice.
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


def _inputs(n, k, norm, fmt, seed):
    wq = synth.q5k_matrix(n, k, synth.stream_key(seed, f"W:split{n}:{k}"), boost_rows=(n // 2,), boost=40.0,
                          fmt=fmt)
    hidden = (synth.normal_f64(k, synth.stream_key(seed, f"H:split{k}")) * 1.3).astype(np.float32).reshape(1, k)
    gamma = synth.normal_f64(k, synth.stream_key(seed, f"G:split{k}"), 1.0, 0.1).astype(np.float32) if norm else None
    return hidden, gamma, wq


def _check(got, am, ref, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= TOL, f"{what}: max|err|={err.max():.3g}"
    if am is not None:
        assert am[0] == int(np.argmax(got[0]))
        if oracle.top2_gap(ref)[0] > GAP:
            assert am[0] == oracle.argmax_first(ref)[0], what


SHAPES = [
    # (n_rows, k, fmt, norm, cap)
    (4099, 13312, "q5_k", True, 20.0),      # 2 chunks of 6,656; a 7-row last tile
    (300, 16384, "q5_k", True, 20.0),       # 4 chunks of 4,096
    (1, 13312, "q5_k", True, 20.0),         # one row: one tile, one CTA per chunk
    (25, 8192, "q5_k", False, 0.0),         # 2 chunks of 4,096, no norm, cap off
    (97, 106496, "q5_k", True, 20.0),       # 16 chunks of 6,656
    (2000, 19968, "q5_k", True, 20.0),      # 3 chunks (the FFN down width)
    (777, 13312, "q4_k", True, 20.0),
    (130, 32768, "q4_k", False, 0.0),       # 8 chunks of 4,096
    (50, 65536, "q5_k", True, 20.0),        # 16 chunks of 4,096: the most the split build takes
    # the K loop (Q4_K, at most 3 chunks, at most 96 rows per CTA)
    (6656, 19968, "q4_k", True, 20.0),      # the FFN down shape: 44 rows per CTA, 3 chunks of 6,656
    (6656, 19968, "q4_k", False, 0.0),
    (2000, 12288, "q4_k", True, 20.0),      # 3 chunks of 4,096
    (1, 19968, "q4_k", True, 20.0),         # one row, one CTA
    (153, 19968, "q4_k", True, 20.0),       # one CTA with two rows, the others one
    (14592, 8192, "q4_k", True, 20.0),      # 96 rows per CTA: the most the K loop takes
    (14593, 8192, "q4_k", True, 20.0),      # one row more: the cross-CTA hand-off
]


@pytest.mark.parametrize("n,k,fmt,norm,cap", SHAPES)
def test_split_k_parity(torch_cuda, n, k, fmt, norm, cap):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    hidden, gamma, wq = _inputs(n, k, norm, fmt, 21)
    scale = synth.LOGIT_SCALE if norm else 1.0
    with mlh.LMHead(n, k, max_batch=1, device=0, fmt=fmt) as head:
        assert head.path_name(1) == "gemv_b1_split"
        assert head.launches_per_forward(1, norm) == 1
        logits, am = head.forward(_dev(torch, hidden), _dev(torch, wq),
                                  None if gamma is None else _dev(torch, gamma), synth.RMS_EPS, scale, cap, True)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        got, am = logits.cpu().numpy(), am.cpu().numpy()
    ref = oracle.lmhead(hidden, gamma, wq, scale, cap, synth.RMS_EPS, fmt=fmt)
    _check(got, am, ref, f"n={n} k={k} {fmt}")


def test_split_k_logprobs(torch_cuda):
    """Logprobs on the split path: the normaliser comes from the separate pass
    over the finished logits (which CTA finishes a row varies between runs)."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 2000, 19968
    hidden, gamma, wq = _inputs(n, k, True, "q5_k", 22)
    with mlh.LMHead(n, k, max_batch=1, device=0) as head:
        assert head.path_name(1) == "gemv_b1_split"
        h, w, g = _dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma)
        lp, lse, am = head.forward_logprobs(h, w, g, synth.RMS_EPS, synth.LOGIT_SCALE, synth.SOFTCAP, True)
        logits, am2 = head.forward(h, w, g, synth.RMS_EPS, synth.LOGIT_SCALE, synth.SOFTCAP, True)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        lp, lse, am, logits, am2 = (t.cpu().numpy() for t in (lp, lse, am, logits, am2))
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
    ref_lp, ref_lse = oracle.log_softmax(ref)
    assert np.abs(lp.astype(np.float64) - ref_lp).max() <= TOL
    assert np.abs(lse.astype(np.float64) - ref_lse).max() <= TOL
    assert np.array_equal(am, am2)
    assert np.abs((lp + lse[:, None]) - logits).max() <= 1e-4 * max(1.0, float(np.abs(lse).max()))


def test_split_k_repeats_bit_for_bit(torch_cuda):
    """Which chunk CTA finishes a tile varies from run to run; the partials are
    added in chunk order, so alternating inputs give the same bits each time,
    and the per-tile counters re-arm."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 3001, 19968
    hidden, gamma, wq = _inputs(n, k, True, "q5_k", 23)
    with mlh.LMHead(n, k, max_batch=1, device=0) as head:
        h1, h2 = _dev(torch, hidden), _dev(torch, hidden[:, ::-1].copy())
        w, g = _dev(torch, wq), _dev(torch, gamma)
        outs = [[t.clone() for t in head.forward(h, w, g)] for h in (h1, h2, h1, h2, h1)]
        torch.cuda.synchronize()
        assert head.device_status() == 0
    for i in (2, 4):
        assert torch.equal(outs[0][0], outs[i][0]) and torch.equal(outs[0][1], outs[i][1])
    assert torch.equal(outs[1][0], outs[3][0])
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
    _check(outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy(), ref, "repeat")


def test_split_k_after_clear_device_status(torch_cuda):
    """The bounded-wait self-test records a fault; the clear re-arms the status
    word and the chunk counters, and the next forward is correct."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 500, 13312
    hidden, gamma, wq = _inputs(n, k, True, "q5_k", 24)
    with mlh.LMHead(n, k, max_batch=1, device=0) as head:
        assert mlh.muse_lmhead_selftest_wait_timeout(head.handle) == 0
        torch.cuda.synchronize()
        assert head.device_status() & mlh.STATUS_WAIT_TIMEOUT
        assert mlh.muse_lmhead_clear_device_status(head.handle) == 0
        torch.cuda.synchronize()
        assert head.device_status() == 0
        logits, am = head.forward(_dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma))
        torch.cuda.synchronize()
        assert head.device_status() == 0
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
    _check(logits.cpu().numpy(), am.cpu().numpy(), ref, "after clear")


def test_k_loop_repeats_and_logprobs(torch_cuda):
    """The K loop: the same bits from forward to forward with alternating
    inputs, and logprobs from the separate pass over its logits."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 6656, 19968
    hidden, gamma, wq = _inputs(n, k, True, "q4_k", 25)
    with mlh.LMHead(n, k, max_batch=1, device=0, fmt="q4_k") as head:
        assert head.path_name(1) == "gemv_b1_split"
        h1, h2 = _dev(torch, hidden), _dev(torch, hidden[:, ::-1].copy())
        w, g = _dev(torch, wq), _dev(torch, gamma)
        outs = [[t.clone() for t in head.forward(h, w, g)] for h in (h1, h2, h1, h2, h1)]
        lp, lse, am = head.forward_logprobs(h1, w, g, synth.RMS_EPS, synth.LOGIT_SCALE, synth.SOFTCAP, True)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        lp, lse, am = (t.cpu().numpy() for t in (lp, lse, am))
    for i in (2, 4):
        assert torch.equal(outs[0][0], outs[i][0]) and torch.equal(outs[0][1], outs[i][1])
    assert torch.equal(outs[1][0], outs[3][0])
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS, fmt="q4_k")
    _check(outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy(), ref, "k loop")
    ref_lp, ref_lse = oracle.log_softmax(ref)
    assert np.abs(lp.astype(np.float64) - ref_lp).max() <= TOL
    assert np.abs(lse.astype(np.float64) - ref_lse).max() <= TOL
    assert am[0] == int(outs[0][1].cpu().numpy()[0])


@pytest.mark.parametrize("n,k,b,path", [
    (1000, 13312, 1, "gemv_b1_split"),
    (1000, 13312, 4, "gemm_tc"),                   # batches above 1 stay on the tensor cores
    (2 ** 25 + 1, 13312, 1, "gemm_tc"),            # n_rows * chunks above 2^26: no partial-sum buffer
    (1000, 17 * 6656, 1, "gemm_tc"),               # 17 chunks: more than the split build takes
    (1000, 8192, 1, "gemv_b1_split"),              # 32 blocks: 2 chunks of 16
    (1000, 39 * 256, 1, "gemv_generic"),           # 39 blocks: neither chunk width, odd
])
def test_split_k_path_choice(torch_cuda, n, k, b, path):
    import q5_lm_head_gb300 as mlh
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
        if b > 1:
            assert head.path_name(1) == "gemv_b1_split"
