"""GPU parity: the CUDA path (through the C-ABI) against the f64 oracle.

Bar, for every logit: |gpu - oracle| <= 2e-3 after the cap (or on the raw
values when the cap is off), and the argmax equal whenever the oracle's top-2
gap exceeds 4e-3 (2 x the tolerance, so the order is then decided).  Inputs are
the seeded workloads of q5k_synth plus randomised small shapes that span several
tiles and a ragged tail.
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


def assert_parity(got_logits, got_argmax, ref, what=""):
    got = got_logits.astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= TOL, f"{what}: max|err|={err.max():.3g} at {worst} gpu={got[worst]} ref={ref[worst]}"
    if got_argmax is not None:
        gap = oracle.top2_gap(ref)
        want = oracle.argmax_first(ref)
        for b in range(ref.shape[0]):
            a = int(got_argmax[b])
            assert 0 <= a < ref.shape[1], what
            # the returned index must hold the largest returned logit (lowest such index)
            assert a == int(np.argmax(got_logits[b])), f"{what}: argmax {a} is not the first max of the logits"
            if gap[b] > GAP:
                assert a == int(want[b]), f"{what}: row {b}: argmax {a} != oracle {want[b]} (gap {gap[b]:.3g})"
    return float(err.max())


def run_case(torch, hidden, gamma, wq, n_rows, k, scale, cap, want_argmax=True, max_batch=None, eps=1e-5):
    import q5_lm_head_gb300 as mlh
    b = hidden.shape[0]
    with mlh.LMHead(n_rows, k, max_batch=max_batch or max(b, 1), device=0) as head:
        out = head.forward(_dev(torch, hidden), _dev(torch, wq), None if gamma is None else _dev(torch, gamma),
                           eps, scale, cap, want_argmax)
        torch.cuda.synchronize()
        assert head.device_status() == 0
    if want_argmax:
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy(), None


# ------------------------------------------------------------- named workloads
@pytest.mark.parametrize("name", ["tiny", "attn_q", "attn_k", "attn_v", "attn_o"])
def test_small_workloads_full_compare(torch_cuda, name):
    wl = synth.WORKLOADS[name]
    hidden, gamma, wq = synth.inputs_for(wl)
    got, am = run_case(torch_cuda, hidden, gamma, wq, wl.n_rows, wl.k, wl.scale, wl.cap, wl.argmax)
    ref = oracle.lmhead(hidden, gamma, wq, wl.scale, wl.cap, synth.RMS_EPS)
    assert_parity(got, am, ref, name)


@pytest.fixture(scope="module")
def lm_weights(torch_cuda):
    """Full LM-head weights (202,048 x 6,656 Q5_K, boosted rows 0/777/200001) on host and device."""
    wl = synth.WORKLOADS["lmhead_b1"]
    wq = synth.weights_for(wl)
    return wq, _dev(torch_cuda, wq)


@pytest.fixture(scope="module")
def lm_weights_plain(torch_cuda):
    wl = synth.WORKLOADS["sweep_b1"]
    wq = synth.weights_for(wl)
    return wq, _dev(torch_cuda, wq)


def _full_case(torch, wl, wq_host, wq_dev):
    import q5_lm_head_gb300 as mlh
    hidden = synth.hidden_for(wl)
    gamma = synth.gamma_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=wl.batch, device=0) as head:
        logits, am = head.forward(_dev(torch, hidden), wq_dev, _dev(torch, gamma), synth.RMS_EPS, wl.scale, wl.cap)
        torch.cuda.synchronize()
        assert head.device_status() == 0
    ref = oracle.lmhead(hidden, gamma, wq_host, wl.scale, wl.cap, synth.RMS_EPS)
    return logits.cpu().numpy(), am.cpu().numpy(), ref


@pytest.mark.parametrize("name", ["lmhead_b1", "lmhead_b8"])
def test_full_lm_head(torch_cuda, lm_weights, name):
    wl = synth.WORKLOADS[name]
    got, am, ref = _full_case(torch_cuda, wl, *lm_weights)
    assert_parity(got, am, ref, name)
    # the boosted rows drive pre-cap values past the cap's knee
    for r in synth.BOOSTED_ROWS:
        assert np.abs(ref[:, r]).max() > 19.0
        assert np.abs(got[:, r]).max() <= 20.0


@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32])
def test_full_lm_head_batch_sweep(torch_cuda, lm_weights_plain, b):
    wl = synth.WORKLOADS[f"sweep_b{b}"]
    got, am, ref = _full_case(torch_cuda, wl, *lm_weights_plain)
    assert_parity(got, am, ref, wl.name)


# ------------------------------------------------------------- randomised shapes
CASES = [
    # (n_rows, k, batch, norm, cap, argmax)
    (1, 256, 1, True, 20.0, True),
    (7, 256, 3, True, 20.0, True),
    (33, 512, 2, False, 0.0, True),
    (4096, 4096, 1, True, 20.0, True),
    (4099, 6656, 1, True, 20.0, True),      # ragged tail of the 12-row tiles
    (1000, 6656, 1, False, 0.0, False),
    (153, 6656, 1, True, 20.0, True),       # even row shares: one row per CTA, two on the first
    (1825, 6656, 1, True, 20.0, True),      # shares of 12 and 13 rows: a full tile and a one-row tile
    (2000, 4096, 1, False, 0.0, False),     # shares on the 16-block build
    (4096, 6656, 5, True, 20.0, True),
    (777, 1024, 32, True, 20.0, True),
    (64, 4096, 16, True, 30.0, True),
    (19600, 1024, 4, True, 20.0, True),     # more 128-row tiles than SMs: tiles shared by two CTAs
    (57857, 1024, 3, False, 0.0, True),     # shared tiles and a one-row last tile
    (1, 512, 2, True, 20.0, True),          # one row on the tensor-core path
    (300, 16384, 1, True, 20.0, True),      # large K, batch 1: tensor-core kernel (no fused build for this K)
    (300, 16640, 1, True, 20.0, True),      # 65 blocks per row, batch 1: generic kernel
    (300, 16384, 2, True, 20.0, True),      # large K on the tensor cores (64 blocks per row)
    (129, 65536, 3, False, 0.0, True),      # 256 blocks per row, cap off
]


@pytest.mark.parametrize("n,k,b,norm,cap,want_argmax", CASES)
def test_random_shapes(torch_cuda, n, k, b, norm, cap, want_argmax):
    key = synth.stream_key(n * 131 + k * 7 + b, "W:random")
    wq = synth.q5k_matrix(n, k, key, boost_rows=(n // 2,), boost=30.0)
    hidden = (synth.normal_f64(b * k, synth.stream_key(b, f"H:random{n}")) * 1.7).astype(np.float32).reshape(b, k)
    gamma = synth.normal_f64(k, synth.stream_key(k, "G:random"), 1.0, 0.1).astype(np.float32) if norm else None
    scale = synth.LOGIT_SCALE if norm else 1.0
    got, am = run_case(torch_cuda, hidden, gamma, wq, n, k, scale, cap, want_argmax)
    ref = oracle.lmhead(hidden, gamma, wq, scale, cap, 1e-5)
    assert_parity(got, am, ref, f"n={n} k={k} b={b}")


# ------------------------------------------------------------- edge cases
def _edge_rows(k):
    """Hidden rows at the edges of the final norm: all zero (x = 0, every logit
    0), one spike of 1e4 over a 1e-3 floor (one activation dominates its
    64-column group), 1e-20 scale (mean(h^2) far below eps), 1e15 scale."""
    base = synth.normal_f64(k, synth.stream_key(11, "H:edge")).astype(np.float32)
    spike = (base * 1e-3).astype(np.float32)
    spike[k // 3] = 1e4
    return np.stack([np.zeros(k, np.float32), spike, (base * 1e-20).astype(np.float32),
                     (base * 1e15).astype(np.float32)])


@pytest.mark.parametrize("b,k,path", [(1, 6656, "gemv_b1"), (4, 6656, "gemm_tc"), (1, 13312, "gemv_b1_split")])
def test_edge_hidden_rows(torch_cuda, b, k, path):
    import q5_lm_head_gb300 as mlh
    n = 3000
    rows = _edge_rows(k)
    wq = synth.q5k_matrix(n, k, synth.stream_key(11, "W:edge"), boost_rows=(7,), boost=40.0)
    gamma = synth.normal_f64(k, synth.stream_key(11, "G:edge"), 1.0, 0.1).astype(np.float32)
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
    batches = [rows[i:i + 1] for i in range(4)] if b == 1 else [rows]
    for hidden in batches:
        got, am = run_case(torch_cuda, hidden, gamma, wq, n, k, synth.LOGIT_SCALE, synth.SOFTCAP, max_batch=b)
        ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
        assert_parity(got, am, ref, f"edge rows on {path}")
        if not hidden[0].any():                       # the zero row: every logit exactly 0, argmax 0
            assert np.all(got[0] == 0.0) and int(am[0]) == 0


def test_all_equal_logits_pick_row_zero(torch_cuda):
    n, k = 1234, 6656
    wq = np.zeros((n, k // 256 * 176), np.uint8)     # every weight is 0 -> every logit is 0
    hidden = synth.normal_f64(k, synth.stream_key(0, "H:tie")).astype(np.float32).reshape(1, k)
    got, am = run_case(torch_cuda, hidden, np.ones(k, np.float32), wq, n, k, 0.196116, 20.0)
    assert np.all(got == 0.0) and int(am[0]) == 0


def test_duplicate_max_rows_pick_the_lower_index(torch_cuda):
    n, k = 3001, 6656
    wq = synth.q5k_matrix(n, k, synth.stream_key(1, "W:dup"))
    hidden = synth.normal_f64(k, synth.stream_key(1, "H:dup")).astype(np.float32).reshape(1, k)
    ref = oracle.lmhead(hidden, None, wq, 1.0, 0.0)
    top = int(np.argmax(ref[0]))
    lo = min(top, 17)
    wq2 = wq.copy()
    wq2[lo] = wq[top]
    wq2[2999] = wq[top]
    got, am = run_case(torch_cuda, hidden, None, wq2, n, k, 1.0, 0.0)
    assert got[0, lo] == got[0, 2999]
    assert int(am[0]) == lo


def test_repeat_calls_are_deterministic_and_rearm_argmax(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    hidden2 = hidden[:, ::-1].copy()
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        l1, a1 = head.forward(_dev(torch, hidden), w_d, g_d)
        l2, a2 = head.forward(_dev(torch, hidden2), w_d, g_d)
        l3, a3 = head.forward(_dev(torch, hidden), w_d, g_d)
        torch.cuda.synchronize()
    assert torch.equal(l1, l3) and torch.equal(a1, a3)
    ref2 = oracle.lmhead(hidden2, gamma, wq, wl.scale, wl.cap)
    assert_parity(l2.cpu().numpy(), a2.cpu().numpy(), ref2, "second input")


@pytest.mark.parametrize("n,k,b", [
    (40000, 6656, 5),     # more tiles than SMs: a tile cut by a range boundary, shared by two CTAs
    (1000, 6656, 8),      # 8 tiles over 104 CTAs: each tile shared by 13
    (300, 16384, 20),     # 32 batch slots, 3 tiles over 96 CTAs
    (257, 65536, 2),      # 3 tiles over every SM, one CTA range across a tile boundary, a one-row last tile
])
def test_tensor_core_shared_tiles_repeat_bit_for_bit(torch_cuda, n, k, b):
    """CTAs share the tiles at their range boundaries and the last to arrive
    finishes them.  Whichever CTA that is, the partial sums are added in a fixed
    order, and the arrival counters re-arm for the next call, so repeated
    forwards (alternating inputs) give the same bits."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wq = synth.q5k_matrix(n, k, synth.stream_key(2, "W:shared"), boost_rows=(n // 3,), boost=40.0)
    hidden = synth.normal_f64(b * k, synth.stream_key(2, "H:shared")).astype(np.float32).reshape(b, k)
    gamma = synth.normal_f64(k, synth.stream_key(2, "G:shared"), 1.0, 0.1).astype(np.float32)
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == "gemm_tc"
        h1, h2 = _dev(torch, hidden), _dev(torch, hidden[::-1].copy())
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        outs = [[t.clone() for t in head.forward(h, w_d, g_d)] for h in (h1, h2, h1, h2, h1)]
        torch.cuda.synchronize()
        assert head.device_status() == 0
    for i in (2, 4):
        assert torch.equal(outs[0][0], outs[i][0]) and torch.equal(outs[0][1], outs[i][1])
    assert torch.equal(outs[1][0], outs[3][0])
    ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
    assert_parity(outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy(), ref, f"shared tiles n={n} k={k} b={b}")


def test_forward_host_matches_device_forward(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=4, device=0) as head:
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        ld, ad = head.forward(_dev(torch, hidden), w_d, g_d)
        # page-locked outputs (written by the kernels through the host mapping)
        lh, ah = head.forward_host(torch.from_numpy(hidden).pin_memory(), w_d, g_d)
        # pageable outputs and input (staged in device memory, copied back)
        lp = torch.full((1, wl.n_rows), float("nan"))
        ap = torch.full((1,), -1, dtype=torch.int32)
        head.forward_host(torch.from_numpy(hidden.copy()), w_d, g_d, logits_host=lp, argmax_host=ap)
        # argmax only, into page-locked memory
        ao = torch.full((1,), -1, dtype=torch.int32).pin_memory()
        st = mlh.muse_lmhead_forward_host(head.handle, torch.from_numpy(hidden).pin_memory().data_ptr(), 1,
                                          g_d.data_ptr(), synth.RMS_EPS, w_d.data_ptr(), synth.LOGIT_SCALE,
                                          synth.SOFTCAP, None, ao.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
    assert torch.equal(ld.cpu(), lh) and torch.equal(ad.cpu(), ah)
    assert torch.equal(ld.cpu(), lp) and torch.equal(ad.cpu(), ap) and torch.equal(ad.cpu(), ao)


@pytest.mark.parametrize("b,k,path", [(4, 6656, "gemm_tc"), (1, 6656, "gemv_b1"), (1, 13312, "gemv_b1_split")])
def test_forward_host_batches_and_repeats(torch_cuda, b, k, path):
    """Host-buffer forwards on the batch-1 (whole and split along K) and
    tensor-core paths, three calls in a row with changing rows: each sees its
    own rows and matches the device forward bit for bit and the oracle within
    the bar."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n = 5000
    wq = synth.q5k_matrix(n, k, synth.stream_key(6, "W:host"), boost_rows=(17,), boost=40.0)
    gamma = synth.normal_f64(k, synth.stream_key(6, "G:host"), 1.0, 0.1).astype(np.float32)
    rows = [synth.normal_f64(b * k, synth.stream_key(6 + i, "H:host")).astype(np.float32).reshape(b, k)
            for i in range(3)]
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
        w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
        outs = [[t.clone() for t in head.forward_host(torch.from_numpy(h).pin_memory(), w_d, g_d)] for h in rows]
        dev = [head.forward(_dev(torch, h), w_d, g_d) for h in rows]
        torch.cuda.synchronize()
        assert head.device_status() == 0
    for (lh, ah), (ld, ad), h in zip(outs, dev, rows):
        assert torch.equal(ld.cpu(), lh) and torch.equal(ad.cpu(), ah)
        assert_parity(lh.numpy(), ah.numpy(), oracle.lmhead(h, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP,
                                                            synth.RMS_EPS), f"host rows b={b}")


def test_two_handles_on_two_streams(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    h2 = np.ascontiguousarray(-hidden)
    w_d, g_d = _dev(torch, wq), _dev(torch, gamma)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with mlh.LMHead(wl.n_rows, wl.k, 1, 0) as a, mlh.LMHead(wl.n_rows, wl.k, 1, 0) as b:
        x1, x2 = _dev(torch, hidden), _dev(torch, h2)
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            r1 = a.forward(x1, w_d, g_d)
        with torch.cuda.stream(s2):
            r2 = b.forward(x2, w_d, g_d)
        torch.cuda.synchronize()
    for (l, am), h in ((r1, hidden), (r2, h2)):
        assert_parity(l.cpu().numpy(), am.cpu().numpy(), oracle.lmhead(h, gamma, wq, wl.scale, wl.cap), "stream")


def test_invalid_arguments_launch_nothing(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    n, k = 64, 512
    wq = _dev(torch, synth.q5k_matrix(n, k, synth.stream_key(0, "W:inv")))
    hid = torch.randn(2, k, device="cuda")
    out = torch.full((2, n), 7.0, device="cuda")
    am = torch.full((2,), -5, dtype=torch.int32, device="cuda")
    with mlh.LMHead(n, k, max_batch=2, device=0) as head:
        h = head.handle
        F = mlh.muse_lmhead_forward
        s = torch.cuda.current_stream().cuda_stream
        assert F(h, hid.data_ptr(), 3, None, 1e-5, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), am.data_ptr(), s) == -3
        assert F(h, hid.data_ptr(), 0, None, 1e-5, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), am.data_ptr(), s) == -3
        assert F(h, hid.data_ptr() + 4, 1, None, 1e-5, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), am.data_ptr(), s) == -4
        assert F(h, hid.data_ptr(), 1, None, 1e-5, wq.data_ptr() + 8, 1.0, 0.0, out.data_ptr(), am.data_ptr(), s) == -4
        assert F(h, hid.data_ptr(), 1, None, 1e-5, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), am.data_ptr() + 2, s) == -4
        assert F(h, hid.data_ptr(), 1, None, 1e-5, wq.data_ptr(), float("nan"), 0.0, out.data_ptr(), None, s) == -5
        assert F(h, hid.data_ptr(), 1, hid.data_ptr(), -1.0, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), None, s) == -5
        assert F(h, 0, 1, None, 1e-5, wq.data_ptr(), 1.0, 0.0, out.data_ptr(), None, s) == -1
        torch.cuda.synchronize()
        assert head.device_status() == 0
    assert torch.all(out == 7.0) and torch.all(am == -5)


def test_init_rejects_bad_device(torch_cuda):
    import q5_lm_head_gb300 as mlh
    with pytest.raises(mlh.MuseError):
        mlh.muse_lmhead_init(999, 10, 256, 1)
