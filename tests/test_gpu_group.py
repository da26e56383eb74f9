"""GPU parity of the grouped batch-1 forward (muse_lmhead_forward_group): up
to four Q5_K matrices against one normed input row in one launch — the
attention block's Q/K/V/gate group ("Chapter 9 — The Muse Glimmer
architecture", Figure 9.1 and §9.8) — against the f64 oracle, matrix by matrix.

Same bar as the LM head: |gpu - oracle| <= 2e-3 on every output (after the cap,
raw when the cap is off).
"""
import numpy as np
import pytest

import oracle
import q5k_synth as synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


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


def _run_group(torch, k, hidden, gamma, mats, eps=synth.RMS_EPS, fmt="q5_k"):
    """mats: list of (weights_host, n_rows, scale, cap).  Returns host outputs."""
    import q5_lm_head_gb300 as mlh
    with mlh.LMHead(1, k, max_batch=1, device=0, fmt=fmt) as head:
        segs = [(_dev(torch, w), n, sc, cp, None) for (w, n, sc, cp) in mats]
        outs = head.forward_group(_dev(torch, hidden), segs, None if gamma is None else _dev(torch, gamma), eps)
        torch.cuda.synchronize()
        assert head.device_status() == 0
        return [o.cpu().numpy() for o in outs]


def _check(got, ref, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert err.max() <= TOL, f"{what}: max|err|={err.max():.3g} at {int(np.argmax(err))}"


def test_attention_qkvg_group(torch_cuda):
    g = synth.GROUPS["attn_qkvg"]
    hidden, gamma, ws = synth.group_inputs(g)
    mats = [(w, n, sc, cp) for w, (_, n, _, sc, cp) in zip(ws, g.segments)]
    outs = _run_group(torch_cuda, g.k, hidden, gamma, mats)
    for (name, n, _, sc, cp), w, got in zip(g.segments, ws, outs):
        ref = oracle.lmhead(hidden, gamma, w, sc, cp, synth.RMS_EPS)[0]
        assert got.shape == (n,)
        _check(got, ref, name)


def test_ffn_gate_up_q4k_group(torch_cuda):
    """The FFN's gate and up projections (two 19,968 x 6,656 Q4_K matrices on
    the ffn_norm-normalised row) in one launch."""
    g = synth.GROUPS["ffn_gate_up_q4k"]
    hidden, gamma, ws = synth.group_inputs(g)
    mats = [(w, n, sc, cp) for w, (_, n, _, sc, cp) in zip(ws, g.segments)]
    outs = _run_group(torch_cuda, g.k, hidden, gamma, mats, fmt=g.fmt)
    for (name, n, _, sc, cp), w, got in zip(g.segments, ws, outs):
        ref = oracle.lmhead(hidden, gamma, w, sc, cp, synth.RMS_EPS, fmt=g.fmt)[0]
        assert got.shape == (n,)
        _check(got, ref, name)


def test_group_from_host_buffers_matches_the_device_call(torch_cuda):
    """muse_lmhead_forward_group_host: pinned outputs (written by the kernel
    through the host mapping), pageable outputs (staged, copied back; the
    staging buffer grows on the second call), the same bits as the device call."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    k = 6656
    rows = (300, 5000, 12)
    hidden = synth.normal_f64(k, synth.stream_key(13, "H:grouphost")).astype(np.float32).reshape(1, k)
    gamma = synth.normal_f64(k, synth.stream_key(13, "G:grouphost"), 1.0, 0.1).astype(np.float32)
    ws = [_dev(torch, synth.q5k_matrix(n, k, synth.stream_key(13, f"W:grouphost{n}"))) for n in rows]
    caps = ((1.0, 0.0), (synth.LOGIT_SCALE, synth.SOFTCAP), (0.5, 2.0))
    with mlh.LMHead(1, k, max_batch=1, device=0) as head:
        g_d = _dev(torch, gamma)
        dev = head.forward_group(_dev(torch, hidden), [(w, n, sc, cp, None) for w, n, (sc, cp) in zip(ws, rows, caps)],
                                 g_d)
        h_pin = torch.from_numpy(hidden).pin_memory()
        pinned = head.forward_group_host(h_pin, [(w, n, sc, cp, None) for w, n, (sc, cp) in zip(ws, rows, caps)],
                                         g_d)
        small = head.forward_group_host(torch.from_numpy(hidden.copy()),       # pageable, one segment
                                        [(ws[0], rows[0], 1.0, 0.0, torch.zeros(rows[0]))], g_d)
        mixed = [torch.zeros(rows[0]), torch.zeros(rows[1]).pin_memory(), torch.zeros(rows[2])]
        head.forward_group_host(h_pin, [(w, n, sc, cp, o) for w, n, (sc, cp), o in zip(ws, rows, caps, mixed)], g_d)
        torch.cuda.synchronize()
        assert head.device_status() == 0
    for d, p, m in zip(dev, pinned, mixed):
        assert torch.equal(d.cpu(), p) and torch.equal(d.cpu(), m)
    assert torch.equal(dev[0].cpu(), small[0])
    for i, (n, (sc, cp)) in enumerate(zip(rows, caps)):
        ref = oracle.lmhead(hidden, gamma, ws[i].cpu().numpy(), sc, cp, synth.RMS_EPS)[0]
        _check(pinned[i].numpy(), ref, f"segment {i}")


@pytest.mark.parametrize("k,rows,caps,norm", [
    (6656, (13, 1, 4099, 256), ((0.5, 3.0), (1.0, 0.0), (synth.LOGIT_SCALE, synth.SOFTCAP), (2.0, 0.0)), True),
    (6656, (25, 12), ((1.0, 0.0), (0.25, 1.0)), False),
    (4096, (300, 7, 12), ((1.0, 0.0), (1.0, 5.0), (0.5, 0.0)), True),
    (4096, (6656,), ((1.0, 0.0),), False),
])
def test_ragged_segments_own_scale_and_cap(torch_cuda, k, rows, caps, norm):
    rng = np.random.default_rng(sum(rows) + k)
    hidden = rng.standard_normal((1, k)).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32) if norm else None
    ws = [synth.q5k_matrix(n, k, synth.stream_key(7, f"W:group{i}:{n}:{k}")) for i, n in enumerate(rows)]
    mats = [(w, n, sc, cp) for w, n, (sc, cp) in zip(ws, rows, caps)]
    outs = _run_group(torch_cuda, k, hidden, gamma, mats)
    for i, (w, n, (sc, cp)) in enumerate(zip(ws, rows, caps)):
        ref = oracle.lmhead(hidden, gamma, w, sc, cp, synth.RMS_EPS)[0]
        _check(outs[i], ref, f"segment {i} ({n} rows)")


def test_one_segment_equals_the_lm_head_forward(torch_cuda):
    """Same kernel arithmetic per row: the grouped call and the plain forward
    give bit-identical outputs."""
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    wl = synth.WORKLOADS["tiny"]
    hidden, gamma, wq = synth.inputs_for(wl)
    with mlh.LMHead(wl.n_rows, wl.k, max_batch=1, device=0) as head:
        h, g, w = _dev(torch, hidden), _dev(torch, gamma), _dev(torch, wq)
        plain = head.forward(h, w, g, synth.RMS_EPS, wl.scale, wl.cap, False)
        grouped = head.forward_group(h, [(w, wl.n_rows, wl.scale, wl.cap, None)], g, synth.RMS_EPS)[0]
        torch.cuda.synchronize()
        assert torch.equal(plain.reshape(-1), grouped)


def test_group_invalid_arguments_launch_nothing(torch_cuda):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    k, n = 6656, 64
    hidden = torch.zeros((k,), dtype=torch.float32, device="cuda")
    w = _dev(torch, synth.q5k_matrix(n, k, synth.stream_key(0, "W:group-invalid")))
    out = torch.full((n + 8,), 7.0, dtype=torch.float32, device="cuda")
    with mlh.LMHead(1, k, max_batch=1, device=0) as head:
        h = head.handle
        wp, op, hp = w.data_ptr(), out.data_ptr(), hidden.data_ptr()
        call = mlh.muse_lmhead_forward_group
        assert call(h, hp, None, 1e-5, [], None) == -2                                   # no segment
        assert call(h, hp, None, 1e-5, [(wp, n, op, 1.0, 0.0)] * 5, None) == -2           # more than four
        assert call(h, hp, None, 1e-5, [(wp, 0, op, 1.0, 0.0)], None) == -2               # n_rows < 1
        assert call(h, hp, None, 1e-5, [(None, n, op, 1.0, 0.0)], None) == -1             # null weights
        assert call(h, hp, None, 1e-5, [(wp, n, None, 1.0, 0.0)], None) == -1             # null out
        assert call(h, None, None, 1e-5, [(wp, n, op, 1.0, 0.0)], None) == -1             # null hidden
        assert call(h, hp, None, 1e-5, [(wp + 8, n, op, 1.0, 0.0)], None) == -4           # weights alignment
        assert call(h, hp, None, 1e-5, [(wp, n, op + 2, 1.0, 0.0)], None) == -4           # out alignment
        assert call(h, hp + 4, None, 1e-5, [(wp, n, op, 1.0, 0.0)], None) == -4           # hidden alignment
        assert call(h, hp, None, 1e-5, [(wp, n, op, float("nan"), 0.0)], None) == -5      # scale
        assert call(h, hp, hp, -1.0, [(wp, n, op, 1.0, 0.0)], None) == -5                 # eps
        torch.cuda.synchronize()
    with mlh.LMHead(1, 512, max_batch=1, device=0) as head512:                            # K with no fused kernel
        assert mlh.muse_lmhead_forward_group(head512.handle, hp, None, 1e-5, [(wp, n, op, 1.0, 0.0)],
                                             None) == -2
    # the host-buffer form checks the same arguments (its input row and outputs are host memory)
    h_host = torch.zeros((k,), dtype=torch.float32)
    o_host = torch.full((n,), 7.0, dtype=torch.float32)
    hh, oh = h_host.data_ptr(), o_host.data_ptr()
    with mlh.LMHead(1, k, max_batch=1, device=0) as head:
        call = mlh.muse_lmhead_forward_group_host
        assert call(head.handle, hh, None, 1e-5, [], None) == -2                          # no segment
        assert call(head.handle, None, None, 1e-5, [(wp, n, oh, 1.0, 0.0)], None) == -1   # null hidden
        assert call(head.handle, hh, None, 1e-5, [(wp, n, None, 1.0, 0.0)], None) == -1   # null out
        assert call(head.handle, hh, None, 1e-5, [(wp + 8, n, oh, 1.0, 0.0)], None) == -4  # weights alignment
        assert call(head.handle, hh, None, 1e-5, [(wp, n, oh + 2, 1.0, 0.0)], None) == -4  # out alignment
        assert call(head.handle, hh, hp, float("inf"), [(wp, n, oh, 1.0, 0.0)], None) == -5  # eps
    with mlh.LMHead(1, 512, max_batch=1, device=0) as head512:
        assert mlh.muse_lmhead_forward_group_host(head512.handle, hh, None, 1e-5, [(wp, n, oh, 1.0, 0.0)],
                                                  None) == -2
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(o_host == 7.0)                             # nothing was written
