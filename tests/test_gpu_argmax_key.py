"""GPU checks of the argmax key (muse_lmhead_set_argmax_key).

The cap is strictly increasing, so greedy selection does not depend on it in
exact arithmetic ("Chapter 20 — Final norm, LM head, and the soft cap", §20.2).
In f32, large pre-cap values collapse onto the same capped float (20.0f from
about 200 up), so the capped key sees ties among them and returns the lowest
index; the pre-cap key (scale * raw) keeps their order.

Each case boosts six rows (d x 60) so that several of them saturate on the
positive side for at least one batch row, then checks on every kernel path:
  * capped key (the default): the index of the first maximum of the returned
    logits;
  * pre-cap key: the oracle's argmax of scale * raw wherever the oracle's
    pre-cap top-2 gap exceeds 4e-3, and a different index from the capped key
    on the saturated ties;
  * the logits do not depend on the key (bit for bit), and the logprobs
    forward ranks with the same key.
"""
import numpy as np
import pytest

import oracle
import q5k_synth as synth

pytestmark = pytest.mark.gpu

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


def _inputs(n, k, b, seed):
    rows = tuple(sorted({(n * i) // 7 + 3 for i in range(6)}))
    wq = synth.q5k_matrix(n, k, synth.stream_key(seed, f"W:precap{n}:{k}"), boost_rows=rows, boost=60.0)
    hidden = synth.normal_f64(b * k, synth.stream_key(seed, f"H:precap{k}")).astype(np.float32).reshape(b, k)
    gamma = synth.normal_f64(k, synth.stream_key(seed, "G:precap"), 1.0, 0.1).astype(np.float32)
    return hidden, gamma, wq


@pytest.mark.parametrize("n,k,b,seed,path", [
    (3000, 6656, 1, 0, "gemv_b1"),
    (3000, 13312, 1, 3, "gemv_b1_split"),
    (3000, 6656, 4, 0, "gemm_tc"),
    (3000, 6912, 2, 2, "gemv_generic"),       # 27 blocks per row
])
def test_capped_and_precap_argmax_keys(torch_cuda, n, k, b, seed, path):
    import q5_lm_head_gb300 as mlh
    torch = torch_cuda
    hidden, gamma, wq = _inputs(n, k, b, seed)
    with mlh.LMHead(n, k, max_batch=b, device=0) as head:
        assert head.path_name(b) == path
        h, w, g = _dev(torch, hidden), _dev(torch, wq), _dev(torch, gamma)
        l_cap, a_cap = [t.clone() for t in head.forward(h, w, g)]
        head.set_argmax_key("precap")
        l_pre, a_pre = [t.clone() for t in head.forward(h, w, g)]
        _, _, a_lp = [t.clone() for t in head.forward_logprobs(h, w, g)]
        head.set_argmax_key("capped")
        l_again, a_again = [t.clone() for t in head.forward(h, w, g)]
        torch.cuda.synchronize()
        assert head.device_status() == 0
        with pytest.raises(ValueError):
            head.set_argmax_key("raw")
        assert mlh.muse_lmhead_set_argmax_key(head.handle, 2) == -5
    assert torch.equal(l_cap, l_pre) and torch.equal(l_cap, l_again) and torch.equal(a_cap, a_again)
    logits = l_cap.cpu().numpy()
    a_cap, a_pre, a_lp = a_cap.cpu().numpy(), a_pre.cpu().numpy(), a_lp.cpu().numpy()
    out, raw = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS, want_raw=True)
    assert np.abs(logits.astype(np.float64) - out).max() <= 2e-3
    v = raw * synth.LOGIT_SCALE                       # the pre-cap values
    gap, want = oracle.top2_gap(v), oracle.argmax_first(v)
    for r in range(b):
        assert a_cap[r] == int(np.argmax(logits[r]))  # first maximum of the returned logits
        if gap[r] > GAP:
            assert a_pre[r] == want[r], f"row {r}"
        assert a_lp[r] == a_pre[r]
    assert np.any(a_cap != a_pre), "no saturated tie separated the two keys"
