"""Weight matrices larger than 4 GiB: every byte offset past 2^32 must be
formed in 64 bits (the batch-1 kernel's bulk-copy sources, the tensor-core
kernel's tensor map and TMA row coordinates, the split kernel's row-strided
chunk copies).  1,600,000 rows x 4,096 columns of Q5_K is 4.5 GB, and so is
800,000 x 8,192; rows near the end are boosted so that the argmax lies past the
4 GiB mark.  Every logit is compared with the f64 oracle (max-abs 2e-3 after
the cap); the argmax as everywhere (the oracle's where its top-2 gap exceeds
4e-3, else the first maximum of the returned logits).
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


def _case(torch, n, k, batches):
    import q5_lm_head_gb300 as mlh
    wq = synth.q5k_matrix(n, k, synth.stream_key(31, f"W:large{k}"), boost_rows=(n // 2, n - 5, n - 1),
                          boost=40.0)
    assert wq.nbytes > 2 ** 32
    gamma = synth.normal_f64(k, synth.stream_key(31, "G:large"), 1.0, 0.1).astype(np.float32)
    w_d = torch.from_numpy(wq).to("cuda")
    g_d = torch.from_numpy(gamma).to("cuda")
    for b, path in batches:
        hidden = synth.normal_f64(b * k, synth.stream_key(31 + b, f"H:large{k}")).astype(np.float32).reshape(b, k)
        with mlh.LMHead(n, k, max_batch=b, device=0) as head:
            assert head.path_name(b) == path
            logits, am = head.forward(torch.from_numpy(hidden).to("cuda"), w_d, g_d)
            torch.cuda.synchronize()
            assert head.device_status() == 0
            got, am = logits.cpu().numpy(), am.cpu().numpy()
        ref = oracle.lmhead(hidden, gamma, wq, synth.LOGIT_SCALE, synth.SOFTCAP, synth.RMS_EPS)
        err = np.abs(got.astype(np.float64) - ref)
        assert err.max() <= TOL, f"{path}: max|err|={err.max():.3g} at row {int(np.argmax(err) % n)}"
        gap, want = oracle.top2_gap(ref), oracle.argmax_first(ref)
        for r in range(b):
            assert am[r] == int(np.argmax(got[r])), path
            if gap[r] > GAP:
                assert am[r] == want[r], path
    del w_d
    torch.cuda.empty_cache()


def test_weights_past_4gib_batch1_and_tensor_cores(torch_cuda):
    _case(torch_cuda, 1_600_000, 4096, [(1, "gemv_b1"), (2, "gemm_tc")])


def test_weights_past_4gib_split_along_k(torch_cuda):
    _case(torch_cuda, 800_000, 8192, [(1, "gemv_b1_split")])
