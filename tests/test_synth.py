"""The seeded input generator: its published definition and the workloads' value ranges."""
import numpy as np

import q5k_synth as synth

M64 = 0xFFFFFFFFFFFFFFFF


def _splitmix64_sequence(state, n):
    """Sequential SplitMix64 as published (Steele, Lea & Flood 2014)."""
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_counter_form_equals_sequential_splitmix64():
    key = synth.stream_key(0, "W:tiny")
    seq = _splitmix64_sequence(key, 50)
    assert [synth.draw(key, i) for i in range(50)] == seq


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.uniform(0, 1e-3, 4000), rng.uniform(2e-4, 5e-2, 4000),
        rng.uniform(0, 6.2e-5, 2000),             # fp16 subnormal range
        np.array([0.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 65504.0, 1.0 + 2.0 ** -11])])
    got = np.array([synth.f64_to_f16_bits(v) for v in vals], np.uint16)
    assert np.array_equal(got, vals.astype(np.float16).view(np.uint16))


def test_rows_are_independent_of_chunking():
    key = synth.stream_key(3, "W:chunk")
    whole = synth.q5k_rows(200, 512, key)
    part = synth.q5k_rows(50, 512, key, row_begin=120)
    assert np.array_equal(whole[120:170], part)


def test_field_ranges():
    w, f = synth.q5k_matrix(400, 1024, synth.stream_key(0, "W:ranges"), boost_rows=(5,), with_fields=True,
                            boost=50.0)
    d = f.d_bits.view(np.float16).astype(np.float64)
    dm = f.dmin_bits.view(np.float16).astype(np.float64)
    normal_rows = np.ones(400, bool)
    normal_rows[5] = False
    assert d[normal_rows].min() >= 2e-4 * (1 - 2 ** -11) and d[normal_rows].max() <= 1e-3 * (1 + 2 ** -11)
    assert d[5].min() >= 1e-2 * (1 - 2 ** -11) and d[5].max() <= 5e-2 * (1 + 2 ** -11)
    assert dm.min() >= 0.0 and dm.max() <= 1e-3 * (1 + 2 ** -11)
    assert f.sc.max() == 63 and f.m.max() == 63 and f.q.max() == 31 and f.q.min() == 0
    counts = np.bincount(f.q.ravel(), minlength=32)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()


def test_hidden_and_gamma_distributions():
    wl = synth.WORKLOADS["lmhead_b8"]
    h = synth.hidden_for(wl)
    assert h.shape == (8, 6656) and h.dtype == np.float32
    rms = np.sqrt(np.mean(h.astype(np.float64) ** 2, axis=1))
    assert rms.min() > 0.45 and rms.max() < 4.3 and rms.max() / rms.min() > 1.5
    g = synth.gamma_for(wl)
    assert abs(g.mean() - 1.0) < 0.01 and abs(g.std() - 0.1) < 0.01
    assert synth.gamma_for(synth.WORKLOADS["attn_q"]) is None


def test_workload_bytes_match_the_roofline_formula():
    for name, wl in synth.WORKLOADS.items():
        nb = wl.k // 256
        bb = {"q5_k": 176, "q4_k": 144}[wl.fmt]
        expect = wl.n_rows * nb * bb + wl.batch * wl.k * 4 + wl.batch * wl.n_rows * 4 + (wl.k * 4 if wl.norm else 0)
        assert wl.algorithmic_bytes() == expect, name
    assert synth.WORKLOADS["lmhead_b1"].algorithmic_bytes() == 925_433_088
    assert synth.WORKLOADS["lmhead_q4k_b1"].weight_bytes == 756_467_712      # the Q4_K head of Chapter 20 §20.7


def test_group_workload_bytes_and_inputs():
    """Grouped workloads: every matrix's weights in the group's format, plus one
    input row, gamma and the outputs; the generated matrices have those sizes."""
    for name, g in synth.GROUPS.items():
        bb = {"q5_k": 176, "q4_k": 144}[g.fmt]
        rows = sum(n for (_, n, _, _, _) in g.segments)
        assert g.weight_bytes == rows * (g.k // 256) * bb, name
        assert g.algorithmic_bytes() == g.weight_bytes + g.k * 4 + rows * 4 + (g.k * 4 if g.norm else 0), name
    ffn = synth.GROUPS["ffn_gate_up_q4k"]
    assert ffn.weight_bytes == 2 * 19_968 * 26 * 144                   # gate and up, Q4_K
    assert synth.GROUPS["attn_qkvg"].weight_bytes == (2 * 4096 + 2 * 256) * 26 * 176
    _, _, ws = synth.group_inputs("attn_qkvg")
    assert [w.shape for w in ws] == [(n, 26 * 176) for (_, n, _, _, _) in synth.GROUPS["attn_qkvg"].segments]
