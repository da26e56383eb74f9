"""Pins of the f64 oracle against what the pages and mathematics fix.

Each test ties one part of the oracle to something other than the oracle
itself: values printed in "Chapter 20 — Final norm, LM head, and the soft cap"
(§20.3 byte bill, §20.7 worked soft-cap example), closed forms of RMSNorm,
hand-built Q5_K blocks, numpy's float16 decoding, a dense numpy matmul over
weights rebuilt from the generator's drawn fields (not from the oracle's
parser), and the order invariance of the cap (§20.2).
"""
import math

import numpy as np
import pytest

import oracle
import q5k_synth as synth
from conftest import read_golden

CAP = 20.0
SCALE = 0.196116


# ----------------------------------------------------------------- soft cap
def test_softcap_worked_values_chapter20():
    rows = read_golden("softcap_worked_example.txt")
    vals = [r for r in rows if r[0] == "value"]
    gaps = [r for r in rows if r[0] == "gap"]
    assert len(vals) == 4 and len(gaps) == 2
    for _, v, printed in vals:
        got = oracle.scale_softcap(float(v), 1.0, CAP)
        assert abs(got - float(printed)) <= 5e-4, (v, got, printed)
    for _, a, b, printed_gap, raw_gap in gaps:
        ga = oracle.scale_softcap(float(a), 1.0, CAP) - oracle.scale_softcap(float(b), 1.0, CAP)
        assert abs(ga - float(printed_gap)) <= 1e-3
        assert abs((float(a) - float(b)) - float(raw_gap)) == 0.0


def test_softcap_strictly_increasing_and_bounded():
    v = np.linspace(-340.0, 340.0, 20001)
    out = np.array([oracle.scale_softcap(x, 1.0, CAP) for x in v])
    assert np.all(np.diff(out) >= 0.0)
    mid = np.abs(v) < 200.0   # well inside binary64 resolution of the flat tails
    assert np.all(np.diff(out[mid]) > 0.0)
    assert np.all(np.abs(out[mid]) < CAP)
    assert np.all(np.abs(out) <= CAP)


def test_softcap_is_identity_near_zero():
    # 20*tanh(v/20) = v - v^3/1200 + ...: within the cubic term for small v
    for v in (1e-6, -3e-4, 0.01, -0.25, 0.5, 1.0):
        got = oracle.scale_softcap(v, 1.0, CAP)
        assert abs(got - v) <= abs(v) ** 3 / 1200.0 * 1.0001 + 1e-18


def test_cap_disabled_leaves_scaled_value():
    for cap in (0.0, -1.0):
        for raw in (-1234.5, -1.0, 0.0, 3.25, 1e6):
            assert oracle.scale_softcap(raw, SCALE, cap) == raw * SCALE


def test_scale_is_applied_before_the_cap():
    # Chapter 9 §9.10: scale first, cap second; the other order caps at 0.196*20
    raw = 100.0
    right = oracle.scale_softcap(raw, SCALE, CAP)
    assert abs(right - 20.0 * math.tanh(raw * SCALE / 20.0)) < 1e-12
    wrong = SCALE * 20.0 * math.tanh(raw / 20.0)
    assert right > 15.0 and wrong < 4.0


def test_logit_scale_is_inverse_sqrt26_to_five_decimals():
    # Chapter 20 §20.5: 0.196116 is 1/sqrt(26) to five decimals
    assert abs(SCALE - 1.0 / math.sqrt(26.0)) < 5e-6


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row_closed_form():
    k = 6656
    c = 0.75
    h = np.full(k, c, np.float32)
    g = synth.normal_f64(k, synth.stream_key(1, "pin-gamma"), 1.0, 0.1).astype(np.float32)
    x = oracle.rmsnorm(h, g, 1e-5)
    cf = float(np.float32(c))
    expect = cf / math.sqrt(cf * cf + 1e-5) * g.astype(np.float64)
    np.testing.assert_allclose(x, expect, rtol=1e-14, atol=0)


def test_rmsnorm_zero_and_single_spike():
    k = 512
    g = np.linspace(0.5, 1.5, k).astype(np.float32)
    assert np.all(oracle.rmsnorm(np.zeros(k, np.float32), g, 1e-5) == 0.0)
    h = np.zeros(k, np.float32)
    h[37] = -3.5
    x = oracle.rmsnorm(h, g, 1e-5)
    expect = -3.5 / math.sqrt(3.5 * 3.5 / k + 1e-5) * float(g[37])
    assert abs(x[37] - expect) <= 1e-14 * abs(expect)
    assert np.count_nonzero(x) == 1


def test_rmsnorm_without_gamma_is_identity():
    h = synth.normal_f64(300, synth.stream_key(2, "pin-h")).astype(np.float32)
    assert np.array_equal(oracle.rmsnorm(h, None), h.astype(np.float64))


def test_rmsnorm_unit_rms_output():
    # with gamma = 1 and eps -> 0 the output has unit root-mean-square
    h = (synth.normal_f64(6656, synth.stream_key(3, "pin-h")) * 3.0).astype(np.float32)
    x = oracle.rmsnorm(h, np.ones(6656, np.float32), 0.0)
    assert abs(math.sqrt(np.mean(x * x)) - 1.0) < 1e-13


# ----------------------------------------------------------------- Q5_K parsing
def test_half_decoding_matches_numpy_float16_everywhere():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[finite]])
    assert np.array_equal(got, ref[finite])


def _blank_block(d=1.0, dmin=0.5):
    blk = np.zeros(176, np.uint8)
    db = np.array([d], np.float16).view(np.uint16)[0]
    mb = np.array([dmin], np.float16).view(np.uint16)[0]
    blk[0], blk[1] = db & 0xFF, db >> 8
    blk[2], blk[3] = mb & 0xFF, mb >> 8
    return blk


def test_all_zero_quants_give_minus_dmin_times_min():
    blk = _blank_block(d=0.00048828125, dmin=0.25)
    # hand-packed scale bytes: m_s = s + 1 for s < 4 (low 6 bits of bytes 4..7),
    # m_s for s >= 4 from high nibble of bytes 8..11 plus top bits of bytes 4..7
    for s in range(4):
        blk[4 + 4 + s] = (s + 1) | (1 << 6)           # m_s = s+1 ; top bits of m_{s+4} = 1
        blk[4 + 8 + s] = (s + 2) << 4                 # low nibble of m_{s+4} = s+2
    expect_m = [1, 2, 3, 4, 16 + 2, 16 + 3, 16 + 4, 16 + 5]
    w = oracle.q5k_dequant_block(blk)
    for e in range(256):
        assert w[e] == -0.25 * expect_m[e // 32]


def test_zero_scales_and_mins_give_zero_weights():
    blk = _blank_block(d=0.75, dmin=0.125)
    blk[16:] = 0xA5   # any quants
    assert np.all(oracle.q5k_dequant_block(blk) == 0.0)


def test_max_quant_and_scale_give_1953_d():
    d = 0.000732421875
    blk = _blank_block(d=d, dmin=0.0)
    blk[4:8] = 0xFF    # sc_0..3 = 63, top bits of sc_4..7 = 3
    blk[12:16] = 0x0F  # low nibble of sc_4..7 = 15 -> 63 ; mins 0
    blk[16:48] = 0xFF  # every high bit set
    blk[48:] = 0xFF    # every nibble 15
    _, _, sc, m, q = oracle.q5k_parse(blk)
    assert list(sc) == [63] * 8 and list(m) == [0] * 8 and np.all(q == 31)
    assert np.all(oracle.q5k_dequant_block(blk) == 1953.0 * d)


@pytest.mark.parametrize("byte", [0, 5, 31, 32, 63, 64, 100, 127])
def test_one_hot_low_nibbles_locate_their_weight(byte):
    for nib in (0, 1):
        blk = _blank_block()
        blk[48 + byte] = 1 << (4 * nib)
        _, _, _, _, q = oracle.q5k_parse(blk)
        s = 2 * (byte // 32) + nib
        e = 32 * s + byte % 32
        expect = np.zeros(256, np.int32)
        expect[e] = 1
        assert np.array_equal(q, expect)


@pytest.mark.parametrize("l", [0, 13, 31])
def test_one_hot_high_bits_locate_their_weight(l):
    for s in range(8):
        blk = _blank_block()
        blk[16 + l] = 1 << s
        _, _, _, _, q = oracle.q5k_parse(blk)
        expect = np.zeros(256, np.int32)
        expect[32 * s + l] = 16
        assert np.array_equal(q, expect)


def test_parse_recovers_every_generated_field():
    w, f = synth.q5k_matrix(24, 1024, synth.stream_key(7, "pin-W"), with_fields=True)
    for i in range(24):
        for kb in range(4):
            d, dmin, sc, m, q = oracle.q5k_parse(w[i, kb * 176:(kb + 1) * 176])
            assert d == float(f.d_bits[i, kb:kb + 1].view(np.float16)[0])
            assert dmin == float(f.dmin_bits[i, kb:kb + 1].view(np.float16)[0])
            assert np.array_equal(sc, f.sc[i, kb]) and np.array_equal(m, f.m[i, kb])
            assert np.array_equal(q, f.q[i, kb])


# ----------------------------------------------------------------- matvec
def _dense_from_fields(f):
    """Dense f64 weights from the generator's drawn fields (numpy float16 decoding)."""
    d = f.d_bits.view(np.float16).astype(np.float64)[:, :, None]
    dm = f.dmin_bits.view(np.float16).astype(np.float64)[:, :, None]
    sc = np.repeat(f.sc.astype(np.float64), 32, axis=2)
    mm = np.repeat(f.m.astype(np.float64), 32, axis=2)
    w = d * sc * f.q.astype(np.float64) - dm * mm
    return w.reshape(w.shape[0], -1)


@pytest.mark.parametrize("n,k,b", [(1, 256, 1), (7, 256, 3), (33, 512, 2), (64, 512, 5)])
def test_matvec_brute_force_against_dense_numpy(n, k, b):
    w, f = synth.q5k_matrix(n, k, synth.stream_key(n * 1000 + k, "pin-mv"), with_fields=True)
    h = synth.normal_f64(b * k, synth.stream_key(b, "pin-mv-h")).astype(np.float32).reshape(b, k)
    out, raw = oracle.lmhead(h, None, w, 1.0, 0.0, want_raw=True)
    dense = _dense_from_fields(f)
    expect = h.astype(np.float64) @ dense.T
    np.testing.assert_allclose(raw, expect, rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, raw)


def test_one_hot_input_picks_a_column():
    n, k = 16, 512
    w, f = synth.q5k_matrix(n, k, synth.stream_key(11, "pin-col"), with_fields=True)
    dense = _dense_from_fields(f)
    for j in (0, 31, 32, 255, 256, 300, 511):
        h = np.zeros((1, k), np.float32)
        h[0, j] = 1.0
        _, raw = oracle.lmhead(h, None, w, 1.0, 0.0, want_raw=True)
        assert np.array_equal(raw[0], dense[:, j])


def test_full_stage_against_textbook_numpy():
    n, k, b = 40, 768, 3
    w, f = synth.q5k_matrix(n, k, synth.stream_key(5, "pin-stage"), with_fields=True)
    h = (synth.normal_f64(b * k, synth.stream_key(5, "pin-stage-h")) * 2.0).astype(np.float32).reshape(b, k)
    g = synth.normal_f64(k, synth.stream_key(5, "pin-stage-g"), 1.0, 0.1).astype(np.float32)
    # boost the weights so some scaled values pass the cap's knee
    out = oracle.lmhead(h, g, w, 30.0, CAP)
    hd = h.astype(np.float64)
    x = hd / np.sqrt(np.mean(hd * hd, axis=1, keepdims=True) + 1e-5) * g.astype(np.float64)
    v = (x @ _dense_from_fields(f).T) * 30.0
    np.testing.assert_allclose(out, CAP * np.tanh(v / CAP), rtol=1e-11, atol=1e-11)
    assert np.abs(v).max() > 20.0


def test_row_subset_equals_full_rows():
    n, k = 50, 512
    w = synth.q5k_matrix(n, k, synth.stream_key(9, "pin-rows"))
    h = synth.normal_f64(2 * k, synth.stream_key(9, "pin-rows-h")).astype(np.float32).reshape(2, k)
    g = np.ones(k, np.float32)
    full = oracle.lmhead(h, g, w, SCALE, CAP)
    rows = [49, 0, 17, 17, 3]
    sub = oracle.lmhead(h, g, w, SCALE, CAP, rows=rows)
    assert np.array_equal(sub, full[:, rows])


def test_threads_do_not_change_results():
    w = synth.q5k_matrix(300, 512, synth.stream_key(4, "pin-thr"))
    h = synth.normal_f64(512, synth.stream_key(4, "pin-thr-h")).astype(np.float32)
    g = np.ones(512, np.float32)
    a = oracle.lmhead(h, g, w, SCALE, CAP, nthreads=1)
    b = oracle.lmhead(h, g, w, SCALE, CAP, nthreads=7)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------- argmax
def test_argmax_is_invariant_under_the_cap():
    n, k = 500, 512
    w = synth.q5k_matrix(n, k, synth.stream_key(12, "pin-arg"), boost_rows=(3, 250), boost=50.0)
    h = synth.normal_f64(4 * k, synth.stream_key(12, "pin-arg-h")).astype(np.float32).reshape(4, k)
    g = np.ones(k, np.float32)
    out, raw = oracle.lmhead(h, g, w, SCALE, CAP, want_raw=True)
    assert np.array_equal(oracle.argmax_first(out), oracle.argmax_first(raw))
    assert np.array_equal(oracle.argmax_first(out), np.argmax(raw * SCALE, axis=1))


def test_argmax_takes_lowest_index_on_ties_and_gap():
    o = np.array([[1.0, 5.0, 5.0, -2.0], [7.0, 7.0, 7.0, 7.0], [0.0, 1.0, 3.0, 2.5]])
    assert list(oracle.argmax_first(o)) == [1, 0, 2]
    assert list(oracle.top2_gap(o)) == [0.0, 0.0, 0.5]


# ----------------------------------------------------------------- byte bill
def test_byte_bill_chapter20():
    bill = {r[0]: int(r[1]) for r in read_golden("lmhead_byte_bill.txt")}
    wl = synth.WORKLOADS["lmhead_b1"]
    assert wl.n_rows == bill["rows"] and wl.k == bill["cols"]
    assert wl.k // synth.BLOCK_WEIGHTS == bill["blocks_per_row"]
    assert bill["blocks_per_row"] * synth.BLOCK_BYTES == bill["bytes_per_row"]
    assert wl.weight_bytes == bill["weight_bytes"]
    assert wl.k * 4 == bill["normed_input_bytes"] and wl.n_rows * 4 == bill["logits_bytes"]
    assert wl.n_rows * bill["blocks_per_row"] * 144 == bill["q4k_weight_bytes"]
    small = synth.q5k_matrix(3, wl.k, synth.stream_key(0, "pin-bill"))
    assert small.shape[1] == bill["bytes_per_row"]


# ----------------------------------------------------------------- log-softmax over the capped logits
def test_log_softmax_hand_cases():
    lp, lse = oracle.log_softmax(np.array([[0.0, 0.0], [0.0, np.log(3.0)], [7.5, 7.5]]))
    assert np.allclose(lp[0], [-np.log(2.0)] * 2, rtol=0, atol=1e-15) and abs(lse[0] - np.log(2.0)) < 1e-15
    assert np.allclose(lp[1], [-np.log(4.0), np.log(3.0) - np.log(4.0)], rtol=0, atol=1e-15)
    assert abs(lse[2] - (7.5 + np.log(2.0))) < 1e-14
    lp1, lse1 = oracle.log_softmax(np.array([[-3.25]]))          # one column: probability 1
    assert lp1[0, 0] == 0.0 and lse1[0] == -3.25


def test_log_softmax_uniform_and_saturated_rows():
    n = 202048
    lp, lse = oracle.log_softmax(np.full((1, n), 20.0))         # all logits at the cap
    assert np.allclose(lp, -np.log(n), rtol=0, atol=1e-12) and abs(lse[0] - (20.0 + np.log(n))) < 1e-12
    lp, _ = oracle.log_softmax(np.array([[20.0, -20.0]]))       # the cap's extremes
    # exact values -log1p(e^-40) and -40 - log1p(e^-40), to f64 resolution at magnitude 20-40
    assert abs(lp[0, 0] - (-np.log1p(np.exp(-40.0)))) < 1e-14
    assert abs(lp[0, 1] - (-40.0 - np.log1p(np.exp(-40.0)))) < 1e-13


def test_log_softmax_sums_to_one_and_is_shift_invariant():
    rng = np.random.default_rng(21)
    o = 20.0 * np.tanh(rng.normal(-1.6, 5.0, size=(3, 50000)) / 20.0)    # capped-logit-like rows
    lp, lse = oracle.log_softmax(o)
    assert np.allclose(np.exp(lp).sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(lp <= 0.0)
    lp2, lse2 = oracle.log_softmax(o + 13.0)
    assert np.allclose(lp2, lp, rtol=0, atol=1e-12) and np.allclose(lse2, lse + 13.0, rtol=0, atol=1e-12)
    # the order of the row is kept, and the argmax has the largest logprob
    assert np.array_equal(np.argmax(lp, axis=1), oracle.argmax_first(o))


# ----------------------------------------------------------------- Q4_K (144-byte blocks)
def _blank_q4k_block(d=1.0, dmin=0.5):
    blk = np.zeros(144, np.uint8)
    blk[:4] = _blank_block(d, dmin)[:4]
    return blk


def test_q4k_all_zero_quants_give_minus_dmin_times_min():
    blk = _blank_q4k_block(d=0.00048828125, dmin=0.25)
    for s in range(4):                                   # same scale-byte packing as Q5_K
        blk[4 + 4 + s] = (s + 1) | (1 << 6)
        blk[4 + 8 + s] = (s + 2) << 4
    expect_m = [1, 2, 3, 4, 16 + 2, 16 + 3, 16 + 4, 16 + 5]
    w = oracle.q4k_dequant_block(blk)
    for e in range(256):
        assert w[e] == -0.25 * expect_m[e // 32]


def test_q4k_zero_scales_give_zero_and_max_gives_945_d():
    blk = _blank_q4k_block(d=0.75, dmin=0.125)
    blk[16:] = 0xA5
    assert np.all(oracle.q4k_dequant_block(blk) == 0.0)
    d = 0.000732421875
    blk = _blank_q4k_block(d=d, dmin=0.0)
    blk[4:8] = 0xFF
    blk[12:16] = 0x0F
    blk[16:] = 0xFF                                       # every nibble 15; there are no high bits
    _, _, sc, m, q = oracle.q4k_parse(blk)
    assert list(sc) == [63] * 8 and list(m) == [0] * 8 and np.all(q == 15)
    assert np.all(oracle.q4k_dequant_block(blk) == 945.0 * d)


@pytest.mark.parametrize("byte", [0, 5, 31, 32, 63, 64, 100, 127])
def test_q4k_one_hot_nibbles_locate_their_weight(byte):
    for nib in (0, 1):
        blk = _blank_q4k_block()
        blk[16 + byte] = 1 << (4 * nib)
        _, _, _, _, q = oracle.q4k_parse(blk)
        expect = np.zeros(256, np.int32)
        expect[32 * (2 * (byte // 32) + nib) + byte % 32] = 1
        assert np.array_equal(q, expect)


def test_q4k_parse_recovers_every_generated_field():
    w, f = synth.q5k_matrix(24, 1024, synth.stream_key(7, "pin-W4"), with_fields=True, fmt="q4_k")
    assert w.shape == (24, 4 * 144) and f.q.max() <= 15
    for i in range(24):
        for kb in range(4):
            d, dmin, sc, m, q = oracle.q4k_parse(w[i, kb * 144:(kb + 1) * 144])
            assert d == float(f.d_bits[i, kb:kb + 1].view(np.float16)[0])
            assert dmin == float(f.dmin_bits[i, kb:kb + 1].view(np.float16)[0])
            assert np.array_equal(sc, f.sc[i, kb]) and np.array_equal(m, f.m[i, kb])
            assert np.array_equal(q, f.q[i, kb])


@pytest.mark.parametrize("n,k,b", [(1, 256, 1), (9, 512, 3), (40, 768, 2)])
def test_q4k_matvec_brute_force_against_dense_numpy(n, k, b):
    w, f = synth.q5k_matrix(n, k, synth.stream_key(n * 1000 + k, "pin-mv4"), with_fields=True, fmt="q4_k")
    h = synth.normal_f64(b * k, synth.stream_key(b, "pin-mv4-h")).astype(np.float32).reshape(b, k)
    out, raw = oracle.lmhead(h, None, w, 1.0, 0.0, want_raw=True, fmt="q4_k")
    np.testing.assert_allclose(raw, h.astype(np.float64) @ _dense_from_fields(f).T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, raw)
    with pytest.raises(ValueError):                       # Q4_K bytes are not a Q5_K matrix of this K
        oracle.lmhead(h, None, w, 1.0, 0.0)


def test_q4k_head_byte_bill():
    bill = {r[0]: int(r[1]) for r in read_golden("lmhead_byte_bill.txt")}
    w = synth.q5k_matrix(2, 6656, synth.stream_key(0, "pin-bill4"), fmt="q4_k")
    assert w.shape[1] * 202048 == bill["q4k_weight_bytes"]
