"""f64 CPU oracle of the Muse Glimmer decode output stage (final RMSNorm ->
Q5_K LM-head matvec -> logit scale -> soft cap -> greedy argmax).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import or call this package.
The CUDA path does not import it, and it does not import the CUDA path; the two
share nothing but the seeded input generator (``q5k_synth``).

The arithmetic is in ``q5k_oracle.c`` (binary64, plain loops, no FMA
contraction); this module loads it and adds the argmax, which follows
"Chapter 20 — Final norm, LM head, and the soft cap" §20.2 (the largest capped
score wins; the cap is strictly increasing, so the index is the same before and
after it).  Ties go to the lowest index: the pages say nothing about ties.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(worked values printed in Chapter 20 §20.7, closed forms, brute force on tiny
shapes against a dense numpy matmul, invariants).  The Q5_K byte layout itself
is the ggml reading (the pages cite an absent chapter for it): agreement with a
real GGUF file's bytes is parity unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q5k_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libq5k_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into an in-tree shared library (gcc -O2, no FP contraction)."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off",
                            "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_half_to_double.restype = dbl
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_q5k_parse.restype = None
        lib.oracle_q5k_parse.argtypes = [vp, vp, vp, vp, vp, vp]
        lib.oracle_q5k_dequant.restype = None
        lib.oracle_q5k_dequant.argtypes = [vp, vp]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rmsnorm.argtypes = [vp, vp, i64, dbl, vp]
        lib.oracle_scale_softcap.restype = dbl
        lib.oracle_scale_softcap.argtypes = [dbl, dbl, dbl]
        lib.oracle_lmhead.restype = i32
        lib.oracle_lmhead.argtypes = [vp, i64, i64, vp, dbl, vp, i64, vp, i64, dbl, dbl, vp, vp, i32]
        lib.oracle_lmhead_fmt.restype = i32
        lib.oracle_lmhead_fmt.argtypes = lib.oracle_lmhead.argtypes + [i32]
        lib.oracle_q4k_parse.restype = None
        lib.oracle_q4k_parse.argtypes = [vp, vp, vp, vp, vp, vp]
        lib.oracle_q4k_dequant.restype = None
        lib.oracle_q4k_dequant.argtypes = [vp, vp]
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def half_to_double(bits: int) -> float:
    return float(_load().oracle_half_to_double(bits))


def q5k_parse(block: np.ndarray):
    """(d, dmin, sc[8], m[8], q[256]) of one 176-byte block."""
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 176
    d = np.zeros(1, np.float64)
    dm = np.zeros(1, np.float64)
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_q5k_parse(_p(blk), _p(d), _p(dm), _p(sc), _p(m), _p(q))
    return float(d[0]), float(dm[0]), sc, m, q


def q5k_dequant_block(block: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 176
    w = np.zeros(256, np.float64)
    _load().oracle_q5k_dequant(_p(blk), _p(w))
    return w


def q5k_dequant_matrix(wq: np.ndarray) -> np.ndarray:
    """Dense f64 [n, k] from Q5_K rows [n, k/256*176] (small matrices only)."""
    n, rb = wq.shape
    nb = rb // 176
    out = np.empty((n, nb * 256), np.float64)
    for i in range(n):
        for kb in range(nb):
            out[i, kb * 256:(kb + 1) * 256] = q5k_dequant_block(wq[i, kb * 176:(kb + 1) * 176])
    return out


def q4k_parse(block: np.ndarray):
    """(d, dmin, sc[8], m[8], q[256]) of one 144-byte Q4_K block."""
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 144
    d = np.zeros(1, np.float64)
    dm = np.zeros(1, np.float64)
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_q4k_parse(_p(blk), _p(d), _p(dm), _p(sc), _p(m), _p(q))
    return float(d[0]), float(dm[0]), sc, m, q


def q4k_dequant_block(block: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 144
    w = np.zeros(256, np.float64)
    _load().oracle_q4k_dequant(_p(blk), _p(w))
    return w


BLOCK_BYTES = {"q5_k": 176, "q4_k": 144}


def rmsnorm(h: np.ndarray, gamma: np.ndarray | None, eps: float = 1e-5) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float32)
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
    x = np.zeros(h.size, np.float64)
    _load().oracle_rmsnorm(_p(h), _p(g), h.size, float(eps), _p(x))
    return x


def scale_softcap(raw: float, scale: float, cap: float) -> float:
    return float(_load().oracle_scale_softcap(float(raw), float(scale), float(cap)))


def lmhead(hidden: np.ndarray, gamma: np.ndarray | None, wq: np.ndarray, scale: float,
           cap: float, eps: float = 1e-5, rows=None, want_raw: bool = False,
           nthreads: int | None = None, fmt: str = "q5_k"):
    """out [B, n_out] f64 (and raw [B, n_out] if want_raw).

    hidden: [B, K] f32; gamma: [K] f32 or None (no norm); wq: [N, K/256*block bytes]
    uint8 in fmt "q5_k" (176-byte blocks) or "q4_k" (144-byte blocks);
    rows: optional list of weight rows to compute (default: all N).
    """
    hidden = np.ascontiguousarray(np.atleast_2d(hidden), dtype=np.float32)
    b, k = hidden.shape
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    n_w = wq.shape[0]
    if wq.shape[1] * 256 != k * BLOCK_BYTES[fmt]:
        raise ValueError("weight row bytes do not match K")
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
    ra = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_out = n_w if ra is None else ra.size
    out = np.zeros((b, n_out), np.float64)
    raw = np.zeros((b, n_out), np.float64) if want_raw else None
    rc = _load().oracle_lmhead_fmt(_p(hidden), b, k, _p(g), float(eps), _p(wq), n_w, _p(ra), n_out,
                                   float(scale), float(cap), _p(raw), _p(out),
                                   nthreads or default_threads(), 1 if fmt == "q4_k" else 0)
    if rc != 0:
        raise RuntimeError(f"oracle_lmhead failed ({rc})")
    return (out, raw) if want_raw else out


def log_softmax(out: np.ndarray):
    """Per row of the capped logits — softmax and logprobs are taken over the
    logits after scale and cap ("Chapter 20 — Final norm, LM head, and the soft
    cap", §20.7; softmax exp(x_i) / sum_j exp(x_j) as defined in "Chapter 9 —
    The Muse Glimmer architecture") — the plain definition in f64:
        M = max_j out_j,  lse = M + log(sum_j exp(out_j - M)),  logprob_j = out_j - lse.
    Returns (logprobs [B, N] f64, lse [B] f64)."""
    o = np.atleast_2d(np.asarray(out, dtype=np.float64))
    m = o.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(o - m).sum(axis=1))
    return o - lse[:, None], lse


def argmax_first(out: np.ndarray) -> np.ndarray:
    """Per row: the lowest index holding the row's maximum."""
    return np.argmax(np.atleast_2d(out), axis=1).astype(np.int64)


def top2_gap(out: np.ndarray) -> np.ndarray:
    """Per row: largest value minus second largest (0 when they tie, inf with one column)."""
    o = np.atleast_2d(out)
    if o.shape[1] < 2:
        return np.full(o.shape[0], np.inf)
    part = np.partition(o, -2, axis=1)
    return part[:, -1] - part[:, -2]
