"""Seeded synthetic inputs for the Muse Glimmer decode output stage.

The generator draws random numbers and lays them out (hidden rows, the final
norm's gamma, Q5_K weight blocks).  It holds none of the output stage's
arithmetic, so both the f64 CPU oracle and the CUDA path can be fed from it
while sharing nothing else.  The C source next to this file states the
generator (counter-form SplitMix64) and the Q5_K byte layout it writes.

Workloads (shapes and value distributions of the Muse Glimmer output head,
"Chapter 20 — Final norm, LM head, and the soft cap" §20.1/§20.3, and of the
attention projections of "Chapter 9 — The Muse Glimmer architecture" §9.3):

* ``tiny``        B=1, N=2,048 rows x K=6,656, RMSNorm + scale + cap + argmax
* ``lmhead_b1``   B=1, N=202,048 x 6,656; rows 0, 777, 200001 get d x 50
* ``lmhead_b8``   B=8, same weights; hidden rows scaled by U(0.5, 4)
* ``attn_q`` ``attn_k`` ``attn_v`` ``attn_o``  projection shapes, B=1, no norm/scale/cap
* ``sweep_b{1,2,4,8,16,32}``  N=202,048 x 6,656, no boosted rows
* ``dflash_verify_b16``  B=16 (the drafted positions), rows scaled by U(0.5, 4)
* ``lmhead_q4k_b1`` ``lmhead_q4k_b8``  the Q4_K head (756.5 MB), B=1 and B=8
* ``ffn_up_q4k`` ``ffn_down_q4k``  one block's FFN shapes in Q4_K, B=1
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libq5k_synth.so")
_lock = threading.Lock()
_lib = None

BLOCK_BYTES = 176
BLOCK_BYTES_Q4K = 144
BLOCK_WEIGHTS = 256


def build(force: bool = False) -> str:
    """Compile synth.c into an in-tree shared library (gcc, no FP contraction)."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off",
                   "-pthread", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, dbl, vp, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.synth_stream_key.restype = u64
        lib.synth_stream_key.argtypes = [u64, u64]
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64]
        lib.synth_f64_to_f16_bits.restype = ctypes.c_uint16
        lib.synth_f64_to_f16_bits.argtypes = [dbl]
        lib.synth_q5k_rows.restype = i32
        lib.synth_q5k_rows.argtypes = [vp, i64, i64, i64, u64, dbl, dbl, dbl, dbl, dbl,
                                       vp, vp, vp, vp, vp, i32]
        lib.synth_q4k_rows.restype = i32
        lib.synth_q4k_rows.argtypes = lib.synth_q5k_rows.argtypes
        lib.synth_normal_f64.restype = None
        lib.synth_normal_f64.argtypes = [vp, i64, u64, dbl, dbl]
        lib.synth_uniform_f64.restype = None
        lib.synth_uniform_f64.argtypes = [vp, i64, u64, dbl, dbl]
        _lib = lib
    return _lib


def tag_id(tag: str) -> int:
    """Fixed 64-bit id of a stream tag (FNV-1a over its UTF-8 bytes)."""
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h = ((h ^ b) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, tag: str) -> int:
    return int(_load().synth_stream_key(seed & 0xFFFFFFFFFFFFFFFF, tag_id(tag)))


def draw(key: int, i: int) -> int:
    return int(_load().synth_draw(key, i))


def f64_to_f16_bits(v: float) -> int:
    return int(_load().synth_f64_to_f16_bits(float(v)))


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


@dataclass
class Q5KFields:
    """Values drawn for each super-block (for tests that build weights independently)."""
    d_bits: np.ndarray      # [n, nb] uint16 (fp16 bit patterns)
    dmin_bits: np.ndarray   # [n, nb] uint16
    sc: np.ndarray          # [n, nb, 8] uint8 (0..63)
    m: np.ndarray           # [n, nb, 8] uint8 (0..63)
    q: np.ndarray           # [n, nb, 256] uint8 (0..31)


D_RANGE = (2e-4, 1e-3)
DMIN_RANGE = (0.0, 1e-3)


def q5k_rows(n_rows: int, k: int, key: int, row_begin: int = 0, d_mult: float = 1.0,
             with_fields: bool = False, out: np.ndarray | None = None, fmt: str = "q5_k"):
    """Rows [row_begin, row_begin + n_rows) of a Q5_K (or, fmt="q4_k", Q4_K)
    matrix with k columns.

    Returns uint8 [n_rows, k // 256 * block bytes] (and Q5KFields if with_fields;
    q is then 0..15 for Q4_K).
    """
    if k % BLOCK_WEIGHTS:
        raise ValueError("k must be a multiple of 256")
    if fmt not in ("q5_k", "q4_k"):
        raise ValueError("fmt must be q5_k or q4_k")
    nb = k // BLOCK_WEIGHTS
    bb = BLOCK_BYTES if fmt == "q5_k" else BLOCK_BYTES_Q4K
    if out is None:
        out = np.empty((n_rows, nb * bb), dtype=np.uint8)
    assert out.shape == (n_rows, nb * bb) and out.dtype == np.uint8 and out.flags.c_contiguous
    f = None
    if with_fields:
        f = Q5KFields(np.empty((n_rows, nb), np.uint16), np.empty((n_rows, nb), np.uint16),
                      np.empty((n_rows, nb, 8), np.uint8), np.empty((n_rows, nb, 8), np.uint8),
                      np.empty((n_rows, nb, 256), np.uint8))
    gen = _load().synth_q5k_rows if fmt == "q5_k" else _load().synth_q4k_rows
    rc = gen(
        _ptr(out), row_begin, row_begin + n_rows, nb, key, D_RANGE[0], D_RANGE[1],
        DMIN_RANGE[0], DMIN_RANGE[1], float(d_mult),
        _ptr(f.d_bits if f else None), _ptr(f.dmin_bits if f else None),
        _ptr(f.sc if f else None), _ptr(f.m if f else None), _ptr(f.q if f else None),
        _threads())
    if rc != 0:
        raise RuntimeError("synth_q5k_rows failed")
    return (out, f) if with_fields else out


def q5k_matrix(n_rows: int, k: int, key: int, boost_rows=(), boost: float = 50.0,
               with_fields: bool = False, out: np.ndarray | None = None, fmt: str = "q5_k"):
    """A whole Q5_K (or Q4_K) matrix; rows in boost_rows have d drawn x boost before fp16 rounding."""
    res = q5k_rows(n_rows, k, key, 0, 1.0, with_fields, out, fmt)
    w, f = (res if with_fields else (res, None))
    for r in boost_rows:
        if not 0 <= r < n_rows:
            continue
        rr = q5k_rows(1, k, key, r, boost, with_fields, None, fmt)
        if with_fields:
            w[r:r + 1], fr = rr
            f.d_bits[r], f.dmin_bits[r], f.sc[r], f.m[r], f.q[r] = fr.d_bits[0], fr.dmin_bits[0], fr.sc[0], fr.m[0], fr.q[0]
        else:
            w[r:r + 1] = rr
    return (w, f) if with_fields else w


def normal_f64(n: int, key: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal_f64(_ptr(out), n, key, float(mean), float(std))
    return out


def uniform_f64(n: int, key: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(_ptr(out), n, key, float(lo), float(hi))
    return out


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------
LOGIT_SCALE = 0.196116          # muse-glimmer.logit_scale (Chapter 20 §20.1, §20.5)
SOFTCAP = 20.0                  # final_logit_softcap (Chapter 20 §20.1)
RMS_EPS = 1e-5                  # output_norm epsilon (Chapter 20 §20.1)
HIDDEN = 6656
VOCAB = 202048
BOOSTED_ROWS = (0, 777, 200001)


@dataclass(frozen=True)
class Workload:
    name: str
    n_rows: int
    k: int
    batch: int
    weight_tag: str
    norm: bool = True
    scale: float = LOGIT_SCALE
    cap: float = SOFTCAP
    argmax: bool = True
    boost_rows: tuple = ()
    row_scale: tuple | None = None   # (lo, hi): hidden row b multiplied by U(lo, hi)
    hidden_tag: str = ""
    gamma_tag: str = "G:lmhead"
    fmt: str = "q5_k"                  # weight blocks: q5_k (176 bytes) or q4_k (144 bytes)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def block_bytes(self) -> int:
        return BLOCK_BYTES if self.fmt == "q5_k" else BLOCK_BYTES_Q4K

    @property
    def weight_bytes(self) -> int:
        return self.n_rows * (self.k // BLOCK_WEIGHTS) * self.block_bytes

    def algorithmic_bytes(self) -> int:
        """Q5_K weights + hidden + gamma + logits: the bytes one forward must move."""
        b = self.weight_bytes + self.batch * self.k * 4 + self.batch * self.n_rows * 4
        if self.norm:
            b += self.k * 4
        return b


def _lm(name, batch, boost=(), row_scale=None):
    return Workload(name, VOCAB, HIDDEN, batch, "W:lmhead", boost_rows=boost,
                    row_scale=row_scale, hidden_tag=f"H:{name}")


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 2048, HIDDEN, 1, "W:tiny", hidden_tag="H:tiny", gamma_tag="G:tiny"),
    "lmhead_b1": _lm("lmhead_b1", 1, BOOSTED_ROWS),
    "lmhead_b8": _lm("lmhead_b8", 8, BOOSTED_ROWS, (0.5, 4.0)),
    "attn_q": Workload("attn_q", 4096, HIDDEN, 1, "W:attn_q", norm=False, scale=1.0, cap=0.0,
                       argmax=False, hidden_tag="H:attn_q"),
    "attn_k": Workload("attn_k", 256, HIDDEN, 1, "W:attn_k", norm=False, scale=1.0, cap=0.0,
                       argmax=False, hidden_tag="H:attn_k"),
    "attn_v": Workload("attn_v", 256, HIDDEN, 1, "W:attn_v", norm=False, scale=1.0, cap=0.0,
                       argmax=False, hidden_tag="H:attn_v"),
    "attn_o": Workload("attn_o", HIDDEN, 4096, 1, "W:attn_o", norm=False, scale=1.0, cap=0.0,
                       argmax=False, hidden_tag="H:attn_o"),
}
for _b in (1, 2, 4, 8, 16, 32):
    WORKLOADS[f"sweep_b{_b}"] = _lm(f"sweep_b{_b}", _b)
# the DFlash verify batch: the target model scores the 16 drafted positions at once
WORKLOADS["dflash_verify_b16"] = _lm("dflash_verify_b16", 16, BOOSTED_ROWS, (0.5, 4.0))
# the Q4_K head alternative (756.5 MB), batch 1, same shapes and boosted rows
WORKLOADS["lmhead_q4k_b1"] = Workload("lmhead_q4k_b1", VOCAB, HIDDEN, 1, "W:lmhead_q4k", boost_rows=BOOSTED_ROWS,
                                      hidden_tag="H:lmhead_q4k_b1", fmt="q4_k")
# the FFN of one block in Q4_K ("Chapter 9 — The Muse Glimmer architecture", Figure 9.1:
# gate and up [6656 -> 19968], down [19968 -> 6656]); batch 1, no norm, scale 1, no cap
FFN_WIDTH = 19968
WORKLOADS["ffn_up_q4k"] = Workload("ffn_up_q4k", FFN_WIDTH, HIDDEN, 1, "W:ffn_up_q4k", norm=False, scale=1.0,
                                   cap=0.0, argmax=False, hidden_tag="H:ffn_up_q4k", fmt="q4_k")
WORKLOADS["ffn_down_q4k"] = Workload("ffn_down_q4k", HIDDEN, FFN_WIDTH, 1, "W:ffn_down_q4k", norm=False,
                                     scale=1.0, cap=0.0, argmax=False, hidden_tag="H:ffn_down_q4k", fmt="q4_k")
WORKLOADS["lmhead_q4k_b8"] = Workload("lmhead_q4k_b8", VOCAB, HIDDEN, 8, "W:lmhead_q4k", boost_rows=BOOSTED_ROWS,
                                      row_scale=(0.5, 4.0), hidden_tag="H:lmhead_q4k_b8", fmt="q4_k")


@dataclass(frozen=True)
class GroupWorkload:
    """Several matrices (all Q5_K or all Q4_K) against one input row in one
    launch.  segments: ((name, n_rows, weight_tag, scale, cap), ...)."""
    name: str
    k: int
    segments: tuple
    norm: bool = True
    hidden_tag: str = ""
    gamma_tag: str = ""
    batch: int = 1
    argmax: bool = False
    fmt: str = "q5_k"

    @property
    def n_rows(self) -> int:
        return sum(s[1] for s in self.segments)

    @property
    def weight_bytes(self) -> int:
        return self.n_rows * (self.k // BLOCK_WEIGHTS) * (BLOCK_BYTES if self.fmt == "q5_k" else BLOCK_BYTES_Q4K)

    def algorithmic_bytes(self) -> int:
        """Weights of every matrix + hidden + gamma + outputs."""
        b = self.weight_bytes + self.k * 4 + self.n_rows * 4
        if self.norm:
            b += self.k * 4
        return b


# The attention block's concurrent group: Q and gate [6656 -> 4096], K and V
# [6656 -> 256] from the attn_norm-normalised residual (no scale, no cap).
GROUPS: dict[str, GroupWorkload] = {
    "attn_qkvg": GroupWorkload("attn_qkvg", HIDDEN,
                               (("q", 4096, "W:attn_q", 1.0, 0.0), ("gate", 4096, "W:attn_gate", 1.0, 0.0),
                                ("k", 256, "W:attn_k", 1.0, 0.0), ("v", 256, "W:attn_v", 1.0, 0.0)),
                               hidden_tag="H:attn_qkvg", gamma_tag="G:attn_norm"),
    # The FFN's gate and up projections [6656 -> 19968] in Q4_K from the
    # ffn_norm-normalised residual: one launch for both (149.5 MB).
    "ffn_gate_up_q4k": GroupWorkload("ffn_gate_up_q4k", HIDDEN,
                                     (("gate", FFN_WIDTH, "W:ffn_gate_q4k", 1.0, 0.0),
                                      ("up", FFN_WIDTH, "W:ffn_up_q4k", 1.0, 0.0)),
                                     hidden_tag="H:ffn_gate_up", gamma_tag="G:ffn_norm", fmt="q4_k"),
}


def group_inputs(g: GroupWorkload | str, seed: int = 0):
    """(hidden [1, K] f32, gamma [K] f32 or None, [weights of each matrix])."""
    if isinstance(g, str):
        g = GROUPS[g]
    h = normal_f64(g.k, stream_key(seed, g.hidden_tag)).reshape(1, g.k).astype(np.float32)
    gam = normal_f64(g.k, stream_key(seed, g.gamma_tag), 1.0, 0.1).astype(np.float32) if g.norm else None
    ws = [q5k_matrix(n, g.k, stream_key(seed, tag), fmt=g.fmt) for (_, n, tag, _, _) in g.segments]
    return h, gam, ws


def hidden_for(w: Workload, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """hidden [B, K] f32: N(0,1), each row optionally scaled by U(lo, hi), rounded once to f32."""
    b = w.batch if batch is None else batch
    h = normal_f64(b * w.k, stream_key(seed, w.hidden_tag)).reshape(b, w.k)
    if w.row_scale is not None:
        s = uniform_f64(b, stream_key(seed, w.hidden_tag + ":rowscale"), *w.row_scale)
        h = h * s[:, None]
    return h.astype(np.float32)


def gamma_for(w: Workload, seed: int = 0) -> np.ndarray | None:
    """output_norm gamma [K] f32 ~ N(1, 0.1), or None for workloads without the norm."""
    if not w.norm:
        return None
    return normal_f64(w.k, stream_key(seed, w.gamma_tag), 1.0, 0.1).astype(np.float32)


def weights_for(w: Workload, seed: int = 0, with_fields: bool = False, out=None):
    return q5k_matrix(w.n_rows, w.k, stream_key(seed, w.weight_tag), w.boost_rows, 50.0,
                      with_fields, out, w.fmt)


def inputs_for(w: Workload | str, seed: int = 0, with_fields: bool = False):
    """(hidden, gamma, weights[, fields]) for a workload."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    h = hidden_for(w, seed)
    g = gamma_for(w, seed)
    wt = weights_for(w, seed, with_fields)
    if with_fields:
        return h, g, wt[0], wt[1]
    return h, g, wt
