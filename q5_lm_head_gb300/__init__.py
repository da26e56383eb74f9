"""Python binding of libmuse_lmhead.so: the Muse Glimmer decode output stage
(final RMSNorm -> Q5_K LM-head matvec -> scale -> soft cap -> argmax) on one
GB300.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  The functions named
``muse_lmhead_*`` mirror the C-ABI in include/muse_lmhead.h one to one (plain
integers for pointers and streams); :class:`LMHead` wraps them for torch
tensors.  If the compiled library is missing, importing works but every call
raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "LMHead", "MuseError", "library_path", "load_library",
    "muse_lmhead_init", "muse_lmhead_forward", "muse_lmhead_forward_host",
    "muse_lmhead_launches_per_forward", "muse_lmhead_path_name", "muse_lmhead_device_status",
    "muse_lmhead_destroy", "muse_lmhead_status_string", "muse_lmhead_forward_b1_noalloc",
    "muse_lmhead_noalloc_device_status",
    "muse_lmhead_forward_group", "muse_lmhead_forward_group_host", "MuseGemvSegment", "MUSE_MAX_SEGMENTS",
    "muse_lmhead_forward_logprobs",
    "muse_lmhead_init_format", "MUSE_FORMAT_Q5_K", "MUSE_FORMAT_Q4_K", "BLOCK_BYTES",
    "muse_lmhead_clear_device_status", "muse_lmhead_selftest_wait_timeout",
    "muse_lmhead_set_argmax_key", "MUSE_ARGMAX_CAPPED", "MUSE_ARGMAX_PRECAP",
    "EXPORTED_SYMBOLS",
    "LOGIT_SCALE", "SOFTCAP", "RMS_EPS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmuse_lmhead.so")

# Constants of the Muse Glimmer checkpoint ("Chapter 20 — Final norm, LM head,
# and the soft cap", §20.1 and §20.5): read from GGUF metadata there, passed as
# call arguments here.
LOGIT_SCALE = 0.196116
SOFTCAP = 20.0
RMS_EPS = 1e-5

EXPORTED_SYMBOLS = (
    "muse_lmhead_init", "muse_lmhead_forward", "muse_lmhead_forward_host",
    "muse_lmhead_launches_per_forward", "muse_lmhead_path_name", "muse_lmhead_device_status",
    "muse_lmhead_destroy", "muse_lmhead_status_string", "muse_lmhead_forward_b1_noalloc",
    "muse_lmhead_noalloc_device_status",
    "muse_lmhead_forward_group", "muse_lmhead_forward_group_host", "muse_lmhead_forward_logprobs",
    "muse_lmhead_init_format",
    "muse_lmhead_clear_device_status", "muse_lmhead_selftest_wait_timeout", "muse_lmhead_set_argmax_key",
)

MUSE_OK = 0
MUSE_MAX_BATCH = 32
MUSE_MAX_SEGMENTS = 4
MUSE_FORMAT_Q5_K = 0
MUSE_FORMAT_Q4_K = 1
FORMATS = {"q5_k": MUSE_FORMAT_Q5_K, "q4_k": MUSE_FORMAT_Q4_K}
BLOCK_BYTES = {"q5_k": 176, "q4_k": 144}
STATUS_WAIT_TIMEOUT = 1
MUSE_ARGMAX_CAPPED = 0      # argmax key: the returned (capped) logit
MUSE_ARGMAX_PRECAP = 1      # argmax key: scale * raw, before the cap
ARGMAX_KEYS = {"capped": MUSE_ARGMAX_CAPPED, "precap": MUSE_ARGMAX_PRECAP}

_lib = None


class MuseGemvSegment(ctypes.Structure):
    """struct muse_gemv_segment of the C header: one matrix of a grouped forward."""
    _fields_ = [("weights", ctypes.c_void_p), ("n_rows", ctypes.c_int64), ("out", ctypes.c_void_p),
                ("scale", ctypes.c_float), ("cap", ctypes.c_float)]


class MuseError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {muse_lmhead_status_string(status)} (status {status})")


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load the compiled library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libmuse_lmhead.so is not built ({LIB_PATH}); run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` or `python q5_lm_head_gb300/_build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.muse_lmhead_init.restype = i32
    lib.muse_lmhead_init.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i32]
    lib.muse_lmhead_init_format.restype = i32
    lib.muse_lmhead_init_format.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i32, i32]
    lib.muse_lmhead_forward.restype = i32
    lib.muse_lmhead_forward.argtypes = [vp, vp, i32, vp, f32, vp, f32, f32, vp, vp, vp]
    lib.muse_lmhead_forward_host.restype = i32
    lib.muse_lmhead_forward_host.argtypes = [vp, vp, i32, vp, f32, vp, f32, f32, vp, vp, vp]
    lib.muse_lmhead_launches_per_forward.restype = i32
    lib.muse_lmhead_launches_per_forward.argtypes = [vp, i32, i32]
    lib.muse_lmhead_path_name.restype = ctypes.c_char_p
    lib.muse_lmhead_path_name.argtypes = [vp, i32]
    lib.muse_lmhead_device_status.restype = i32
    lib.muse_lmhead_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.muse_lmhead_destroy.restype = None
    lib.muse_lmhead_destroy.argtypes = [vp]
    lib.muse_lmhead_status_string.restype = ctypes.c_char_p
    lib.muse_lmhead_status_string.argtypes = [i32]
    lib.muse_lmhead_forward_b1_noalloc.restype = i32
    lib.muse_lmhead_forward_b1_noalloc.argtypes = [i32, vp, vp, f32, vp, i64, i64, f32, f32, vp, vp, vp]
    lib.muse_lmhead_noalloc_device_status.restype = i32
    lib.muse_lmhead_noalloc_device_status.argtypes = [i32, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.muse_lmhead_clear_device_status.restype = i32
    lib.muse_lmhead_clear_device_status.argtypes = [vp, vp]
    lib.muse_lmhead_selftest_wait_timeout.restype = i32
    lib.muse_lmhead_selftest_wait_timeout.argtypes = [vp, vp]
    lib.muse_lmhead_set_argmax_key.restype = i32
    lib.muse_lmhead_set_argmax_key.argtypes = [vp, i32]
    lib.muse_lmhead_forward_logprobs.restype = i32
    lib.muse_lmhead_forward_logprobs.argtypes = [vp, vp, i32, vp, f32, vp, f32, f32, vp, vp, vp, vp]
    lib.muse_lmhead_forward_group.restype = i32
    lib.muse_lmhead_forward_group.argtypes = [vp, vp, vp, f32, ctypes.POINTER(MuseGemvSegment), i32, vp]
    lib.muse_lmhead_forward_group_host.restype = i32
    lib.muse_lmhead_forward_group_host.argtypes = [vp, vp, vp, f32, ctypes.POINTER(MuseGemvSegment), i32, vp]
    _lib = lib
    return lib


# ------------------------------------------------------------ same-named C-ABI calls
def muse_lmhead_init(device: int, n_rows: int, k: int, max_batch: int) -> int:
    """Returns the handle (an integer) or raises MuseError."""
    h = ctypes.c_void_p()
    st = load_library().muse_lmhead_init(ctypes.byref(h), device, n_rows, k, max_batch)
    if st != MUSE_OK:
        raise MuseError(st, "muse_lmhead_init")
    return h.value


def muse_lmhead_init_format(device: int, n_rows: int, k: int, max_batch: int, fmt: int) -> int:
    """Returns the handle (an integer) or raises MuseError."""
    h = ctypes.c_void_p()
    st = load_library().muse_lmhead_init_format(ctypes.byref(h), device, n_rows, k, max_batch, fmt)
    if st != MUSE_OK:
        raise MuseError(st, "muse_lmhead_init_format")
    return h.value


def muse_lmhead_forward(h: int, hidden: int, batch: int, gamma: int | None, eps: float, weights: int,
                        scale: float, cap: float, logits: int, argmax: int | None, stream: int | None) -> int:
    return load_library().muse_lmhead_forward(h, hidden, batch, gamma, eps, weights, scale, cap, logits,
                                              argmax, stream)


def muse_lmhead_forward_host(h: int, hidden_host: int, batch: int, gamma: int | None, eps: float,
                             weights: int, scale: float, cap: float, logits_host: int | None,
                             argmax_host: int | None, stream: int | None) -> int:
    return load_library().muse_lmhead_forward_host(h, hidden_host, batch, gamma, eps, weights, scale, cap,
                                                   logits_host, argmax_host, stream)


def muse_lmhead_launches_per_forward(h: int, batch: int, with_norm: bool) -> int:
    return load_library().muse_lmhead_launches_per_forward(h, batch, int(bool(with_norm)))


def muse_lmhead_path_name(h: int, batch: int) -> str | None:
    r = load_library().muse_lmhead_path_name(h, batch)
    return None if r is None else r.decode()


def muse_lmhead_device_status(h: int) -> int:
    v = ctypes.c_uint32()
    st = load_library().muse_lmhead_device_status(h, ctypes.byref(v))
    if st != MUSE_OK:
        raise MuseError(st, "muse_lmhead_device_status")
    return v.value


def muse_lmhead_destroy(h: int | None) -> None:
    if h:
        load_library().muse_lmhead_destroy(h)


def muse_lmhead_forward_b1_noalloc(device: int, hidden: int, gamma: int | None, eps: float, weights: int,
                                   n_rows: int, k: int, scale: float, cap: float, logits: int,
                                   argmax: int | None, stream: int | None) -> int:
    """Batch-1 forward without a handle that allocates no device memory (see the C header)."""
    return load_library().muse_lmhead_forward_b1_noalloc(device, hidden, gamma, eps, weights, n_rows, k, scale,
                                                         cap, logits, argmax, stream)


def muse_lmhead_noalloc_device_status(device: int, stream: int | None) -> int:
    """Status word of the no-alloc forward on `device`, read after the work
    queued on `stream` and cleared (see the C header); raises on a failed read."""
    v = ctypes.c_uint32()
    st = load_library().muse_lmhead_noalloc_device_status(device, stream, ctypes.byref(v))
    if st != MUSE_OK:
        raise MuseError(st, "muse_lmhead_noalloc_device_status")
    return v.value


def muse_lmhead_status_string(status: int) -> str:
    return load_library().muse_lmhead_status_string(status).decode()


# ------------------------------------------------------------ torch-facing wrapper
def muse_lmhead_clear_device_status(h: int, stream: int | None = None) -> int:
    return load_library().muse_lmhead_clear_device_status(h, stream)


def muse_lmhead_set_argmax_key(h: int | None, key: int) -> int:
    return load_library().muse_lmhead_set_argmax_key(h, key)


def muse_lmhead_selftest_wait_timeout(h: int, stream: int | None = None) -> int:
    return load_library().muse_lmhead_selftest_wait_timeout(h, stream)


def muse_lmhead_forward_logprobs(h: int, hidden: int, batch: int, gamma: int | None, eps: float, weights: int,
                                 scale: float, cap: float, logprobs: int, lse: int | None, argmax: int | None,
                                 stream: int | None) -> int:
    return load_library().muse_lmhead_forward_logprobs(h, hidden, batch, gamma, eps, weights, scale, cap,
                                                       logprobs, lse, argmax, stream)


def muse_lmhead_forward_group(h: int | None, hidden: int, gamma: int | None, eps: float, segments,
                              stream: int | None) -> int:
    """segments: sequence of (weights_ptr, n_rows, out_ptr, scale, cap)."""
    arr = (MuseGemvSegment * max(1, len(segments)))()
    for i, (w, n, o, sc, cp) in enumerate(segments):
        arr[i] = MuseGemvSegment(w, n, o, sc, cp)
    return load_library().muse_lmhead_forward_group(h, hidden, gamma, eps, arr, len(segments), stream)


def muse_lmhead_forward_group_host(h: int | None, hidden_host: int, gamma: int | None, eps: float, segments,
                                   stream: int | None) -> int:
    """segments: sequence of (weights_ptr (device), n_rows, out_ptr (host), scale, cap)."""
    arr = (MuseGemvSegment * max(1, len(segments)))()
    for i, (w, n, o, sc, cp) in enumerate(segments):
        arr[i] = MuseGemvSegment(w, n, o, sc, cp)
    return load_library().muse_lmhead_forward_group_host(h, hidden_host, gamma, eps, arr, len(segments), stream)


class LMHead:
    """A handle for one [n_rows x k] Q5_K (or, fmt="q4_k", Q4_K) matrix and batches up to max_batch."""

    def __init__(self, n_rows: int, k: int, max_batch: int = MUSE_MAX_BATCH, device: int | None = None,
                 fmt: str = "q5_k"):
        import torch
        if fmt not in FORMATS:
            raise ValueError(f"fmt must be one of {sorted(FORMATS)}")
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.n_rows, self.k, self.max_batch = int(n_rows), int(k), int(max_batch)
        self.fmt, self.block_bytes = fmt, BLOCK_BYTES[fmt]
        self.handle = muse_lmhead_init_format(self.device, self.n_rows, self.k, self.max_batch, FORMATS[fmt])

    def close(self):
        if getattr(self, "handle", None):
            muse_lmhead_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _check(self, t, name, dtype, shape=None):
        import torch
        if t.dtype != dtype or not t.is_contiguous() or t.device.type != "cuda" or t.device.index != self.device:
            raise ValueError(f"{name}: need a contiguous {dtype} tensor on cuda:{self.device}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
        return t.data_ptr()

    def forward(self, hidden, weights, gamma=None, eps: float = RMS_EPS, scale: float = LOGIT_SCALE,
                cap: float = SOFTCAP, want_argmax: bool = True, logits=None, argmax=None, stream=None):
        """logits [B, n_rows] f32 (and argmax [B] int32) for hidden [B, k] f32 on the GPU."""
        import torch
        if hidden.dim() == 1:
            hidden = hidden.unsqueeze(0)
        b = hidden.shape[0]
        hp = self._check(hidden, "hidden", torch.float32, (b, self.k))
        wp = self._check(weights, "weights", torch.uint8)
        if weights.numel() != self.n_rows * (self.k // 256) * self.block_bytes:
            raise ValueError("weights: wrong number of bytes for this handle")
        gp = None if gamma is None else self._check(gamma, "gamma", torch.float32, (self.k,))
        if logits is None:
            logits = torch.empty((b, self.n_rows), dtype=torch.float32, device=hidden.device)
        lp = self._check(logits, "logits", torch.float32, (b, self.n_rows))
        ap = None
        if want_argmax:
            if argmax is None:
                argmax = torch.empty((b,), dtype=torch.int32, device=hidden.device)
            ap = self._check(argmax, "argmax", torch.int32, (b,))
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = muse_lmhead_forward(self.handle, hp, b, gp, float(eps), wp, float(scale), float(cap), lp, ap,
                                 s.cuda_stream)
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_forward")
        return (logits, argmax) if want_argmax else logits

    def forward_host(self, hidden_host, weights, gamma=None, eps: float = RMS_EPS, scale: float = LOGIT_SCALE,
                     cap: float = SOFTCAP, logits_host=None, argmax_host=None, stream=None):
        """Host-memory forward: hidden_host [B, k] f32 CPU tensor (pinned for speed); returns CPU tensors.
        Pinned output tensors (the default) are written by the kernels directly through the
        device's mapping of host memory; pageable ones are filled by a copy after the kernels."""
        import torch
        if hidden_host.dim() == 1:
            hidden_host = hidden_host.unsqueeze(0)
        if hidden_host.device.type != "cpu" or hidden_host.dtype != torch.float32 or not hidden_host.is_contiguous():
            raise ValueError("hidden_host: need a contiguous f32 CPU tensor")
        b = hidden_host.shape[0]
        if logits_host is None:
            logits_host = torch.empty((b, self.n_rows), dtype=torch.float32, pin_memory=True)
        if argmax_host is None:
            argmax_host = torch.empty((b,), dtype=torch.int32, pin_memory=True)
        wp = self._check(weights, "weights", torch.uint8)
        gp = None if gamma is None else self._check(gamma, "gamma", torch.float32, (self.k,))
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = muse_lmhead_forward_host(self.handle, hidden_host.data_ptr(), b, gp, float(eps), wp, float(scale),
                                      float(cap), logits_host.data_ptr(), argmax_host.data_ptr(), s.cuda_stream)
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_forward_host")
        return logits_host, argmax_host

    def forward_logprobs(self, hidden, weights, gamma=None, eps: float = RMS_EPS, scale: float = LOGIT_SCALE,
                         cap: float = SOFTCAP, want_argmax: bool = True, logprobs=None, lse=None, argmax=None,
                         stream=None):
        """(logprobs [B, n_rows], lse [B][, argmax [B]]): log-softmax of the capped logits."""
        import torch
        if hidden.dim() == 1:
            hidden = hidden.unsqueeze(0)
        b = hidden.shape[0]
        hp = self._check(hidden, "hidden", torch.float32, (b, self.k))
        wp = self._check(weights, "weights", torch.uint8)
        if weights.numel() != self.n_rows * (self.k // 256) * self.block_bytes:
            raise ValueError("weights: wrong number of bytes for this handle")
        gp = None if gamma is None else self._check(gamma, "gamma", torch.float32, (self.k,))
        if logprobs is None:
            logprobs = torch.empty((b, self.n_rows), dtype=torch.float32, device=hidden.device)
        lp = self._check(logprobs, "logprobs", torch.float32, (b, self.n_rows))
        if lse is None:
            lse = torch.empty((b,), dtype=torch.float32, device=hidden.device)
        sp = self._check(lse, "lse", torch.float32, (b,))
        ap = None
        if want_argmax:
            if argmax is None:
                argmax = torch.empty((b,), dtype=torch.int32, device=hidden.device)
            ap = self._check(argmax, "argmax", torch.int32, (b,))
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = muse_lmhead_forward_logprobs(self.handle, hp, b, gp, float(eps), wp, float(scale), float(cap), lp, sp,
                                          ap, s.cuda_stream)
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_forward_logprobs")
        return (logprobs, lse, argmax) if want_argmax else (logprobs, lse)

    def forward_group(self, hidden, segments, gamma=None, eps: float = RMS_EPS, stream=None):
        """Up to four matrices against one input row in one launch.

        hidden [k] (or [1, k]) f32 on the GPU; segments: sequence of
        (weights uint8 tensor, n_rows, scale, cap, out or None).  Returns the
        list of outputs ([n_rows] f32 each)."""
        import torch
        h = hidden.reshape(-1)
        hp = self._check(h, "hidden", torch.float32, (self.k,))
        gp = None if gamma is None else self._check(gamma, "gamma", torch.float32, (self.k,))
        outs, descs = [], []
        for (w, n, scale, cap, out) in segments:
            wp = self._check(w, "weights", torch.uint8)
            if w.numel() != n * (self.k // 256) * self.block_bytes:
                raise ValueError("weights: wrong number of bytes for n_rows")
            if out is None:
                out = torch.empty((n,), dtype=torch.float32, device=hidden.device)
            op = self._check(out, "out", torch.float32, (n,))
            outs.append(out)
            descs.append((wp, n, op, float(scale), float(cap)))
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = muse_lmhead_forward_group(self.handle, hp, gp, float(eps), descs, s.cuda_stream)
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_forward_group")
        return outs

    def forward_group_host(self, hidden_host, segments, gamma=None, eps: float = RMS_EPS, stream=None):
        """The grouped forward from host memory: hidden_host [k] (or [1, k]) f32
        CPU tensor; segments: sequence of (weights uint8 tensor on the GPU,
        n_rows, scale, cap, out CPU tensor or None).  Outputs default to pinned
        CPU tensors, which the kernel writes directly; returns them."""
        import torch
        h = hidden_host.reshape(-1)
        if h.device.type != "cpu" or h.dtype != torch.float32 or not h.is_contiguous() or h.numel() != self.k:
            raise ValueError("hidden_host: need a contiguous f32 CPU tensor of k values")
        gp = None if gamma is None else self._check(gamma, "gamma", torch.float32, (self.k,))
        outs, descs = [], []
        for (w, n, scale, cap, out) in segments:
            wp = self._check(w, "weights", torch.uint8)
            if w.numel() != n * (self.k // 256) * self.block_bytes:
                raise ValueError("weights: wrong number of bytes for n_rows")
            if out is None:
                out = torch.empty((n,), dtype=torch.float32, pin_memory=True)
            if out.device.type != "cpu" or out.dtype != torch.float32 or not out.is_contiguous() or out.numel() != n:
                raise ValueError("out: need a contiguous f32 CPU tensor of n_rows values")
            outs.append(out)
            descs.append((wp, n, out.data_ptr(), float(scale), float(cap)))
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = muse_lmhead_forward_group_host(self.handle, h.data_ptr(), gp, float(eps), descs, s.cuda_stream)
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_forward_group_host")
        return outs

    def set_argmax_key(self, key: str) -> None:
        """"capped" (the returned logit; the default) or "precap" (scale * raw, before the cap)."""
        if key not in ARGMAX_KEYS:
            raise ValueError(f"argmax key: one of {sorted(ARGMAX_KEYS)}")
        st = muse_lmhead_set_argmax_key(self.handle, ARGMAX_KEYS[key])
        if st != MUSE_OK:
            raise MuseError(st, "muse_lmhead_set_argmax_key")

    def path_name(self, batch: int) -> str | None:
        return muse_lmhead_path_name(self.handle, batch)

    def launches_per_forward(self, batch: int, with_norm: bool) -> int:
        return muse_lmhead_launches_per_forward(self.handle, batch, with_norm)

    def device_status(self) -> int:
        return muse_lmhead_device_status(self.handle)
