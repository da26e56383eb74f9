"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
symbol the public header declares, and rejects bad arguments before touching
CUDA (host-only validation paths; no compute call is made)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muse_lmhead.h")


@pytest.fixture(scope="module")
def lib():
    from q5_lm_head_gb300 import _build
    import q5_lm_head_gb300 as mlh
    _build.build()
    return mlh.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muse_lmhead_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("muse_lmhead_init", "muse_lmhead_forward", "muse_lmhead_destroy",
                     "muse_lmhead_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import q5_lm_head_gb300 as mlh
    out = subprocess.run(["nm", "-D", "--defined-only", mlh.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (muse_lmhead_\w+)$", out, flags=re.M))
    declared = set(_declared_functions())
    assert declared <= exported, declared - exported
    assert set(mlh.EXPORTED_SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name)


def test_status_strings(lib):
    import q5_lm_head_gb300 as mlh
    for code in range(0, -9, -1):
        s = mlh.muse_lmhead_status_string(code)
        assert s and s != "unknown status"
    assert mlh.muse_lmhead_status_string(-99) == "unknown status"


def test_validation_fails_closed_without_cuda(lib):
    # every rejection below happens before the library makes any CUDA call
    vp = ctypes.c_void_p
    h = vp()
    assert lib.muse_lmhead_init(None, 0, 10, 256, 1) == -1
    assert lib.muse_lmhead_init(ctypes.byref(h), 0, 0, 256, 1) == -2      # n_rows < 1
    assert lib.muse_lmhead_init(ctypes.byref(h), 0, 10, 300, 1) == -2     # k % 256
    assert lib.muse_lmhead_init(ctypes.byref(h), 0, 10, 0, 1) == -2
    assert lib.muse_lmhead_init(ctypes.byref(h), 0, 10, 256, 0) == -3     # max_batch
    assert lib.muse_lmhead_init(ctypes.byref(h), 0, 10, 256, 33) == -3
    assert lib.muse_lmhead_init_format(ctypes.byref(h), 0, 10, 256, 1, 2) == -5   # unknown weight format
    assert lib.muse_lmhead_init_format(None, 0, 10, 256, 1, 1) == -1
    assert h.value is None
    assert lib.muse_lmhead_forward(None, 16, 1, None, 1e-5, 16, 1.0, 0.0, 16, None, None) == -1
    assert lib.muse_lmhead_forward_host(None, 16, 1, None, 1e-5, 16, 1.0, 0.0, 16, None, None) == -1
    assert lib.muse_lmhead_launches_per_forward(None, 1, 1) == -1
    import q5_lm_head_gb300 as mlh
    seg = (mlh.MuseGemvSegment * 1)()
    assert lib.muse_lmhead_forward_group(None, 16, None, 1e-5, seg, 1, None) == -1
    assert lib.muse_lmhead_forward_group_host(None, 16, None, 1e-5, seg, 1, None) == -1
    assert lib.muse_lmhead_forward_logprobs(None, 16, 1, None, 1e-5, 16, 1.0, 0.0, 16, None, None, None) == -1
    assert lib.muse_lmhead_clear_device_status(None, None) == -1
    assert lib.muse_lmhead_selftest_wait_timeout(None, None) == -1
    assert lib.muse_lmhead_path_name(None, 1) is None
    assert lib.muse_lmhead_set_argmax_key(None, 0) == -1
    lib.muse_lmhead_destroy(None)


def test_binding_fails_loudly_when_library_missing(tmp_path, monkeypatch):
    import q5_lm_head_gb300 as mlh
    monkeypatch.setattr(mlh, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(mlh, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        mlh.load_library()
