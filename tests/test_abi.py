"""The C-ABI library builds, loads, exports every entry point include/*.h
declares, and rejects bad arguments on the host.

No test here launches a kernel: every call either fails host-side validation or
has no work, so none reaches the GPU (these run without one).
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

from grammar_constrained_logit_gb300 import _lib, build  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(lp_\w+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_header_is_plain_c(tmp_path):
    """include/lp.h is a C header: a C99 file that includes it and names its types
    compiles with the system C compiler (no C++ in the interface)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if cc is None or not os.path.isdir(cuda_inc):
        pytest.skip("no C compiler or CUDA headers")
    src = tmp_path / "use_lp.c"
    src.write_text('#include "lp.h"\n'
                   "int main(void) {\n"
                   "  lp_sampling_params p = {0};\n"
                   "  lp_dtype d = LP_BF16;\n"
                   "  (void)p; (void)d;\n"
                   "  return (int)LP_OK;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only",
                        f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda_inc}", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_header_declares_the_entry_points():
    assert set(_lib.EXPORTS) <= _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        s = lib.lp_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.lp_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation


def _apply(lib, **kw):
    a = dict(logits=FAKE, dt=2, B=4, cols=64, stride=64, bm=FAKE, bm_rows=4, words=2,
             bm_stride=2, vocab=-1, idx=None, n=0)
    a.update(kw)
    return lib.lp_apply_token_bitmask(a["logits"], a["dt"], a["B"], a["cols"], a["stride"],
                                      a["bm"], a["bm_rows"], a["words"], a["bm_stride"],
                                      a["vocab"], a["idx"], a["n"], None)


@pytest.mark.parametrize("kw", [
    dict(B=-1), dict(cols=-1), dict(stride=63), dict(words=-1), dict(bm_stride=1),
    dict(vocab=65), dict(vocab=70, words=2, cols=100, stride=100), dict(n=-1),
    dict(n=3, idx=None), dict(bm_rows=3), dict(bm_rows=-1), dict(logits=None),
    dict(bm=None),
])
def test_apply_rejects(lib, kw):
    assert _apply(lib, **kw) == _lib.LP_ERR_INVALID_ARGUMENT


def test_apply_unsupported_dtype(lib):
    assert _apply(lib, dt=7) == _lib.LP_ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("kw", [dict(B=0), dict(vocab=0), dict(idx=FAKE, n=0),
                                dict(B=0, logits=None, bm=None)])
def test_apply_no_work_is_ok(lib, kw):
    assert _apply(lib, **kw) == _lib.LP_OK


def _rows(lib, **kw):
    a = dict(logits=FAKE, dt=2, B=4, cols=64, stride=64, bm=FAKE, bm_rows=4, words=2,
             bm_stride=2, vocab=-1, flags=None, has=None)
    a.update(kw)
    return lib.lp_apply_token_bitmask_rows(a["logits"], a["dt"], a["B"], a["cols"], a["stride"],
                                           a["bm"], a["bm_rows"], a["words"], a["bm_stride"],
                                           a["vocab"], a["flags"], a["has"], None)


@pytest.mark.parametrize("kw", [
    dict(B=-1), dict(cols=-1), dict(stride=63), dict(words=-1), dict(bm_stride=1),
    dict(vocab=65), dict(bm_rows=3), dict(logits=None), dict(bm=None),
    dict(logits=None, has=FAKE), dict(bm=None, flags=FAKE, has=FAKE),
])
def test_apply_rows_rejects(lib, kw):
    # every rejection happens before the report is zeroed: nothing is enqueued
    assert _rows(lib, **kw) == _lib.LP_ERR_INVALID_ARGUMENT


def test_apply_rows_unsupported_dtype(lib):
    assert _rows(lib, dt=5) == _lib.LP_ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("kw", [dict(B=0), dict(B=0, has=FAKE), dict(vocab=0),
                                dict(vocab=0, logits=None, bm=None)])
def test_apply_rows_no_work_is_ok(lib, kw):
    assert _rows(lib, **kw) == _lib.LP_OK


def _oop(lib, **kw):
    a = dict(out=ctypes.c_void_p(0x2000), out_stride=64, logits=FAKE, dt=0, B=4, cols=64,
             stride=64, bm=FAKE, bm_rows=4, words=2, bm_stride=2, fill=-1.0, vocab=-1,
             idx=None, n=0)
    a.update(kw)
    return lib.lp_apply_packed_bitmask(a["out"], a["out_stride"], a["logits"], a["dt"], a["B"],
                                       a["cols"], a["stride"], a["bm"], a["bm_rows"],
                                       a["words"], a["bm_stride"], a["fill"], a["vocab"],
                                       a["idx"], a["n"], None)


@pytest.mark.parametrize("kw", [dict(out_stride=10), dict(out=None), dict(logits=None),
                                dict(bm=None), dict(stride=3), dict(vocab=100)])
def test_out_of_place_rejects(lib, kw):
    assert _oop(lib, **kw) == _lib.LP_ERR_INVALID_ARGUMENT


def test_out_of_place_no_work(lib):
    assert _oop(lib, B=0) == _lib.LP_OK
    assert _oop(lib, cols=0, stride=0, out_stride=0) == _lib.LP_OK


def _params():
    p = _lib.SamplingParams()
    p.temperature_scalar, p.top_k_scalar, p.top_p_scalar, p.min_p_scalar = 1.0, 0, 1.0, 0.0
    return p


WS = ctypes.c_void_p(0x100000)  # 256-byte aligned; never dereferenced
WSN = 1 << 40


def test_sample_validation(lib):
    p = _params()
    out = ctypes.c_void_p(0x3000)
    call = lambda logits, dt, B, V, stride, params, o, ws=WS, wsn=WSN: lib.lp_sample(  # noqa: E731
        logits, dt, B, V, stride, params, o, ws, wsn, None)
    assert call(FAKE, 0, -1, 10, 10, ctypes.byref(p), out) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(FAKE, 0, 2, 10, 9, ctypes.byref(p), out) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(FAKE, 5, 2, 10, 10, ctypes.byref(p), out) == _lib.LP_ERR_UNSUPPORTED_DTYPE
    assert call(FAKE, 0, 2, 10, 10, None, out) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(FAKE, 0, 2, 10, 10, ctypes.byref(p), None) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(None, 0, 0, 10, 10, ctypes.byref(p), None, None, 0) == _lib.LP_OK
    # sizes past the kernels' 32-bit index range are refused before any launch
    huge = 2**31
    assert call(FAKE, 1, 2, huge, huge, ctypes.byref(p), out) == _lib.LP_ERR_TOO_LARGE
    assert call(FAKE, 1, 2**28, 8, 8, ctypes.byref(p), out) == _lib.LP_ERR_TOO_LARGE
    # the workspace: present, 256-byte aligned and at least the stated size
    need = lib.lp_sample_workspace_bytes(0, 2, 10)
    assert need > 0
    assert call(FAKE, 0, 2, 10, 10, ctypes.byref(p), out, None, WSN) == \
        _lib.LP_ERR_INVALID_ARGUMENT
    assert call(FAKE, 0, 2, 10, 10, ctypes.byref(p), out, WS, need - 1) == \
        _lib.LP_ERR_INVALID_ARGUMENT
    assert call(FAKE, 0, 2, 10, 10, ctypes.byref(p), out, ctypes.c_void_p(0x100010), WSN) == \
        _lib.LP_ERR_INVALID_ARGUMENT


def test_workspace_bytes(lib):
    f = lib.lp_sample_workspace_bytes
    assert f(0, 0, 1000) == 0
    assert f(7, 4, 1000) == -1 and f(0, -1, 10) == -1 and f(0, 1, -1) == -1
    for dt in (0, 1, 2):
        sizes = [f(dt, B, V) for B, V in ((1, 1003), (64, 128256), (256, 131072), (1024, 202048))]
        assert all(n > 0 and n % 256 == 0 for n in sizes)
        assert sizes == sorted(sizes)  # more rows or tokens never need less
    # monotone on a fine grid of shapes (tile halving rounds up, so a naive plan
    # could need more scratch for a narrower vocabulary, e.g. 98304 vs 131072)
    Bs = (1, 3, 64, 255, 256, 1000, 1024, 5000, 16384, 40000)
    Vs = (1, 33, 1003, 8192, 32000, 65536, 98304, 100000, 131072, 202048, 262144, 1 << 20)
    for dt in (0, 1, 2):
        grid = [[f(dt, B, V) for V in Vs] for B in Bs]
        for row in grid:
            assert row == sorted(row)
        for col in zip(*grid):
            assert list(col) == sorted(col)
    # bounded: tile summaries and slots are a few percent of the logits, the pool
    # at most 128 MB
    for dt, eb in ((0, 4), (2, 2)):
        for B, V in ((1 << 20, 131072), (4096, 32000), (64, 1 << 24)):
            assert f(dt, B, V) < B * V * eb * 7 // 100 + (130 << 20)


def test_mask_and_sample_validation(lib):
    p = _params()
    out = ctypes.c_void_p(0x3000)
    call = lambda **kw: lib.lp_mask_and_sample(  # noqa: E731
        kw.get("logits", FAKE), 2, kw.get("B", 4), kw.get("cols", 64), kw.get("stride", 64),
        kw.get("bm", FAKE), kw.get("bm_rows", 4), kw.get("words", 2), kw.get("bm_stride", 2),
        kw.get("vocab", -1), kw.get("idx", None), kw.get("n", 0), ctypes.byref(p), out,
        kw.get("ws", WS), kw.get("wsn", WSN), None)
    assert call(vocab=65) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(bm_rows=3) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(n=2) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(bm_stride=1) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(stride=10) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(B=0) == _lib.LP_OK
    assert call(ws=None) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(wsn=16) == _lib.LP_ERR_INVALID_ARGUMENT


def _upload(lib, **kw):
    a = dict(dev=FAKE, dstride=4, host=FAKE, hstride=4, rows=3, words=4, dflags=None,
             hflags=None)
    a.update(kw)
    return lib.lp_upload_bitmask(a["dev"], a["dstride"], a["host"], a["hstride"], a["rows"],
                                 a["words"], a["dflags"], a["hflags"], None, None)


@pytest.mark.parametrize("kw", [dict(rows=-1), dict(words=-1), dict(dstride=3), dict(hstride=2),
                                dict(dflags=FAKE), dict(hflags=FAKE), dict(dev=None),
                                dict(host=None)])
def test_upload_rejects(lib, kw):
    assert _upload(lib, **kw) == _lib.LP_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("kw", [dict(rows=0), dict(words=0, dev=None, host=None)])
def test_upload_no_work_is_ok(lib, kw):
    assert _upload(lib, **kw) == _lib.LP_OK


def test_mask_and_sample_slots_validation(lib):
    p = _params()
    out = ctypes.c_void_p(0x3000)
    call = lambda **kw: lib.lp_mask_and_sample_slots(  # noqa: E731
        kw.get("logits", FAKE), 2, kw.get("B", 8), 64, 64, FAKE, 8, 2, 2, -1, None, 0,
        ctypes.byref(p), kw.get("rps", 4), kw.get("seeds", None), out, kw.get("ws", WS),
        kw.get("wsn", WSN), None)
    assert call(rps=0) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(rps=-2) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(rps=3) == _lib.LP_ERR_INVALID_ARGUMENT   # 8 rows are not slots of 3
    assert call(ws=None) == _lib.LP_ERR_INVALID_ARGUMENT
    assert call(B=0) == _lib.LP_OK
    assert call(B=0, rps=5) == _lib.LP_OK


def test_philox_validation(lib):
    assert lib.lp_philox4x32_10(None, None, None, -1, None) == _lib.LP_ERR_INVALID_ARGUMENT
    assert lib.lp_philox4x32_10(None, None, None, 0, None) == _lib.LP_OK
    assert lib.lp_philox4x32_10(None, FAKE, FAKE, 3, None) == _lib.LP_ERR_INVALID_ARGUMENT


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "nope.so"))
