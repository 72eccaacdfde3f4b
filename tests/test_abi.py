"""The C ABI library builds, loads and exports what include/ewg.h declares (no GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

import embedding_weight_grad_gb300 as ewg
from embedding_weight_grad_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ewg.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return ewg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ewg_[a-z_]+)\s*\(", src)))


def header_defines():
    out = {}
    for m in re.finditer(r"#define\s+(EWG_[A-Z0-9_]+)\s+(.+)", open(HEADER).read()):
        val = m.group(2).split("/*")[0].strip()
        try:
            out[m.group(1)] = int(eval(val.replace("(", " ( ").replace(")", " ) ")))
        except Exception:
            pass
    return out


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    nm = subprocess.run(["nm", "-D", "--defined-only", ewg.library_path()], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ewg_[a-z_]+)\b", nm))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_debug_hooks_only_in_the_checked_build():
    """include/ewg_debug.h declares test hooks that libewg_debug.so exports and libewg.so
    does not."""
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "ewg_debug.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(ewg_[a-z_]+)\s*\(", src)))
    assert names == ["ewg_debug_lookback_probe"]
    dbg = cuda_build.build(debug=True)
    nm = lambda path: set(re.findall(r"\bT (ewg_[a-z_]+)\b", subprocess.run(
        ["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout))
    assert set(names) <= nm(dbg)
    assert not set(names) & nm(ewg.library_path())


def test_constants_match_binding():
    d = header_defines()
    assert d["EWG_MIN_TOKENS"] == ewg.MIN_TOKENS == 3073
    assert d["EWG_MAX_TOKENS"] == ewg.MAX_TOKENS
    assert d["EWG_NROWS"] == ewg.NROWS == 10
    assert (d["EWG_INT32"], d["EWG_INT64"], d["EWG_BF16"], d["EWG_FP32"]) == (0, 1, 2, 3)
    assert d["EWG_OK"] == ewg.OK and d["EWG_ERR_ID_OUT_OF_RANGE"] == ewg.ERR_ID_OUT_OF_RANGE


def test_host_only_entry_points(lib):
    assert lib.ewg_version() == 1
    assert lib.ewg_status_string(0) == b"EWG_OK"
    assert lib.ewg_status_string(4) == b"EWG_ERR_ID_OUT_OF_RANGE"
    assert lib.ewg_status_string(99) == b"EWG_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    # out of range -> 0
    assert ewg.workspace_bytes(0, 256) == 0
    assert ewg.workspace_bytes(4096, 12) == 0
    assert ewg.workspace_bytes(ewg.MAX_TOKENS + 1, 256) == 0
    # grows with tokens and hidden; holds the fp32 partial rows of up to 2n/11 + 1 chunks
    for n, h in [(4096, 256), (8192, 7168), (65536, 7168), (131072, 8192)]:
        b = ewg.workspace_bytes(n, h)
        assert b % 256 == 0
        assert b >= (2 * n // 11 + 1) * h * 4 + n * 64
        assert b < (2 * n // 11 + 1) * h * 4 * 1.1 + n * 200 + (1 << 20)
    assert ewg.workspace_bytes(8192, 7168) < ewg.workspace_bytes(8193, 7168)
    assert ewg.workspace_bytes(8192, 7168) < ewg.workspace_bytes(8192, 7176)


def test_host_workspace_bytes(lib):
    # the ordinary workspace plus 256-aligned copies of ids and grad; 0 when unsupported
    n, h = 8192, 7168
    base = ewg.workspace_bytes(n, h)
    got = lib.ewg_host_workspace_bytes(n, h, 1, 2)          # int64 ids, bf16 grad
    assert got % 256 == 0 and got >= base + n * 8 + n * h * 2
    assert got < base + n * 8 + n * h * 2 + 512
    assert lib.ewg_host_workspace_bytes(n, h, 0, 3) >= base + n * 4 + n * h * 4
    assert lib.ewg_host_workspace_bytes(n, h, 2, 2) == 0     # ids dtype not an integer
    assert lib.ewg_host_workspace_bytes(n, h, 1, 1) == 0     # grad dtype not a float
    assert lib.ewg_host_workspace_bytes(0, h, 1, 2) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """With the shared library absent the binding raises instead of computing anything."""
    import importlib
    mod = importlib.reload(ewg)
    monkeypatch.setattr(mod, "_LIB_PATH", str(tmp_path / "libewg.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(ImportError):
        mod.lib()
