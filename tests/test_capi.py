"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
every call here returns before touching the device)."""
import ctypes
import glob
import os
import re

import pytest

from paged_kv_cache_06_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?!typedef)[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, re.M):
            if m.group(1) not in ("if", "while", "sizeof", "defined"):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("paged_kv_append", "paged_attention_decode", "paged_attention_workspace_size",
              "paged_attention_padded_decode", "pkv_status_string", "pkv_check_error",
              "pkv_bm_create", "pkv_bm_admit", "pkv_bm_append_slot", "pkv_bm_free"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ops.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    assert ops.status_string(0) == "PKV_OK"
    assert ops.status_string(3) == "PKV_ERR_WORKSPACE"
    assert ops.status_string(12345) == "PKV_ERR_UNKNOWN"
    assert ops.lib().pkv_abi_version() >= 1


def test_workspace_size_host_arithmetic():
    ws = ops.workspace_size(32, 12, 2, 128, 4096, 64)
    assert ws > 0 and ws % 256 == 0
    assert ops.workspace_size(32, 12, 2, 128, 8192, 64) >= ws  # grows with the bound
    assert ops.workspace_size(32, 12, 2, 64, 4096, 64) == 0   # head_dim 64 not built
    assert ops.workspace_size(32, 12, 5, 128, 4096, 64) == 0  # 12 % 5 != 0
    assert ops.workspace_size(32, 12, 1, 128, 4096, 64) == 0  # group of 12 > 8


FAKE = ctypes.c_void_p(0x100000)  # aligned, non-null; never dereferenced by these calls


def _decode(**kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, rows=4, hq=12, hk=2, d=128, bs=16,
             scale=0.088, mbpr=16, nb=64, msl=200, ws=FAKE, wsb=0, err=None, stream=None)
    a.update(kw)
    return ops.lib().paged_attention_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["sl"],
                                            a["rows"], a["hq"], a["hk"], a["d"], a["bs"], a["scale"],
                                            a["mbpr"], a["nb"], a["msl"], a["ws"], a["wsb"],
                                            a["err"], a["stream"])


def test_decode_rejects_bad_arguments_before_launch():
    assert _decode(d=64) == UNSUPPORTED
    assert _decode(hq=12, hk=1) == UNSUPPORTED
    assert _decode(hq=12, hk=5) == INVALID
    assert _decode(out=None) == INVALID
    assert _decode(bt=None) == INVALID
    assert _decode(q=ctypes.c_void_p(0x100008)) == INVALID     # not 16-byte aligned
    assert _decode(msl=16 * 16 + 1) == INVALID                 # beyond the table
    assert _decode(bs=0) == INVALID
    assert _decode(scale=float("nan")) == INVALID
    assert _decode(wsb=0) == WORKSPACE
    assert _decode(ws=None, wsb=1 << 30) == WORKSPACE
    assert _decode(rows=0, out=None) == 0                      # nothing to do


def test_append_rejects_bad_arguments_before_launch():
    f = ops.lib().paged_kv_append
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 12, 16, 16, 64, None, None) == UNSUPPORTED
    assert f(None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 16, 64, None, None) == INVALID
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 0, 16, 64, None, None) == INVALID
    assert f(None, None, None, None, None, None, 0, 2, 128, 16, 16, 64, None, None) == 0


def test_padded_rejects_bad_arguments_before_launch():
    f = ops.lib().paged_attention_padded_decode
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 12, 2, 96, 0.1, FAKE, 1 << 30, None, None) == UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 12, 2, 128, 0.1, FAKE, 0, None, None) == WORKSPACE
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 256, 12, 2, 128, 0.1, FAKE, 1 << 30, None, None) == INVALID


def test_ops_refuse_cpu_tensors():
    import torch
    x = torch.zeros(4, 12, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        ops.decode(x, x, x, x, x, x, 0.1, 16, x)
