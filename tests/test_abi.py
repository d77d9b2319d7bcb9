"""The C ABI library builds, loads and exports every symbol the header
declares; host-side argument checks reject bad calls before any CUDA work
(these paths need no GPU)."""
import ctypes
import os
import re

import pytest

from mla_decode_attention_kv_gb300 import _ffi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return _ffi.lib(path)


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "mla_dcp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text))


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert {"mla_dcp_decode_partial", "mla_lse_combine", "mla_vup", "mla_lse_combine_vup",
            "mla_gather_kv", "mla_get_error_string"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mla_dcp.h but not exported"
    assert set(_ffi.SIGNATURES) == names


def test_error_strings(lib):
    assert lib.mla_get_error_string(0) == b"ok"
    for code in range(1, 8):
        assert lib.mla_get_error_string(code) != b"unknown status"
    assert lib.mla_device_error_string(1).startswith(b"block_table")
    assert lib.mla_device_error_string(3).startswith(b"seq_lens")
    assert lib.mla_version() >= 100


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)       # 8-byte aligned only


def _partial(lib, **over):
    args = dict(q_abs=FAKE, q_pe=FAKE, kv=FAKE, table=FAKE, lens=FAKE, cur=None, B=2, q=1,
                H=128, nb=10, bs=32, mb=5, S=2, scale=0.07, idt=0, pdt=0, o=FAKE, l=FAKE,
                err=None, ws=None, wsb=0)
    args.update(over)
    a = args
    return lib.mla_dcp_decode_partial(a["q_abs"], a["q_pe"], a["kv"], a["table"], a["lens"],
                                      a["cur"], a["B"], a["q"], a["H"], a["nb"], a["bs"],
                                      a["mb"], a["S"], a["scale"], a["idt"], a["pdt"], a["o"],
                                      a["l"], a["err"], a["ws"], a["wsb"], None)


def test_partial_host_checks(lib):
    assert _partial(lib, q_abs=None) == 1
    assert _partial(lib, idt=2) == 3                 # fp32 inputs unsupported
    assert _partial(lib, pdt=7) == 3
    assert _partial(lib, H=129) == 2
    assert _partial(lib, q=0) == 2
    assert _partial(lib, q=65) == 2
    assert _partial(lib, scale=0.0) == 2
    assert _partial(lib, S=0) == 5
    assert _partial(lib, S=65) == 5
    assert _partial(lib, bs=48) == 6
    assert _partial(lib, kv=ODD) == 4
    assert _partial(lib, ws=ctypes.c_void_p(0x10010), wsb=1 << 20) == 4   # workspace not 256-aligned


def _partial_fp8(lib, kv_scale=0.01, **over):
    args = dict(q_abs=FAKE, q_pe=FAKE, kv=FAKE, table=FAKE, lens=FAKE, cur=None, B=2, q=1,
                H=128, nb=10, bs=32, mb=5, S=2, scale=0.07, idt=0, pdt=0, o=FAKE, l=FAKE,
                err=None, ws=None, wsb=0, slices=1)
    args.update(over)
    a = args
    return lib.mla_dcp_decode_partial_fp8(a["q_abs"], a["q_pe"], a["kv"], a["table"], a["lens"],
                                          a["cur"], a["B"], a["q"], a["H"], a["nb"], a["bs"],
                                          a["mb"], a["S"], a["scale"], kv_scale, a["idt"],
                                          a["pdt"], a["o"], a["l"], a["err"], a["ws"], a["wsb"],
                                          a["slices"], None)


def test_partial_fp8_host_checks(lib):
    """The E4M3-cache entry point runs the same checks, plus kv_scale."""
    assert _partial_fp8(lib, q_abs=None) == 1
    assert _partial_fp8(lib, idt=2) == 3
    assert _partial_fp8(lib, H=129) == 2
    assert _partial_fp8(lib, q=65) == 2
    assert _partial_fp8(lib, S=65) == 5
    assert _partial_fp8(lib, bs=48) == 6
    assert _partial_fp8(lib, kv=ODD) == 4
    assert _partial_fp8(lib, kv_scale=0.0) == 2
    assert _partial_fp8(lib, kv_scale=-1.0) == 2
    assert _partial_fp8(lib, kv_scale=float("inf")) == 2
    assert _partial_fp8(lib, kv_scale=float("nan")) == 2
    assert _partial_fp8(lib, kv_scale=1e38, scale=1e3) == 2     # scale * kv_scale overflows
    assert _partial_fp8(lib, slices=3) == 2                     # 3 does not divide 128


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.mla_dcp_decode_partial_workspace_size(0, 1, 2, 0) == 0
    assert lib.mla_dcp_decode_partial_workspace_size(2, 65, 2, 0) == 0
    assert lib.mla_dcp_decode_partial_workspace_size(2, 1, 65, 1) == 0


def test_combine_vup_gather_host_checks(lib):
    assert lib.mla_lse_combine(None, FAKE, 2, None, None, 4, 8, 0, 0, FAKE, None, None) == 1
    assert lib.mla_lse_combine(FAKE, FAKE, 2, FAKE, None, 4, 8, 0, 0, FAKE, None, None) == 1
    assert lib.mla_lse_combine(FAKE, FAKE, 0, None, None, 4, 8, 0, 0, FAKE, None, None) == 5
    assert lib.mla_lse_combine(FAKE, FAKE, 2, None, None, 4, 200, 0, 0, FAKE, None, None) == 2
    assert lib.mla_lse_combine(FAKE, FAKE, 2, None, None, 4, 8, 5, 0, FAKE, None, None) == 3
    assert lib.mla_lse_combine(ODD, FAKE, 2, None, None, 4, 8, 0, 0, FAKE, None, None) == 4
    assert lib.mla_vup(FAKE, FAKE, 4, 8, 2, FAKE, None, None) == 3      # fp32 MMA unsupported
    assert lib.mla_vup(FAKE, FAKE, 0, 8, 0, FAKE, None, None) == 2
    assert lib.mla_vup(None, FAKE, 4, 8, 0, FAKE, None, None) == 1
    assert lib.mla_lse_combine_vup(FAKE, FAKE, 70, None, None, FAKE, 4, 8, 0, 0, FAKE, None,
                                   None, None, None) == 5
    assert lib.mla_gather_kv(FAKE, FAKE, FAKE, 0, 4, 32, 2, 64, FAKE, None, None) == 2
    assert lib.mla_gather_kv(FAKE, FAKE, FAKE, 2, 4, 32, 2, 64, ODD, None, None) == 4
