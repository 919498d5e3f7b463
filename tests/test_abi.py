"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mla_paged.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(mla_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_paged_decode", "mla_paged_prefill", "mla_workspace_bytes", "mla_status_string",
              "mla_read_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(lib.library_path())
    for n in declared_functions():
        assert hasattr(handle, n), n


def _dims(lib, **kw):
    d = dict(batch=2, num_qo_heads=16, num_pages=4, page_size=64, num_kv_indices=10, total_q=0,
             num_workers=4)
    d.update(kw)
    return lib.make_dims(**d)


FAKE = 0x10000  # never dereferenced: every case below fails before any CUDA call


def _decode(lib, dims, ptrs=None, ws_bytes=1 << 30, ws=FAKE):
    p = dict(q_nope=FAKE, q_pe=FAKE, ckv=FAKE, kpe=FAKE, indptr=FAKE, indices=FAKE, out=FAKE, lse=FAKE)
    p.update(ptrs or {})
    v = ctypes.c_void_p
    return lib.lib().mla_paged_decode(v(p["q_nope"]), v(p["q_pe"]), v(p["ckv"]), v(p["kpe"]),
                                      v(p["indptr"]), v(p["indices"]), 0.1, v(p["out"]), v(p["lse"]),
                                      ctypes.byref(dims) if dims is not None else None,
                                      v(ws), ws_bytes, 0, None)


def test_host_argument_errors(lib):
    assert _decode(lib, None) == -1                                       # MLA_ERR_NULL
    assert _decode(lib, _dims(lib, num_qo_heads=0)) == -2                 # MLA_ERR_DIMS
    assert _decode(lib, _dims(lib, num_qo_heads=129)) == -2
    assert _decode(lib, _dims(lib, page_size=0)) == -2
    assert _decode(lib, _dims(lib, num_pages=1 << 20, page_size=1 << 12)) == -2
    d = _dims(lib)
    d.head_dim_ckv = 576
    assert _decode(lib, d) == -2
    assert _decode(lib, _dims(lib), {"q_pe": 0}) == -1
    assert _decode(lib, _dims(lib), {"indices": 0}) == -1
    assert _decode(lib, _dims(lib), {"ckv": FAKE + 8}) == -3              # MLA_ERR_ALIGN
    assert _decode(lib, _dims(lib), ws_bytes=16) == -4                    # MLA_ERR_WORKSPACE
    assert _decode(lib, _dims(lib), ws=0) == -4
    # An empty batch is a no-op that succeeds without a device.
    assert _decode(lib, _dims(lib, batch=0, num_kv_indices=0)) == 0


def test_prefill_needs_qo_indptr(lib):
    v = ctypes.c_void_p
    d = _dims(lib, total_q=5)
    st = lib.lib().mla_paged_prefill(v(FAKE), v(FAKE), v(FAKE), v(FAKE), None, v(FAKE), v(FAKE), 0.1,
                                     v(FAKE), v(FAKE), ctypes.byref(d), v(FAKE), 1 << 30, 0, None)
    assert st == -1


def test_workspace_size_grows_with_workers_and_heads(lib):
    a = lib.workspace_bytes(_dims(lib, num_workers=4, num_qo_heads=16), False)
    b = lib.workspace_bytes(_dims(lib, num_workers=8, num_qo_heads=16), False)
    c = lib.workspace_bytes(_dims(lib, num_workers=8, num_qo_heads=128), False)
    assert 0 < a < b < c
    # partial outputs dominate: workers x 2 slots x heads x 512 fp32
    assert c >= 8 * 2 * 128 * 512 * 4
    assert lib.workspace_bytes(_dims(lib, num_qo_heads=0), False) == 0


def test_status_strings(lib):
    for code in range(0, -10, -1):
        s = lib.string_of(code)
        assert s.startswith("MLA_")


def _mtp(lib, dims, q_len, ws_bytes=1 << 30):
    v = ctypes.c_void_p
    return lib.lib().mla_paged_decode_mtp(v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), 0.1, v(FAKE),
                                          v(FAKE), ctypes.byref(dims), q_len, v(FAKE), ws_bytes, 0, None)


def test_mtp_host_argument_errors(lib):
    assert _mtp(lib, _dims(lib, num_qo_heads=16), 0) == -2          # q_len < 1
    assert _mtp(lib, _dims(lib, num_qo_heads=16), 9) == -2          # 9 x 16 rows > 128
    assert _mtp(lib, _dims(lib, num_qo_heads=128), 2) == -2
    assert _mtp(lib, _dims(lib, num_qo_heads=16), 8, ws_bytes=16) == -4
    assert _mtp(lib, _dims(lib, num_qo_heads=16, batch=0, num_kv_indices=0), 4) == 0


def test_mtp_workspace_is_decode_workspace_of_packed_rows(lib):
    for h, q in ((16, 4), (32, 4), (8, 3), (128, 1)):
        a = lib.workspace_bytes_mtp(_dims(lib, num_qo_heads=h), q)
        b = lib.workspace_bytes(_dims(lib, num_qo_heads=h * q), False)
        assert a == b > 0
    assert lib.workspace_bytes_mtp(_dims(lib, num_qo_heads=16), 9) == 0
    assert lib.workspace_bytes_mtp(_dims(lib, num_qo_heads=16), 0) == 0
