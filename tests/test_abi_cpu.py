"""The C-ABI library builds, loads and exports every symbol include/mla.h
declares; host-side argument checks reject bad calls before touching a GPU.
No compute call is made here (no GPU in this environment)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def L():
    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api
    return api.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def header_define(name):
    m = re.search(rf"#define\s+{name}\s+(\d+)", open(HEADER).read())
    return int(m.group(1))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("mla_get_metadata", "mla_absorb_q", "mla_decode_paged", "mla_out_proj", "mla_read_device_error",
              "mla_workspace_size", "mla_default_num_parts"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in mla.h but not exported by libmla.so"


def test_library_is_built_for_sm_103a(L):
    from mla_paged_kv_absorbed_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_schedule_constants_match_header_and_oracle_tests(L):
    from mla_paged_kv_absorbed_gb300 import api
    ovh, min_split = api.mla_schedule_constants()
    assert ovh == header_define("MLA_SCHED_PIECE_OVERHEAD")
    assert min_split == header_define("MLA_SCHED_MIN_SPLIT_PAGES")


def test_version_is_declared_one(L):
    L.mla_version.restype = ctypes.c_int
    assert L.mla_version() == 101
    assert "1.1 (101)" in open(os.path.join(ROOT, "include", "mla.h")).read()


def test_status_strings(L):
    from mla_paged_kv_absorbed_gb300 import api
    for code in range(6):
        assert api.status_string(code).startswith("MLA_")
    assert "unknown" in api.status_string(99)


def test_workspace_size_formula(L):
    from mla_paged_kv_absorbed_gb300 import api
    for B, s_q, H, parts in ((128, 1, 128, 76), (132, 2, 128, 38), (2, 1, 16, 5)):
        rows = (B + parts) * s_q * H
        lse = (rows * 4 + 255) // 256 * 256
        assert api.mla_workspace_size(B, s_q, H, parts) == 256 + lse + rows * 512 * 4
    assert api.mla_workspace_size(0, 1, 128, 76) == 0
    assert api.mla_workspace_size(4, 3, 128, 76) == 0
    assert api.mla_workspace_size(4, 1, 100, 76) == 0


def test_bad_arguments_are_rejected_on_the_host(L):
    null = ctypes.c_void_p(0)
    assert L.mla_get_metadata(null, 4, 1, 128, 1, 8, null, null, null) == 1
    assert L.mla_absorb_q(null, null, null, 4, 1, 128, null) == 1
    assert L.mla_out_proj(null, null, null, 4, 1, 128, null) == 1
    assert L.mla_decode_paged(null, null, 1, null, 1, null, 1, 1, 128, null, null, 1, ctypes.c_float(0.1), 1,
                              null, null, null, 0, null) == 1
    assert L.mla_debug_mma(null, null, 64, 64, 1, 0, null, null) == 1
    assert L.mla_rope_append(null, null, null, null, 1, null, 1, 1, 1, 128, ctypes.c_float(10000.0), null) == 1
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    # a rope base that is not > 1
    assert L.mla_rope_append(p, p, p, p, 1, p, 1, 1, 1, 128, ctypes.c_float(1.0), null) == 1
    # INT8 cache entry points: missing records or scales, empty or unaligned inputs
    assert L.mla_decode_paged_q8(p, null, p, 1, p, 1, p, 1, 1, 128, p, p, 1, ctypes.c_float(0.1), 1,
                                 p, p, p, 1 << 20, null) == 1
    assert L.mla_decode_paged_q8(p, p, null, 1, p, 1, p, 1, 1, 128, p, p, 1, ctypes.c_float(0.1), 1,
                                 p, p, p, 1 << 20, null) == 1
    # the fused decode + output projection: missing weight or output, unaligned weight
    F = ctypes.c_float(0.1)
    assert L.mla_decode_out_proj(p, p, 1, p, 1, p, 1, 1, 128, p, p, 1, F, 1, null, p, p, p, p, 1 << 20, null) == 1
    assert L.mla_decode_out_proj(p, p, 1, p, 1, p, 1, 1, 128, p, p, 1, F, 1, p, p, null, p, p, 1 << 20, null) == 1
    assert L.mla_decode_out_proj(p, p, 1, p, 1, p, 1, 1, 128, p, p, 1, F, 1, ctypes.c_void_p(buf_addr(buf) + 4), p,
                                 p, p, p, 1 << 20, null) == 1
    assert L.mla_quantize_cache(p, ctypes.c_longlong(0), p, p, null) == 1
    assert L.mla_quantize_cache(null, ctypes.c_longlong(4), p, p, null) == 1
    odd = ctypes.c_void_p(buf_addr(buf) + 4)
    assert L.mla_quantize_cache(odd, ctypes.c_longlong(4), p, p, null) == 1
    assert L.mla_rope_append_q8(p, p, p, p, 1, null, p, 1, 1, 1, 128, ctypes.c_float(10000.0), null) == 1
    assert L.mla_rope_append_q8(p, p, p, p, 1, p, null, 1, 1, 1, 128, ctypes.c_float(10000.0), null) == 1
    # the no-allocation decode checks every argument before it touches its scratch:
    # bad arguments are rejected without any CUDA call; well-formed ones get past
    # the checks and only then fail here, where there is no GPU (MLA_ERR_CUDA)
    q = ctypes.c_void_p(buf_addr(buf))
    na = L.mla_decode_paged_noalloc
    na.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    na.restype = ctypes.c_int
    assert na(null, q, 1, q, 1, q, 1, 1, 128, q, q, 1, F, 1, q, q, null, null) == 1  # no query
    assert na(q, q, 1, q, 1, q, 1, 3, 128, q, q, 1, F, 1, q, q, null, null) == 1  # s_q outside {1, 2}
    assert na(q, q, 1, q, 1, q, 1, 1, 128, q, q, 1, ctypes.c_float(0.0), 1, q, q, null, null) == 1  # scale 0
    assert na(odd, q, 1, q, 1, q, 1, 1, 128, q, q, 1, F, 1, q, q, null, null) == 1  # unaligned query
    assert na(q, q, 1, q, 1, q, 1, 1, 128, q, q, 1, F, 1, q, q, null, null) == 3


def buf_addr(buf):
    return ctypes.addressof(buf) + ((16 - ctypes.addressof(buf) % 16) % 16)


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from mla_paged_kv_absorbed_gb300 import api
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(RuntimeError, match="libmla.so not found"):
        api.lib()
