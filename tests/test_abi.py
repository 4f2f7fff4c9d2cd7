"""The C-ABI library: it builds, loads, exports every entry point declared in
include/mla.h, and rejects bad arguments on the host before launching anything.
No test here needs a GPU or runs a kernel."""
import ctypes
import os
import re
import shutil

import pytest

import mla_latent_kv_04_gb300 as M
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def _declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h, encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = re.sub(r"typedef[^;]*;", "", src, flags=re.S)
        for m in re.finditer(r"\b(mla_[A-Za-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(M.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.fail("libmla.so is not built and nvcc is unavailable")
        from mla_latent_kv_04_gb300 import build
        build.build()
    return M.lib()


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for f in ("mla_absorb_weights", "mla_append_cache", "mla_decode", "mla_output_proj"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(M.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_python_binding_names_match_header():
    for n in _declared_functions():
        if n in ("mla_decode_ex",):
            continue
        assert hasattr(M, n), n


def test_status_strings(lib):
    assert M.mla_status_string(0) == "ok"
    assert "workspace" in M.mla_status_string(3)
    assert M.mla_version() >= 100


def _cfg(**kw):
    c = M.make_config(W.V2, "bf16", "bf16")
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,code", [
    ("num_heads", 0, M.MLA_ERR_INVALID),
    ("d_rope", 63, M.MLA_ERR_INVALID),
    ("page_size", 128, M.MLA_ERR_UNSUPPORTED),
    ("rope_interleaved", 0, M.MLA_ERR_UNSUPPORTED),
    ("cache_dtype", M.MLA_F32, M.MLA_ERR_UNSUPPORTED),
    ("act_dtype", 7, M.MLA_ERR_INVALID),
])
def test_bad_config_is_rejected_before_any_launch(lib, field, value, code):
    n = ctypes.c_size_t(0)
    st = lib.mla_decode_workspace_size(ctypes.byref(_cfg(**{field: value})), 4, 1, None,
                                       ctypes.byref(n))
    assert st == code


def test_fp8_needs_a_scale(lib):
    c = _cfg(cache_dtype=M.MLA_FP8_E4M3, cache_scale=0.0)
    n = ctypes.c_size_t(0)
    assert lib.mla_decode_workspace_size(ctypes.byref(c), 4, 1, None, ctypes.byref(n)) == M.MLA_ERR_INVALID


def test_null_pointers_and_small_workspace_are_rejected(lib):
    c = _cfg()
    # null inputs
    st = lib.mla_decode(ctypes.byref(c), None, None, None, None, 1, None, 1, None, 1, 1, None, None,
                        None, 0, None)
    assert st == M.MLA_ERR_INVALID
    # all pointers non-null but no workspace: a fake non-null address is never dereferenced
    fake = ctypes.c_void_p(256)
    st = lib.mla_decode(ctypes.byref(c), fake, fake, fake, fake, 1, fake, 1, fake, 1, 1, fake, fake,
                        None, 0, None)
    assert st == M.MLA_ERR_WORKSPACE
    st = lib.mla_output_proj(ctypes.byref(c), fake, fake, 2, fake, None, 0, None)
    assert st == M.MLA_ERR_WORKSPACE
    st = lib.mla_append_cache_latent(ctypes.byref(c), None, None, 3, None, None, None, 1, 1, None, 1,
                                     1, None, None)
    assert st == M.MLA_ERR_INVALID
    # T == 0 is a no-op that touches nothing
    st = lib.mla_append_cache_latent(ctypes.byref(c), None, None, 0, None, None, None, 1, 1, None, 1,
                                     1, None, None)
    assert st == M.MLA_OK


def test_workspace_grows_with_batch(lib):
    c = _cfg()
    a = M.mla_decode_workspace_size(c, 4, 1, num_workers=8)
    b = M.mla_decode_workspace_size(c, 64, 2, num_workers=8)
    assert b > a > 0
    assert M.mla_output_proj_workspace_size(c, 32) == 32 * 5120 * 4 + 256
    # the bf16 append sums its split-K partials on chip: no scratch
    assert M.mla_append_cache_workspace_size(c, 32) == 0


def test_query_call_validates_before_any_launch(lib):
    c = _cfg()
    n = ctypes.c_size_t(0)
    assert lib.mla_query_workspace_size(ctypes.byref(c), 0, 4, ctypes.byref(n)) == M.MLA_ERR_INVALID
    assert lib.mla_query_workspace_size(ctypes.byref(c), 1536, 4, ctypes.byref(n)) == M.MLA_OK
    # an fp32 accumulator as wide as the widest of the three products, a status word, c^Q
    assert n.value == 4 * (128 * 128) * 4 + 256 + 4 * 1536 * 2
    fake = ctypes.c_void_p(256)
    st = lib.mla_query_from_hidden(ctypes.byref(c), 1536, None, fake, fake, fake, 4, fake, fake,
                                   fake, n.value, None)
    assert st == M.MLA_ERR_INVALID
    st = lib.mla_query_from_hidden(ctypes.byref(c), 1536, fake, fake, fake, fake, 4, fake, fake,
                                   None, 0, None)
    assert st == M.MLA_ERR_WORKSPACE
    st = lib.mla_query_from_hidden(ctypes.byref(c), 1536, fake, fake, fake, fake, 4, fake, fake,
                                   ctypes.c_void_p(256 + 16), n.value, None)
    assert st == M.MLA_ERR_INVALID          # workspace not 256-byte aligned
    # T == 0 is a no-op that touches nothing
    st = lib.mla_query_from_hidden(ctypes.byref(c), 1536, None, None, None, None, 0, None, None,
                                   None, 0, None)
    assert st == M.MLA_OK


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    # no silent fallback: a missing libmla.so is an error at the first call
    monkeypatch.setattr(M, "LIB_PATH", str(tmp_path / "missing" / "libmla.so"))
    monkeypatch.setattr(M, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="not built"):
        M.lib()


def test_decode_options_are_validated(lib):
    fake = ctypes.c_void_p(256)
    args = lambda c, o: (ctypes.byref(c), fake, fake, fake, fake, 4, fake, 1, fake, 1, 1, fake, fake,  # noqa: E731
                         fake, 1 << 20, ctypes.byref(o), None)
    bad_kernel = M.MlaDecodeOpts(num_workers=0, kernel=7)
    assert lib.mla_decode_ex(*args(_cfg(), bad_kernel)) == M.MLA_ERR_INVALID
    bad_workers = M.MlaDecodeOpts(num_workers=-1, kernel=0)
    assert lib.mla_decode_ex(*args(_cfg(), bad_workers)) == M.MLA_ERR_INVALID
    # the tensor-core kernel asked for on a shape it does not cover
    tc_on_f32 = M.MlaDecodeOpts(num_workers=0, kernel=M.KERNEL_TC)
    c32 = M.make_config(W.TINY, "f32", "f32")
    assert lib.mla_decode_ex(*args(c32, tc_on_f32)) == M.MLA_ERR_UNSUPPORTED


def test_unfolded_projection_validates_before_any_launch(lib):
    c = _cfg()
    fake = ctypes.c_void_p(256)
    n = ctypes.c_size_t(0)
    assert lib.mla_output_proj_unfolded_workspace_size(ctypes.byref(c), 3, ctypes.byref(n)) == M.MLA_OK
    # an fp32 accumulator [rows][d], a status word and u [rows][H*d_v] (bf16), each 256-aligned
    assert n.value == 3 * 5120 * 4 + 256 + 3 * 128 * 128 * 2
    assert lib.mla_output_proj_unfolded(ctypes.byref(c), None, fake, fake, 3, fake, fake, n.value,
                                        None) == M.MLA_ERR_INVALID
    assert lib.mla_output_proj_unfolded(ctypes.byref(c), fake, fake, fake, 3, fake, fake, n.value - 1,
                                        None) == M.MLA_ERR_WORKSPACE
    assert lib.mla_output_proj_unfolded(ctypes.byref(c), None, None, None, 0, None, None, 0,
                                        None) == M.MLA_OK


def test_block_scaled_fp8_cache_rows(lib):
    c = _cfg(cache_dtype=M.MLA_FP8_E4M3_B128)
    assert M.mla_cache_row_bytes(c) == 512 + 4 * 4 + 2 * 64        # codes, 4 fp32 scales, bf16 k_pe
    assert M.mla_cache_row_bytes(_cfg()) == 576 * 2
    n = ctypes.c_size_t(0)
    odd = _cfg(cache_dtype=M.MLA_FP8_E4M3_B128, d_latent=320)
    assert lib.mla_cache_row_bytes(ctypes.byref(odd), ctypes.byref(n)) == M.MLA_ERR_UNSUPPORTED
    f32 = M.make_config(W.TINY, "f32", "f32")
    f32.cache_dtype = M.MLA_FP8_E4M3_B128
    assert lib.mla_cache_row_bytes(ctypes.byref(f32), ctypes.byref(n)) == M.MLA_ERR_UNSUPPORTED
