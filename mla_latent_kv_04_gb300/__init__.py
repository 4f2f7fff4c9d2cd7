"""Python binding of libmla, the C-ABI weight-absorbed MLA decode library for GB300.

Argument marshalling only: each function takes torch tensors that already live on
the GPU, checks their dtype/shape/contiguity, and passes raw pointers and sizes to
the C entry point of the same name declared in include/mla.h. Every step of the
computation runs in the library's CUDA kernels; there is no fallback path. When
libmla.so has not been built the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_GUARD = 5
MLA_ERR_TIMEOUT = 6

MLA_F32 = 0
MLA_BF16 = 1
MLA_FP8_E4M3 = 2
MLA_FP8_E4M3_B128 = 3

KERNEL_AUTO = 0
KERNEL_SIMT = 1
KERNEL_TC = 2

_DTYPE_CODES = {"f32": MLA_F32, "bf16": MLA_BF16, "fp8_e4m3": MLA_FP8_E4M3,
                "fp8_e4m3_b128": MLA_FP8_E4M3_B128}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" + (f" ({detail})" if detail else ""))


class MlaConfig(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int), ("d_model", ctypes.c_int), ("d_latent", ctypes.c_int),
        ("d_rope", ctypes.c_int), ("d_nope", ctypes.c_int), ("d_v", ctypes.c_int),
        ("page_size", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("rope_theta", ctypes.c_float), ("rope_interleaved", ctypes.c_int),
        ("act_dtype", ctypes.c_int), ("cache_dtype", ctypes.c_int), ("cache_scale", ctypes.c_float),
    ]


class MlaDecodeOpts(ctypes.Structure):
    _fields_ = [("num_workers", ctypes.c_int), ("kernel", ctypes.c_int),
                ("attn_events", ctypes.c_void_p * 2), ("wait_limit_us", ctypes.c_int),
                ("withhold_page", ctypes.c_int)]


_lib_handle = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_CFG = ctypes.POINTER(MlaConfig)

_SIGNATURES = {
    "mla_absorb_weights": (_I, [_CFG, _P, _P, _P, _P, _P, _P]),
    "mla_append_cache": (_I, [_CFG, _P, _P, _I, _P, _P, _P, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "mla_append_cache_workspace_size": (_I, [_CFG, _I, ctypes.POINTER(_SZ)]),
    "mla_append_cache_latent": (_I, [_CFG, _P, _P, _I, _P, _P, _P, _I, _I, _P, _I, _I, _P, _P]),
    "mla_decode_workspace_size": (_I, [_CFG, _I, _I, ctypes.POINTER(MlaDecodeOpts),
                                       ctypes.POINTER(_SZ)]),
    "mla_decode": (_I, [_CFG, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, _P, _SZ, _P]),
    "mla_decode_ex": (_I, [_CFG, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, _P, _SZ,
                           ctypes.POINTER(MlaDecodeOpts), _P]),
    "mla_decode_noalloc": (_I, [_CFG, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, _P]),
    "mla_decode_noalloc_status": (_I, [_P, ctypes.POINTER(_I)]),
    "mla_output_proj_workspace_size": (_I, [_CFG, _I, ctypes.POINTER(_SZ)]),
    "mla_output_proj": (_I, [_CFG, _P, _P, _I, _P, _P, _SZ, _P]),
    "mla_output_proj_unfolded_workspace_size": (_I, [_CFG, _I, ctypes.POINTER(_SZ)]),
    "mla_output_proj_unfolded": (_I, [_CFG, _P, _P, _P, _I, _P, _P, _SZ, _P]),
    "mla_cache_row_bytes": (_I, [_CFG, ctypes.POINTER(_SZ)]),
    "mla_query_workspace_size": (_I, [_CFG, _I, _I, ctypes.POINTER(_SZ)]),
    "mla_query_from_hidden": (_I, [_CFG, _I, _P, _P, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "mla_read_device_status": (_I, [_P, _P, ctypes.POINTER(_I)]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_version": (_I, []),
    "mla_kernel_launches": (ctypes.c_uint64, []),
}


def lib():
    """The loaded libmla.so (raises RuntimeError when it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmla.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    try:
        return lib().mla_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def mla_status_string(status: int) -> str:
    return status_string(status)


def mla_last_error() -> str:
    return lib().mla_last_error().decode()


def mla_version() -> int:
    return lib().mla_version()


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MlaError(status, where, mla_last_error())


def make_config(dims, act: str = "bf16", cache: str = "bf16", cache_scale: float = 1.0,
                softmax_scale: float = 0.0, rope_theta: float = 10000.0) -> MlaConfig:
    """Config from an object with num_heads/d_model/d_latent/d_rope/d_nope/d_v/page_size."""
    return MlaConfig(dims.num_heads, dims.d_model, dims.d_latent, dims.d_rope, dims.d_nope, dims.d_v,
                     dims.page_size, float(softmax_scale), float(rope_theta), 1,
                     _DTYPE_CODES[act], _DTYPE_CODES[cache], float(cache_scale))


# ----------------------------------------------------------------------------- marshalling

def _torch():
    import torch
    return torch


def _act_dtype(cfg):
    t = _torch()
    return t.float32 if cfg.act_dtype == MLA_F32 else t.bfloat16


def _cache_dtypes(cfg):
    t = _torch()
    if cfg.cache_dtype == MLA_F32:
        return (t.float32,)
    if cfg.cache_dtype == MLA_BF16:
        return (t.bfloat16,)
    return (t.uint8, t.float8_e4m3fn)


def _cache_row_elems(cfg):
    """Elements of the cache tensor per token row: d_c + d_r, or the row's bytes for the
    block-scaled fp8 cache (a uint8 tensor)."""
    if cfg.cache_dtype == MLA_FP8_E4M3_B128:
        return cfg.d_latent + cfg.d_latent // 32 + 2 * cfg.d_rope
    return cfg.d_latent + cfg.d_rope


def _ptr(x, name, dtypes=None, numel=None, allow_none=False):
    if x is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and x.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {x.dtype}, expected one of {dtypes}")
    if numel is not None and x.numel() != numel:
        raise ValueError(f"{name} has {x.numel()} elements, expected {numel}")
    return ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _opts(num_workers, kernel, attn_events=None, wait_limit_us=0, withhold_page=0):
    o = MlaDecodeOpts(int(num_workers), int(kernel))
    o.wait_limit_us = int(wait_limit_us)
    o.withhold_page = int(withhold_page)
    if attn_events is not None:
        o.attn_events[0] = attn_events[0].cuda_event
        o.attn_events[1] = attn_events[1].cuda_event
    return o


def mla_kernel_launches() -> int:
    return int(lib().mla_kernel_launches())


# ----------------------------------------------------------------------------- entry points

def mla_absorb_weights(cfg, W_UK, W_UV, W_O, W_UK_abs, W_comb, stream=None):
    a = (_act_dtype(cfg),)
    H, d_c, d_n, d_v, d = cfg.num_heads, cfg.d_latent, cfg.d_nope, cfg.d_v, cfg.d_model
    _check(lib().mla_absorb_weights(
        ctypes.byref(cfg), _ptr(W_UK, "W_UK", a, d_c * H * d_n), _ptr(W_UV, "W_UV", a, d_c * H * d_v),
        _ptr(W_O, "W_O", a, H * d_v * d), _ptr(W_UK_abs, "W_UK_abs", a, H * d_n * d_c),
        _ptr(W_comb, "W_comb", a, H * d_c * d), _stream(stream)), "mla_absorb_weights")


def _i32(t):
    return (_torch().int32,)


def mla_append_cache_workspace_size(cfg, T) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mla_append_cache_workspace_size(ctypes.byref(cfg), int(T), ctypes.byref(n)),
           "mla_append_cache_workspace_size")
    return int(n.value)


def mla_append_cache(cfg, h, W_DKV_KR, req_ids, positions, block_table, cache, dev_status=None,
                     workspace=None, stream=None):
    """workspace: uint8 device tensor of mla_append_cache_workspace_size bytes (None if 0)."""
    a = (_act_dtype(cfg),)
    T = req_ids.numel()
    D = cfg.d_latent + cfg.d_rope
    batch, max_pages = block_table.shape
    num_pages = cache.numel() // (cfg.page_size * _cache_row_elems(cfg))
    _check(lib().mla_append_cache(
        ctypes.byref(cfg), _ptr(h, "h", a, T * cfg.d_model), _ptr(W_DKV_KR, "W_DKV_KR", a, cfg.d_model * D),
        T, _ptr(req_ids, "req_ids", _i32(0), T), _ptr(positions, "positions", _i32(0), T),
        _ptr(block_table, "block_table", _i32(0)), batch, max_pages,
        _ptr(cache, "cache", _cache_dtypes(cfg), num_pages * cfg.page_size * _cache_row_elems(cfg)), num_pages,
        _ptr(dev_status, "dev_status", _i32(0), allow_none=True),
        _ptr(workspace, "workspace", (_torch().uint8,), allow_none=True),
        0 if workspace is None else workspace.numel(), _stream(stream)),
        "mla_append_cache")


def mla_append_cache_latent(cfg, c_kv, k_pe, req_ids, positions, block_table, cache, rotate=True,
                            dev_status=None, stream=None):
    a = (_act_dtype(cfg),)
    T = req_ids.numel()
    D = cfg.d_latent + cfg.d_rope
    batch, max_pages = block_table.shape
    num_pages = cache.numel() // (cfg.page_size * _cache_row_elems(cfg))
    _check(lib().mla_append_cache_latent(
        ctypes.byref(cfg), _ptr(c_kv, "c_kv", a, T * cfg.d_latent), _ptr(k_pe, "k_pe", a, T * cfg.d_rope),
        T, _ptr(req_ids, "req_ids", _i32(0), T), _ptr(positions, "positions", _i32(0), T),
        _ptr(block_table, "block_table", _i32(0)), batch, max_pages,
        _ptr(cache, "cache", _cache_dtypes(cfg), num_pages * cfg.page_size * _cache_row_elems(cfg)), num_pages,
        1 if rotate else 0, _ptr(dev_status, "dev_status", _i32(0), allow_none=True),
        _stream(stream)), "mla_append_cache_latent")


def mla_decode_workspace_size(cfg, batch, q_len, num_workers=0, kernel=KERNEL_AUTO) -> int:
    n = ctypes.c_size_t(0)
    o = _opts(num_workers, kernel)
    _check(lib().mla_decode_workspace_size(ctypes.byref(cfg), int(batch), int(q_len), ctypes.byref(o),
                                           ctypes.byref(n)), "mla_decode_workspace_size")
    return int(n.value)


def mla_decode(cfg, q_nope, q_pe, W_UK_abs, cache, block_table, seq_lens, out_latent, lse,
               workspace, num_workers=0, kernel=KERNEL_AUTO, stream=None, attn_events=None,
               wait_limit_us=0, withhold_page=0):
    """attn_events: optional pair of torch.cuda.Event recorded around the attention kernel.
    wait_limit_us, withhold_page: testing hooks of the tensor-core kernel's failure path
    (see mla_decode_opts in include/mla.h)."""
    a = (_act_dtype(cfg),)
    t = _torch()
    batch, q_len = q_nope.shape[0], q_nope.shape[1]
    H, d_c, d_r, d_n = cfg.num_heads, cfg.d_latent, cfg.d_rope, cfg.d_nope
    D = d_c + d_r
    num_pages = cache.numel() // (cfg.page_size * _cache_row_elems(cfg))
    max_pages = block_table.shape[1]
    o = _opts(num_workers, kernel, attn_events, wait_limit_us, withhold_page)
    _check(lib().mla_decode_ex(
        ctypes.byref(cfg), _ptr(q_nope, "q_nope", a, batch * q_len * H * d_n),
        _ptr(q_pe, "q_pe", a, batch * q_len * H * d_r),
        _ptr(W_UK_abs, "W_UK_abs", a, H * d_n * d_c),
        _ptr(cache, "cache", _cache_dtypes(cfg), num_pages * cfg.page_size * _cache_row_elems(cfg)), num_pages,
        _ptr(block_table, "block_table", _i32(0), batch * max_pages), max_pages,
        _ptr(seq_lens, "seq_lens", _i32(0), batch), batch, q_len,
        _ptr(out_latent, "out_latent", a, batch * q_len * H * d_c),
        _ptr(lse, "lse", (t.float32,), batch * q_len * H),
        _ptr(workspace, "workspace", (t.uint8,)), workspace.numel(), ctypes.byref(o),
        _stream(stream)), "mla_decode")


def mla_decode_noalloc(cfg, q_nope, q_pe, W_UK_abs, cache, block_table, seq_lens, out_latent, lse,
                       stream=None):
    """mla_decode with the library's fixed 64 MiB device scratch array instead of a workspace,
    for callers that cannot allocate device memory at decode time. Calls sharing the array
    must be ordered on the GPU; the first call on a device must come before any capture."""
    a = (_act_dtype(cfg),)
    t = _torch()
    batch, q_len = q_nope.shape[0], q_nope.shape[1]
    H, d_c, d_r, d_n = cfg.num_heads, cfg.d_latent, cfg.d_rope, cfg.d_nope
    D = d_c + d_r
    num_pages = cache.numel() // (cfg.page_size * _cache_row_elems(cfg))
    max_pages = block_table.shape[1]
    _check(lib().mla_decode_noalloc(
        ctypes.byref(cfg), _ptr(q_nope, "q_nope", a, batch * q_len * H * d_n),
        _ptr(q_pe, "q_pe", a, batch * q_len * H * d_r),
        _ptr(W_UK_abs, "W_UK_abs", a, H * d_n * d_c),
        _ptr(cache, "cache", _cache_dtypes(cfg), num_pages * cfg.page_size * _cache_row_elems(cfg)), num_pages,
        _ptr(block_table, "block_table", _i32(0), batch * max_pages), max_pages,
        _ptr(seq_lens, "seq_lens", _i32(0), batch), batch, q_len,
        _ptr(out_latent, "out_latent", a, batch * q_len * H * d_c),
        _ptr(lse, "lse", (t.float32,), batch * q_len * H), _stream(stream)), "mla_decode_noalloc")


def mla_decode_noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device status of the last
    mla_decode_noalloc on the current device."""
    code = ctypes.c_int(0)
    _check(lib().mla_decode_noalloc_status(_stream(stream), ctypes.byref(code)),
           "mla_decode_noalloc_status")
    return int(code.value)


def mla_output_proj_workspace_size(cfg, rows) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mla_output_proj_workspace_size(ctypes.byref(cfg), int(rows), ctypes.byref(n)),
           "mla_output_proj_workspace_size")
    return int(n.value)


def mla_output_proj(cfg, out_latent, W_comb, out, workspace, stream=None):
    a = (_act_dtype(cfg),)
    K = cfg.num_heads * cfg.d_latent
    rows = out_latent.numel() // K
    _check(lib().mla_output_proj(
        ctypes.byref(cfg), _ptr(out_latent, "out_latent", a, rows * K),
        _ptr(W_comb, "W_comb", a, K * cfg.d_model), rows, _ptr(out, "out", a, rows * cfg.d_model),
        _ptr(workspace, "workspace", (_torch().uint8,)), workspace.numel(), _stream(stream)),
        "mla_output_proj")


def mla_output_proj_unfolded_workspace_size(cfg, rows) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mla_output_proj_unfolded_workspace_size(ctypes.byref(cfg), int(rows),
                                                         ctypes.byref(n)),
           "mla_output_proj_unfolded_workspace_size")
    return int(n.value)


def mla_output_proj_unfolded(cfg, out_latent, W_UV, W_O, out, workspace, stream=None):
    a = (_act_dtype(cfg),)
    K = cfg.num_heads * cfg.d_latent
    HV = cfg.num_heads * cfg.d_v
    rows = out_latent.numel() // K
    _check(lib().mla_output_proj_unfolded(
        ctypes.byref(cfg), _ptr(out_latent, "out_latent", a, rows * K),
        _ptr(W_UV, "W_UV", a, cfg.d_latent * HV), _ptr(W_O, "W_O", a, HV * cfg.d_model), rows,
        _ptr(out, "out", a, rows * cfg.d_model),
        _ptr(workspace, "workspace", (_torch().uint8,)), workspace.numel(), _stream(stream)),
        "mla_output_proj_unfolded")


def mla_cache_row_bytes(cfg) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mla_cache_row_bytes(ctypes.byref(cfg), ctypes.byref(n)), "mla_cache_row_bytes")
    return int(n.value)


def mla_query_workspace_size(cfg, d_q, T) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().mla_query_workspace_size(ctypes.byref(cfg), int(d_q), int(T), ctypes.byref(n)),
           "mla_query_workspace_size")
    return int(n.value)


def mla_query_from_hidden(cfg, d_q, h, W_DQ, W_UQ, W_QR, q_nope, q_pe, workspace, stream=None):
    """h [T][d_model] -> q_nope [T][H][d_n], q_pe [T][H][d_r] (not rotated)."""
    a = (_act_dtype(cfg),)
    d, H = cfg.d_model, cfg.num_heads
    T = h.numel() // d
    _check(lib().mla_query_from_hidden(
        ctypes.byref(cfg), int(d_q), _ptr(h, "h", a, T * d), _ptr(W_DQ, "W_DQ", a, d * d_q),
        _ptr(W_UQ, "W_UQ", a, d_q * H * cfg.d_nope), _ptr(W_QR, "W_QR", a, d * H * cfg.d_rope), T,
        _ptr(q_nope, "q_nope", a, T * H * cfg.d_nope), _ptr(q_pe, "q_pe", a, T * H * cfg.d_rope),
        _ptr(workspace, "workspace", (_torch().uint8,)), workspace.numel(), _stream(stream)),
        "mla_query_from_hidden")


def mla_read_device_status(status_word, stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device status code."""
    code = ctypes.c_int(0)
    _check(lib().mla_read_device_status(_ptr(status_word, "status_word"), _stream(stream),
                                        ctypes.byref(code)), "mla_read_device_status")
    return int(code.value)
