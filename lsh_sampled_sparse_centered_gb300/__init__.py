"""Python binding of libmagicpig (LSH-sampled sparse decode attention on one GB300).

Argument marshalling only: every function forwards to the C entry point of the same
name in ``include/magicpig.h``. Tensors are passed as device pointers; PyTorch
supplies device memory and streams. The shared library must have been built
(``python lsh_sampled_sparse_centered_gb300/build.py`` or ``__graft_entry__.build()``);
importing this package without it raises ImportError, and there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Union

_PKG = os.path.dirname(os.path.abspath(__file__))
# MP_BOUNDS_CHECK=1 loads the bounds-checking build (kernels test data-derived indices
# and set MP_STATUS_BAD_INDEX instead of touching memory outside their buffers)
BOUNDS_CHECK = os.environ.get("MP_BOUNDS_CHECK") == "1"
LIB_PATH = os.path.join(_PKG, "_lib", "libmagicpig_check.so" if BOUNDS_CHECK else "libmagicpig.so")

MP_OK = 0
MP_ERR_INVALID_ARG = -1
MP_ERR_UNSUPPORTED = -2
MP_ERR_CAPACITY = -3
MP_ERR_CUDA = -4
MP_ERR_INJECTED = -5
MP_ERR_SCRATCH = -6

MP_STATUS_W_NOT_BF16 = 0x1
MP_STATUS_WAIT_TIMEOUT = 0x2
MP_STATUS_APPEND_GAP = 0x4
MP_STATUS_NOT_BUILT = 0x8
MP_STATUS_BAD_INDEX = 0x10

MP_DTYPE_F32 = 0
MP_DTYPE_BF16 = 1
MP_MATCH_AUTO = 0
MP_MATCH_CSR = 1
MP_MATCH_SCAN = 2

EXACT_FLAG = 0x80000000

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                      "`python lsh_sampled_sparse_centered_gb300/build.py`" + (" --check" if BOUNDS_CHECK else ""))
_lib = ctypes.CDLL(LIB_PATH)


class mp_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "layers", "batch", "kv_heads", "q_heads", "head_dim", "K", "L", "n_sink", "window",
        "capacity", "dtype", "w_per_layer", "match_mode", "threshold", "no_centering", "center_query")] + [
        ("reserved", ctypes.c_int32 * 2)]


class mp_tables_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "total_bytes", "header", "center", "beta", "ones", "negbeta_f32", "wt_f32", "wt_bf16", "center_parts", "codes",
        "csr_offsets", "csr_ids", "planes", "logu_lut")] + [(n, ctypes.c_int32) for n in (
        "n_buckets", "parts", "tc_cols", "match_mode", "cap_words")]


class mp_decode_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "total_bytes", "q_codes", "list_len", "sample_count", "lists", "partials", "counters",
        "sample_bits")] + [
        (n, ctypes.c_int32) for n in ("splits_max", "reserved")]


class mp_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("total_ms", ctypes.c_double)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_CFG = ctypes.POINTER(mp_config)
_SIGS = {
    "mp_abi_version": (ctypes.c_int, []),
    "mp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mp_config_check": (ctypes.c_int, [_CFG]),
    "mp_tables_layout_get": (ctypes.c_int, [_CFG, ctypes.POINTER(mp_tables_layout)]),
    "mp_decode_layout_get": (ctypes.c_int, [_CFG, ctypes.POINTER(mp_decode_layout)]),
    "mp_build_tables": (ctypes.c_int, [_CFG, _P, _I, _P, _P, _P]),
    "mp_append": (ctypes.c_int, [_CFG, _P, _P, _I, _P]),
    "mp_decode_attention": (ctypes.c_int, [_CFG, _P, _P, _P, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "mp_decode_step": (ctypes.c_int, [_CFG, _P, _P, _P, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "mp_decode_attention_static": (ctypes.c_int, [_CFG, _P, _P, _P, _I, _P, _P, _P]),
    "mp_get_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "mp_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "mp_profile_read": (ctypes.c_int, [ctypes.POINTER(mp_kernel_time), ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


class MagicPigError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({mp_status_string(code)})")
        self.code = code


def _ptr(x) -> Optional[int]:
    """Device address of a tensor argument (ints pass through as raw addresses). The
    kernels read and write these addresses directly, so a host tensor or a strided
    view is refused here rather than handed to the GPU."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if getattr(x, "is_cuda", True) is False:
        raise ValueError("tensor arguments must be CUDA tensors (device memory)")
    if hasattr(x, "is_contiguous") and not x.is_contiguous():
        raise ValueError("tensor arguments must be contiguous (dense row-major layout)")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc != MP_OK:
        raise MagicPigError(fn, rc)
    return rc


def make_config(*, layers: int, batch: int, kv_heads: int, q_heads: int, head_dim: int, K: int, L: int,
                n_sink: int, window: int, capacity: int, dtype: Union[int, str], w_per_layer: bool = False,
                match_mode: int = MP_MATCH_AUTO, threshold: int = 2, centering: bool = True,
                center_query: bool = False) -> mp_config:
    if isinstance(dtype, str):
        dtype = MP_DTYPE_BF16 if dtype == "bf16" else MP_DTYPE_F32
    return mp_config(layers, batch, kv_heads, q_heads, head_dim, K, L, n_sink, window, capacity, int(dtype),
                     int(bool(w_per_layer)), match_mode, threshold, 0 if centering else 1,
                     int(bool(center_query)))


def mp_abi_version() -> int:
    return _lib.mp_abi_version()


def mp_status_string(code: int) -> str:
    return _lib.mp_status_string(code).decode()


def mp_config_check(cfg: mp_config) -> int:
    return _lib.mp_config_check(ctypes.byref(cfg))


def mp_tables_layout_get(cfg: mp_config) -> mp_tables_layout:
    out = mp_tables_layout()
    _check("mp_tables_layout_get", _lib.mp_tables_layout_get(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def mp_decode_layout_get(cfg: mp_config) -> mp_decode_layout:
    out = mp_decode_layout()
    _check("mp_decode_layout_get", _lib.mp_decode_layout_get(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def mp_build_tables(cfg: mp_config, keys, n_prefill: int, W, tables, stream=None) -> int:
    return _check("mp_build_tables", _lib.mp_build_tables(
        ctypes.byref(cfg), _ptr(keys), n_prefill, _ptr(W), _ptr(tables), _stream(stream)))


def mp_append(cfg: mp_config, tables, keys, pos: int, stream=None) -> int:
    return _check("mp_append", _lib.mp_append(ctypes.byref(cfg), _ptr(tables), _ptr(keys), pos,
                                              _stream(stream)))


def mp_decode_attention(cfg: mp_config, tables, keys, values, n: int, q, out, scratch,
                        scratch_bytes: Optional[int] = None, stream=None) -> int:
    if scratch_bytes is None:
        scratch_bytes = scratch.numel() * scratch.element_size()
    return _check("mp_decode_attention", _lib.mp_decode_attention(
        ctypes.byref(cfg), _ptr(tables), _ptr(keys), _ptr(values), n, _ptr(q), _ptr(out), _ptr(scratch),
        scratch_bytes, _stream(stream)))


def mp_decode_step(cfg: mp_config, tables, keys, values, pos: int, q, out, scratch,
                   scratch_bytes: Optional[int] = None, stream=None) -> int:
    if scratch_bytes is None:
        scratch_bytes = scratch.numel() * scratch.element_size()
    return _check("mp_decode_step", _lib.mp_decode_step(
        ctypes.byref(cfg), _ptr(tables), _ptr(keys), _ptr(values), pos, _ptr(q), _ptr(out), _ptr(scratch),
        scratch_bytes, _stream(stream)))


MP_STATIC_SCRATCH_BYTES = 32 << 20


def mp_decode_attention_static(cfg: mp_config, tables, keys, values, n: int, q, out, stream=None) -> int:
    """mp_decode_attention with the library's built-in scratch array (no caller scratch)."""
    return _check("mp_decode_attention_static", _lib.mp_decode_attention_static(
        ctypes.byref(cfg), _ptr(tables), _ptr(keys), _ptr(values), n, _ptr(q), _ptr(out), _stream(stream)))


def mp_get_status(tables, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check("mp_get_status", _lib.mp_get_status(_ptr(tables), ctypes.byref(v), _stream(stream)))
    return v.value


def mp_profile_enable(on: bool) -> int:
    return _check("mp_profile_enable", _lib.mp_profile_enable(int(bool(on))))


def mp_profile_read() -> dict:
    """{kernel name: (launches, total_ms)} of the launches recorded since enabling."""
    buf = (mp_kernel_time * 32)()
    n = ctypes.c_int32(0)
    _check("mp_profile_read", _lib.mp_profile_read(buf, 32, ctypes.byref(n)))
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(32, n.value))}


def call_raw(name: str, *args) -> int:
    """Call an entry point with already-marshalled ctypes arguments; returns the code."""
    return getattr(_lib, name)(*args)
