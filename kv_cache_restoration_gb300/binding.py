"""ctypes binding of libhcr.so: the C ABI of include/hcr.h under the same names.

Argument marshalling only -- every step of a restore runs in the library's
CUDA kernels.  Tensors are passed by their device pointers; the library
never sees a torch type.  There is no CPU fallback: if libhcr.so is missing,
importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from .build import LIB

HCR_OK = 0
HCR_ERR_INVALID_ARG = 1
HCR_ERR_UNSUPPORTED = 2
HCR_ERR_CUDA = 3
HCR_ERR_OOM = 4
HCR_ERR_WORKSPACE = 5
HCR_ERR_DEVICE_BOUNDS = 6
HCR_ERR_TIMEOUT = 7

HCR_NORM_RMS, HCR_NORM_LAYER = 0, 1
HCR_ROPE_NONE, HCR_ROPE_ROTATE_HALF = 0, 1
HCR_DTYPE_BF16, HCR_DTYPE_FP16 = 0, 1

HCR_DEVERR_BLOCK_ID = 1 << 0
HCR_DEVERR_LOGICAL_BLOCK = 1 << 1
HCR_DEVERR_POSITION = 1 << 2
HCR_DEVERR_SEQLENS = 1 << 3
HCR_DEVERR_TIMEOUT = 1 << 4


class hcr_model_dims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("norm", ctypes.c_int32),
                ("norm_eps", ctypes.c_float), ("rope", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("max_position", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("has_kv_bias", ctypes.c_int32)]


class hcr_cache_layout(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("layer_stride_elems", ctypes.c_int64)]


class hcr_chunk_source(ctypes.Structure):
    _fields_ = [("store", ctypes.c_void_p), ("chunk_tokens", ctypes.c_int32),
                ("num_chunks", ctypes.c_int32), ("chunk_table", ctypes.c_void_p),
                ("max_chunks", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p),
                ("start_pos", ctypes.c_void_p)]


class hcr_layer_costs(ctypes.Structure):
    _fields_ = [("restore_s", ctypes.c_double), ("hidden_copy_s", ctypes.c_double),
                ("kv_copy_s", ctypes.c_double), ("kv_place_s", ctypes.c_double)]


class hcr_layer_split(ctypes.Structure):
    _fields_ = [("hidden_layers", ctypes.c_int32), ("kv_layers", ctypes.c_int32),
                ("transfer_s", ctypes.c_double), ("compute_s", ctypes.c_double),
                ("predicted_s", ctypes.c_double)]


class hcr_codec_params(ctypes.Structure):
    _fields_ = [("bins", ctypes.c_float * 3), ("group_tokens", ctypes.c_int32)]


def codec_params(bins=(0.5, 1.0, 1.5), group_tokens: int = 10) -> hcr_codec_params:
    return hcr_codec_params((ctypes.c_float * 3)(*bins), group_tokens)


class HcrError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB):
        raise ImportError(
            f"{LIB} is missing: the CUDA library must be built first "
            "(python -m kv_cache_restoration_gb300.build); there is no CPU fallback")
    return ctypes.CDLL(LIB)


lib = _load()

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_RESTORE_ARGTYPES = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp,
                     ctypes.POINTER(hcr_cache_layout), _vp, ctypes.c_size_t, _vp]

lib.hcr_create.argtypes = [ctypes.POINTER(hcr_model_dims)] + [ctypes.POINTER(_vp)] * 6 + [
    ctypes.POINTER(_vp)]
lib.hcr_create.restype = ctypes.c_int
lib.hcr_destroy.argtypes = [_vp]
lib.hcr_destroy.restype = None
lib.hcr_workspace_bytes.argtypes = [_vp, _i32, _i32]
lib.hcr_workspace_bytes.restype = ctypes.c_size_t
for _name in ("hcr_restore", "hcr_restore_prepare", "hcr_restore_project"):
    getattr(lib, _name).argtypes = _RESTORE_ARGTYPES
    getattr(lib, _name).restype = ctypes.c_int
lib.hcr_restore_streamed.argtypes = _RESTORE_ARGTYPES[:13] + [_vp, ctypes.c_size_t, _i32, _vp,
                                                            ctypes.c_size_t, _vp]
lib.hcr_restore_streamed.restype = ctypes.c_int
lib.hcr_save_hidden.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _vp,
                                _i32, _vp]
lib.hcr_save_hidden.restype = ctypes.c_int
lib.hcr_restore_streamed_chunks.argtypes = [_vp, ctypes.POINTER(hcr_chunk_source)] + \
    _RESTORE_ARGTYPES[2:13] + [_vp, ctypes.c_size_t, _i32, _vp, ctypes.c_size_t, _vp]
lib.hcr_restore_streamed_chunks.restype = ctypes.c_int
for _name in ("hcr_load_kv", "hcr_save_kv"):
    getattr(lib, _name).argtypes = _RESTORE_ARGTYPES
    getattr(lib, _name).restype = ctypes.c_int
lib.hcr_plan_layer_split.argtypes = [ctypes.POINTER(hcr_layer_costs), _i32,
                                     ctypes.POINTER(hcr_layer_split)]
lib.hcr_plan_layer_split.restype = ctypes.c_int
lib.hcr_profile_layer_costs.argtypes = [_vp, _i32, _i32, _i32, _vp,
                                        ctypes.POINTER(hcr_layer_costs)]
lib.hcr_profile_layer_costs.restype = ctypes.c_int
lib.hcr_restore_streamed_split.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                           _vp, _i32, _vp, _vp, ctypes.POINTER(hcr_cache_layout),
                                           _vp, ctypes.c_size_t, _i32, _vp, ctypes.c_size_t, _vp]
lib.hcr_restore_streamed_split.restype = ctypes.c_int
lib.hcr_encode_hidden.argtypes = [_vp, ctypes.POINTER(hcr_codec_params), _vp, _i32, _i32, _i32,
                                  _i32, _vp, _vp, _vp, _vp]
lib.hcr_encode_hidden.restype = ctypes.c_int
lib.hcr_decode_hidden.argtypes = [_vp, ctypes.POINTER(hcr_codec_params), _vp, _vp, _i32, _i32,
                                  _i32, _i32, _vp, _vp, _vp]
lib.hcr_decode_hidden.restype = ctypes.c_int
lib.hcr_restore_streamed_encoded.argtypes = [_vp, ctypes.POINTER(hcr_codec_params), _vp, _vp,
                                             _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp,
                                             _vp, ctypes.POINTER(hcr_cache_layout), _vp,
                                             ctypes.c_size_t, _i32, _vp, ctypes.c_size_t, _vp]
lib.hcr_restore_streamed_encoded.restype = ctypes.c_int
lib.hcr_encoded_workspace_bytes.argtypes = [_vp, _i32, _i32]
lib.hcr_encoded_workspace_bytes.restype = ctypes.c_size_t
lib.hcr_restore_encoded.argtypes = [_vp, ctypes.POINTER(hcr_codec_params), _vp, _vp] + \
    _RESTORE_ARGTYPES[2:]
lib.hcr_restore_encoded.restype = ctypes.c_int
lib.hcr_restore_no_alloc.argtypes = _RESTORE_ARGTYPES[:13] + [_vp]
lib.hcr_restore_no_alloc.restype = ctypes.c_int
HCR_NO_ALLOC_SCRATCH_BYTES = 16 << 20
lib.hcr_check_device_error.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
lib.hcr_check_device_error.restype = ctypes.c_int
lib.hcr_status_string.argtypes = [ctypes.c_int]
lib.hcr_status_string.restype = ctypes.c_char_p
lib.hcr_last_error.argtypes = []
lib.hcr_last_error.restype = ctypes.c_char_p
lib.hcr_project_variant.argtypes = [_vp, _i32, _i32]
lib.hcr_project_variant.restype = _i32
lib.hcr_num_sms.argtypes = [_vp]
lib.hcr_num_sms.restype = _i32
lib.hcr_debug_timeout_record.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
lib.hcr_debug_timeout_record.restype = ctypes.c_int
lib.hcr_debug_fused_stats.argtypes = [_vp, _i32, _i32, ctypes.c_size_t]
lib.hcr_debug_fused_stats.restype = _i32
lib.hcr_debug_plan.argtypes = [ctypes.POINTER(hcr_model_dims), _i32, _i32, _i32, _i32, _i32,
                               ctypes.c_size_t, _vp]
lib.hcr_debug_plan.restype = ctypes.c_int
lib.hcr_debug_swap_plan.argtypes = [_i32, _vp]
lib.hcr_debug_swap_plan.restype = ctypes.c_int
lib.hcr_debug_set_variant.argtypes = [_vp, _i32]
lib.hcr_debug_set_variant.restype = ctypes.c_int
lib.hcr_debug_set_stall.argtypes = [_vp, _i32]
lib.hcr_debug_set_stall.restype = ctypes.c_int


def hcr_status_string(status: int) -> str:
    return lib.hcr_status_string(status).decode()


def hcr_last_error() -> str:
    return lib.hcr_last_error().decode()


def _check(status: int, where: str) -> int:
    if status != HCR_OK:
        raise HcrError(status, where, f"{hcr_status_string(status)} -- {hcr_last_error()}")
    return status


def _ptr(x) -> Optional[int]:
    """Device (or host) address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptr_array(xs: Optional[Sequence]):
    if xs is None:
        return None
    arr = (_vp * len(xs))(*[_ptr(x) for x in xs])
    return arr


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream   # torch.cuda.Stream


def hcr_create(dims: hcr_model_dims, gamma, beta, w_k, w_v, b_k=None, b_v=None, *,
               check: bool = True):
    """Returns (status, handle address or None).  Raises HcrError if check and status != OK."""
    out = _vp()
    arrays = [_ptr_array(x) for x in (gamma, beta, w_k, w_v, b_k, b_v)]
    casted = [ctypes.cast(a, ctypes.POINTER(_vp)) if a is not None else None for a in arrays]
    st = lib.hcr_create(ctypes.byref(dims), *casted, ctypes.byref(out))
    if check:
        _check(st, "hcr_create")
    return st, out.value


def hcr_destroy(handle) -> None:
    lib.hcr_destroy(handle)


def hcr_workspace_bytes(handle, n_tokens: int, n_layers_in_range: int) -> int:
    return lib.hcr_workspace_bytes(handle, n_tokens, n_layers_in_range)


def _restore_call(fn, name, handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                  start_pos, block_table, max_blocks_per_req, k_cache, v_cache, layout,
                  workspace, workspace_bytes, stream, check):
    st = fn(handle, _ptr(hidden), layer_begin, layer_end, n_req, n_tokens, _ptr(cu_seqlens),
            _ptr(start_pos), _ptr(block_table), max_blocks_per_req, _ptr(k_cache),
            _ptr(v_cache), ctypes.byref(layout) if layout is not None else None,
            _ptr(workspace), workspace_bytes, _stream_ptr(stream))
    if check:
        _check(st, name)
    return st


def hcr_restore(handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                block_table, max_blocks_per_req, k_cache, v_cache, layout, workspace,
                workspace_bytes, stream=None, *, check: bool = True) -> int:
    return _restore_call(lib.hcr_restore, "hcr_restore", handle, hidden, layer_begin, layer_end,
                         n_req, n_tokens, cu_seqlens, start_pos, block_table,
                         max_blocks_per_req, k_cache, v_cache, layout, workspace,
                         workspace_bytes, stream, check)


def hcr_restore_prepare(handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                        start_pos, block_table, max_blocks_per_req, k_cache, v_cache, layout,
                        workspace, workspace_bytes, stream=None, *, check: bool = True) -> int:
    return _restore_call(lib.hcr_restore_prepare, "hcr_restore_prepare", handle, hidden,
                         layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                         block_table, max_blocks_per_req, k_cache, v_cache, layout, workspace,
                         workspace_bytes, stream, check)


def hcr_restore_project(handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                        start_pos, block_table, max_blocks_per_req, k_cache, v_cache, layout,
                        workspace, workspace_bytes, stream=None, *, check: bool = True) -> int:
    return _restore_call(lib.hcr_restore_project, "hcr_restore_project", handle, hidden,
                         layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                         block_table, max_blocks_per_req, k_cache, v_cache, layout, workspace,
                         workspace_bytes, stream, check)


def hcr_restore_streamed(handle, hidden_host, layer_begin, layer_end, n_req, n_tokens,
                         cu_seqlens, start_pos, block_table, max_blocks_per_req, k_cache, v_cache,
                         layout, staging, staging_bytes, layers_per_chunk, workspace,
                         workspace_bytes, stream=None, *, check: bool = True) -> int:
    """Layer-pipelined restore: hidden states in (pinned) host memory, copied in
    chunks of layers into a device staging ring while earlier chunks restore."""
    st = lib.hcr_restore_streamed(
        handle, _ptr(hidden_host), layer_begin, layer_end, n_req, n_tokens, _ptr(cu_seqlens),
        _ptr(start_pos), _ptr(block_table), max_blocks_per_req, _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(layout) if layout is not None else None, _ptr(staging), staging_bytes,
        layers_per_chunk, _ptr(workspace), workspace_bytes, _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_streamed")
    return st


def hcr_restore_streamed_chunks(handle, source: hcr_chunk_source, layer_begin, layer_end, n_req,
                                n_tokens, cu_seqlens, start_pos, block_table, max_blocks_per_req,
                                k_cache, v_cache, layout, staging, staging_bytes,
                                layers_per_chunk, workspace, workspace_bytes, stream=None, *,
                                check: bool = True) -> int:
    """Layer-pipelined restore from a host chunk store (hcr_save_hidden's layout)."""
    st = lib.hcr_restore_streamed_chunks(
        handle, ctypes.byref(source), layer_begin, layer_end, n_req, n_tokens, _ptr(cu_seqlens),
        _ptr(start_pos), _ptr(block_table), max_blocks_per_req, _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(layout) if layout is not None else None, _ptr(staging), staging_bytes,
        layers_per_chunk, _ptr(workspace), workspace_bytes, _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_streamed_chunks")
    return st


def hcr_load_kv(handle, kv, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                block_table, max_blocks_per_req, k_cache, v_cache, layout, workspace,
                workspace_bytes, stream=None, *, check: bool = True) -> int:
    """Places saved K/V rows ([layers][2][tokens][d_kv]) into the paged cache."""
    return _restore_call(lib.hcr_load_kv, "hcr_load_kv", handle, kv, layer_begin, layer_end,
                         n_req, n_tokens, cu_seqlens, start_pos, block_table,
                         max_blocks_per_req, k_cache, v_cache, layout, workspace,
                         workspace_bytes, stream, check)


def hcr_save_kv(handle, kv, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                block_table, max_blocks_per_req, k_cache, v_cache, layout, workspace,
                workspace_bytes, stream=None, *, check: bool = True) -> int:
    """Copies the requests' K/V rows out of the paged cache ([layers][2][tokens][d_kv])."""
    return _restore_call(lib.hcr_save_kv, "hcr_save_kv", handle, kv, layer_begin, layer_end,
                         n_req, n_tokens, cu_seqlens, start_pos, block_table,
                         max_blocks_per_req, k_cache, v_cache, layout, workspace,
                         workspace_bytes, stream, check)


def hcr_plan_layer_split(costs: hcr_layer_costs, n_layers: int) -> hcr_layer_split:
    """Min-max layer split between hidden-state restore and K/V load (host only)."""
    out = hcr_layer_split()
    _check(lib.hcr_plan_layer_split(ctypes.byref(costs), n_layers, ctypes.byref(out)),
           "hcr_plan_layer_split")
    return out


def hcr_profile_layer_costs(handle, n_tokens: int, layers_per_chunk: int, reps: int,
                            stream=None) -> hcr_layer_costs:
    """Per-layer costs measured on the current GPU for n_tokens tokens."""
    out = hcr_layer_costs()
    _check(lib.hcr_profile_layer_costs(handle, n_tokens, layers_per_chunk, reps,
                                       _stream_ptr(stream), ctypes.byref(out)),
           "hcr_profile_layer_costs")
    return out


def hcr_restore_streamed_split(handle, hidden_host, kv_host, layer_begin, split_layer, layer_end,
                               n_req, n_tokens, cu_seqlens, start_pos, block_table,
                               max_blocks_per_req, k_cache, v_cache, layout, staging,
                               staging_bytes, layers_per_chunk, workspace, workspace_bytes,
                               stream=None, *, check: bool = True) -> int:
    """Layer-split streamed restore: hidden states below split_layer, saved K/V above."""
    st = lib.hcr_restore_streamed_split(
        handle, _ptr(hidden_host), _ptr(kv_host), layer_begin, split_layer, layer_end, n_req,
        n_tokens, _ptr(cu_seqlens), _ptr(start_pos), _ptr(block_table), max_blocks_per_req,
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout) if layout is not None else None,
        _ptr(staging), staging_bytes, layers_per_chunk, _ptr(workspace), workspace_bytes,
        _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_streamed_split")
    return st


def hcr_encode_hidden(handle, params: hcr_codec_params, hidden, layer_begin, layer_end, n_req,
                      n_tokens, cu_seqlens, codes, scales, stream=None, *,
                      check: bool = True) -> int:
    """Anchor + delta codec: hidden [layers][tokens][d] -> int8 codes + float32 scales."""
    st = lib.hcr_encode_hidden(handle, ctypes.byref(params), _ptr(hidden), layer_begin,
                               layer_end, n_req, n_tokens, _ptr(cu_seqlens), _ptr(codes),
                               _ptr(scales), _stream_ptr(stream))
    if check:
        _check(st, "hcr_encode_hidden")
    return st


def hcr_decode_hidden(handle, params: hcr_codec_params, codes, scales, layer_begin, layer_end,
                      n_req, n_tokens, cu_seqlens, hidden, stream=None, *,
                      check: bool = True) -> int:
    """Inverse of hcr_encode_hidden, into the storage dtype."""
    st = lib.hcr_decode_hidden(handle, ctypes.byref(params), _ptr(codes), _ptr(scales),
                               layer_begin, layer_end, n_req, n_tokens, _ptr(cu_seqlens),
                               _ptr(hidden), _stream_ptr(stream))
    if check:
        _check(st, "hcr_decode_hidden")
    return st


def hcr_encoded_workspace_bytes(handle, n_tokens: int, n_layers_in_range: int) -> int:
    return lib.hcr_encoded_workspace_bytes(handle, n_tokens, n_layers_in_range)


def hcr_restore_encoded(handle, params: hcr_codec_params, codes, scales, layer_begin, layer_end,
                        n_req, n_tokens, cu_seqlens, start_pos, block_table, max_blocks_per_req,
                        k_cache, v_cache, layout, workspace, workspace_bytes, stream=None, *,
                        check: bool = True) -> int:
    """hcr_restore from the codec's encoded form in device memory, decoded
    inside the restore kernels."""
    st = lib.hcr_restore_encoded(
        handle, ctypes.byref(params), _ptr(codes), _ptr(scales), layer_begin, layer_end, n_req,
        n_tokens, _ptr(cu_seqlens), _ptr(start_pos), _ptr(block_table), max_blocks_per_req,
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout) if layout is not None else None,
        _ptr(workspace), workspace_bytes, _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_encoded")
    return st


def encoded_staging_bytes(n_tokens: int, d_model: int, layers_per_chunk: int, slots: int) -> int:
    """Staging hcr_restore_streamed_encoded needs for `slots` slots of
    `layers_per_chunk` layers (codes, scales and decoded hidden states each)."""
    def a(x):
        return (x + 255) // 256 * 256
    c = layers_per_chunk
    return slots * (a(c * n_tokens * d_model) + a(c * n_tokens * 4) + a(c * n_tokens * d_model * 2))


def hcr_restore_streamed_encoded(handle, params: hcr_codec_params, codes_host, scales_host,
                                 layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                                 block_table, max_blocks_per_req, k_cache, v_cache, layout,
                                 staging, staging_bytes, layers_per_chunk, workspace,
                                 workspace_bytes, stream=None, *, check: bool = True) -> int:
    """Layer-pipelined restore from the codec's encoded form in host memory."""
    st = lib.hcr_restore_streamed_encoded(
        handle, ctypes.byref(params), _ptr(codes_host), _ptr(scales_host), layer_begin,
        layer_end, n_req, n_tokens, _ptr(cu_seqlens), _ptr(start_pos), _ptr(block_table),
        max_blocks_per_req, _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(layout) if layout is not None else None, _ptr(staging), staging_bytes,
        layers_per_chunk, _ptr(workspace), workspace_bytes, _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_streamed_encoded")
    return st


def hcr_save_hidden(handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                    start_pos, chunk_table, max_chunks_per_req, chunk_tokens, chunk_store,
                    num_chunks, stream=None, *, check: bool = True) -> int:
    """Scatter layer inputs into fixed-size, token-before-layer chunks."""
    st = lib.hcr_save_hidden(handle, _ptr(hidden), layer_begin, layer_end, n_req, n_tokens,
                             _ptr(cu_seqlens), _ptr(start_pos), _ptr(chunk_table),
                             max_chunks_per_req, chunk_tokens, _ptr(chunk_store), num_chunks,
                             _stream_ptr(stream))
    if check:
        _check(st, "hcr_save_hidden")
    return st


def hcr_restore_no_alloc(handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                         start_pos, block_table, max_blocks_per_req, k_cache, v_cache, layout,
                         stream=None, *, check: bool = True) -> int:
    """hcr_restore with the library's built-in scratch array (no workspace argument)."""
    st = lib.hcr_restore_no_alloc(handle, _ptr(hidden), layer_begin, layer_end, n_req, n_tokens,
                                  _ptr(cu_seqlens), _ptr(start_pos), _ptr(block_table),
                                  max_blocks_per_req, _ptr(k_cache), _ptr(v_cache),
                                  ctypes.byref(layout) if layout is not None else None,
                                  _stream_ptr(stream))
    if check:
        _check(st, "hcr_restore_no_alloc")
    return st


def hcr_check_device_error(handle, stream=None):
    """Returns (status, raw HCR_DEVERR_* bits); never raises for device errors."""
    flags = ctypes.c_uint32(0)
    st = lib.hcr_check_device_error(handle, _stream_ptr(stream), ctypes.byref(flags))
    return st, flags.value


def hcr_project_variant(handle, n_tokens: int, n_layers: int) -> int:
    """Tile variant the projection uses: 1 single CTAs, 2 CTA pairs, 3 CTA pairs
    with weight rows as M and chunks of up to 320 tokens as N (host-only)."""
    return lib.hcr_project_variant(handle, n_tokens, n_layers)


def hcr_debug_fused_stats(handle, n_tokens: int, n_layers: int, workspace_bytes: int) -> int:
    """0, or the layers the prepare kernel still computes when the projection
    computes the rest of the norm statistics (host-only)."""
    return lib.hcr_debug_fused_stats(handle, n_tokens, n_layers, workspace_bytes)


def hcr_debug_plan(dims, n_tokens: int, n_layers: int, num_sms: int, pair_clusters: int,
                   swap_clusters: int, workspace_bytes: int) -> tuple:
    """(tile variant, fused statistics' prepare layers or 0) of a restore on a
    device with the given unit counts (host-only, no handle)."""
    out = (ctypes.c_int32 * 2)()
    st = lib.hcr_debug_plan(ctypes.byref(dims), n_tokens, n_layers, num_sms, pair_clusters,
                            swap_clusters, workspace_bytes, out)
    if st != 0:
        raise RuntimeError(hcr_last_error())
    return int(out[0]), int(out[1])


def hcr_debug_swap_plan(n_tokens: int) -> dict:
    """The weight-row tiles' chunks and TMEM slots for n_tokens (host-only)."""
    out = (ctypes.c_int32 * 6)()
    st = lib.hcr_debug_swap_plan(n_tokens, out)
    if st != 0:
        raise RuntimeError(hcr_last_error())
    keys = ("chunk", "n_chunks", "last_n", "slot_cols", "n_slots", "ok")
    return dict(zip(keys, (int(v) for v in out)))


def hcr_num_sms(handle) -> int:
    return lib.hcr_num_sms(handle)


def hcr_debug_timeout_record(handle, stream=None):
    """(status, [which wait, CTA, thread, a, b, parity]) of the first wait that gave up."""
    out = (ctypes.c_uint32 * 6)()
    st = lib.hcr_debug_timeout_record(handle, _stream_ptr(stream), out)
    return st, list(out)


def hcr_debug_set_variant(handle, variant: int) -> int:
    """Testing hook: 0 automatic, 1 single-CTA tiles, 2 CTA-pair tiles, 3 CTA-pair
    tiles with weight rows as M (128-wide heads only)."""
    return lib.hcr_debug_set_variant(handle, variant)


def hcr_debug_set_stall(handle, enable: bool) -> int:
    """Testing hook: make restores through `handle` run into the bounded-wait timeout."""
    return lib.hcr_debug_set_stall(handle, 1 if enable else 0)
