"""A small owner object over the C ABI: one handle plus a reusable workspace.

PyTorch is used only to hold device memory (the workspace) and to name the
stream; every computation runs inside libhcr.so.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import binding as B

_DTYPE = {"bf16": B.HCR_DTYPE_BF16, "fp16": B.HCR_DTYPE_FP16}
_TORCH = {B.HCR_DTYPE_BF16: torch.bfloat16, B.HCR_DTYPE_FP16: torch.float16}


def make_dims(n_layers: int, d_model: int, n_heads: int, n_kv_heads: int, head_dim: int,
              norm: str = "rms", norm_eps: float = 1e-5, rope: bool = True,
              rope_theta: float = 1e4, max_position: int = 1, dtype: str = "bf16",
              has_kv_bias: bool = False) -> B.hcr_model_dims:
    return B.hcr_model_dims(
        n_layers, d_model, n_heads, n_kv_heads, head_dim,
        B.HCR_NORM_LAYER if norm == "ln" else B.HCR_NORM_RMS, norm_eps,
        B.HCR_ROPE_ROTATE_HALF if rope else B.HCR_ROPE_NONE, rope_theta, max(1, max_position),
        _DTYPE[dtype], 1 if has_kv_bias else 0)


class Restorer:
    """Holds a packed model (hcr_create) and restores caches from hidden states.

    params: per layer, an object with gamma, beta, w_k, w_v, b_k, b_v device
    tensors (beta/b_k/b_v may be None), in the dims' storage dtype.
    """

    def __init__(self, dims: B.hcr_model_dims, params: Sequence):
        self.dims = dims
        L = dims.n_layers
        if len(params) != L:
            raise ValueError(f"{len(params)} layer parameter sets for {L} layers")
        ln = dims.norm == B.HCR_NORM_LAYER
        _, self.handle = B.hcr_create(
            dims, [p.gamma for p in params], [p.beta for p in params] if ln else None,
            [p.w_k for p in params], [p.w_v for p in params],
            [p.b_k for p in params] if dims.has_kv_bias else None,
            [p.b_v for p in params] if dims.has_kv_bias else None)
        self._ws: Optional[torch.Tensor] = None

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH[self.dims.dtype]

    def workspace(self, n_tokens: int, n_layers: int, device) -> torch.Tensor:
        need = B.hcr_workspace_bytes(self.handle, n_tokens, n_layers)
        if self._ws is None or self._ws.numel() < need:
            # torch's caching allocator hands out 512-byte-aligned blocks
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def _check_tensors(self, hidden, cu_seqlens, start_pos, block_table, k_cache, v_cache):
        """The library reads raw pointers: shapes are the caller's contract, but
        layout, dtype and device mistakes are caught here."""
        dt = self.torch_dtype
        for name, t, want in (("hidden", hidden, dt), ("k_cache", k_cache, dt),
                              ("v_cache", v_cache, dt), ("cu_seqlens", cu_seqlens, torch.int32),
                              ("start_pos", start_pos, torch.int32),
                              ("block_table", block_table, torch.int32)):
            if not isinstance(t, torch.Tensor):
                raise TypeError(f"{name} must be a torch.Tensor")
            if not t.is_cuda:
                raise ValueError(f"{name} must be on a CUDA device")
            if t.dtype != want:
                raise TypeError(f"{name} must be {want}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if hidden.dim() != 3 or hidden.shape[-1] != self.dims.d_model:
            raise ValueError(f"hidden must be [layers][tokens][{self.dims.d_model}]")

    def _args(self, hidden, layer_begin, layer_end, cu_seqlens, start_pos, block_table,
              k_cache, v_cache, num_blocks, block_size, layer_stride_elems, workspace):
        self._check_tensors(hidden, cu_seqlens, start_pos, block_table, k_cache, v_cache)
        n_req = int(start_pos.numel())
        n_tokens = int(hidden.shape[-2]) if hidden is not None and hidden.dim() >= 2 else 0
        nl = layer_end - layer_begin
        if workspace is None:
            dev = (hidden if hidden is not None else k_cache).device
            workspace = self.workspace(n_tokens, max(nl, 1), dev)
        layout = B.hcr_cache_layout(num_blocks, block_size, layer_stride_elems)
        return (self.handle, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                start_pos, block_table, int(block_table.shape[-1]), k_cache, v_cache, layout,
                workspace, workspace.numel())

    def restore(self, hidden, layer_begin, layer_end, cu_seqlens, start_pos, block_table,
                k_cache, v_cache, num_blocks, block_size, layer_stride_elems=0, stream=None,
                workspace=None, stage: str = "all", check: bool = True) -> int:
        """hidden: [layer_end-layer_begin][T][d]; caches: base of layer layer_begin."""
        args = self._args(hidden, layer_begin, layer_end, cu_seqlens, start_pos, block_table,
                          k_cache, v_cache, num_blocks, block_size, layer_stride_elems,
                          workspace)
        if stream is None:
            stream = torch.cuda.current_stream()
        fn = {"all": B.hcr_restore, "prepare": B.hcr_restore_prepare,
              "project": B.hcr_restore_project}[stage]
        return fn(*args, stream, check=check)

    # --- the other entry points: thin wrappers that own staging buffers ----
    def _stream(self, stream):
        return torch.cuda.current_stream() if stream is None else stream

    def _staging(self, nbytes: int, device) -> torch.Tensor:
        st = getattr(self, "_stage_buf", None)
        if st is None or st.numel() < nbytes or st.device != torch.device(device):
            self._stage_buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self._stage_buf

    def restore_streamed(self, hidden_host, layer_begin, layer_end, cu_seqlens, start_pos,
                         block_table, k_cache, v_cache, num_blocks, block_size,
                         layers_per_chunk: int = 4, slots: int = 3, layer_stride_elems=0,
                         stream=None) -> int:
        """Layer-pipelined restore from hidden states in (pinned) host memory,
        [layer_end-layer_begin][T][d]."""
        if hidden_host.is_cuda:
            raise ValueError("hidden_host must be in host memory")
        dev = k_cache.device
        T, d = int(hidden_host.shape[-2]), self.dims.d_model
        c = max(1, min(layers_per_chunk, layer_end - layer_begin))
        staging = self._staging(slots * c * T * d * 2, dev)
        ws = self.workspace(T, c, dev)
        return B.hcr_restore_streamed(
            self.handle, hidden_host, layer_begin, layer_end, int(start_pos.numel()), T,
            cu_seqlens, start_pos, block_table, int(block_table.shape[-1]), k_cache, v_cache,
            B.hcr_cache_layout(num_blocks, block_size, layer_stride_elems), staging,
            staging.numel(), layers_per_chunk, ws, ws.numel(), self._stream(stream))

    def save_hidden(self, hidden, layer_begin, layer_end, cu_seqlens, start_pos, chunk_table,
                    chunk_tokens, chunk_store, stream=None) -> int:
        """Layer inputs into a chunk store [num_chunks][n_layers][chunk_tokens][d]
        (device or pinned host memory)."""
        return B.hcr_save_hidden(self.handle, hidden, layer_begin, layer_end,
                                 int(start_pos.numel()), int(hidden.shape[-2]), cu_seqlens,
                                 start_pos, chunk_table, int(chunk_table.shape[-1]),
                                 chunk_tokens, chunk_store, int(chunk_store.shape[0]),
                                 self._stream(stream))

    def _kv(self, fn, kv, layer_begin, layer_end, cu_seqlens, start_pos, block_table, k_cache,
            v_cache, num_blocks, block_size, layer_stride_elems, stream):
        T = int(kv.shape[-2])
        ws = self.workspace(T, 1, k_cache.device)
        return fn(self.handle, kv, layer_begin, layer_end, int(start_pos.numel()), T, cu_seqlens,
                  start_pos, block_table, int(block_table.shape[-1]), k_cache, v_cache,
                  B.hcr_cache_layout(num_blocks, block_size, layer_stride_elems), ws, ws.numel(),
                  self._stream(stream))

    def save_kv(self, kv, layer_begin, layer_end, cu_seqlens, start_pos, block_table, k_cache,
                v_cache, num_blocks, block_size, layer_stride_elems=0, stream=None) -> int:
        """K/V rows out of the paged cache into kv [layers][2][T][d_kv]."""
        return self._kv(B.hcr_save_kv, kv, layer_begin, layer_end, cu_seqlens, start_pos,
                        block_table, k_cache, v_cache, num_blocks, block_size,
                        layer_stride_elems, stream)

    def load_kv(self, kv, layer_begin, layer_end, cu_seqlens, start_pos, block_table, k_cache,
                v_cache, num_blocks, block_size, layer_stride_elems=0, stream=None) -> int:
        """K/V rows kv [layers][2][T][d_kv] back into the paged cache."""
        return self._kv(B.hcr_load_kv, kv, layer_begin, layer_end, cu_seqlens, start_pos,
                        block_table, k_cache, v_cache, num_blocks, block_size,
                        layer_stride_elems, stream)

    def encode(self, hidden, layer_begin, layer_end, cu_seqlens, n_req, codes=None, scales=None,
               bins=(0.5, 1.0, 1.5), group_tokens: int = 10, stream=None):
        """Hidden-state codec: returns (codes int8 [Lr][T][d], scales float32 [Lr][T])."""
        Lr, T, d = (int(x) for x in hidden.shape)
        if codes is None:
            codes = torch.empty((Lr, T, d), dtype=torch.int8, device=hidden.device)
        if scales is None:
            scales = torch.zeros((Lr, T), dtype=torch.float32, device=hidden.device)
        B.hcr_encode_hidden(self.handle, B.codec_params(bins, group_tokens), hidden, layer_begin,
                            layer_end, n_req, T, cu_seqlens, codes, scales, self._stream(stream))
        return codes, scales

    def decode(self, codes, scales, layer_begin, layer_end, cu_seqlens, n_req, out=None,
               bins=(0.5, 1.0, 1.5), group_tokens: int = 10, stream=None):
        """Inverse of encode, into the storage dtype."""
        if out is None:
            out = torch.empty(tuple(codes.shape), dtype=self.torch_dtype, device=codes.device)
        B.hcr_decode_hidden(self.handle, B.codec_params(bins, group_tokens), codes, scales,
                            layer_begin, layer_end, n_req, int(codes.shape[-2]), cu_seqlens, out,
                            self._stream(stream))
        return out

    def encoded_workspace(self, n_tokens: int, n_layers: int, device) -> torch.Tensor:
        need = B.hcr_encoded_workspace_bytes(self.handle, n_tokens, n_layers)
        ws = getattr(self, "_enc_ws", None)
        if ws is None or ws.numel() < need or ws.device != torch.device(device):
            self._enc_ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._enc_ws

    def restore_encoded(self, codes, scales, layer_begin, layer_end, cu_seqlens, start_pos,
                        block_table, k_cache, v_cache, num_blocks, block_size,
                        bins=(0.5, 1.0, 1.5), group_tokens: int = 10, layer_stride_elems=0,
                        stream=None, workspace=None, check: bool = True) -> int:
        """Restore from the codec's form in device memory (codes int8
        [Lr][T][d], scales float32 [Lr][T]), decoded inside the kernels."""
        dt = self.torch_dtype
        for name, t, want in (("codes", codes, torch.int8), ("scales", scales, torch.float32),
                              ("k_cache", k_cache, dt), ("v_cache", v_cache, dt),
                              ("cu_seqlens", cu_seqlens, torch.int32),
                              ("start_pos", start_pos, torch.int32),
                              ("block_table", block_table, torch.int32)):
            if not isinstance(t, torch.Tensor) or not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if t.dtype != want:
                raise TypeError(f"{name} must be {want}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if codes.dim() != 3 or codes.shape[-1] != self.dims.d_model:
            raise ValueError(f"codes must be [layers][tokens][{self.dims.d_model}]")
        T = int(codes.shape[-2])
        nl = layer_end - layer_begin
        if workspace is None:
            workspace = self.encoded_workspace(T, max(nl, 1), codes.device)
        return B.hcr_restore_encoded(
            self.handle, B.codec_params(bins, group_tokens), codes, scales, layer_begin,
            layer_end, int(start_pos.numel()), T, cu_seqlens, start_pos, block_table,
            int(block_table.shape[-1]), k_cache, v_cache,
            B.hcr_cache_layout(num_blocks, block_size, layer_stride_elems), workspace,
            workspace.numel(), self._stream(stream), check=check)

    def plan_split(self, n_tokens: int, layers_per_chunk: int = 4, reps: int = 5, stream=None):
        """Profiles the per-layer costs on this GPU and returns (costs, split)."""
        costs = B.hcr_profile_layer_costs(self.handle, n_tokens, layers_per_chunk, reps,
                                          self._stream(stream))
        return costs, B.hcr_plan_layer_split(costs, self.dims.n_layers)

    def check(self, stream=None):
        if stream is None:
            stream = torch.cuda.current_stream()
        return B.hcr_check_device_error(self.handle, stream)

    def close(self):
        if self.handle:
            B.hcr_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
