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
