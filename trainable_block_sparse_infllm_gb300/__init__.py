"""InfLLM v2 block-sparse attention for GB300 (sm_103a): Python binding.

The compute path is the CUDA library ``libinfllmv2.so`` behind the C ABI in
``include/infllmv2.h``; this module only passes torch tensors' device
pointers, sizes and the current stream to it.  PyTorch provides device
memory and streams.  Entry points mirror the C names:

    compress_keys        stage 1, semantic-kernel key means
    select_blocks        stage 2, block relevance and top-k
    sparse_attn_decode   stage 3 for decode / speculative verification
    sparse_attn_prefill  stage 3 for prefill
    append_kv            write the newest tokens' keys and values to the caches
    decode_step          stages 1-3 for the newest token(s), one launch when n_q = 1
    append_decode_step   the cache append and stages 1-3 for one new token, one launch
    coarse_means, select_blocks_coarse_lse
                         the coarse-kernel LSE approximation (prefill path)
    sparse_attn_backward dq, dk, dv of stage 3 with the selection held fixed

Method: "MiniCPM4: Ultra-Efficient LLMs on End Devices", section "InfLLM v2:
Trainable Sparse Attention for Both Prefilling and Decoding".
"""

from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import (InfLLMv2Error, OP_BACKWARD, OP_DECODE, OP_DECODE_STEP, OP_PREFILL, OP_SELECT,  # noqa: F401
                   Params, DEVICE_BAD_KV_LEN, DEVICE_BOUNDS, DEVICE_TIMEOUT)

__all__ = [
    "Params", "InfLLMv2Error", "make_params", "num_kernels", "max_selected", "workspace_size",
    "alloc_kc", "alloc_workspace", "compress_keys", "select_blocks", "sparse_attn_decode",
    "sparse_attn_prefill", "decode_step", "coarse_means", "alloc_kcc", "select_blocks_coarse_lse",
    "sparse_attn_backward", "append_kv", "append_decode_step", "get_device_status", "OP_SELECT", "OP_DECODE", "OP_PREFILL",
    "OP_DECODE_STEP", "OP_BACKWARD", "DECODE_MAX_NQ", "is_checked_build", "test_hooks",
]

DECODE_MAX_NQ = 16


def make_params(batch: int, n_kv_heads: int, max_kv_len: int, topk: int,
                includes_forced: bool = True, n_init: int = 1, n_local: int = 2,
                score_scale: float | None = None, attn_scale: float | None = None) -> Params:
    p = Params()
    _lib.lib.infllmv2_default_params(ctypes.byref(p), batch, n_kv_heads, max_kv_len, topk,
                                     1 if includes_forced else 0)
    p.n_init_blocks = n_init
    p.n_local_blocks = n_local
    if score_scale is not None:
        p.score_scale = score_scale
    if attn_scale is not None:
        p.attn_scale = attn_scale
    return p


def num_kernels(p: Params) -> int:
    return int(_lib.lib.infllmv2_num_kernels(ctypes.byref(p)))


def max_selected(p: Params) -> int:
    k = int(_lib.lib.infllmv2_max_selected(ctypes.byref(p)))
    if k < 0:
        raise InfLLMv2Error(_lib.INVALID_ARGUMENT, _lib.lib.infllmv2_last_error().decode())
    return k


def workspace_size(p: Params, n_q: int, op: int) -> int:
    return int(_lib.lib.infllmv2_workspace_size(ctypes.byref(p), n_q, op))


def _ptr(t: torch.Tensor | None, host_ok: bool = False):
    """Device pointer of ``t``.  host_ok: a pinned host tensor is accepted too
    (for outputs the kernels write with ordinary stores)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise InfLLMv2Error(_lib.INVALID_ARGUMENT, "tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise InfLLMv2Error(_lib.INVALID_ARGUMENT, "tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def alloc_kc(p: Params, device=None) -> torch.Tensor:
    """Compressed-key buffer bf16 [B, Hkv, 2, n_c(max_kv_len), 128] (hi and lo planes)."""
    return torch.empty((p.batch, p.n_kv_heads, 2, max(num_kernels(p), 0), p.head_dim),
                       dtype=torch.bfloat16, device=device)


def alloc_workspace(p: Params, n_q: int, op: int, device=None) -> torch.Tensor | None:
    n = workspace_size(p, n_q, op)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def compress_keys(p: Params, k_cache: torch.Tensor, kv_lens: torch.Tensor, kc: torch.Tensor,
                  kernel_begin: int = 0, kernel_end: int = -1, stream=None) -> torch.Tensor:
    _lib.check(_lib.lib.infllmv2_compress_keys(ctypes.byref(p), _ptr(k_cache), _ptr(kv_lens),
                                               kernel_begin, kernel_end, _ptr(kc), _stream(stream)))
    return kc


def select_blocks(p: Params, q: torch.Tensor, kc: torch.Tensor, kv_lens: torch.Tensor,
                  block_idx: torch.Tensor, n_selected: torch.Tensor,
                  block_scores: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None):
    n_q = q.shape[1]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _lib.check(_lib.lib.infllmv2_select_blocks(ctypes.byref(p), _ptr(q), n_q, _ptr(kc), _ptr(kv_lens),
                                               _ptr(block_idx), _ptr(n_selected), _ptr(block_scores),
                                               _ptr(workspace), ws_bytes, _stream(stream)))
    return block_idx, n_selected


def select_blocks_static(p: Params, q: torch.Tensor, kc: torch.Tensor, kv_lens: torch.Tensor,
                         block_idx: torch.Tensor, n_selected: torch.Tensor,
                         block_scores: torch.Tensor | None = None, stream=None):
    """select_blocks with the library's built-in scratch instead of a workspace.

    For embedders that cannot hand over device scratch at the call site
    (start-up-planned device memory, C hosts without a device allocator).
    At most 8 MiB of scratch; calls that overlap on the GPU share it.
    """
    n_q = q.shape[1]
    _lib.check(_lib.lib.infllmv2_select_blocks_static(ctypes.byref(p), _ptr(q), n_q, _ptr(kc), _ptr(kv_lens),
                                                      _ptr(block_idx), _ptr(n_selected), _ptr(block_scores),
                                                      _stream(stream)))
    return block_idx, n_selected


def _attn(fn, p, q, k_cache, v_cache, kv_lens, block_idx, n_selected, out, lse, workspace, stream):
    n_q = q.shape[1]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _lib.check(fn(ctypes.byref(p), _ptr(q), n_q, _ptr(k_cache), _ptr(v_cache), _ptr(kv_lens),
                  _ptr(block_idx), _ptr(n_selected), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                  _stream(stream)))
    return out, lse


def sparse_attn_decode(p: Params, q, k_cache, v_cache, kv_lens, block_idx, n_selected, out,
                       lse=None, workspace=None, stream=None):
    return _attn(_lib.lib.infllmv2_sparse_attn_decode, p, q, k_cache, v_cache, kv_lens, block_idx,
                 n_selected, out, lse, workspace, stream)


def sparse_attn_prefill(p: Params, q, k_cache, v_cache, kv_lens, block_idx, n_selected, out,
                        lse=None, workspace=None, stream=None):
    return _attn(_lib.lib.infllmv2_sparse_attn_prefill, p, q, k_cache, v_cache, kv_lens, block_idx,
                 n_selected, out, lse, workspace, stream)


def alloc_kcc(p: Params, coarse: int, device=None) -> torch.Tensor:
    """Coarse-window means bf16 [B, Hkv, 2, max_kv_len // coarse, 128] (hi and lo planes)."""
    return torch.empty((p.batch, p.n_kv_heads, 2, p.max_kv_len // coarse, p.head_dim),
                       dtype=torch.bfloat16, device=device)


def coarse_means(p: Params, k_cache: torch.Tensor, kv_lens: torch.Tensor, coarse: int, kcc: torch.Tensor,
                 stream=None) -> torch.Tensor:
    _lib.check(_lib.lib.infllmv2_coarse_means(ctypes.byref(p), _ptr(k_cache), _ptr(kv_lens), coarse, _ptr(kcc),
                                              _stream(stream)))
    return kcc


def select_blocks_coarse_lse(p: Params, q: torch.Tensor, kc: torch.Tensor, coarse: int, kcc: torch.Tensor,
                             kv_lens: torch.Tensor, block_idx: torch.Tensor, n_selected: torch.Tensor,
                             block_scores: torch.Tensor | None = None, stream=None):
    """select_blocks (prefill path) with the LSE over coarse windows of `coarse` keys."""
    n_q = q.shape[1]
    _lib.check(_lib.lib.infllmv2_select_blocks_coarse_lse(ctypes.byref(p), _ptr(q), n_q, _ptr(kc), coarse, _ptr(kcc),
                                                          _ptr(kv_lens), _ptr(block_idx), _ptr(n_selected),
                                                          _ptr(block_scores), _stream(stream)))
    return block_idx, n_selected


def decode_step(p: Params, q, k_cache, v_cache, kv_lens, kc, block_idx, n_selected, out,
                lse=None, workspace=None, stream=None):
    """Newest kernel mean(s), selection and attention for the last n_q tokens.

    ``kc`` must hold every kernel that ends before those tokens; the ones that
    end inside them are recomputed and written back.  ``out`` and ``lse`` may
    be pinned host tensors: the step then stores its result straight to host
    memory."""
    n_q = q.shape[1]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _lib.check(_lib.lib.infllmv2_decode_step(ctypes.byref(p), _ptr(q), n_q, _ptr(k_cache), _ptr(v_cache),
                                             _ptr(kv_lens), _ptr(kc), _ptr(block_idx), _ptr(n_selected),
                                             _ptr(out, host_ok=True), _ptr(lse, host_ok=True), _ptr(workspace),
                                             ws_bytes, _stream(stream)))
    return block_idx, n_selected, out, lse


def append_kv(p: Params, k_new, v_new, kv_lens, k_cache, v_cache, q_src=None, q_dst=None, stream=None):
    """Write k_new / v_new [B, Hkv, n_q, d] to cache rows kv_lens - n_q .. kv_lens - 1 and, if given,
    copy q_src to q_dst.  k_new, v_new and q_src may be pinned host tensors."""
    n_q = k_new.shape[2]
    _lib.check(_lib.lib.infllmv2_append_kv(ctypes.byref(p), n_q, _ptr(k_new, host_ok=True),
                                           _ptr(v_new, host_ok=True), _ptr(kv_lens), _ptr(k_cache),
                                           _ptr(v_cache), _ptr(q_src, host_ok=True), _ptr(q_dst), _stream(stream)))
    return k_cache, v_cache


def append_decode_step(p: Params, q, k_new, v_new, k_cache, v_cache, kv_lens, kc, block_idx, n_selected, out,
                       lse=None, stream=None):
    """append_kv then decode_step for one new token per sequence, as one launch.

    ``q`` [B, 1, Hq, d], ``k_new`` / ``v_new`` [B, Hkv, 1, d] may be pinned host
    tensors, like ``out`` and ``lse``; the token's key and value go to cache
    rows kv_lens - 1."""
    _lib.check(_lib.lib.infllmv2_append_decode_step(
        ctypes.byref(p), _ptr(q, host_ok=True), q.shape[1], _ptr(k_new, host_ok=True), _ptr(v_new, host_ok=True),
        _ptr(k_cache), _ptr(v_cache), _ptr(kv_lens), _ptr(kc), _ptr(block_idx), _ptr(n_selected),
        _ptr(out, host_ok=True), _ptr(lse, host_ok=True), _stream(stream)))
    return block_idx, n_selected, out, lse


def sparse_attn_backward(p: Params, q, k_cache, v_cache, kv_lens, block_idx, n_selected, out, lse, dout,
                         dq, dk, dv, workspace, stream=None):
    """dq, dk, dv (fp32) of the block-sparse attention for upstream ``dout``,
    with ``out`` and ``lse`` from the forward call on the same inputs."""
    n_q = q.shape[1]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _lib.check(_lib.lib.infllmv2_sparse_attn_backward(
        ctypes.byref(p), _ptr(q), n_q, _ptr(k_cache), _ptr(v_cache), _ptr(kv_lens), _ptr(block_idx),
        _ptr(n_selected), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        ws_bytes, _stream(stream)))
    return dq, dk, dv


def is_checked_build() -> bool:
    """True when the loaded library is the checked build (INFLLMV2_CHECKED)."""
    return bool(_lib.lib.infllmv2_is_checked_build())


def test_hooks(flags: int) -> None:
    """Fault injection of the checked build's tests (infllmv2_test_hooks)."""
    _lib.check(_lib.lib.infllmv2_test_hooks(flags))


def get_device_status(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _lib.check(_lib.lib.infllmv2_get_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def default_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)
