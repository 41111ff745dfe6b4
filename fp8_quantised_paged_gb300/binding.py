"""FP8-quantised paged decode attention for GB300 (sm_103a).

Two calls, both hand-written CUDA kernels behind a C ABI (``include/fp8pa.h``):

* :func:`kv_append_quant` -- absmax-scale each new token's K/V rows, round
  them to E4M3 or E5M2 (or symmetric INT8 codes) and scatter codes and
  scales into the paged cache.
* :func:`paged_decode_attention` -- grouped-query (or shared-latent MLA)
  attention of one query token per request over its paged FP8 cache, split
  across the GPU and merged.

These wrappers only check torch tensors and pass their device pointers and
the current CUDA stream to the library.  PyTorch provides memory and streams;
all arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native as N
from ._native import (E4M3, E5M2, INT8, OUT_BF16, OUT_F32, SCALE_CHANNEL_STATIC, SCALE_MX_BLOCK,
                      SCALE_SEGMENT, SCALE_TOKEN_GROUP, SCALE_TOKEN_HEAD, SEGMENT_TOKENS,
                      Fp8paError)

__all__ = ["kv_append_quant", "kv_append_quant_segment", "segment_scale_heads",
           "kv_channel_scales", "kv_channel_absmax_update",
           "kv_scales_from_absmax", "paged_decode_attention", "paged_multiquery_attention",
           "decode_step", "decode_workspace_bytes", "get_device_error", "set_decode_workers",
           "version", "E4M3", "E5M2", "INT8", "SCALE_TOKEN_HEAD", "SCALE_CHANNEL_STATIC",
           "SCALE_TOKEN_GROUP", "SCALE_MX_BLOCK", "SCALE_SEGMENT", "SEGMENT_TOKENS", "OUT_BF16",
           "OUT_F32", "Fp8paError"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class _Nop:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


_NOP = _Nop()


def _on(dev):
    """Make `dev` current for a call (a no-op when it already is)."""
    return _NOP if dev.index == torch.cuda.current_device() else torch.cuda.device(dev)


def _scale_dtype(scale_mode):
    """fp32 scales, or E8M0 exponent bytes for the MX block mode."""
    return torch.uint8 if scale_mode == SCALE_MX_BLOCK else torch.float32


def _need(t, dtype, name, device=None):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def version() -> int:
    return int(N.lib.fp8pa_version())


def set_decode_workers(workers: int) -> None:
    N.check(N.lib.fp8pa_set_decode_workers(int(workers)), "set_decode_workers")


def kv_append_quant(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, fmt=E4M3,
                    scale_mode=SCALE_TOKEN_HEAD, group_size=64, stream=None):
    """k, v: bf16 [num_tokens, Hkv, D] (v may be None for the MLA latent);
    slot_mapping: int32 [num_tokens]; caches: uint8 [num_blocks, Hkv, bs, D];
    scales: float32 per the scale mode, uint8 E8M0 exponents for SCALE_MX_BLOCK
    (see include/fp8pa.h)."""
    _need(k, torch.bfloat16, "k")
    dev = k.device
    _need(v, torch.bfloat16, "v", dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    _need(k_cache, torch.uint8, "k_cache", dev)
    _need(v_cache, torch.uint8, "v_cache", dev)
    _need(k_scale, _scale_dtype(scale_mode), "k_scale", dev)
    _need(v_scale, _scale_dtype(scale_mode), "v_scale", dev)
    n, hkv, d = k.shape
    nb, _, bs, _ = k_cache.shape
    with _on(dev):
        rc = N.lib.fp8pa_kv_append_quant(_ptr(k), _ptr(v), _ptr(slot_mapping), n, hkv, d, fmt,
                                         scale_mode, group_size, _ptr(k_cache), _ptr(v_cache),
                                         _ptr(k_scale), _ptr(v_scale), nb, bs, _stream(stream))
    N.check(rc, "kv_append_quant")


def segment_scale_heads(n_kv_heads: int) -> int:
    """Row length of a SCALE_SEGMENT scale tensor: KV heads rounded up to 4."""
    return (n_kv_heads + 3) // 4 * 4


def kv_append_quant_segment(k, v, slot_mapping, seq_offsets, seq_start_pos, k_cache, v_cache,
                            k_scale, v_scale, seg_state, fmt=E4M3, stream=None):
    """Append with block-wise cumulative rescaling (SCALE_SEGMENT).
    k, v: bf16 [num_tokens, Hkv, D] (v may be None); seq_offsets: int32
    [num_seqs + 1]; seq_start_pos: int32 [num_seqs] (each sequence's cached
    length before the call); scales: float32 [num_blocks, round_up(Hkv, 4)];
    seg_state: float32 [num_seqs, 2, Hkv, 2], carried between calls (see
    include/fp8pa.h)."""
    _need(k, torch.bfloat16, "k")
    dev = k.device
    _need(v, torch.bfloat16, "v", dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    _need(seq_offsets, torch.int32, "seq_offsets", dev)
    _need(seq_start_pos, torch.int32, "seq_start_pos", dev)
    _need(k_cache, torch.uint8, "k_cache", dev)
    _need(v_cache, torch.uint8, "v_cache", dev)
    _need(k_scale, torch.float32, "k_scale", dev)
    _need(v_scale, torch.float32, "v_scale", dev)
    _need(seg_state, torch.float32, "seg_state", dev)
    n, hkv, d = k.shape
    nb, _, bs, _ = k_cache.shape
    ns = seq_start_pos.numel()
    if seq_offsets.numel() != ns + 1 or tuple(seg_state.shape) != (ns, 2, hkv, 2):
        raise ValueError("seq_offsets must have num_seqs + 1 entries and seg_state "
                         "[num_seqs, 2, Hkv, 2]")
    if tuple(k_scale.shape) != (nb, segment_scale_heads(hkv)):
        raise ValueError("k_scale must be [num_blocks, round_up(Hkv, 4)]")
    with _on(dev):
        rc = N.lib.fp8pa_kv_append_quant_segment(
            _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(seq_offsets), _ptr(seq_start_pos), ns,
            hkv, d, fmt, _ptr(seg_state), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
            _ptr(v_scale), nb, bs, _stream(stream))
    N.check(rc, "kv_append_quant_segment")


def kv_channel_scales(x, fmt=E5M2, out=None, stream=None):
    """Static per-channel scales max(absmax over tokens / FMAX, 1e-12) of a
    bf16 [N, Hkv, D] tensor; returns float32 [Hkv, D]."""
    _need(x, torch.bfloat16, "x")
    n, hkv, d = x.shape
    if out is None:
        out = torch.empty((hkv, d), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, "out", x.device)
    with torch.cuda.device(x.device):
        rc = N.lib.fp8pa_kv_channel_scales(_ptr(x), n, hkv, d, fmt, _ptr(out), _stream(stream))
    N.check(rc, "kv_channel_scales")
    return out


def kv_channel_absmax_update(x, running_absmax, stream=None):
    """Fold a prefill batch x (bf16 [N, Hkv, D]) into a running per-channel
    absmax (float32 [Hkv, D], zero-initialised by the caller)."""
    _need(x, torch.bfloat16, "x")
    _need(running_absmax, torch.float32, "running_absmax", x.device)
    n, hkv, d = x.shape
    with torch.cuda.device(x.device):
        rc = N.lib.fp8pa_kv_channel_absmax_update(_ptr(x), n, hkv, d, _ptr(running_absmax),
                                                  _stream(stream))
    N.check(rc, "kv_channel_absmax_update")
    return running_absmax


def kv_scales_from_absmax(absmax, fmt=E5M2, out=None, stream=None):
    """Static scales max(absmax / FMAX, 1e-12) from a running absmax."""
    _need(absmax, torch.float32, "absmax")
    if out is None:
        out = torch.empty_like(absmax)
    _need(out, torch.float32, "out", absmax.device)
    with torch.cuda.device(absmax.device):
        rc = N.lib.fp8pa_kv_scales_from_absmax(_ptr(absmax), absmax.numel(), fmt, _ptr(out),
                                               _stream(stream))
    N.check(rc, "kv_scales_from_absmax")
    return out


def decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, head_dim_v, block_size,
                           max_blocks_per_seq, device=None, q_len=1) -> int:
    """Workspace bytes for the decode (q_len = 1) or a causal chunk of q_len
    queries per request (paged_multiquery_attention, decode_step)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        nbytes = int(N.lib.fp8pa_multiquery_workspace_bytes(batch, q_len, n_q_heads, n_kv_heads,
                                                            head_dim, head_dim_v, block_size,
                                                            max_blocks_per_seq))
    if nbytes == 0:
        raise Fp8paError(N.ERR_UNSUPPORTED, "decode_workspace_bytes")
    return nbytes


def paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                           n_kv_heads, sm_scale, fmt=E4M3, scale_mode=SCALE_TOKEN_HEAD,
                           group_size=64, head_dim_v=None, out=None, out_dtype=None,
                           workspace=None, stream=None):
    """q: bf16 [B, Hq, Dk]; caches/scales as written by kv_append_quant
    (v_cache/v_scale may be the same tensors as k_cache/k_scale for MLA);
    block_tables: int32 [B, max_blocks]; seq_lens: int32 [B].
    Returns out [B, Hq, Dv] (bf16 unless out_dtype=torch.float32)."""
    _need(q, torch.bfloat16, "q")
    dev = q.device
    for t, dt, name in ((k_cache, torch.uint8, "k_cache"), (v_cache, torch.uint8, "v_cache"),
                        (k_scale, _scale_dtype(scale_mode), "k_scale"),
                        (v_scale, _scale_dtype(scale_mode), "v_scale"),
                        (block_tables, torch.int32, "block_tables"),
                        (seq_lens, torch.int32, "seq_lens")):
        _need(t, dt, name, dev)
    B, hq, dk = q.shape
    dv = dk if head_dim_v is None else head_dim_v
    nb, _, bs, _ = k_cache.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty((B, hq, dv), dtype=out_dtype or torch.bfloat16, device=dev)
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or float32")
    _need(out, out.dtype, "out", dev)
    with _on(dev):
        if workspace is None:
            need = int(N.lib.fp8pa_decode_workspace_bytes(B, hq, n_kv_heads, dk, dv, bs,
                                                          max_blocks))
            if need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        # need == 0 means the shapes are rejected: the call below returns the
        # precise status code.
        _need(workspace, torch.uint8, "workspace", dev)
        rc = N.lib.fp8pa_paged_decode_attention(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), max_blocks, _ptr(seq_lens), B, bs, hq, n_kv_heads, dk, dv, fmt,
            scale_mode, group_size, float(sm_scale), nb, _ptr(out), odt, _ptr(workspace),
            0 if workspace is None else workspace.numel(), _stream(stream))
    N.check(rc, "paged_decode_attention")
    return out


def paged_multiquery_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                               n_kv_heads, sm_scale, fmt=E4M3, scale_mode=SCALE_TOKEN_HEAD,
                               group_size=64, head_dim_v=None, out=None, out_dtype=None,
                               workspace=None, stream=None):
    """A causal chunk of q_len queries per request: q bf16 [B, q_len, Hq, Dk],
    the chunk already appended to the cache, seq_lens counting it.  Query i
    sees the first seq_lens[b] - (q_len - 1 - i) tokens.
    Returns out [B, q_len, Hq, Dv]."""
    _need(q, torch.bfloat16, "q")
    dev = q.device
    for t, dt, name in ((k_cache, torch.uint8, "k_cache"), (v_cache, torch.uint8, "v_cache"),
                        (k_scale, _scale_dtype(scale_mode), "k_scale"),
                        (v_scale, _scale_dtype(scale_mode), "v_scale"),
                        (block_tables, torch.int32, "block_tables"),
                        (seq_lens, torch.int32, "seq_lens")):
        _need(t, dt, name, dev)
    B, qlen, hq, dk = q.shape
    dv = dk if head_dim_v is None else head_dim_v
    nb, _, bs, _ = k_cache.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty((B, qlen, hq, dv), dtype=out_dtype or torch.bfloat16, device=dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or float32")
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _need(out, out.dtype, "out", dev)
    with _on(dev):
        if workspace is None:
            need = int(N.lib.fp8pa_multiquery_workspace_bytes(B, qlen, hq, n_kv_heads, dk, dv,
                                                              bs, max_blocks))
            if need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _need(workspace, torch.uint8, "workspace", dev)
        rc = N.lib.fp8pa_paged_multiquery_attention(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), max_blocks, _ptr(seq_lens), B, qlen, bs, hq, n_kv_heads, dk, dv,
            fmt, scale_mode, group_size, float(sm_scale), nb, _ptr(out), odt, _ptr(workspace),
            0 if workspace is None else workspace.numel(), _stream(stream))
    N.check(rc, "paged_multiquery_attention")
    return out


def decode_step(k_new, v_new, slot_mapping, q, k_cache, v_cache, k_scale, v_scale,
                block_tables, seq_lens, n_kv_heads, sm_scale, fmt=E4M3,
                scale_mode=SCALE_TOKEN_HEAD, group_size=64, head_dim_v=None, out=None,
                out_dtype=None, workspace=None, stream=None):
    """Append the new rows (as kv_append_quant), then attend (as
    paged_decode_attention for q [B, Hq, Dk], or paged_multiquery_attention
    for q [B, q_len, Hq, Dk]) in one call.  For MLA pass v_new=None and
    v_cache/v_scale equal to k_cache/k_scale.  Returns out."""
    _need(q, torch.bfloat16, "q")
    dev = q.device
    _need(k_new, torch.bfloat16, "k_new", dev)
    _need(v_new, torch.bfloat16, "v_new", dev)
    for t, dt, name in ((k_cache, torch.uint8, "k_cache"), (v_cache, torch.uint8, "v_cache"),
                        (k_scale, _scale_dtype(scale_mode), "k_scale"),
                        (v_scale, _scale_dtype(scale_mode), "v_scale"),
                        (block_tables, torch.int32, "block_tables"),
                        (seq_lens, torch.int32, "seq_lens"),
                        (slot_mapping, torch.int32, "slot_mapping")):
        _need(t, dt, name, dev)
    multi = q.dim() == 4
    B, qlen, hq, dk = q.shape if multi else (q.shape[0], 1, q.shape[1], q.shape[2])
    dv = dk if head_dim_v is None else head_dim_v
    nb, _, bs, _ = k_cache.shape
    max_blocks = block_tables.shape[1]
    n_new = k_new.shape[0]
    if out is None:
        shape = (B, qlen, hq, dv) if multi else (B, hq, dv)
        out = torch.empty(shape, dtype=out_dtype or torch.bfloat16, device=dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or float32")
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _need(out, out.dtype, "out", dev)
    with _on(dev):
        if workspace is None:
            need = int(N.lib.fp8pa_multiquery_workspace_bytes(B, qlen, hq, n_kv_heads, dk, dv,
                                                              bs, max_blocks))
            if need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _need(workspace, torch.uint8, "workspace", dev)
        rc = N.lib.fp8pa_decode_step(
            _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n_new, _ptr(q), _ptr(k_cache),
            _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), max_blocks,
            _ptr(seq_lens), B, qlen, bs, hq, n_kv_heads, dk, dv, fmt, scale_mode, group_size,
            float(sm_scale), nb, _ptr(out), odt, _ptr(workspace),
            0 if workspace is None else workspace.numel(), _stream(stream))
    N.check(rc, "decode_step")
    return out


def get_device_error(stream=None, device=None) -> int:
    """Synchronise the stream, then read and clear the device error word."""
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        N.check(N.lib.fp8pa_get_device_error(_stream(stream), ctypes.byref(flags)),
                "get_device_error")
    return int(flags.value)
