"""FP8-quantised paged decode attention for GB300 (sm_103a).

Two calls, both hand-written CUDA kernels behind a C ABI (``include/fp8pa.h``):

* ``kv_append_quant`` -- absmax-scale each new token's K/V rows, round them
  to E4M3 or E5M2 (or symmetric INT8 codes) and scatter codes and scales
  into the paged cache.
* ``paged_decode_attention`` -- grouped-query (or shared-latent MLA)
  attention of one query token per request over its paged FP8 cache, split
  across the GPU and merged.

The torch-facing wrappers live in :mod:`.binding` and are re-exported here
on first use, so that importing the input generators (:mod:`.workloads`)
does not need the native library.  Using any wrapper loads ``libfp8pa.so``
and raises if it is missing: there is no fallback path.
"""
_API = ("kv_append_quant", "kv_append_quant_segment", "segment_scale_heads",
        "kv_channel_scales", "kv_channel_absmax_update",
        "kv_scales_from_absmax", "paged_decode_attention", "paged_multiquery_attention",
        "decode_step",
        "decode_workspace_bytes", "get_device_error", "set_decode_workers", "version",
        "E4M3", "E5M2", "INT8", "SCALE_TOKEN_HEAD", "SCALE_CHANNEL_STATIC", "SCALE_TOKEN_GROUP",
        "SCALE_MX_BLOCK", "SCALE_SEGMENT", "SEGMENT_TOKENS",
        "OUT_BF16", "OUT_F32", "Fp8paError")

__all__ = list(_API)


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
