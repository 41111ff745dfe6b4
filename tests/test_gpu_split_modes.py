"""GPU parity of the MX block-scaled, INT8 and multi-query paths at every kind
of page range the planner can cut: one range over the whole batch (a warp's
ring is reused across many pages and the range crosses every request
boundary), two ranges, ranges of a handful of pages, ranges of about one page,
and the device's own split.  Each run is compared with the FP64 oracle (f32
output, the unmodified 4e-3 / 2e-3 bounds), with codes and scales bit-exact,
and the runs must agree with each other to fp32 rounding.

The cases follow the pages' workloads: the Llama-3-70B-shaped layer (64 query
/ 8 KV heads) with its cache in MX blocks of 32 and 16 ("FP8混合精度推理全链路
部署实战", ybb.press, sec. 7.1) and in INT8 codes (an INT8 KV cache is named as
a serving option on the third page, inference-engine settings); the ragged
E5M2 workload with static channel scales in INT8; the MLA latent in INT8; and
causal chunks of 2 to 4 queries ("Llama 3 70B FP8 deployment", dpshk.com,
sec. 3.3 chunked prefill and sec. 4.3 speculative verify) on the grouped-query
layout, where the chunk's query warps walk the same pages, and on the latent
layout."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WORKERS = (1, 2, 7, 64, 0)

# name: (base workload, fmt or None, scale mode or None, group size or None, q_len)
VARIANTS = {
    "mx32_e4m3": (2, W.E4M3, W.SCALE_MX_BLOCK, 32, 1),
    "mx16_e5m2": (2, W.E5M2, W.SCALE_MX_BLOCK, 16, 1),
    "int8_token_head": (2, W.INT8, None, None, 1),
    "int8_static_channel": (4, W.INT8, None, None, 1),
    "int8_mla_latent": (5, W.INT8, None, None, 1),
    "chunk2_gqa": (2, None, None, None, 2),
    "chunk4_gqa": (2, None, None, None, 4),
    "chunk3_static_packed": (4, None, None, None, 3),
    "chunk4_mx32": (2, W.E4M3, W.SCALE_MX_BLOCK, 32, 4),
    "chunk3_int8": (2, W.INT8, None, None, 3),
    "chunk2_mla": (5, None, None, None, 2),
    "chunk4_mla_int8": (5, W.INT8, None, None, 4),
}


def make_variant(name, size="small"):
    idx, fmt, mode, gs, q_len = VARIANTS[name]
    w = W.make_workload(idx, size)
    if fmt is not None:
        w.fmt = fmt
    if mode is not None:
        w.scale_mode, w.group_size = mode, gs
    w.name = f"{w.name}_{name}"
    return w, q_len


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    yield F
    F.set_decode_workers(0)


@pytest.mark.parametrize("name", list(VARIANTS))
def test_variant_at_every_split(F, name):
    from gpu_util import (check_close, gpu_attention, gpu_cache, gpu_multiquery, oracle_attention,
                          oracle_cache, oracle_multiquery)
    w, q_len = make_variant(name)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    for got, want, what in zip(g, o, ("K codes", "V codes", "K scales", "V scales")):
        if want is not None:
            a = got.cpu().numpy()
            assert np.array_equal(a.view(np.uint8), np.ascontiguousarray(want).view(np.uint8)), what
    if q_len == 1:
        q = W.queries(w)
        ref = oracle_attention(w, q, o)
        run = lambda: gpu_attention(w, F, q, g, out_dtype=torch.float32)
    else:
        q = W.chunk_queries(w, q_len)
        ref = oracle_multiquery(w, q, o, q_len)
        run = lambda: gpu_multiquery(w, F, q, g, out_dtype=torch.float32)
    flag = 4 if bool((w.seq_lens < q_len).any()) else 0  # a request shorter than the chunk
    outs = []
    try:
        for workers in WORKERS:
            F.set_decode_workers(workers)
            got = run()
            assert F.get_device_error() == flag, f"workers={workers}"
            check_close(got, ref, bf16_out=False, what=f"{name} workers={workers}")
            outs.append(got)
    finally:
        F.set_decode_workers(0)
    # Splits may differ by fp32 rounding (and, on the latent tensor-core
    # path, by the rounding of 16-bit hi + lo operand parts), whose size
    # follows the magnitude of the values summed (up to x50 outliers here),
    # not of each output element.
    tol = 1e-4 * np.abs(outs[0]).max()
    for workers, got in zip(WORKERS[1:], outs[1:]):
        diff = np.abs(got - outs[0]).max()
        assert diff <= tol, f"workers={workers}: max difference {diff:.3g} > {tol:.3g}"
