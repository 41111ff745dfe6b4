"""The decode entry point for callers that cannot allocate device memory
(fp8pa_paged_decode_attention_static_ws) against the FP64 oracle and the
regular entry point.

Such callers -- a plugin given only its input and output buffers, or a
server that forbids allocation after start-up -- cannot provide the
workspace the regular decode needs, so this variant takes its scratch from
a static array inside the library.  The test calls both through the C ABI
and checks the variant twice in a row (the array keeps the previous call's
contents, which must not matter), plus the size limit.  This file is named
to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_ws_call(N, w, q, caches, bt, sl, out, out_dtype):
    kc, vc, ks, vs = caches
    return N.lib.fp8pa_paged_decode_attention_static_ws(
        _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt), w.max_blocks, _p(sl), w.batch,
        w.block_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.head_dim_v, w.fmt, w.scale_mode,
        w.group_size, ctypes.c_float(w.sm_scale), w.num_blocks, _p(out), out_dtype,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _regular_call(N, w, q, caches, bt, sl, out, out_dtype, ws):
    kc, vc, ks, vs = caches
    return N.lib.fp8pa_paged_decode_attention(
        _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt), w.max_blocks, _p(sl), w.batch,
        w.block_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.head_dim_v, w.fmt, w.scale_mode,
        w.group_size, ctypes.c_float(w.sm_scale), w.num_blocks, _p(out), out_dtype, _p(ws),
        ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_static_workspace_matches_oracle_and_regular_entry_point(idx):
    """Llama-shaped layer, ragged E5M2 with static channel scales, and the MLA
    latent (small sizes): the static-workspace call is checked against the
    FP64 oracle directly, and is bit-identical to the regular entry point
    (same kernels, same split), on two calls in a row."""
    import fp8_quantised_paged_gb300 as F
    from fp8_quantised_paged_gb300 import _native as N
    from gpu_util import DEV, check_close, gpu_cache, oracle_attention, oracle_cache, to_dev_bf16

    torch.cuda.set_device(0)
    F.set_decode_workers(0)
    F.get_device_error()
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    caches = gpu_cache(w, F, kvs)
    q_bits = W.queries(w)
    want = oracle_attention(w, q_bits, oracle_cache(w, kvs))
    q = to_dev_bf16(q_bits)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    need = N.lib.fp8pa_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                              w.head_dim_v, w.block_size, w.max_blocks)
    if need > 32 << 20:
        pytest.skip(f"this device's split needs {need} bytes, more than the static array")
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    shape = (w.batch, w.n_q_heads, w.head_dim_v)
    for out_dtype, tdt in ((N.OUT_F32, torch.float32), (N.OUT_BF16, torch.bfloat16)):
        bf16 = tdt == torch.bfloat16
        ref = torch.empty(shape, dtype=tdt, device=DEV)
        assert _regular_call(N, w, q, caches, bt, sl, ref, out_dtype, ws) == 0
        ref_np = ref.float().cpu().numpy().astype(np.float64)
        for call in range(2):  # two calls in a row share the static array
            out = torch.full(shape, float("nan"), dtype=tdt, device=DEV)
            assert _static_ws_call(N, w, q, caches, bt, sl, out, out_dtype) == 0
            torch.cuda.synchronize()
            got = out.float().cpu().numpy().astype(np.float64)
            check_close(got, want, bf16_out=bf16, what=f"static workspace cfg{idx} call {call}")
            assert np.array_equal(got, ref_np), "differs from the regular entry point"
    assert F.get_device_error() == 0


def test_static_workspace_rejects_shapes_beyond_its_size():
    import fp8_quantised_paged_gb300 as F
    from fp8_quantised_paged_gb300 import _native as N
    from gpu_util import DEV, gpu_cache, to_dev_bf16

    torch.cuda.set_device(0)
    w = W.make_workload(2, "small")
    caches = gpu_cache(w, F)
    q = to_dev_bf16(W.queries(w))
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.zeros((w.batch, w.n_q_heads, w.head_dim_v), dtype=torch.float32, device=DEV)
    try:
        F.set_decode_workers(1 << 20)  # a split so fine its partials need > 32 MiB
        assert _static_ws_call(N, w, q, caches, bt, sl, out, N.OUT_F32) == N.ERR_WORKSPACE
    finally:
        F.set_decode_workers(0)
    torch.cuda.synchronize()
    assert (out == 0).all()  # nothing was launched
