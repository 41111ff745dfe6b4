"""GPU parity of the causal-chunk (multi-query) attention against the FP64
oracle: every (request, query) row is a decode row over its visible prefix,
seq_lens[b] - (q_len - 1 - i) tokens of the paged FP8 cache."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    return F


@pytest.mark.parametrize("idx,q_len", [(1, 3), (2, 4), (3, 2), (4, 3), (5, 2)])
def test_multiquery_matches_oracle(F, idx, q_len):
    from gpu_util import check_close, gpu_cache, gpu_multiquery, oracle_cache, oracle_multiquery
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    qc = W.chunk_queries(w, q_len)
    ref = oracle_multiquery(w, qc, o, q_len)
    short = bool((w.seq_lens < q_len).any())
    got = gpu_multiquery(w, F, qc, g)
    check_close(got, ref, bf16_out=True, what=f"cfg{idx} q_len={q_len} bf16")
    # a request shorter than the chunk is out of contract and flagged
    assert F.get_device_error() == (4 if short else 0)
    got32 = gpu_multiquery(w, F, qc, g, out_dtype=torch.float32)
    check_close(got32, ref, bf16_out=False, what=f"cfg{idx} q_len={q_len} f32")
    assert F.get_device_error() == (4 if short else 0)


@pytest.mark.parametrize("idx", [1, 5])
def test_multiquery_of_one_is_the_decode(F, idx):
    """q_len = 1 runs the same kernels as the decode call: identical bits."""
    from gpu_util import gpu_attention, gpu_cache, gpu_multiquery
    w = W.make_workload(idx, "small")
    g = gpu_cache(w, F)
    q = W.queries(w)
    a = gpu_attention(w, F, q, g, out_dtype=torch.float32)
    b = gpu_multiquery(w, F, q[:, None], g, out_dtype=torch.float32)[:, 0]
    assert np.array_equal(a, b)
    assert F.get_device_error() == 0


def test_chunk_longer_than_request_is_flagged(F):
    """Request 0 holds 3 tokens and the chunk is 5 long: its first two
    queries see nothing (zero rows) and the call raises the length flag."""
    from gpu_util import check_close, gpu_cache, gpu_multiquery, oracle_cache, oracle_multiquery
    w = W.make_workload(1, "small")
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[0] = 3
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    q_len = 5
    qc = W.chunk_queries(w, q_len)
    got = gpu_multiquery(w, F, qc, g, out_dtype=torch.float32)
    assert F.get_device_error() == 4
    ref = oracle_multiquery(w, qc, o, q_len)
    assert (got[0, :2] == 0).all()
    check_close(got, ref, bf16_out=False, what="short request")


def test_bad_q_len_is_rejected(F):
    from gpu_util import DEV
    w = W.make_workload(1, "small")
    kc = torch.zeros((w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim), dtype=torch.uint8,
                     device=DEV)
    ks = torch.zeros((w.num_blocks, w.n_kv_heads, w.block_size, 1), dtype=torch.float32,
                     device=DEV)
    q = torch.zeros((w.batch, 0, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(F.Fp8paError) as e:
        F.paged_multiquery_attention(q, kc, kc, ks, ks,
                                     torch.from_numpy(w.block_tables).to(DEV),
                                     torch.from_numpy(w.seq_lens).to(DEV), w.n_kv_heads,
                                     w.sm_scale, out_dtype=torch.float32,
                                     workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert e.value.code == -3
