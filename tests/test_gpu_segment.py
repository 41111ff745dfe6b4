"""GPU parity of the block-wise cumulative rescaling (the segment scale mode,
"DeepSeek V4 950: whole-network FP8 dataflow", 2kiu.com/news/4508674,
sec. 4.3): the append's codes, page scales and carried state are bit-exact
with the oracle however the tokens are split into calls (a prefill call and
then a decode step, random chunks mixing sequences, a call longer than the
kernel's 32-segment window); attention over the segment-scaled cache meets
the oracle's tolerance on the grouped-query and latent layouts, at every
kind of split, and for causal chunks."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4, E5, I8, SEG = W.E4M3, W.E5M2, W.INT8, W.SCALE_SEGMENT

# name, lengths, hq, hkv, d, bs, fmt
CASES = [
    ("seg_llama_heads", [2100, 1024, 1025, 7, 3000], 64, 8, 128, 16, E4),
    ("seg_g4_d64_bs32_e5m2", [1, 31, 1023, 1024, 2049], 8, 2, 64, 32, E5),
    ("seg_g3_hkv3_bs64_int8", [64, 65, 1100, 2048], 9, 3, 128, 64, I8),
    ("seg_g1_hkv5_d64_bs16", [500, 1500, 2500], 5, 5, 64, 16, E4),
    ("seg_mla_32_heads", [300, 1025, 2100], 32, 1, 576, 64, E4),
    ("seg_mla_64_heads_e5m2", [129, 1100, 64], 64, 1, 576, 64, E5),
]


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    yield F
    F.set_decode_workers(0)


def _case(case):
    name, lens, hq, hkv, d, bs, fmt = case
    return W.make_shape_case(name, lens, hq, hkv, d, bs, fmt, SEG, seed=5000 + CASES.index(case))


def _same(got, want, what):
    assert np.array_equal(got.cpu().numpy().view(np.uint8),
                          np.ascontiguousarray(want).view(np.uint8)), what


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_segment_append_and_decode_match_oracle(F, case):
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    w = _case(case)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)      # prefill call, then a one-token decode-step call
    o = oracle_cache(w, kvs)      # one call per request
    for got, want, what in zip(g, o, ("K codes", "V codes", "K page scales", "V page scales")):
        _same(got, want, what)
    q = W.queries(w)
    ref = oracle_attention(w, q, o)
    check_close(gpu_attention(w, F, q, g), ref, bf16_out=True, what=f"{w.name} bf16")
    outs = []
    try:
        for workers in (1, 2, 7, 64, 0):
            F.set_decode_workers(workers)
            got = gpu_attention(w, F, q, g, out_dtype=torch.float32)
            check_close(got, ref, bf16_out=False, what=f"{w.name} f32 workers={workers}")
            outs.append(got)
    finally:
        F.set_decode_workers(0)
    tol = 1e-4 * np.abs(outs[0]).max()
    for got in outs[1:]:
        assert np.abs(got - outs[0]).max() <= tol
    assert F.get_device_error() == 0


@pytest.mark.parametrize("case", [CASES[0], CASES[4]], ids=lambda c: c[0])
def test_segment_multiquery_matches_oracle(F, case):
    from gpu_util import check_close, gpu_cache, gpu_multiquery, oracle_cache, oracle_multiquery
    w = _case(case)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    qc = W.chunk_queries(w, 3)
    check_close(gpu_multiquery(w, F, qc, g, out_dtype=torch.float32),
                oracle_multiquery(w, qc, o, 3), bf16_out=False, what=f"{w.name} q_len=3")
    assert F.get_device_error() == 0


def test_segment_append_in_random_chunks(F):
    """The tokens of four sequences appended in random chunks, each call
    mixing sequences at different positions: codes, page scales and the
    carried (running absmax, segment scale) state equal the oracle's
    one-call result bit for bit."""
    from gpu_util import DEV, to_dev_bf16
    w = _case(CASES[0])
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    o = [np.zeros((w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim), np.uint8)
         for _ in range(2)]
    hp = oracle.segment_scale_heads(w.n_kv_heads)
    os_ = [np.zeros((w.num_blocks, hp), np.float32) for _ in range(2)]
    ost = np.zeros((w.batch, 2, w.n_kv_heads, 2), np.float32)
    lens = [int(L) for L in w.seq_lens]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    oracle.kv_append_quant_segment(np.concatenate([k for k, _ in kvs]),
                                   np.concatenate([v for _, v in kvs]),
                                   np.concatenate([W.token_slots(w, b, 0, L)
                                                   for b, L in enumerate(lens)]),
                                   off, [0] * w.batch, w.fmt, ost, o[0], o[1], os_[0], os_[1],
                                   w.block_size)
    kc = torch.zeros(o[0].shape, dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((w.num_blocks, hp), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    state = torch.zeros((w.batch, 2, w.n_kv_heads, 2), dtype=torch.float32, device=DEV)
    rng = np.random.default_rng(17)
    cuts = []
    for b, L in enumerate(lens):
        c = np.unique(np.concatenate([[0, L], rng.integers(1, max(L, 2), size=5)]))
        cuts.append([(int(a), int(e)) for a, e in zip(c[:-1], c[1:]) if e > a])
    while any(cuts):
        rows = [b for b in range(w.batch) if cuts[b]]
        parts = [(b, *cuts[b].pop(0)) for b in rows]
        sub = state[rows].contiguous()
        F.kv_append_quant_segment(
            to_dev_bf16(np.concatenate([kvs[b][0][a:e] for b, a, e in parts])),
            to_dev_bf16(np.concatenate([kvs[b][1][a:e] for b, a, e in parts])),
            torch.from_numpy(np.concatenate([W.token_slots(w, b, a, e) for b, a, e in parts])
                             ).to(DEV),
            torch.from_numpy(np.concatenate([[0], np.cumsum([e - a for _, a, e in parts])])
                             .astype(np.int32)).to(DEV),
            torch.from_numpy(np.array([a for _, a, _ in parts], np.int32)).to(DEV),
            kc, vc, ks, vs, sub, fmt=w.fmt)
        state[rows] = sub
    _same(kc, o[0], "K codes")
    _same(vc, o[1], "V codes")
    _same(ks, os_[0], "K page scales")
    _same(vs, os_[1], "V page scales")
    _same(state, ost, "carried state")
    assert F.get_device_error() == 0


def test_segment_append_longer_than_the_kernel_window(F):
    """One call of 40,000 tokens (39 segments: more than the 32-segment
    window the kernel holds in shared memory at a time)."""
    from gpu_util import gpu_cache, oracle_cache
    w = W.make_shape_case("seg_long_call", [40000, 900], 4, 1, 64, 16, E4, SEG, seed=5100)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs, step=False, back=0)
    o = oracle_cache(w, kvs)
    for got, want, what in zip(g, o, ("K codes", "V codes", "K page scales", "V page scales")):
        _same(got, want, what)
    assert F.get_device_error() == 0


def test_segment_mode_is_rejected_where_positions_are_missing(F):
    """The generic append and the one-call decode step have no token
    positions: the segment mode returns FP8PA_ERR_UNSUPPORTED there."""
    from gpu_util import DEV, to_dev_bf16
    w = _case(CASES[0])
    k = to_dev_bf16(W.request_kv(w, 0)[0][:4])
    kc = torch.zeros((w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim), dtype=torch.uint8,
                     device=DEV)
    ks = torch.zeros((w.num_blocks, F.segment_scale_heads(w.n_kv_heads)), dtype=torch.float32,
                     device=DEV)
    with pytest.raises(F.Fp8paError) as e:
        F.kv_append_quant(k, k, torch.arange(4, dtype=torch.int32, device=DEV), kc, kc, ks, ks,
                          scale_mode=SEG)
    assert e.value.code == -4
