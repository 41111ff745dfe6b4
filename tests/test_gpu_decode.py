"""GPU parity of paged decode attention against the FP64 oracle computed
from the same codes and scales: every output at oracle-sized shapes, sampled
rows at the full workload sizes, split-count independence and edge cases."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    yield F
    F.set_decode_workers(0)


ALL = [1, 2, 3, 4, 5]


@pytest.mark.parametrize("idx", ALL)
def test_decode_small_matches_oracle(F, idx):
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    assert np.array_equal(g[0].cpu().numpy(), o[0])  # same codes on both sides
    q = W.queries(w)
    ref = oracle_attention(w, q, o)
    got = gpu_attention(w, F, q, g)
    check_close(got, ref, bf16_out=True, what=f"cfg{idx} bf16")
    got32 = gpu_attention(w, F, q, g, out_dtype=torch.float32)
    check_close(got32, ref, bf16_out=False, what=f"cfg{idx} f32")
    assert F.get_device_error() == 0


@pytest.mark.parametrize("idx", [1, 3, 4, 5])
def test_decode_independent_of_split_count(F, idx):
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    q = W.queries(w)
    ref = oracle_attention(w, q, oracle_cache(w, kvs))
    outs = []
    try:
        for workers in (1, 2, 7, 64, 1000, 0):
            F.set_decode_workers(workers)
            o = gpu_attention(w, F, q, g, out_dtype=torch.float32)
            check_close(o, ref, bf16_out=False, what=f"workers={workers}")
            outs.append(o)
    finally:
        F.set_decode_workers(0)
    # Splits may differ by fp32 rounding and, on the latent tensor-core path,
    # by the rounding of P's and V^'s 16-bit hi + lo parts: bounded against
    # the output's scale.
    tol = 1e-4 * np.abs(outs[0]).max()
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= tol


def test_decode_edges(F):
    """seq_len 0 gives zeros; a bad block id is masked and flagged; a length
    past the block table is clamped and flagged; nothing traps."""
    from gpu_util import DEV, gpu_cache, oracle_attention, oracle_cache, check_close, to_dev_bf16
    w = W.make_workload(2, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    q = W.queries(w)
    kc, vc, ks, vs = g

    def run(bt, sl):
        return F.paged_decode_attention(to_dev_bf16(q), kc, vc, ks, vs,
                                        torch.from_numpy(bt).to(DEV), torch.from_numpy(sl).to(DEV),
                                        w.n_kv_heads, w.sm_scale, out_dtype=torch.float32)

    sl = w.seq_lens.copy()
    sl[1] = 0
    out = run(w.block_tables, sl).cpu().numpy()
    assert (out[1] == 0).all()
    assert F.get_device_error() == 0
    w2 = W.make_workload(2, "small")
    w2.seq_lens = sl
    check_close(out[[0, 2]], oracle_attention(w2, q, o)[[0, 2]], bf16_out=False)

    bt = w.block_tables.copy()
    bt[0, 3] = w.num_blocks + 5      # out of the pool: that page is masked
    out = run(bt, w.seq_lens).cpu().numpy()
    assert F.get_device_error() == 2  # FP8PA_DEVERR_BLOCK_RANGE
    assert np.isfinite(out).all()
    check_close(out[1:], oracle_attention(w, q, o)[1:], bf16_out=False)

    sl = w.seq_lens.copy()
    sl[2] = w.block_tables.shape[1] * w.block_size + 100
    out = run(w.block_tables, sl).cpu().numpy()
    assert F.get_device_error() & 4   # FP8PA_DEVERR_SEQ_LEN
    assert np.isfinite(out).all()


def test_decode_bad_arguments_return_codes(F):
    from gpu_util import DEV, to_dev_bf16
    w = W.make_workload(1, "small")
    q = to_dev_bf16(W.queries(w))
    kc = torch.zeros((w.num_blocks, 1, 16, 64), dtype=torch.uint8, device=DEV)
    ks = torch.zeros((w.num_blocks, 1, 16, 1), dtype=torch.float32, device=DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    with pytest.raises(F.Fp8paError) as e:
        F.paged_decode_attention(q, kc, kc, ks, ks, bt, sl, 3, 0.125)  # 4 % 3 != 0
    assert e.value.code == -3
    with pytest.raises(F.Fp8paError) as e:
        F.paged_decode_attention(q, kc, kc, ks, ks, bt, sl, 1, 0.125, fmt=9)
    assert e.value.code == -2
    small_ws = torch.zeros(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(F.Fp8paError) as e:
        F.paged_decode_attention(q, kc, kc, ks, ks, bt, sl, 1, 0.125, workspace=small_ws)
    assert e.value.code == -5
    assert F.get_device_error() == 0


def _full_size_sampled(F, w, sample, q_len=1):
    """Full-size workload `w` through the GPU path in the bench's launch
    configuration: every request's first L - q_len tokens are appended, then
    one fp8pa_decode_step call appends the last q_len tokens of each request
    and attends (a causal chunk when q_len > 1).  The oracle rebuilds only the
    sampled requests in a compact pool and checks their codes, scales and
    outputs (bf16, as the bench writes them)."""
    from gpu_util import DEV, check_close, n_scale_groups, oracle_multiquery, scale_dtype, \
        to_dev_bf16
    nb, hkv, bs, d = w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device=DEV)
    vc = None if w.mla else torch.zeros_like(kc)
    kv_sample = {}
    if w.scale_mode == W.SCALE_CHANNEL_STATIC:
        allk = [W.request_kv(w, b) for b in range(w.batch)]
        ks = F.kv_channel_scales(to_dev_bf16(np.concatenate([k for k, _ in allk])), w.fmt)
        vs = F.kv_channel_scales(to_dev_bf16(np.concatenate([v for _, v in allk])), w.fmt)
        oks = oracle.kv_channel_scales(np.concatenate([k for k, _ in allk]), w.fmt)
        ovs = oracle.kv_channel_scales(np.concatenate([v for _, v in allk]), w.fmt)
        assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
        assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))
        get = lambda b: allk[b]
    else:
        ks = torch.zeros((nb, hkv, bs, n_scale_groups(w)), dtype=scale_dtype(w), device=DEV)
        vs = None if w.mla else torch.zeros_like(ks)
        get = lambda b: W.request_kv(w, b)
    last_k, last_v, last_slots = [], [], []
    for b in range(w.batch):
        k, v = get(b)
        L = int(w.seq_lens[b])
        n = max(L - q_len, 0)
        if b in sample:
            kv_sample[b] = (k, v)
        if n > 0:
            F.kv_append_quant(to_dev_bf16(k[:n]), None if v is None else to_dev_bf16(v[:n]),
                              torch.from_numpy(W.token_slots(w, b, 0, n)).to(DEV), kc, vc, ks,
                              vs, fmt=w.fmt, scale_mode=w.scale_mode, group_size=w.group_size)
        last_k.append(k[n:L])
        if v is not None:
            last_v.append(v[n:L])
        last_slots.append(W.token_slots(w, b, n, L))
    q = W.queries(w) if q_len == 1 else W.chunk_queries(w, q_len)
    vc_, vs_ = (kc, ks) if w.mla else (vc, vs)
    out = F.decode_step(to_dev_bf16(np.concatenate(last_k)),
                        None if w.mla else to_dev_bf16(np.concatenate(last_v)),
                        torch.from_numpy(np.concatenate(last_slots).astype(np.int32)).to(DEV),
                        to_dev_bf16(q), kc, vc_, ks, vs_, torch.from_numpy(w.block_tables).to(DEV),
                        torch.from_numpy(w.seq_lens).to(DEV), hkv, w.sm_scale, fmt=w.fmt,
                        scale_mode=w.scale_mode, group_size=w.group_size,
                        head_dim_v=w.head_dim_v)
    got = out.float().cpu().numpy().astype(np.float64)
    assert F.get_device_error() == 0
    # Compact oracle pool holding only the sampled requests' blocks.
    for b in sample:
        k, v = kv_sample[b]
        L = int(w.seq_lens[b])
        nbl = (L + bs - 1) // bs
        blocks = torch.from_numpy(w.block_tables[b, :nbl].astype(np.int64)).to(DEV)
        cw = W.make_workload(w.index, "full")
        cw.fmt, cw.scale_mode, cw.group_size = w.fmt, w.scale_mode, w.group_size
        cw.batch = 1
        cw.seq_lens = np.array([L], np.int32)
        cw.block_tables = np.arange(nbl, dtype=np.int32)[None]
        cw.num_blocks = nbl
        okc = np.zeros((nbl, hkv, bs, d), np.uint8)
        ovc = None if w.mla else np.zeros_like(okc)
        if w.scale_mode == W.SCALE_CHANNEL_STATIC:
            oks2, ovs2 = oks, ovs
        else:
            oks2 = np.zeros((nbl, hkv, bs, ks.shape[-1]), scale_dtype(w, torch_side=False))
            ovs2 = None if w.mla else np.zeros_like(oks2)
        slots = W.token_slots(cw, 0, 0, L)
        assert oracle.kv_append_quant(k, v, slots, w.fmt, w.scale_mode, w.group_size, okc, ovc,
                                      oks2, ovs2, bs) == 0
        assert np.array_equal(kc[blocks].cpu().numpy(), okc), f"request {b}: K codes differ"
        if not w.mla:
            assert np.array_equal(vc[blocks].cpu().numpy(), ovc), f"request {b}: V codes differ"
        if w.scale_mode != W.SCALE_CHANNEL_STATIC:
            assert np.array_equal(ks[blocks].cpu().numpy().view(np.uint8),
                                  oks2.view(np.uint8)), f"request {b}: K scales differ"
            if not w.mla:
                assert np.array_equal(vs[blocks].cpu().numpy().view(np.uint8),
                                      ovs2.view(np.uint8)), f"request {b}: V scales differ"
        if w.mla:
            ovc, ovs2 = okc, oks2
        if q_len == 1:
            ref = oracle.paged_decode_attention(q[b:b + 1], okc, ovc, oks2, ovs2,
                                                cw.block_tables, cw.seq_lens, bs, hkv,
                                                w.head_dim_v, w.fmt, w.scale_mode, w.group_size,
                                                w.sm_scale)
        else:
            ref = oracle_multiquery(cw, q[b:b + 1], (okc, ovc, oks2, ovs2), q_len)
        check_close(got[b:b + 1], ref, bf16_out=True, what=f"{w.name} request {b}")


@pytest.mark.slow
def test_full_llama70b_layer_sampled(F):
    _full_size_sampled(F, W.make_workload(2, "full"), sample=(0, 7, 11))


@pytest.mark.slow
def test_full_long_context_sampled(F):
    _full_size_sampled(F, W.make_workload(3, "full"), sample=(2,))


@pytest.mark.slow
def test_full_ragged_e5m2_sampled(F):
    w = W.make_workload(4, "full")
    order = np.argsort(w.seq_lens)
    _full_size_sampled(F, w, sample=(int(order[0]), int(order[len(order) // 2]),
                                     int(order[-1])))


@pytest.mark.slow
def test_full_mla_latent_sampled(F):
    _full_size_sampled(F, W.make_workload(5, "full"), sample=(0, 31))


def _llama_variant(fmt=None, mode=None, gs=None, tag=""):
    w = W.make_workload(2, "full")
    if fmt is not None:
        w.fmt = fmt
    if mode is not None:
        w.scale_mode, w.group_size = mode, gs
    w.name += tag
    return w


@pytest.mark.slow
def test_full_llama70b_layer_mx32_sampled(F):
    """The bench's --mx-block 32 launch, checked on sampled requests."""
    _full_size_sampled(F, _llama_variant(W.E4M3, W.SCALE_MX_BLOCK, 32, "_mx32"), sample=(0, 11))


@pytest.mark.slow
def test_full_llama70b_layer_int8_sampled(F):
    """The bench's --kv-fmt int8 launch, checked on sampled requests."""
    _full_size_sampled(F, _llama_variant(W.INT8, tag="_int8"), sample=(3, 11))


@pytest.mark.slow
def test_full_llama70b_layer_chunk4_sampled(F):
    """The bench's --q-len 4 launch (a causal chunk of 4 queries per request:
    the tensor-core kernel with all 4 queries x 8 heads on the MMA columns),
    checked on sampled requests."""
    _full_size_sampled(F, _llama_variant(tag="_chunk4"), sample=(0, 5), q_len=4)


@pytest.mark.slow
def test_full_llama70b_layer_chunk8_sampled(F):
    """The bench's --q-len 8 launch (each chunk planned as two requests of 4
    queries on the tensor-core kernel), checked on sampled requests."""
    _full_size_sampled(F, _llama_variant(tag="_chunk8"), sample=(2, 11), q_len=8)


def test_bounded_wait_gives_up_and_reports(F):
    """Failure detection without a fault: a warp waiting on a barrier that
    nothing completes gives up after its cycle limit (here ~1 ms), records
    the timeout bit and returns; the context stays usable."""
    import time
    from fp8_quantised_paged_gb300 import _native as N
    F.get_device_error()
    t0 = time.perf_counter()
    N.check(N.lib.fp8pa_selftest_bounded_wait(2_000_000, None), "selftest")
    assert F.get_device_error() == N.DEVERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the device still runs work afterwards
    x = torch.ones(4, device="cuda:0")
    assert float((x * 2).sum()) == 8.0
