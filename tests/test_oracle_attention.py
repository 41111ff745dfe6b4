"""Pins for the oracle's FP64 attention: closed forms (zero query gives the
mean of V, one token gives that token's V, weights sum to one), invariance
to physical block placement, agreement with torch's scaled-dot-product
attention (a library routine) on the dequantised cache, and the split-K
merge algebra."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

TORCH_T = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def build_cache(w):
    """Fill a cache for every token of every request through the oracle's
    append (static channel scales calibrated by the oracle when needed)."""
    nb, hkv, bs, d = w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim
    ng = d // w.group_size if w.scale_mode in (W.SCALE_TOKEN_GROUP, W.SCALE_MX_BLOCK) else 1
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = None if w.mla else np.zeros_like(kc)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    if w.scale_mode == W.SCALE_CHANNEL_STATIC:
        ks = oracle.kv_channel_scales(np.concatenate([k for k, _ in kvs]), w.fmt)
        vs = oracle.kv_channel_scales(np.concatenate([v for _, v in kvs]), w.fmt)
    else:
        sdt = np.uint8 if w.scale_mode == W.SCALE_MX_BLOCK else np.float32
        ks = np.zeros((nb, hkv, bs, ng), sdt)
        vs = None if w.mla else np.zeros_like(ks)
    for b, (k, v) in enumerate(kvs):
        slots = W.token_slots(w, b, 0, int(w.seq_lens[b]))
        assert oracle.kv_append_quant(k, v, slots, w.fmt, w.scale_mode, w.group_size, kc, vc,
                                      ks, vs, bs) == 0
    if w.mla:
        vc, vs = kc, ks
    return kc, vc, ks, vs


def dequant_request(w, cache, scale, b):
    """[L, Hkv, D] float64 through torch's float8 decode (INT8: the byte less
    128), not the oracle's."""
    L = int(w.seq_lens[b])
    t = np.arange(L)
    blk = w.block_tables[b, t // w.block_size]
    off = t % w.block_size
    codes = torch.from_numpy(cache[blk, :, off, :].copy())          # [L, Hkv, D]
    if w.fmt == oracle.INT8:
        vals = codes.to(torch.float64) - 128.0
    else:
        vals = codes.view(TORCH_T[w.fmt]).to(torch.float64)
    if w.scale_mode == W.SCALE_TOKEN_HEAD:
        s = torch.from_numpy(scale[blk, :, off, 0].astype(np.float64))[..., None]
    elif w.scale_mode == W.SCALE_TOKEN_GROUP:
        s = torch.from_numpy(scale[blk, :, off, :].astype(np.float64))
        s = s.repeat_interleave(w.group_size, dim=-1)
    elif w.scale_mode == W.SCALE_MX_BLOCK:   # E8M0 bytes: 2^(byte - 127)
        s = torch.from_numpy(np.exp2(scale[blk, :, off, :].astype(np.float64) - 127.0))
        s = s.repeat_interleave(w.group_size, dim=-1)
    else:
        s = torch.from_numpy(scale.astype(np.float64))[None]
    return vals * s


def run_oracle(w, q, kc, vc, ks, vs, **kw):
    return oracle.paged_decode_attention(q, kc, vc, ks, vs, w.block_tables, w.seq_lens,
                                         w.block_size, w.n_kv_heads, w.head_dim_v, w.fmt,
                                         w.scale_mode, w.group_size, w.sm_scale, **kw)


def sdpa_reference(w, q, kc, vc, ks, vs):
    qf = torch.from_numpy(W.bf16_bits_to_f32(q).astype(np.float64))
    out = np.zeros((w.batch, w.n_q_heads, w.head_dim_v))
    G = w.n_q_heads // w.n_kv_heads
    for b in range(w.batch):
        K = dequant_request(w, kc, ks, b)                            # [L, Hkv, D]
        V = dequant_request(w, vc, vs, b)[..., :w.head_dim_v]
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)           # [Hq, L, D]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qf[b][:, None, :], K, V, scale=w.sm_scale)
        out[b] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_matches_torch_sdpa(idx):
    w = W.make_workload(idx, "small")
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    got = run_oracle(w, q, kc, vc, ks, vs)
    ref = sdpa_reference(w, q, kc, vc, ks, vs)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-10), np.abs(got - ref).max()


def test_zero_query_gives_mean_of_v():
    w = W.make_workload(2, "small")
    kc, vc, ks, vs = build_cache(w)
    q = np.zeros((w.batch, w.n_q_heads, w.head_dim), np.uint16)
    got = run_oracle(w, q, kc, vc, ks, vs)
    G = w.n_q_heads // w.n_kv_heads
    for b in range(w.batch):
        V = dequant_request(w, vc, vs, b).numpy()                   # [L, Hkv, D]
        mean = V.mean(axis=0)
        for h in range(w.n_q_heads):
            assert np.allclose(got[b, h], mean[h // G], rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_v():
    w = W.make_workload(1, "small")
    w.seq_lens = np.ones_like(w.seq_lens)
    kc, vc, ks, vs = build_cache(w)
    got = run_oracle(w, W.queries(w), kc, vc, ks, vs)
    for b in range(w.batch):
        v0 = dequant_request(w, vc, vs, b).numpy()[0]
        assert np.array_equal(got[b], np.repeat(v0, w.n_q_heads // w.n_kv_heads, axis=0))


def test_weights_sum_to_one_and_follow_scores():
    w = W.make_workload(1, "small")
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    for b in range(w.batch):
        for h in range(w.n_q_heads):
            p = oracle.attention_weights(q, kc, ks, w.block_tables, w.seq_lens, w.block_size,
                                         w.n_kv_heads, w.fmt, w.scale_mode, w.group_size,
                                         w.sm_scale, b, h)
            assert p.size == w.seq_lens[b]
            assert abs(p.sum() - 1.0) < 1e-12 and (p > 0).all()
            K = dequant_request(w, kc, ks, b).numpy()[:, h // 4]
            z = K @ W.bf16_bits_to_f32(q[b, h]).astype(np.float64) * w.sm_scale
            assert np.argmax(p) == np.argmax(z)
            i, j = np.argsort(z)[-2:]
            assert math.isclose(p[j] / p[i], math.exp(z[j] - z[i]), rel_tol=1e-9)


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_paged_equals_contiguous_under_block_permutation(idx):
    w = W.make_workload(idx, "small")
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    base = run_oracle(w, q, kc, vc, ks, vs)
    rng = np.random.default_rng(99)
    perm = rng.permutation(w.num_blocks)        # new position of each physical block
    inv = np.argsort(perm)
    w2 = W.make_workload(idx, "small")
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    w2.block_tables = w2.block_tables.astype(np.int32)
    kc2 = kc[inv].copy()
    ks2 = ks[inv].copy() if ks.ndim == 4 else ks
    vc2 = kc2 if w.mla else vc[inv].copy()
    vs2 = ks2 if w.mla else (vs[inv].copy() if vs.ndim == 4 else vs)
    moved = run_oracle(w2, q, kc2, vc2, ks2, vs2)
    assert np.array_equal(base, moved)
    # two requests whose tables name the same physical blocks (a shared
    # prefix) see the same keys: their outputs agree for the same query.
    w3 = W.make_workload(idx, "small")
    w3.block_tables[1] = w3.block_tables[0]
    w3.seq_lens[1] = w3.seq_lens[0]
    q3 = q.copy()
    q3[1] = q3[0]
    o3 = run_oracle(w3, q3, kc, vc, ks, vs)
    assert np.array_equal(o3[0], o3[1])


@pytest.mark.parametrize("idx", [1, 3, 5])
def test_split_merge_equals_two_pass(idx):
    w = W.make_workload(idx, "small")
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    base = run_oracle(w, q, kc, vc, ks, vs)
    for chunk in (1, 7, 16, 100, 10 ** 6):
        sm = oracle.attention_split_merge(q, kc, vc, ks, vs, w.block_tables, w.seq_lens,
                                          w.block_size, w.n_kv_heads, w.head_dim_v, w.fmt,
                                          w.scale_mode, w.group_size, w.sm_scale, chunk)
        assert np.allclose(sm, base, rtol=1e-12, atol=1e-12)


def test_empty_sequence_and_sampled_rows():
    w = W.make_workload(2, "small")
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    full = run_oracle(w, q, kc, vc, ks, vs)
    rows = np.array([0, 70, 191], np.int32)
    part = run_oracle(w, q, kc, vc, ks, vs, rows=rows, num_threads=2)
    assert np.array_equal(part, full.reshape(-1, w.head_dim_v)[rows])
    w.seq_lens[2] = 0
    z = run_oracle(w, q, kc, vc, ks, vs)
    assert (z[2] == 0).all() and np.array_equal(z[:2], full[:2])


def test_gqa_group_of_one_is_plain_mha():
    # G = 1: every query head reads its own KV head.
    w = W.make_workload(2, "small")
    w.n_q_heads = w.n_kv_heads
    kc, vc, ks, vs = build_cache(w)
    q = W.queries(w)
    got = run_oracle(w, q, kc, vc, ks, vs)
    assert np.allclose(got, sdpa_reference(w, q, kc, vc, ks, vs), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("idx,q_len", [(2, 3), (4, 4), (5, 2)])
def test_multiquery_rows_are_a_causal_chunk(idx, q_len):
    """A chunk of q_len queries over a cache that already holds the chunk:
    running every (request, query) as a decode row over its visible prefix
    equals causal attention of the chunk (torch SDPA with a boolean mask) --
    the reading under which the multi-query call is checked."""
    w = W.make_workload(idx, "small")
    kc, vc, ks, vs = build_cache(w)
    qc = W.chunk_queries(w, q_len)                                   # [B, q_len, Hq, D]
    # decode rows: request b's table repeated, query i sees L - (q_len - 1 - i)
    tables = np.repeat(w.block_tables, q_len, axis=0)
    lens = np.array([max(0, int(L) - (q_len - 1 - i)) for L in w.seq_lens for i in range(q_len)],
                    np.int32)
    got = oracle.paged_decode_attention(
        qc.reshape(-1, w.n_q_heads, w.head_dim), kc, vc, ks, vs, tables, lens, w.block_size,
        w.n_kv_heads, w.head_dim_v, w.fmt, w.scale_mode, w.group_size, w.sm_scale)
    got = got.reshape(w.batch, q_len, w.n_q_heads, w.head_dim_v)
    G = w.n_q_heads // w.n_kv_heads
    # a row that sees no token is zero (a request shorter than the chunk)
    assert (got.reshape(-1, w.n_q_heads, w.head_dim_v)[lens == 0] == 0).all()
    checked = 0
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        if L < q_len:
            continue
        checked += 1
        K = dequant_request(w, kc, ks, b).permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = dequant_request(w, vc, vs, b)[..., :w.head_dim_v]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qf = torch.from_numpy(W.bf16_bits_to_f32(qc[b]).astype(np.float64)).permute(1, 0, 2)
        t = torch.arange(L)[None, :]
        pos = torch.arange(L - q_len, L)[:, None]          # the chunk's own positions
        mask = t <= pos                                     # [q_len, L]
        o = torch.nn.functional.scaled_dot_product_attention(qf, K, V, attn_mask=mask,
                                                             scale=w.sm_scale)
        ref = o.permute(1, 0, 2).numpy()
        assert np.allclose(got[b], ref, rtol=1e-10, atol=1e-10), np.abs(got[b] - ref).max()
    assert checked >= w.batch - 1


@pytest.mark.parametrize("fmt,gs", [(W.E4M3, 32), (W.E5M2, 16)])
def test_mx_block_attention_matches_torch_sdpa(fmt, gs):
    """Block-scaled (MX) cache: attention over the dequantised cache,
    decode(code) * 2^(byte - 127), against float64 SDPA."""
    w = W.make_shape_case("mx", [1, 15, 16, 17, 53], 16, 4, 128, 16, fmt, W.SCALE_MX_BLOCK,
                          seed=31, group_size=gs)
    kc, vc, ks, vs = build_cache(w)
    assert ks.dtype == np.uint8 and ks.shape[-1] == 128 // gs
    q = W.queries(w)
    got = run_oracle(w, q, kc, vc, ks, vs)
    ref = sdpa_reference(w, q, kc, vc, ks, vs)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-10), np.abs(got - ref).max()


@pytest.mark.parametrize("mode,hq,hkv,d,bs", [(W.SCALE_TOKEN_HEAD, 16, 4, 128, 16),
                                             (W.SCALE_CHANNEL_STATIC, 8, 2, 64, 32),
                                             (W.SCALE_TOKEN_GROUP, 32, 1, 576, 64)])
def test_int8_attention_matches_torch_sdpa(mode, hq, hkv, d, bs):
    """INT8 caches (token-head, static channel and per-latent-group scales):
    attention over the dequantised cache, integer code * scale, against
    float64 SDPA."""
    w = W.make_shape_case("int8", [1, bs - 1, bs, bs + 1, 3 * bs + 5], hq, hkv, d, bs, W.INT8,
                          mode, seed=41)
    kc, vc, ks, vs = build_cache(w)
    for b in range(w.batch):  # written codes are bytes 1 .. 255 (integers -127 .. 127)
        t = np.arange(int(w.seq_lens[b]))
        assert kc[w.block_tables[b, t // bs], :, t % bs, :].min() >= 1
    q = W.queries(w)
    got = run_oracle(w, q, kc, vc, ks, vs)
    ref = sdpa_reference(w, q, kc, vc, ks, vs)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-10), np.abs(got - ref).max()
