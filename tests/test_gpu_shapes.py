"""GPU parity over the supported shape space beyond the five named
workloads: block sizes 16/32/64, head_dim 64/128, GQA group sizes 1, 2, 3, 4
and 8, KV-head counts that are not a power of two or need several head sets
per CTA, both formats with both GQA scale modes, KV-head counts up to 24,
and the latent layout with 32 and 64 query heads.  Static scales with 1, 2
or 4 query heads per KV head run the packed kernel (q's high and low parts
in one MMA), at head_dim 64 and 128.  INT8 codes run through the same
layouts (token-head, static, latent).  Every output is compared with the FP64 oracle;
lengths include 1, block_size - 1, block_size, block_size + 1 and several
pages with a ragged tail."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4, E5, I8 = W.E4M3, W.E5M2, W.INT8
TH, CS, TG, MX = W.SCALE_TOKEN_HEAD, W.SCALE_CHANNEL_STATIC, W.SCALE_TOKEN_GROUP, W.SCALE_MX_BLOCK

# name, hq, hkv, d, bs, fmt, mode
CASES = [
    ("mha_g1_bs64_e4m3", 8, 8, 128, 64, E4, TH),
    ("g2_hkv16_e5m2_token", 32, 16, 128, 16, E5, TH),
    ("g3_hkv3_d64_bs32_static", 9, 3, 64, 32, E4, CS),
    ("g8_d64_bs64_e5m2_static", 64, 8, 64, 64, E5, CS),
    ("g2_hkv24_bs32_e4m3_static", 48, 24, 128, 32, E4, CS),
    ("g4_hkv2_d128_bs16_e5m2_token", 8, 2, 128, 16, E5, TH),
    ("g2_hkv10_d64_bs16_e4m3_token", 20, 10, 64, 16, E4, TH),
    ("g1_hkv13_d128_bs64_e5m2_static", 13, 13, 128, 64, E5, CS),
    ("mla_32_heads_e4m3", 32, 1, 576, 64, E4, TG),
    ("mla_64_heads_e5m2", 64, 1, 576, 64, E5, TG),
    ("g4_hkv2_d64_bs16_e4m3_static", 8, 2, 64, 16, E4, CS),
    ("g1_hkv4_d64_bs64_e5m2_static", 4, 4, 64, 64, E5, CS),
    ("int8_g8_d128_bs16_token", 64, 8, 128, 16, I8, TH),
    ("int8_g4_hkv2_d64_bs32_static", 8, 2, 64, 32, I8, CS),
    ("int8_g3_hkv3_d128_bs64_static", 9, 3, 128, 64, I8, CS),
    ("int8_g2_hkv4_d64_bs16_token", 8, 4, 64, 16, I8, TH),
    ("int8_mla_32_heads", 32, 1, 576, 64, I8, TG),
    ("mla_192_heads_e4m3", 192, 1, 576, 64, E4, TG),
]


def _lens(bs):
    return [1, bs - 1, bs, bs + 1, 3 * bs + 5]


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    return F


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_shape_matches_oracle(F, case):
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    name, hq, hkv, d, bs, fmt, mode = case
    w = W.make_shape_case(name, _lens(bs), hq, hkv, d, bs, fmt, mode,
                          seed=2000 + CASES.index(case))
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    assert np.array_equal(g[0].cpu().numpy(), o[0]), "K codes"
    if not w.mla:
        assert np.array_equal(g[1].cpu().numpy(), o[1]), "V codes"
    q = W.queries(w)
    ref = oracle_attention(w, q, o)
    check_close(gpu_attention(w, F, q, g), ref, bf16_out=True, what=f"{name} bf16")
    check_close(gpu_attention(w, F, q, g, out_dtype=torch.float32), ref, bf16_out=False,
                what=f"{name} f32")
    assert F.get_device_error() == 0


@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[8], CASES[10], CASES[12], CASES[16]],
                         ids=lambda c: c[0])
def test_shape_multiquery_matches_oracle(F, case):
    from gpu_util import check_close, gpu_cache, gpu_multiquery, oracle_cache, oracle_multiquery
    name, hq, hkv, d, bs, fmt, mode = case
    lens = [L for L in _lens(bs) if L >= 3]
    w = W.make_shape_case(name, lens, hq, hkv, d, bs, fmt, mode,
                          seed=2000 + CASES.index(case))
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    qc = W.chunk_queries(w, 3)
    check_close(gpu_multiquery(w, F, qc, g, out_dtype=torch.float32),
                oracle_multiquery(w, qc, o, 3), bf16_out=False, what=f"{name} q_len=3")
    assert F.get_device_error() == 0


# MX block-scaled caches: name, hq, hkv, d, bs, fmt, group_size
MX_CASES = [
    ("mx32_e4m3_d128_bs16_g8", 64, 8, 128, 16, E4, 32),
    ("mx16_e5m2_d64_bs32_g4", 16, 4, 64, 32, E5, 16),
    ("mx16_e4m3_d128_bs64_g8", 16, 2, 128, 64, E4, 16),
    ("mx32_e5m2_d64_bs16_g8", 8, 1, 64, 16, E5, 32),
]


@pytest.mark.parametrize("case", MX_CASES, ids=[c[0] for c in MX_CASES])
def test_mx_block_matches_oracle(F, case):
    """Block exponents and codes bit-exact; attention (bf16 and f32 outputs,
    and a 3-query chunk) within tolerance of the oracle."""
    from gpu_util import (check_close, gpu_attention, gpu_cache, gpu_multiquery, oracle_attention,
                          oracle_cache, oracle_multiquery)
    name, hq, hkv, d, bs, fmt, gs = case
    w = W.make_shape_case(name, _lens(bs), hq, hkv, d, bs, fmt, MX,
                          seed=3000 + MX_CASES.index(case), group_size=gs)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    for got, want, what in zip(g, o, ("K codes", "V codes", "K exponents", "V exponents")):
        assert np.array_equal(got.cpu().numpy(), want), what
    q = W.queries(w)
    ref = oracle_attention(w, q, o)
    check_close(gpu_attention(w, F, q, g), ref, bf16_out=True, what=f"{name} bf16")
    check_close(gpu_attention(w, F, q, g, out_dtype=torch.float32), ref, bf16_out=False,
                what=f"{name} f32")
    qc = W.chunk_queries(w, 3)
    short = bool((w.seq_lens < 3).any())
    check_close(gpu_multiquery(w, F, qc, g, out_dtype=torch.float32),
                oracle_multiquery(w, qc, o, 3), bf16_out=False, what=f"{name} q_len=3")
    assert F.get_device_error() == (4 if short else 0)


def test_large_batch_matches_oracle(F):
    """3,000 requests of 1..64 tokens (the planner's scans run ~100 warp
    passes; most ranges cross many requests), checked in full."""
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 65, size=3000)
    w = W.make_shape_case("large_batch", lens, 8, 2, 64, 16, E4, TH, seed=4242)
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    q = W.queries(w)
    check_close(gpu_attention(w, F, q, g, out_dtype=torch.float32), oracle_attention(w, q, o),
                bf16_out=False, what="large batch")
    assert F.get_device_error() == 0


# name, hq, hkv, d, bs, fmt, mode, group size
FAR_CASES = [
    ("gqa_token_head", 16, 2, 128, 16, E4, TH, None),
    ("gqa_mx32", 16, 2, 128, 16, E5, MX, 32),
    ("mla_latent", 32, 1, 576, 64, E4, TG, None),
]


@pytest.mark.parametrize("case", FAR_CASES, ids=[c[0] for c in FAR_CASES])
def test_blocks_beyond_4gib_of_cache(F, case):
    """Maximum-size addressing: the requests' blocks sit past the first 4 GiB
    of the code cache (block ids offset by `off`), so every code, scale and
    page address of the append and the decode needs 64-bit arithmetic.  The
    oracle sees the same cache with the offset removed (attention is
    invariant to where the blocks are)."""
    import dataclasses
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    name, hq, hkv, d, bs, fmt, mode, gs = case
    w = W.make_shape_case(name, [1, bs + 1, 3 * bs + 5], hq, hkv, d, bs, fmt, mode,
                          seed=2100 + FAR_CASES.index(case), group_size=gs)
    block_bytes = hkv * bs * d
    off = -(-(1 << 32) // block_bytes)  # first block id at or past 4 GiB
    far = dataclasses.replace(
        w, num_blocks=w.num_blocks + off,
        block_tables=np.where(w.block_tables >= 0, w.block_tables + off, -1).astype(np.int32))
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    try:
        g = gpu_cache(far, F, kvs)
        o = oracle_cache(w, kvs)
        assert np.array_equal(g[0][off:].cpu().numpy(), o[0]), "K codes"
        assert np.array_equal(g[2][off:].cpu().numpy(), o[2]), "K scales"
        if not w.mla:
            assert np.array_equal(g[1][off:].cpu().numpy(), o[1]), "V codes"
        q = W.queries(w)
        check_close(gpu_attention(far, F, q, g, out_dtype=torch.float32),
                    oracle_attention(w, q, o), bf16_out=False, what=f"{name} past 4 GiB")
        assert F.get_device_error() == 0
    finally:
        g = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("gs", [16, 32])
@pytest.mark.parametrize("fmt", [E4, E5])
def test_mx_blocks_spanning_the_f16_factor_range(F, gs, fmt):
    """Blocks of one token whose exponents lie up to 2^40 below the token's
    largest (and all-zero blocks), so the decode's per-block factors
    2^(e_k - e_max) take normal f16 values, f16 subnormals (2^-15 .. 2^-24)
    and 0: exponents and codes bit-exact, attention (f32) within tolerance
    of the oracle."""
    from gpu_util import check_close, gpu_attention, gpu_cache, oracle_attention, oracle_cache
    d, bs = 128, 16
    w = W.make_shape_case(f"mx{gs}_factor_range", [1, bs - 1, 3 * bs + 5, 70], 16, 2, d, bs,
                          fmt, MX, seed=3300 + gs + fmt, group_size=gs)
    rng = np.random.default_rng(3300 + gs + fmt)
    pw = np.array([0, -6, -12, -15, -18, -21, -24, -26, -40], np.float32)
    kvs = []
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        pair = []
        for _ in range(2):
            x = rng.standard_normal((L, w.n_kv_heads, d)).astype(np.float32)
            xb = x.reshape(L, w.n_kv_heads, d // gs, gs)
            f = np.exp2(rng.choice(pw, size=(L, w.n_kv_heads, d // gs))).astype(np.float32)
            f[rng.random(f.shape) < 0.1] = 0.0  # all-zero blocks
            xb *= f[..., None]
            pair.append(W.f32_to_bf16_bits(x))
        kvs.append(tuple(pair))
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    for got, want, what in zip(g, o, ("K codes", "V codes", "K exponents", "V exponents")):
        assert np.array_equal(got.cpu().numpy(), want), what
    q = W.queries(w)
    check_close(gpu_attention(w, F, q, g, out_dtype=torch.float32), oracle_attention(w, q, o),
                bf16_out=False, what=f"mx{gs} factor range f32")
    assert F.get_device_error() == 0
