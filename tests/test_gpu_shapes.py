"""GPU parity over the supported shape space beyond the five named
workloads: block sizes 16/32/64, head_dim 64/128, GQA group sizes 1, 2, 3, 4
and 8, KV-head counts that are not a power of two or need several head sets
per CTA, both formats with both GQA scale modes, KV-head counts up to 24,
and the latent layout with 32 and 64 query heads.  Every output is compared with the FP64 oracle;
lengths include 1, block_size - 1, block_size, block_size + 1 and several
pages with a ragged tail."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4, E5 = W.E4M3, W.E5M2
TH, CS, TG = W.SCALE_TOKEN_HEAD, W.SCALE_CHANNEL_STATIC, W.SCALE_TOKEN_GROUP

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


@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[8]], ids=lambda c: c[0])
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
