"""GPU parity of causal chunks on the grouped-query layout where they run
on the tensor-core kernel (FP8 codes, one scale per token and KV head,
head_dim 128, G x qw = 16 or 32 columns for qw queries of the chunk, qw the
largest such divisor of q_len): every (request, query) row against the FP64
oracle over its visible prefix, seq_lens[b] - (q_len - 1 - i) tokens ("Llama
3 70B FP8 deployment", dpshk.com, sec. 3.3: chunked prefill).  Block sizes
16, 32 and 64, both FP8 formats, 2 to 32 query heads per KV head, chunks
taken whole or as 2, 3 or 8 planned requests of qw queries, ragged lengths
that start steps mid-page and end them mid-step, and every kind of split."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4, E5, TH = W.E4M3, W.E5M2, W.SCALE_TOKEN_HEAD

# name, lengths, hq, hkv, bs, fmt, q_len
CASES = [
    ("g8_q4_bs16_e4m3", [300, 129, 1025, 4], 64, 8, 16, E4, 4),
    ("g8_q2_bs32_e5m2", [2, 700, 128, 257], 16, 2, 32, E5, 2),
    ("g4_q4_bs64_e4m3", [1100, 63, 65, 500], 8, 2, 64, E4, 4),
    ("g4_q8_bs16_e5m2", [900, 8, 300], 12, 3, 16, E5, 8),
    ("g2_q8_bs32_e4m3", [640, 1300, 33], 8, 4, 32, E4, 8),
    ("g8_q4_hkv1_bs64_e5m2", [2050, 777], 8, 1, 64, E5, 4),
    # chunks split into planned requests of qw < q_len queries
    ("g8_q8_qw4_bs16_e4m3", [700, 129, 1030, 9], 16, 2, 16, E4, 8),
    ("g16_q4_qw2_bs32_e5m2", [513, 77, 300], 32, 2, 32, E5, 4),
    ("g32_q3_qw1_bs64_e4m3", [400, 65, 130], 32, 1, 64, E4, 3),
    ("g16_q3_qw1_bs16_e5m2", [260, 33, 3], 16, 1, 16, E5, 3),
]


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    yield F
    F.set_decode_workers(0)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_chunk_on_tensor_cores_matches_oracle(F, case):
    from gpu_util import check_close, gpu_cache, gpu_multiquery, oracle_cache, oracle_multiquery
    name, lens, hq, hkv, bs, fmt, q_len = case
    w = W.make_shape_case(name, lens, hq, hkv, 128, bs, fmt, TH, seed=7300 + CASES.index(case))
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    qc = W.chunk_queries(w, q_len)
    ref = oracle_multiquery(w, qc, o, q_len)
    short = bool((w.seq_lens < q_len).any())
    outs = []
    try:
        for workers in (1, 2, 7, 64, 0):
            F.set_decode_workers(workers)
            got = gpu_multiquery(w, F, qc, g, out_dtype=torch.float32)
            check_close(got, ref, bf16_out=False, what=f"{name} workers={workers}")
            outs.append(got)
            # a request shorter than the chunk is out of contract and flagged
            assert F.get_device_error() == (4 if short else 0)
    finally:
        F.set_decode_workers(0)
    got = gpu_multiquery(w, F, qc, g)
    check_close(got, ref, bf16_out=True, what=f"{name} bf16")
    assert F.get_device_error() == (4 if short else 0)
    tol = 1e-4 * np.abs(outs[0]).max()
    for x in outs[1:]:
        assert np.abs(x - outs[0]).max() <= tol


def _finite_codes(fmt):
    b = np.arange(256, dtype=np.uint8)
    keep = (b & 0x7F) != 0x7F if fmt == E4 else (b & 0x7C) != 0x7C
    return b[keep]


def _small_codes(fmt):
    """Codes with exponent field 0 (subnormal) or 1 (smallest normal)."""
    b = _finite_codes(fmt)
    e = (b >> 3) & 0xF if fmt == E4 else (b >> 2) & 0x1F
    return b[e <= 1]


# fmt, code set, q_len, bs
CODE_CASES = [(E4, "all", 4, 16), (E4, "small", 2, 32), (E5, "all", 2, 64), (E5, "small", 4, 16)]


@pytest.mark.parametrize("case", CODE_CASES, ids=lambda c: f"{'e4m3' if c[0] == E4 else 'e5m2'}"
                                                            f"_{c[1]}_codes_q{c[2]}_bs{c[3]}")
def test_chunk_on_tensor_cores_over_every_code(F, case):
    """Caches written directly, not through the append: K and V codes drawn
    from all finite bytes of the format, or only from the subnormal and
    smallest normal ones, with a free-ranging fp32 scale per (token, KV
    head), so that the kernel's conversion of every code (sign, exponent,
    mantissa, subnormals) and its scaling meet the oracle's definitions."""
    from gpu_util import DEV, check_close, gpu_multiquery, oracle_multiquery
    fmt, which, q_len, bs = case
    idx = CODE_CASES.index(case)
    w = W.make_shape_case(f"chunk_codes_{which}", [700, 129, 64], 16, 2, 128, bs, fmt, TH,
                          seed=7400 + idx)
    rng = np.random.default_rng(7500 + idx)
    pool = _finite_codes(fmt) if which == "all" else _small_codes(fmt)
    top = np.abs(torch.from_numpy(pool).view(
        torch.float8_e4m3fn if fmt == E4 else torch.float8_e5m2).float().numpy()).max()
    shape = (w.num_blocks, w.n_kv_heads, bs, 128)
    kc, vc = (rng.choice(pool, size=shape).astype(np.uint8) for _ in range(2))
    # scales 2^U(-2, 2) (a full 24-bit mantissa) over the largest code of the set
    ks, vs = ((np.exp2(rng.uniform(-2.0, 2.0, size=shape[:3] + (1,))) / top).astype(np.float32)
              for _ in range(2))
    qc = W.chunk_queries(w, q_len)
    ref = oracle_multiquery(w, qc, (kc, vc, ks, vs), q_len)
    dev = tuple(torch.from_numpy(x).to(DEV) for x in (kc, vc, ks, vs))
    try:
        for workers in (1, 0):
            F.set_decode_workers(workers)
            got = gpu_multiquery(w, F, qc, dev, out_dtype=torch.float32)
            check_close(got, ref, bf16_out=False, what=f"{w.name} workers={workers}")
    finally:
        F.set_decode_workers(0)
    assert F.get_device_error() == 0
