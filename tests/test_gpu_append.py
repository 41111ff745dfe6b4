"""GPU parity of the append step: FP8 codes, scales and slot placement must
be bit-exact with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()  # clear
    return F


def _assert_codes_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
    assert bad.size == 0, (f"{what}: {bad.size} mismatches, first at flat {bad[0]}: "
                           f"gpu {got.reshape(-1)[bad[0]]:#04x} oracle {want.reshape(-1)[bad[0]]:#04x}")


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_append_matches_oracle(F, idx):
    from gpu_util import gpu_cache, oracle_cache
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    g = gpu_cache(w, F, kvs)
    o = oracle_cache(w, kvs)
    assert F.get_device_error() == 0
    _assert_codes_equal(g[0].cpu().numpy(), o[0], "k codes")
    assert np.array_equal(g[2].cpu().numpy().view(np.uint32), o[2].view(np.uint32)), "k scales"
    if not w.mla:
        _assert_codes_equal(g[1].cpu().numpy(), o[1], "v codes")
        assert np.array_equal(g[3].cpu().numpy().view(np.uint32), o[3].view(np.uint32))


def _all_bf16_rows(d):
    """Every bf16 bit pattern once, as rows of d values."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits.reshape(-1, 1, d)


@pytest.mark.parametrize("fmt", [W.E4M3, W.E5M2, W.INT8])
@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7, 0.3, 1000.0])
def test_every_bf16_pattern_static_scale(F, fmt, scale):
    """Static scale: code = fp8(x / s) (or the INT8 rounding) for all 65,536
    bf16 inputs."""
    from gpu_util import DEV, to_dev_bf16
    d = 128
    x = _all_bf16_rows(d)
    n = x.shape[0]
    s = np.full((1, d), scale, np.float32)
    kc = torch.zeros((n, 1, 1, d), dtype=torch.uint8, device=DEV)
    slots = torch.arange(n, dtype=torch.int32, device=DEV)
    F.kv_append_quant(to_dev_bf16(x), None, slots, kc, None, torch.from_numpy(s).to(DEV), None,
                      fmt=fmt, scale_mode=W.SCALE_CHANNEL_STATIC)
    got = kc.cpu().numpy().reshape(-1)
    okc = np.zeros((n, 1, 1, d), np.uint8)
    oracle.kv_append_quant(x, None, np.arange(n, dtype=np.int32), fmt, W.SCALE_CHANNEL_STATIC, d,
                           okc, None, s.copy(), None, 1)
    want = okc.reshape(-1)
    xf = W.bf16_bits_to_f32(x.reshape(-1))
    nan_in = np.isnan(xf)
    # NaN inputs: any NaN code is a correct answer (INT8 has none: any code);
    # everything else is unique.
    if fmt != W.INT8:
        assert np.isnan(oracle.fp8_decode(got[nan_in], fmt)).all()
    _assert_codes_equal(got[~nan_in], want[~nan_in], f"fmt={fmt} scale={scale}")


@pytest.mark.parametrize("fmt", [W.E4M3, W.E5M2, W.INT8])
def test_every_finite_bf16_pattern_dynamic_rows(F, fmt):
    """Dynamic per-row scales over rows that together hold every finite bf16."""
    from gpu_util import DEV, to_dev_bf16
    d = 128
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xf = W.bf16_bits_to_f32(bits)
    fin = bits[np.isfinite(xf)]
    rng = np.random.default_rng(1)
    fin = rng.permutation(fin)
    pad = (-fin.size) % (2 * d)
    fin = np.concatenate([fin, np.zeros(pad, np.uint16)])
    x = fin.reshape(-1, 2, d)  # [tokens, hkv=2, d]
    n = x.shape[0]
    bs = 16
    nb = (n + bs - 1) // bs + 1
    kc = torch.zeros((nb, 2, bs, d), dtype=torch.uint8, device=DEV)
    ks = torch.zeros((nb, 2, bs, 1), dtype=torch.float32, device=DEV)
    slots = rng.permutation(nb * bs)[:n].astype(np.int32)
    F.kv_append_quant(to_dev_bf16(x), None, torch.from_numpy(slots).to(DEV), kc, None, ks, None,
                      fmt=fmt, scale_mode=W.SCALE_TOKEN_HEAD)
    okc = np.zeros((nb, 2, bs, d), np.uint8)
    oks = np.zeros((nb, 2, bs, 1), np.float32)
    oracle.kv_append_quant(x, None, slots, fmt, W.SCALE_TOKEN_HEAD, d, okc, None, oks, None, bs)
    _assert_codes_equal(kc.cpu().numpy(), okc, "codes")
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))


def test_edges_zero_rows_skip_and_bad_slots(F):
    from gpu_util import DEV, to_dev_bf16
    d, hkv, bs, nb = 64, 2, 16, 4
    x = np.zeros((5, hkv, d), np.uint16)
    x[1] = 0x8000                      # a row of -0.0
    x[2, 0, 3] = 0x3F80                # one 1.0 among zeros
    x[3, 1, :] = 0x4300                # 128.0 everywhere
    slots = np.array([0, 5, -1, 63, 64], np.int32)  # -1 skipped, 64 past the pool
    for fmt in (W.E4M3, W.E5M2):
        kc = torch.full((nb, hkv, bs, d), 0xAA, dtype=torch.uint8, device=DEV)
        vc = torch.full_like(kc, 0xAA)
        ks = torch.full((nb, hkv, bs, 1), -1.0, dtype=torch.float32, device=DEV)
        vs = torch.full_like(ks, -1.0)
        F.kv_append_quant(to_dev_bf16(x), to_dev_bf16(x), torch.from_numpy(slots).to(DEV), kc,
                          vc, ks, vs, fmt=fmt)
        assert F.get_device_error() == 1   # FP8PA_DEVERR_SLOT_RANGE
        okc = np.full((nb, hkv, bs, d), 0xAA, np.uint8)
        ovc = okc.copy()
        oks = np.full((nb, hkv, bs, 1), -1.0, np.float32)
        ovs = oks.copy()
        assert oracle.kv_append_quant(x, x, slots, fmt, W.SCALE_TOKEN_HEAD, d, okc, ovc, oks, ovs,
                                      bs) == 1
        _assert_codes_equal(kc.cpu().numpy(), okc, "k")
        _assert_codes_equal(vc.cpu().numpy(), ovc, "v")
        assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
        # -0.0 keeps its sign; a zero row gets the 1e-12 floor
        assert (kc[0, 1, 5].cpu().numpy() == 0x80).all()
        assert ks[0, 0, 0, 0].item() == np.float32(1e-12)


def test_channel_scales_match_oracle(F):
    from gpu_util import DEV, to_dev_bf16
    w = W.make_workload(4, "small")
    ks = np.concatenate([W.request_kv(w, b)[0] for b in range(w.batch)])
    for fmt in (W.E4M3, W.E5M2):
        got = F.kv_channel_scales(to_dev_bf16(ks), fmt).cpu().numpy()
        want = oracle.kv_channel_scales(ks, fmt)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_running_absmax_calibration_matches_oracle(F):
    """Online calibration: folding prefill batches into a running absmax in
    any order gives the one-shot static scales of all tokens, bit for bit."""
    from gpu_util import DEV, to_dev_bf16
    w = W.make_workload(4, "small")
    ks = [W.request_kv(w, b)[0] for b in range(w.batch)]
    for fmt in (W.E4M3, W.E5M2):
        amax = torch.zeros((w.n_kv_heads, w.head_dim), dtype=torch.float32, device=DEV)
        for b in (3, 0, 5, 1, 4, 2):          # batches arrive in any order
            F.kv_channel_absmax_update(to_dev_bf16(ks[b]), amax)
        got = F.kv_scales_from_absmax(amax, fmt).cpu().numpy()
        want = oracle.kv_channel_scales(np.concatenate(ks), fmt)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        # scale_out may alias the running absmax
        amax2 = amax.clone()
        F.kv_scales_from_absmax(amax2, fmt, out=amax2)
        assert np.array_equal(amax2.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("fmt", [W.E4M3, W.E5M2])
@pytest.mark.parametrize("gs", [16, 32])
def test_every_finite_bf16_pattern_mx_blocks(F, fmt, gs):
    """MX block mode over rows that together hold every finite bf16 value:
    E8M0 block exponents and codes bit-exact with the oracle."""
    from gpu_util import DEV, to_dev_bf16
    d = 128
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xf = W.bf16_bits_to_f32(bits)
    fin = bits[np.isfinite(xf)]
    rng = np.random.default_rng(gs + fmt)
    fin = rng.permutation(fin)
    pad = (-fin.size) % (2 * d)
    fin = np.concatenate([fin, np.zeros(pad, np.uint16)])
    x = fin.reshape(-1, 2, d)
    n, bs = x.shape[0], 16
    nb = (n + bs - 1) // bs + 1
    kc = torch.zeros((nb, 2, bs, d), dtype=torch.uint8, device=DEV)
    ke = torch.zeros((nb, 2, bs, d // gs), dtype=torch.uint8, device=DEV)
    slots = rng.permutation(nb * bs)[:n].astype(np.int32)
    F.kv_append_quant(to_dev_bf16(x), None, torch.from_numpy(slots).to(DEV), kc, None, ke, None,
                      fmt=fmt, scale_mode=W.SCALE_MX_BLOCK, group_size=gs)
    okc = np.zeros((nb, 2, bs, d), np.uint8)
    oke = np.zeros((nb, 2, bs, d // gs), np.uint8)
    oracle.kv_append_quant(x, None, slots, fmt, W.SCALE_MX_BLOCK, gs, okc, None, oke, None, bs)
    _assert_codes_equal(kc.cpu().numpy(), okc, "codes")
    assert np.array_equal(ke.cpu().numpy(), oke), "exponents"


@pytest.mark.parametrize("fmt", [W.E4M3, W.E5M2, W.INT8])
@pytest.mark.parametrize("mode", [W.SCALE_TOKEN_HEAD, W.SCALE_TOKEN_GROUP])
def test_bulk_rows_every_finite_bf16_pattern(F, fmt, mode):
    """A call of more than 16K rows (the persistent streaming kernel) whose
    rows hold every finite bf16 value many times over, in shuffled rows and
    slots, with -0.0 entries and all-zero rows among them: codes and scales
    bit-exact with the oracle."""
    from gpu_util import DEV, to_dev_bf16
    d, hkv, bs, gs = 128, 8, 16, 32
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = bits[np.isfinite(W.bf16_bits_to_f32(bits))]
    rng = np.random.default_rng(7)
    n = 2304                                  # tokens: 2304 x 8 heads x (K, V) rows
    vals = np.concatenate([rng.permutation(fin) for _ in range(2 * n * hkv * d // fin.size + 1)])
    x = vals[:2 * n * hkv * d].reshape(2, n, hkv, d).copy()
    x[0, 5] = 0x8000                          # a token of -0.0 rows
    x[1, 9, 3] = 0                            # an all-zero row
    nb = n // bs + 3
    slots = rng.permutation(nb * bs)[:n].astype(np.int32)
    ng = d // gs if mode == W.SCALE_TOKEN_GROUP else 1
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((nb, hkv, bs, ng), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    F.kv_append_quant(to_dev_bf16(x[0]), to_dev_bf16(x[1]), torch.from_numpy(slots).to(DEV), kc,
                      vc, ks, vs, fmt=fmt, scale_mode=mode, group_size=gs)
    assert F.get_device_error() == 0
    okc = np.zeros((nb, hkv, bs, d), np.uint8)
    ovc = okc.copy()
    oks = np.zeros((nb, hkv, bs, ng), np.float32)
    ovs = oks.copy()
    assert oracle.kv_append_quant(x[0], x[1], slots, fmt, mode, gs, okc, ovc, oks, ovs, bs) == 0
    _assert_codes_equal(kc.cpu().numpy(), okc, "k codes")
    _assert_codes_equal(vc.cpu().numpy(), ovc, "v codes")
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32)), "k scales"
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32)), "v scales"


@pytest.mark.parametrize("fmt", [W.E4M3, W.E5M2, W.INT8])
@pytest.mark.parametrize("mode", [W.SCALE_TOKEN_HEAD, W.SCALE_TOKEN_GROUP])
@pytest.mark.parametrize("n_tokens", [40, 2100])
def test_dynamic_rows_with_infinities_and_nans(F, fmt, mode, n_tokens):
    """Rows (or groups) holding +-inf get an infinite scale, and their codes
    come from the exact division x / inf (0 of x's sign, NaN for an infinite
    x); NaN entries leave the absmax alone.  Small calls (the one-step
    kernel) and calls above 16K rows (the streaming kernel).  Codes and
    scales match the oracle; where the quotient is NaN any NaN code is
    accepted; INT8 codes a NaN quotient as 0 on both sides."""
    from gpu_util import DEV, to_dev_bf16
    d, hkv, bs, gs = 128, 4, 16, 32
    rng = np.random.default_rng(11 + n_tokens)
    xf = rng.standard_normal((2, n_tokens, hkv, d)).astype(np.float32)
    x = W.f32_to_bf16_bits(xf).reshape(2, n_tokens, hkv, d)
    flat = x.reshape(-1)
    for pat in (0x7F80, 0xFF80, 0x7FC0):       # +inf, -inf, NaN
        idx = rng.choice(flat.size, size=max(4, flat.size // 997), replace=False)
        flat[idx] = pat
    nb = n_tokens // bs + 2
    slots = rng.permutation(nb * bs)[:n_tokens].astype(np.int32)
    ng = d // gs if mode == W.SCALE_TOKEN_GROUP else 1
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((nb, hkv, bs, ng), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    F.kv_append_quant(to_dev_bf16(x[0]), to_dev_bf16(x[1]), torch.from_numpy(slots).to(DEV), kc,
                      vc, ks, vs, fmt=fmt, scale_mode=mode, group_size=gs)
    assert F.get_device_error() == 0
    okc = np.zeros((nb, hkv, bs, d), np.uint8)
    ovc = okc.copy()
    oks = np.zeros((nb, hkv, bs, ng), np.float32)
    ovs = oks.copy()
    assert oracle.kv_append_quant(x[0], x[1], slots, fmt, mode, gs, okc, ovc, oks, ovs, bs) == 0
    for got, want, what in ((kc, okc, "k"), (vc, ovc, "v")):
        got = got.cpu().numpy().reshape(-1)
        want = want.reshape(-1)
        nan_want = np.isnan(oracle.fp8_decode(want, fmt)) if fmt != W.INT8 else None
        if nan_want is not None:
            assert np.isnan(oracle.fp8_decode(got[nan_want], fmt)).all(), what
            _assert_codes_equal(got[~nan_want], want[~nan_want], what)
        else:
            _assert_codes_equal(got, want, what)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32)), "k scales"
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32)), "v scales"
