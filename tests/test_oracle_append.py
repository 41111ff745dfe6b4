"""Pins for the oracle's append step: hand-worked rows with exact
power-of-two scales, group independence, static channel scales, the slot
scatter, and the channel calibration."""
import json
import os

import numpy as np

import oracle
from fp8_quantised_paged_gb300.workloads import f32_to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden", "append_rows.json")
FMTS = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}


def _gold():
    with open(GOLD) as f:
        return json.load(f)


def _bf16(x):
    b = f32_to_bf16_bits(np.asarray(x, np.float32))
    # every golden value is exactly representable in bf16
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), np.float32(x))
    return b


def _empty_cache(nb, hkv, bs, d, ngroups=1):
    return (np.zeros((nb, hkv, bs, d), np.uint8), np.zeros((nb, hkv, bs, d), np.uint8),
            np.zeros((nb, hkv, bs, ngroups), np.float32),
            np.zeros((nb, hkv, bs, ngroups), np.float32))


def test_token_head_rows():
    for row in _gold()["token_head"]:
        fmt = FMTS[row["fmt"]]
        x = _bf16(row["x"])
        d = x.size
        k = x.reshape(1, 1, d)
        v = (x ^ np.uint16(0x8000)).reshape(1, 1, d)  # V is the negated row
        kc, vc, ks, vs = _empty_cache(2, 1, 4, d)
        slot = np.array([4 + 2], np.int32)             # block 1, offset 2
        bad = oracle.kv_append_quant(k, v, slot, fmt, oracle.SCALE_TOKEN_HEAD, d, kc, vc,
                                     ks, vs, block_size=4)
        assert bad == 0
        assert ks[1, 0, 2, 0] == np.float32(row["scale"]) == vs[1, 0, 2, 0]
        assert list(kc[1, 0, 2]) == row["codes"]
        assert list(vc[1, 0, 2]) == [c ^ 0x80 for c in row["codes"]]
        # nothing else was written
        mask = np.ones(kc.shape, bool)
        mask[1, 0, 2] = False
        assert not kc[mask].any() and not vc[mask].any()


def test_scale_is_absmax_over_fmax():
    # absmax 2.0 -> 2/448 and 2/57344 in fp32 (division, then the 1e-12 floor)
    x = _bf16([1.0, -2.0, 0.5, 0.0])
    assert oracle.absmax_scale(x, oracle.E4M3) == np.float32(2.0) / np.float32(448.0)
    assert oracle.absmax_scale(x, oracle.E5M2) == np.float32(2.0) / np.float32(57344.0)
    assert oracle.absmax_scale(x, oracle.INT8) == np.float32(2.0) / np.float32(127.0)
    assert oracle.absmax_scale(_bf16([0.0, -0.0]), oracle.E4M3) == np.float32(1e-12)


def test_token_group_rows_are_independent():
    g = _gold()["token_group"]
    gs, d = g["group_size"], 128
    x = np.zeros(d, np.float32)
    for i, val in g["nonzero"].items():
        x[int(i)] = val
    k = _bf16(x).reshape(1, 1, d)
    kc, _, ks, _ = _empty_cache(1, 1, 2, d, ngroups=d // gs)
    oracle.kv_append_quant(k, None, np.array([1], np.int32), oracle.E4M3,
                           oracle.SCALE_TOKEN_GROUP, gs, kc, None, ks, None, block_size=2)
    assert list(ks[0, 0, 1]) == g["scales"]
    for i, c in g["codes_nonzero"].items():
        assert kc[0, 0, 1, int(i)] == c
    # changing group 1 leaves group 0's codes and scale untouched
    x2 = x.copy()
    x2[64:] *= 64.0
    k2 = _bf16(x2).reshape(1, 1, d)
    kc2, _, ks2, _ = _empty_cache(1, 1, 2, d, ngroups=d // gs)
    oracle.kv_append_quant(k2, None, np.array([1], np.int32), oracle.E4M3,
                           oracle.SCALE_TOKEN_GROUP, gs, kc2, None, ks2, None, block_size=2)
    assert np.array_equal(kc2[0, 0, 1, :64], kc[0, 0, 1, :64]) and ks2[0, 0, 1, 0] == ks[0, 0, 1, 0]
    assert ks2[0, 0, 1, 1] == 128.0 and np.array_equal(kc2[0, 0, 1, 64:], kc[0, 0, 1, 64:])


def test_channel_static_power_of_two_scales():
    rng = np.random.default_rng(3)
    hkv, d = 2, 32
    x = f32_to_bf16_bits(rng.standard_normal((5, hkv, d)).astype(np.float32) * 40)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    e = rng.integers(-3, 4, size=(hkv, d))
    s = np.exp2(e).astype(np.float32)
    kc = np.zeros((3, hkv, 4, d), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.array([0, 5, 6, -1, 11], np.int32)
    oracle.kv_append_quant(x, x, slots, oracle.E5M2, oracle.SCALE_CHANNEL_STATIC, d, kc, vc,
                           s.copy(), s.copy(), block_size=4)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        want = oracle.fp8_encode(xf[t] * np.exp2(-e).astype(np.float32), oracle.E5M2)
        assert np.array_equal(kc[sl // 4, :, sl % 4], want)
        assert np.array_equal(vc[sl // 4, :, sl % 4], want)


def test_slot_scatter_skip_and_bounds():
    hkv, d, bs, nb = 2, 16, 4, 3
    n = 6
    # token t carries the constant value t+1 in every element, so each
    # stored row names the token that wrote it.
    x = np.stack([np.full((hkv, d), t + 1, np.float32) for t in range(n)])
    k = f32_to_bf16_bits(x)
    slots = np.array([11, -1, 0, 7, 12, 5], np.int32)  # 12 is past the pool
    kc, vc, ks, vs = _empty_cache(nb, hkv, bs, d)
    bad = oracle.kv_append_quant(k, k, slots, oracle.E4M3, oracle.SCALE_TOKEN_HEAD, d, kc, vc,
                                 ks, vs, block_size=bs)
    assert bad == 1
    written = {}
    for blk in range(nb):
        for off in range(bs):
            if ks[blk, 0, off, 0] != 0:
                written[blk * bs + off] = ks[blk, 0, off, 0] * 448.0
    want = {11: 1.0, 0: 3.0, 7: 4.0, 5: 6.0}
    assert set(written) == set(want)
    for sl, val in want.items():
        assert abs(written[sl] - val) < 1e-5 * val
        assert (kc[sl // bs, :, sl % bs] == 0x7E).all()


def test_channel_calibration():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, 3, 16)).astype(np.float32)
    x[17, 1, 4] = -900.0
    b = f32_to_bf16_bits(x)
    xf = (b.astype(np.uint32) << 16).view(np.float32)
    s = oracle.kv_channel_scales(b, oracle.E5M2)
    assert s.shape == (3, 16)
    assert s[1, 4] == np.float32(900.0) / np.float32(57344.0)
    i = (2, 9)
    assert s[i] == np.abs(xf[:, i[0], i[1]]).max() / np.float32(57344.0)
    z = oracle.kv_channel_scales(np.zeros((4, 1, 16), np.uint16), oracle.E4M3)
    assert (z == np.float32(1e-12)).all()


# ---------------------------------------------------------------- MX block mode
def _mx_append(x_rows, fmt, gs):
    """Append rows [n, d] (bf16 bits) for one KV head with MX block scales."""
    n, d = x_rows.shape
    kc = np.zeros((n, 1, 1, d), np.uint8)
    ks = np.zeros((n, 1, 1, d // gs), np.uint8)
    assert oracle.kv_append_quant(x_rows.reshape(n, 1, d), None, np.arange(n, dtype=np.int32),
                                  fmt, oracle.SCALE_MX_BLOCK, gs, kc, None, ks, None, 1) == 0
    return kc.reshape(n, d), ks.reshape(n, d // gs)


def test_mx_block_hand_worked():
    """E4M3, blocks of 32: absmax 448 -> e = 0, codes are the plain cast;
    absmax 500 -> e = 0 too and 500 saturates to 448 (0x7E); absmax 1 ->
    e = -8, so 1.0 -> 256 (0x78) and 0.5 -> 128 (0x70); an all-zero block
    takes e = -127 (byte 0) and zero codes."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0], x[0, 1] = 448.0, -2.0           # block 0
    x[0, 32], x[0, 33] = 500.0, -1.0         # block 1
    x[0, 64], x[0, 65] = 1.0, 0.5            # block 2
    kc, ks = _mx_append(_bf16(x), oracle.E4M3, 32)
    assert list(ks[0]) == [127, 127, 119, 0]
    assert kc[0, 0] == 0x7E and kc[0, 1] == 0xC0      # 448, -2.0
    assert kc[0, 32] == 0x7E and kc[0, 33] == 0xB8    # 500 -> 448, -1.0
    assert kc[0, 64] == 0x78 and kc[0, 65] == 0x70    # 256, 128
    assert not kc[0, 96:].any()


def test_mx_block_matches_numpy_torch_restatement():
    """Every block of seeded heavy-tailed rows against an independent
    restatement: e from numpy's frexp, codes from torch's float8 cast of
    x * 2^-e (clamped to the finite range first: torch's e4m3fn cast does not
    saturate)."""
    import torch
    rng = np.random.default_rng(7)
    for fmt, tdt, fmax, emax in ((oracle.E4M3, torch.float8_e4m3fn, 448.0, 8),
                                 (oracle.E5M2, torch.float8_e5m2, 57344.0, 15)):
        for gs in (16, 32):
            x = rng.standard_t(2.0, size=(64, 128)).astype(np.float32)
            x *= np.exp2(rng.integers(-20, 20, size=(64, 1))).astype(np.float32)
            x[3, :gs] = 0.0                                  # an all-zero block
            xb = f32_to_bf16_bits(x)
            kc, ks = _mx_append(xb, fmt, gs)
            xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            blocks = xf.reshape(64, 128 // gs, gs)
            amax = np.abs(blocks).max(axis=2)
            _, E = np.frexp(amax)
            e = np.where(amax > 0, E - 1 - emax, -127).clip(-127, 127)
            assert np.array_equal(ks.astype(np.int64) - 127, e)
            scaled = np.clip(blocks * np.exp2(-e)[..., None], -fmax, fmax)
            want = torch.from_numpy(scaled.astype(np.float32)).to(tdt).view(torch.uint8).numpy()
            assert np.array_equal(kc.reshape(64, 128 // gs, gs), want), (fmt, gs)
