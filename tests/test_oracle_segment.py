"""Pins for the oracle's block-wise cumulative rescaling (the segment scale
mode): "DeepSeek V4 950: whole-network FP8 dataflow" (2kiu.com/news/4508674)
sec. 4.3 cuts the KV cache into length blocks, keeps a cumulative scale per
block and refreshes an extra offset every 1024 tokens.  Reading: per
(sequence, K or V, KV head) a running absmax R over every appended token;
the token at a position that is a multiple of 1024 opens a segment whose
scale is frozen as max(R / FMAX, 1e-12); every token of the segment is coded
with it.

The pins: a hand-worked sequence whose expected codes and page scales are
written out from the E4M3 definition (not from the oracle's encoder); a jump
in range at token 1024 changes only the later segment's scale; the result
does not depend on how the tokens are split into calls (one call, one token
per call, random chunks, sequences interleaved); rows of equal absmax give
the per-(token, head) mode's codes; scales never decrease along a sequence;
and attention over the segment-scaled cache equals torch's float64 SDPA on
the cache dequantised through torch's float8 types."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

SEG = oracle.SEGMENT_TOKENS


def bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


# A row of exact E4M3 values (absmax 448) and its codes at scale 1, 2 and
# (for the row doubled) at scale 1, from the format's bit fields
# (S.EEEE.MMM, bias 7; 448 = 1.75 * 2^8 is the largest finite value).
BASE = [448.0, -448.0, 1.0, 0.5, 0.25, -2.0, 3.0] + [0.0] * 9
CODES_S1 = [0x7E, 0xFE, 0x38, 0x30, 0x28, 0xC0, 0x44] + [0x00] * 9
CODES_S2 = [0x76, 0xF6, 0x30, 0x28, 0x20, 0xB8, 0x3C] + [0x00] * 9   # BASE / 2
CODES_2X_S1 = [0x7E, 0xFE, 0x40, 0x38, 0x30, 0xC8, 0x4C] + [0x00] * 9  # 2*BASE, 896 saturates


def _one_sequence(rows, bs=16):
    """Append `rows` (float [L, D]) as one sequence of one KV head (K only)
    through blocks 0, 1, 2, ... in one call."""
    L, d = rows.shape
    nb = (L + bs - 1) // bs
    k = bf16(rows)[:, None, :]
    kc = np.zeros((nb, 1, bs, d), np.uint8)
    ks = np.zeros((nb, oracle.segment_scale_heads(1)), np.float32)
    st = np.zeros((1, 2, 1, 2), np.float32)
    slots = np.arange(L, dtype=np.int32)
    assert oracle.kv_append_quant_segment(k, None, slots, [0, L], [0], oracle.E4M3, st, kc, None,
                                          ks, None, bs) == 0
    return kc.reshape(nb * bs, d)[:L], ks[:, 0], st


def test_hand_worked_segments():
    """2100 tokens of BASE; token 500 doubled (absmax 896, a spike inside
    segment 0).  Segment 0's scale is frozen at token 0 (448 / 448 = 1), so
    the spike saturates; it raises the running absmax, so segments 1 and 2
    open at 896 / 448 = 2."""
    rows = np.tile(np.array(BASE, np.float32), (2100, 1))
    rows[500] *= 2.0
    codes, page_scales, st = _one_sequence(rows)
    assert list(codes[0]) == CODES_S1
    assert list(codes[1023]) == CODES_S1
    assert list(codes[500]) == CODES_2X_S1
    assert list(codes[1024]) == CODES_S2
    assert list(codes[2099]) == CODES_S2
    assert (page_scales[:64] == 1.0).all()          # tokens 0..1023
    assert (page_scales[64:] == 2.0).all()          # tokens 1024..2099
    assert st[0, 0, 0, 0] == 896.0 and st[0, 0, 0, 1] == 2.0


def test_jump_at_token_1024_changes_only_the_later_segment():
    rows = np.tile(np.array(BASE, np.float32), (1100, 1))
    rows[1024] *= 10.0                              # absmax 4480 -> scale 10
    codes, page_scales, _ = _one_sequence(rows)
    assert (page_scales[:64] == 1.0).all()
    assert (page_scales[64:] == 10.0).all()
    assert all(list(codes[t]) == CODES_S1 for t in (0, 511, 1023))
    # BASE / 10 after token 1024: 448 / 10 = 44.8 lies in [32, 64), where
    # E4M3 steps by 4; the nearest value is 44 = 1.375 * 2^5: exponent field
    # 5 + 7 = 12, mantissa field 3.
    assert codes[1025][0] == (12 << 3) | 3
    assert codes[1024][0] == 0x7E                   # the opening row itself: 4480 / 10


def _random_case(seed, lens, hkv=2, d=32, bs=16, spike_p=0.002):
    rng = np.random.default_rng(seed)
    seqs = []
    for L in lens:
        x = rng.standard_normal((L, 2, hkv, d)).astype(np.float32)
        x *= rng.uniform(0.5, 3.0, size=(1, 2, hkv, 1)).astype(np.float32)
        spikes = rng.random((L, 2, hkv)) < spike_p
        x[spikes] *= 40.0
        seqs.append(bf16(x))
    need = [(L + bs - 1) // bs for L in lens]
    perm = rng.permutation(sum(need) + 3)
    tables, pos = [], 0
    for n in need:
        tables.append(perm[pos:pos + n])
        pos += n
    return seqs, tables, sum(need) + 3


def _append(seqs, tables, nb, calls, hkv=2, d=32, bs=16, fmt=oracle.E4M3):
    """Replay `calls`: a list of calls, each a list of (sequence, t0, t1)."""
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros_like(kc)
    hp = oracle.segment_scale_heads(hkv)
    ks = np.zeros((nb, hp), np.float32)
    vs = np.zeros_like(ks)
    state = np.zeros((len(seqs), 2, hkv, 2), np.float32)
    for call in calls:
        k, v, slots, off, start, rows_state = [], [], [], [0], [], []
        for (r, t0, t1) in call:
            x = seqs[r][t0:t1]
            k.append(x[:, 0])
            v.append(x[:, 1])
            t = np.arange(t0, t1)
            slots.append((tables[r][t // bs] * bs + t % bs).astype(np.int32))
            off.append(off[-1] + (t1 - t0))
            start.append(t0)
            rows_state.append(r)
        st = np.ascontiguousarray(state[rows_state])
        assert oracle.kv_append_quant_segment(np.concatenate(k), np.concatenate(v),
                                              np.concatenate(slots), off, start, fmt, st, kc, vc,
                                              ks, vs, bs) == 0
        state[rows_state] = st
    return kc, vc, ks, vs, state


def test_independent_of_how_tokens_are_split_into_calls():
    lens = [2500, 1024, 7, 3100]
    seqs, tables, nb = _random_case(11, lens)
    whole = [[(r, 0, L) for r, L in enumerate(lens)]]
    ref = _append(seqs, tables, nb, whole)
    # one token per call, the sequences interleaved (a decode loop)
    steps = []
    for t in range(max(lens)):
        steps.append([(r, t, t + 1) for r, L in enumerate(lens) if t < L])
    got = _append(seqs, tables, nb, steps)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)
    # random chunks per sequence, calls mixing sequences
    rng = np.random.default_rng(3)
    cuts = []
    for r, L in enumerate(lens):
        c = np.unique(np.concatenate([[0, L], rng.integers(1, L, size=6)]))
        cuts.append([(r, int(a), int(b)) for a, b in zip(c[:-1], c[1:])])
    calls = []
    while any(cuts):
        calls.append([c.pop(0) for c in cuts if c])
    got = _append(seqs, tables, nb, calls)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


def test_equal_row_absmax_gives_the_token_head_codes():
    """When every row has the same absmax A, every segment's scale is
    A / FMAX, which is also each token's own scale in the per-(token, head)
    mode: the codes must agree with that (separately pinned) mode."""
    rng = np.random.default_rng(5)
    L, hkv, d, bs = 1500, 2, 32, 16
    x = rng.uniform(-3.0, 3.0, size=(L, hkv, d)).astype(np.float32)
    x[:, :, 7] = 3.5                                  # every row's absmax
    kb = bf16(x)
    slots = np.arange(L, dtype=np.int32)
    nb = (L + bs - 1) // bs
    for fmt in (oracle.E4M3, oracle.E5M2, oracle.INT8):
        kc = np.zeros((nb, hkv, bs, d), np.uint8)
        ks = np.zeros((nb, oracle.segment_scale_heads(hkv)), np.float32)
        st = np.zeros((1, 2, hkv, 2), np.float32)
        oracle.kv_append_quant_segment(kb, None, slots, [0, L], [0], fmt, st, kc, None, ks, None,
                                       bs)
        kc2 = np.zeros_like(kc)
        ks2 = np.zeros((nb, hkv, bs, 1), np.float32)
        oracle.kv_append_quant(kb, None, slots, fmt, oracle.SCALE_TOKEN_HEAD, d, kc2, None, ks2,
                               None, bs)
        assert np.array_equal(kc, kc2)
        assert np.array_equal(ks[:, :hkv], ks2[:, :, 0, 0])


def test_scales_never_decrease_along_a_sequence():
    lens = [5000, 2049]
    seqs, tables, nb = _random_case(21, lens, spike_p=0.01)
    kc, vc, ks, vs, state = _append(seqs, tables, nb, [[(r, 0, L) for r, L in enumerate(lens)]])
    for r, L in enumerate(lens):
        for sc in (ks, vs):
            per_page = sc[tables[r], :2]
            assert (np.diff(per_page, axis=0) >= 0).all()
            # constant within each segment of 64 pages
            for s0 in range(0, len(per_page), SEG // 16):
                seg = per_page[s0:s0 + SEG // 16]
                assert (seg == seg[0]).all()


def test_a_new_sequence_restarts_the_running_absmax():
    """A state row reused for a new sequence (position 0) forgets the old one."""
    seqs, tables, nb = _random_case(31, [1200], spike_p=0.0)
    big = seqs[0].copy()
    big[:] = bf16(W.bf16_bits_to_f32(big) * 100.0)
    kc, vc, ks, vs, _ = _append([seqs[0]], tables, nb, [[(0, 0, 1200)]])
    # the same state row first used by a large sequence, then restarted
    kc2 = np.zeros_like(kc)
    vc2 = np.zeros_like(vc)
    ks2 = np.zeros_like(ks)
    vs2 = np.zeros_like(vs)
    st = np.zeros((1, 2, 2, 2), np.float32)
    for x in (big, seqs[0]):
        t = np.arange(1200)
        slots = (tables[0][t // 16] * 16 + t % 16).astype(np.int32)
        oracle.kv_append_quant_segment(x[:, 0], x[:, 1], slots, [0, 1200], [0], oracle.E4M3, st,
                                       kc2, vc2, ks2, vs2, 16)
    for a, b in ((kc, kc2), (vc, vc2), (ks, ks2), (vs, vs2)):
        assert np.array_equal(a, b)


def test_attention_over_segment_scales_matches_sdpa():
    """Decode attention (GQA, 8 query / 2 KV heads) over a segment-scaled
    cache equals float64 SDPA over the cache dequantised through torch's
    float8 type and the page scales."""
    lens = [2100, 333, 1025]
    hkv, d, bs, hq = 2, 32, 16, 8
    seqs, tables, nb = _random_case(41, lens, hkv=hkv, d=d)
    kc, vc, ks, vs, _ = _append(seqs, tables, nb, [[(r, 0, L) for r, L in enumerate(lens)]])
    width = max(len(t) for t in tables)
    bt = np.full((len(lens), width), -1, np.int32)
    for r, t in enumerate(tables):
        bt[r, :len(t)] = t
    rng = np.random.default_rng(9)
    q = bf16(rng.standard_normal((len(lens), hq, d)))
    sm = 1.0 / np.sqrt(d)
    got = oracle.paged_decode_attention(q, kc, vc, ks, vs, bt, np.array(lens, np.int32), bs, hkv,
                                        d, oracle.E4M3, oracle.SCALE_SEGMENT, d, sm)
    G = hq // hkv
    for r, L in enumerate(lens):
        t = np.arange(L)
        blk = bt[r, t // bs]
        off = t % bs

        def deq(cache, scale):
            c = torch.from_numpy(cache[blk, :, off, :].copy()).view(torch.float8_e4m3fn)
            s = torch.from_numpy(scale[blk, :hkv].astype(np.float64))[..., None]
            return (c.to(torch.float64) * s).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qf = torch.from_numpy(W.bf16_bits_to_f32(q[r]).astype(np.float64))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qf, deq(kc, ks), deq(vc, vs),
                                                               scale=sm)[:, 0, :]
        assert np.allclose(got[r], ref.numpy(), rtol=1e-10, atol=1e-12)
