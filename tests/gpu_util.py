"""Helpers shared by the GPU parity tests: fill a cache on the GPU through
the library and the same cache on the host through the oracle, from the
same seeded inputs, and compare within the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp8_quantised_paged_gb300 import workloads as W

DEV = "cuda:0"

# Attention tolerance: max-abs 4e-3 and rel-L2 2e-3 against the FP64 oracle
# computed from the same codes and scales.  A bf16 output adds what rounding
# the exact result to bf16 alone costs: half a bf16 ulp of the reference per
# element, and the norm of (bf16(ref) - ref) to the rel-L2 bound.
ATOL = 4e-3
RTOL_L2 = 2e-3


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 8)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """x rounded to fp32, then to bf16 (nearest, ties to even), as float64."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    return W.bf16_bits_to_f32(W.f32_to_bf16_bits(x32)).astype(np.float64)


def check_close(got, ref, bf16_out=True, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + (half_ulp_bf16(ref) if bf16_out else 0.0)
    worst = np.argmax(err - bound)
    assert (err <= bound).all(), (f"{what}: max excess {float((err - bound).flat[worst]):.3g} at "
                                  f"{np.unravel_index(worst, err.shape)}; max abs "
                                  f"{err.max():.3g}")
    den = np.linalg.norm(ref)
    allow = np.linalg.norm(round_bf16(ref) - ref) if bf16_out else 0.0
    diff = np.linalg.norm(got - ref)
    rel = diff / den if den > 0 else diff
    assert diff <= RTOL_L2 * den + allow, (f"{what}: rel-L2 {rel:.3g} (bound {RTOL_L2:g} + "
                                           f"bf16 rounding {allow / max(den, 1e-300):.3g})")
    return float(err.max()), float(rel)


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def n_scale_groups(w):
    grouped = (W.SCALE_TOKEN_GROUP, W.SCALE_MX_BLOCK)
    return w.head_dim // w.group_size if w.scale_mode in grouped else 1


def scale_dtype(w, torch_side=True):
    """E8M0 bytes for the MX block mode, fp32 scales otherwise."""
    if w.scale_mode == W.SCALE_MX_BLOCK:
        return torch.uint8 if torch_side else np.uint8
    return torch.float32 if torch_side else np.float32


def gpu_cache(w, F, kvs=None, step=True, back=1):
    """Prefill all but the last `back` tokens of every request with one
    append call, then (step=True, back=1) append each request's last token
    with a second call (the decode step).  Returns device tensors
    (k_cache, v_cache, k_scale, v_scale)."""
    nb, hkv, bs, d = w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device=DEV)
    vc = None if w.mla else torch.zeros_like(kc)
    if kvs is None:
        kvs = [W.request_kv(w, b) for b in range(w.batch)]
    if w.scale_mode == W.SCALE_SEGMENT:
        return _gpu_cache_segment(w, F, kvs, kc, vc, step, back)
    if w.scale_mode == W.SCALE_CHANNEL_STATIC:
        ks = F.kv_channel_scales(to_dev_bf16(np.concatenate([k for k, _ in kvs])), w.fmt)
        vs = F.kv_channel_scales(to_dev_bf16(np.concatenate([v for _, v in kvs])), w.fmt)
    else:
        ks = torch.zeros((nb, hkv, bs, n_scale_groups(w)), dtype=scale_dtype(w), device=DEV)
        vs = None if w.mla else torch.zeros_like(ks)
    pk, pv, ps = [], [], []
    for b, (k, v) in enumerate(kvs):
        L = int(w.seq_lens[b])
        n = max(L - back, 0)
        pk.append(k[:n])
        if v is not None:
            pv.append(v[:n])
        ps.append(W.token_slots(w, b, 0, n))
    F.kv_append_quant(to_dev_bf16(np.concatenate(pk)),
                      None if w.mla else to_dev_bf16(np.concatenate(pv)),
                      torch.from_numpy(np.concatenate(ps)).to(DEV), kc, vc, ks, vs, fmt=w.fmt,
                      scale_mode=w.scale_mode, group_size=w.group_size)
    if not step:
        return (kc, kc, ks, ks) if w.mla else (kc, vc, ks, vs)
    sk = np.stack([k[-1] for k, _ in kvs])
    sv = None if w.mla else np.stack([v[-1] for _, v in kvs])
    F.kv_append_quant(to_dev_bf16(sk), None if w.mla else to_dev_bf16(sv),
                      torch.from_numpy(W.step_slots(w)).to(DEV), kc, vc, ks, vs, fmt=w.fmt,
                      scale_mode=w.scale_mode, group_size=w.group_size)
    if w.mla:
        vc, vs = kc, ks
    return kc, vc, ks, vs


def _gpu_cache_segment(w, F, kvs, kc, vc, step, back):
    """The segment-scale cache: one prefill call over every request (all but
    its last `back` tokens), then (step=True) one decode-step call appending
    each request's last token at its position, with the running state
    carried between the calls."""
    nb, hkv = w.num_blocks, w.n_kv_heads
    hp = F.segment_scale_heads(hkv)
    ks = torch.zeros((nb, hp), dtype=torch.float32, device=DEV)
    vs = None if w.mla else torch.zeros_like(ks)
    state = torch.zeros((w.batch, 2, hkv, 2), dtype=torch.float32, device=DEV)
    lens = [int(L) for L in w.seq_lens]
    n = [max(L - back, 0) for L in lens]

    def call(rows_k, rows_v, slots, counts, starts):
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        F.kv_append_quant_segment(to_dev_bf16(np.concatenate(rows_k)),
                                  None if w.mla else to_dev_bf16(np.concatenate(rows_v)),
                                  torch.from_numpy(np.concatenate(slots).astype(np.int32)).to(DEV),
                                  torch.from_numpy(off).to(DEV),
                                  torch.from_numpy(np.asarray(starts, np.int32)).to(DEV),
                                  kc, vc, ks, vs, state, fmt=w.fmt)
    call([k[:m] for (k, _), m in zip(kvs, n)],
         None if w.mla else [v[:m] for (_, v), m in zip(kvs, n)],
         [W.token_slots(w, b, 0, m) for b, m in enumerate(n)], n, [0] * w.batch)
    if step:
        call([k[m:L] for (k, _), m, L in zip(kvs, n, lens)],
             None if w.mla else [v[m:L] for (_, v), m, L in zip(kvs, n, lens)],
             [W.token_slots(w, b, m, L) for b, (m, L) in enumerate(zip(n, lens))],
             [L - m for m, L in zip(n, lens)], n)
    if w.mla:
        return kc, kc, ks, ks
    return kc, vc, ks, vs


def oracle_cache(w, kvs=None, requests=None):
    """The same cache built by the oracle on the host (all requests, or only
    `requests`; static channel scales always from every request)."""
    nb, hkv, bs, d = w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = None if w.mla else np.zeros_like(kc)
    if kvs is None:
        kvs = [W.request_kv(w, b) for b in range(w.batch)]
    if w.scale_mode == W.SCALE_SEGMENT:
        hp = oracle.segment_scale_heads(hkv)
        ks = np.zeros((nb, hp), np.float32)
        vs = None if w.mla else np.zeros_like(ks)
        for b, (k, v) in enumerate(kvs):
            if requests is not None and b not in requests:
                continue
            L = int(w.seq_lens[b])
            st = np.zeros((1, 2, hkv, 2), np.float32)
            assert oracle.kv_append_quant_segment(k, v, W.token_slots(w, b, 0, L), [0, L], [0],
                                                  w.fmt, st, kc, vc, ks, vs, bs) == 0
        return (kc, kc, ks, ks) if w.mla else (kc, vc, ks, vs)
    if w.scale_mode == W.SCALE_CHANNEL_STATIC:
        ks = oracle.kv_channel_scales(np.concatenate([k for k, _ in kvs]), w.fmt)
        vs = oracle.kv_channel_scales(np.concatenate([v for _, v in kvs]), w.fmt)
    else:
        ks = np.zeros((nb, hkv, bs, n_scale_groups(w)), scale_dtype(w, torch_side=False))
        vs = None if w.mla else np.zeros_like(ks)
    for b, (k, v) in enumerate(kvs):
        if requests is not None and b not in requests:
            continue
        slots = W.token_slots(w, b, 0, int(w.seq_lens[b]))
        assert oracle.kv_append_quant(k, v, slots, w.fmt, w.scale_mode, w.group_size, kc, vc,
                                      ks, vs, bs) == 0
    if w.mla:
        vc, vs = kc, ks
    return kc, vc, ks, vs


def oracle_attention(w, q, caches, rows=None):
    kc, vc, ks, vs = caches
    return oracle.paged_decode_attention(q, kc, vc, ks, vs, w.block_tables, w.seq_lens,
                                         w.block_size, w.n_kv_heads, w.head_dim_v, w.fmt,
                                         w.scale_mode, w.group_size, w.sm_scale, rows=rows)


def gpu_attention(w, F, q_bits, caches, out_dtype=torch.bfloat16):
    kc, vc, ks, vs = caches
    out = F.paged_decode_attention(to_dev_bf16(q_bits), kc, vc, ks, vs,
                                   torch.from_numpy(w.block_tables).to(DEV),
                                   torch.from_numpy(w.seq_lens).to(DEV), w.n_kv_heads,
                                   w.sm_scale, fmt=w.fmt, scale_mode=w.scale_mode,
                                   group_size=w.group_size, head_dim_v=w.head_dim_v,
                                   out_dtype=out_dtype)
    return out.float().cpu().numpy().astype(np.float64)


def expand_multiquery(w, q_len):
    """A causal chunk as plain decode rows: (request b, query i) becomes one
    virtual request with b's block table and visible length
    seq_lens[b] - (q_len - 1 - i), floored at 0."""
    tables = np.repeat(w.block_tables, q_len, axis=0)
    i = np.tile(np.arange(q_len), w.batch)
    lens = np.repeat(w.seq_lens.astype(np.int64), q_len) - (q_len - 1 - i)
    return tables, np.maximum(lens, 0).astype(np.int32)


def oracle_multiquery(w, q_chunk, caches, q_len):
    """Oracle rows of the chunk: [B, q_len, Hq, Dv]."""
    kc, vc, ks, vs = caches
    tables, lens = expand_multiquery(w, q_len)
    q = q_chunk.reshape(w.batch * q_len, w.n_q_heads, w.head_dim)
    out = oracle.paged_decode_attention(q, kc, vc, ks, vs, tables, lens, w.block_size,
                                        w.n_kv_heads, w.head_dim_v, w.fmt, w.scale_mode,
                                        w.group_size, w.sm_scale)
    return out.reshape(w.batch, q_len, w.n_q_heads, w.head_dim_v)


def gpu_multiquery(w, F, q_chunk, caches, out_dtype=torch.bfloat16):
    kc, vc, ks, vs = caches
    out = F.paged_multiquery_attention(to_dev_bf16(q_chunk), kc, vc, ks, vs,
                                       torch.from_numpy(w.block_tables).to(DEV),
                                       torch.from_numpy(w.seq_lens).to(DEV), w.n_kv_heads,
                                       w.sm_scale, fmt=w.fmt, scale_mode=w.scale_mode,
                                       group_size=w.group_size, head_dim_v=w.head_dim_v,
                                       out_dtype=out_dtype)
    return out.float().cpu().numpy().astype(np.float64)
