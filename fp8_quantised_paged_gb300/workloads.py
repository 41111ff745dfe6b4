"""Seeded synthetic workloads for FP8 paged decode attention.

This module only makes inputs: shapes, block tables, slot numbers, sequence
lengths and bf16 bit patterns drawn from seeded numpy generators.  It holds
none of the method's arithmetic (no scale, no FP8 rounding, no attention),
so both the CUDA path and the CPU oracle can take their inputs from it.

Every request draws its K/V rows from its own generator (seeded by the
workload seed and the request index), so any request can be regenerated on
its own to check sampled outputs of a full-size run.

The five workloads follow the shapes the source pages discuss:
  1 tiny GQA       - a small correctness case (4 q heads / 1 KV head, D=64).
  2 Llama-3-70B    - one decode layer, 64 q / 8 KV heads, D=128, 16K context
                     ("Llama 3 70B FP8 deployment", dpshk.com/news/5605006,
                     sec. 1.2 and sec. 2.2).
  3 long split-K   - 128K context, 4 requests (same page, sec. 2.2 table of
                     context lengths).
  4 ragged E5M2    - 64 requests with log-uniform lengths, E5M2 codes and
                     static per-channel scales ("DeepSeek V4 950",
                     2kiu.com/news/4508674, sec. 2.1 and sec. 3.2; paged KV
                     per "DeepSeek-V4.1 512K", hotelren.com/news/5711065,
                     sec. 3.3).
  5 MLA latent     - one shared 576-dim latent (512 + 64 rope) per token,
                     128 query heads, one scale per 64-dim group
                     ("DeepSeek V4 950", sec. 2.2).
The pages measure on serving traces (ShareGPT, long-document QA) that are
not available here; these seeded inputs stand in for their shapes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

E4M3, E5M2, INT8 = 0, 1, 2
SCALE_TOKEN_HEAD, SCALE_CHANNEL_STATIC, SCALE_TOKEN_GROUP, SCALE_MX_BLOCK = 0, 1, 2, 3
SCALE_SEGMENT = 4  # one scale per (page, KV head), refreshed every 1024 tokens


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    index: int
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    head_dim_v: int
    block_size: int
    fmt: int
    scale_mode: int
    group_size: int
    sm_scale: float
    seq_lens: np.ndarray          # int32 [B], includes the token appended this step
    block_tables: np.ndarray      # int32 [B, max_blocks]; unused entries are -1
    num_blocks: int
    seed: int
    mla: bool = False
    params: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    def describe(self) -> dict:
        return {"workload": self.name, "batch": self.batch, "n_q_heads": self.n_q_heads,
                "n_kv_heads": self.n_kv_heads, "head_dim": self.head_dim,
                "head_dim_v": self.head_dim_v, "block_size": self.block_size,
                "kv_fmt": {E4M3: "e4m3", E5M2: "e5m2", INT8: "int8"}[self.fmt],
                "scale_mode": ["token_head", "channel_static", "token_group",
                               f"mx_block_{self.group_size}", "segment_1024"][self.scale_mode],
                "kv_tokens": self.total_tokens, "num_blocks": self.num_blocks}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def _tables(rng, lens, bs, pool, mode):
    """Hand out physical blocks: a seeded permutation of the pool ("perm")
    or a uniform draw without replacement ("draw"), in request order."""
    need = [int(math.ceil(L / bs)) for L in lens]
    total = sum(need)
    assert total <= pool, (total, pool)
    if mode == "perm":
        ids = rng.permutation(pool)[:total]
    else:
        ids = rng.choice(pool, size=total, replace=False)
    width = max(1, max(need))
    bt = np.full((len(lens), width), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = ids[pos:pos + n]
        pos += n
    return bt


# Full-size recipes (the shapes each workload is quoted on) and the small
# variants used where the oracle must cover every output.
_FULL = {
    1: dict(batch=4, hq=4, hkv=1, d=64, bs=16),
    2: dict(batch=12, hq=64, hkv=8, d=128, bs=16, L=16384),
    3: dict(batch=4, hq=64, hkv=8, d=128, bs=16, L=131072),
    4: dict(batch=64, hq=32, hkv=8, d=128, bs=32, Lmax=32768),
    5: dict(batch=32, hq=128, hkv=1, d=576, dv=512, bs=64, L=8192),
}


def make_workload(index: int, size: str = "full", seed: int | None = None) -> Workload:
    """Build workload `index` (1..5).  size="full" is the quoted shape;
    size="small" keeps heads, dims, format and block size but shortens and
    raggeds the sequences so the FP64 oracle can check every output."""
    assert index in _FULL and size in ("full", "small")
    f = _FULL[index]
    seed = 1000 + index if seed is None else seed
    g = _rng(seed, 0)
    B, hq, hkv, d, bs = f["batch"], f["hq"], f["hkv"], f["d"], f["bs"]
    dv = f.get("dv", d)
    params: dict = {}
    if index == 1:
        lens = g.integers(17, 201, size=B)
        pool, mode = 64, "perm"
        fmt, smode, gs, sm = E4M3, SCALE_TOKEN_HEAD, d, 1.0 / 8.0
        # one channel in 64 (1%, rounded up) per (K/V, kv head) is scaled x20
        params["hot_channels"] = g.integers(0, d, size=(2, hkv))
    elif index in (2, 3):
        if size == "full":
            lens = np.full(B, f["L"])
        else:
            B = 3
            lens = np.array([1000, 517, 33])
        need = int(sum(math.ceil(L / bs) for L in lens))
        if index == 2:
            pool, mode = (need, "perm") if size == "full" else (int(need * 1.25), "perm")
            params["std"] = g.uniform(0.5, 4.0, size=(2, hkv))
            params["outlier_p"], params["outlier_x"] = 0.001, 50.0
        else:
            pool, mode = int(math.ceil(need * 1.25)), "draw"
            params["std"] = np.ones((2, hkv))
            params["outlier_p"], params["outlier_x"] = 0.01, 30.0
        fmt, smode, gs, sm = E4M3, SCALE_TOKEN_HEAD, d, 1.0 / math.sqrt(d)
    elif index == 4:
        if size == "full":
            u = g.uniform(0.0, math.log(f["Lmax"]), size=B)
            lens = np.clip(np.rint(np.exp(u)), 1, f["Lmax"])
        else:
            B = 6
            lens = np.array([1, 31, 32, 33, 700, 95])
        pool = int(sum(math.ceil(L / bs) for L in lens))
        mode = "perm"
        fmt, smode, gs, sm = E5M2, SCALE_CHANNEL_STATIC, d, 1.0 / math.sqrt(d)
        params["heavy_heads"] = g.choice(hkv, size=2, replace=False)
    else:
        if size == "full":
            lens = np.full(B, f["L"])
            pool = B * (f["L"] // bs)
        else:
            B = 2
            lens = np.array([300, 129])
            pool = int(sum(math.ceil(L / bs) for L in lens)) + 3
        mode = "perm"
        fmt, smode, gs, sm = E4M3, SCALE_TOKEN_GROUP, 64, 1.0 / math.sqrt(192.0)
        params["group_std"] = g.uniform(0.5, 3.0, size=d // 64)
    lens = np.asarray(lens, dtype=np.int32)
    bt = _tables(g, lens, bs, pool, mode)
    names = {1: "tiny_gqa", 2: "llama3_70b_layer_decode", 3: "long_context_split_k",
             4: "ragged_e5m2_static_channel", 5: "mla_latent_decode"}
    name = names[index] + ("" if size == "full" else "_small")
    return Workload(index=index, name=name, batch=B, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                    head_dim_v=dv, block_size=bs, fmt=fmt, scale_mode=smode, group_size=gs,
                    sm_scale=sm, seq_lens=lens, block_tables=bt, num_blocks=pool, seed=seed,
                    mla=(index == 5), params=params)


def make_shape_case(name: str, batch_lens, hq: int, hkv: int, d: int, bs: int, fmt: int,
                    scale_mode: int, seed: int, dv: int | None = None,
                    group_size: int | None = None) -> Workload:
    """A small seeded workload of any supported shape (parity matrix cases):
    the given ragged lengths, a permuted pool with 2 spare blocks, values
    N(0, 1) times a per-(K/V, kv head) spread U(0.5, 2) with 0.5% outliers x20.
    d = 576 builds the shared-latent layout (one latent, 64-dim groups)."""
    g = _rng(seed, 0)
    lens = np.asarray(batch_lens, dtype=np.int32)
    mla = d == 576
    pool = int(sum(math.ceil(int(L) / bs) for L in lens)) + 2
    bt = _tables(g, lens, bs, pool, "perm")
    params = {"std": g.uniform(0.5, 2.0, size=(2, hkv)), "outlier_p": 0.005, "outlier_x": 20.0}
    dk_eff = 192.0 if mla else float(d)
    return Workload(index=0, name=name, batch=len(lens), n_q_heads=hq, n_kv_heads=hkv,
                    head_dim=d, head_dim_v=(dv or (512 if mla else d)), block_size=bs, fmt=fmt,
                    scale_mode=scale_mode, group_size=group_size or (64 if mla else d),
                    sm_scale=1.0 / math.sqrt(dk_eff), seq_lens=lens, block_tables=bt,
                    num_blocks=pool, seed=seed, mla=mla, params=params)


def request_kv(w: Workload, b: int):
    """bf16 bits of request b's K and V rows, [L_b, Hkv, D] each (V is None
    for the MLA workload, whose single latent serves as K and V)."""
    L = int(w.seq_lens[b])
    hkv, d = w.n_kv_heads, w.head_dim
    rng = _rng(w.seed, 1, b)
    shape = (L, hkv, d)
    outs = []
    for which in range(1 if w.mla else 2):
        if w.index == 1:
            x = rng.standard_normal(shape, dtype=np.float32)
            hot = w.params["hot_channels"][which]
            for h in range(hkv):
                x[:, h, hot[h]] *= 20.0
        elif w.index in (0, 2, 3):
            x = rng.standard_normal(shape, dtype=np.float32)
            x *= w.params["std"][which].astype(np.float32)[None, :, None]
            n = x.size
            k = int(rng.binomial(n, w.params["outlier_p"]))
            idx = rng.integers(0, n, size=k)
            x.reshape(-1)[idx] *= np.float32(w.params["outlier_x"])
        elif w.index == 4:
            x = rng.standard_normal(shape, dtype=np.float32)
            for h in w.params["heavy_heads"]:
                x[:, h, :] = rng.standard_t(3.0, size=(L, d)).astype(np.float32)
        else:
            x = rng.standard_normal(shape, dtype=np.float32)
            gstd = np.repeat(w.params["group_std"].astype(np.float32), 64)
            x *= gstd[None, None, :]
        outs.append(f32_to_bf16_bits(x))
    return (outs[0], None) if w.mla else (outs[0], outs[1])


def queries(w: Workload) -> np.ndarray:
    """bf16 bits of the step's queries, [B, Hq, Dk], ~N(0, 1)."""
    rng = _rng(w.seed, 2)
    return f32_to_bf16_bits(rng.standard_normal((w.batch, w.n_q_heads, w.head_dim),
                                                dtype=np.float32))


def chunk_queries(w: Workload, q_len: int) -> np.ndarray:
    """bf16 bits of a causal chunk's queries, [B, q_len, Hq, Dk], ~N(0, 1)
    (the chunk is the last q_len cached tokens of each request)."""
    rng = _rng(w.seed, 5, q_len)
    return f32_to_bf16_bits(rng.standard_normal((w.batch, q_len, w.n_q_heads, w.head_dim),
                                                dtype=np.float32))


def token_slots(w: Workload, b: int, t0: int, t1: int) -> np.ndarray:
    """Slot numbers (block id * block_size + offset) of tokens [t0, t1) of
    request b under its block table."""
    t = np.arange(t0, t1, dtype=np.int64)
    blk = w.block_tables[b, t // w.block_size].astype(np.int64)
    return (blk * w.block_size + t % w.block_size).astype(np.int32)


def step_slots(w: Workload) -> np.ndarray:
    """Slots of the one token each request appends this step (its last)."""
    return np.array([token_slots(w, b, int(L) - 1, int(L))[0] for b, L in enumerate(w.seq_lens)],
                    dtype=np.int32)


def step_kv(w: Workload):
    """bf16 bits of the appended token's K/V rows, [B, Hkv, D] each."""
    ks, vs = [], []
    for b in range(w.batch):
        k, v = request_kv(w, b)
        ks.append(k[-1])
        if v is not None:
            vs.append(v[-1])
    return np.stack(ks), (np.stack(vs) if vs else None)
