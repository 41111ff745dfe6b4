"""The one-call decode step (append, then attention, with the planner inside
the append's launch) against the two calls it replaces: the same cache bits
and the same output bits, and the oracle's result within tolerance."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    return F


def _chunk(w, kvs, q_len):
    """The last q_len rows of every request, their slots (request-major)."""
    ks, vs, slots = [], [], []
    for b, (k, v) in enumerate(kvs):
        L = int(w.seq_lens[b])
        n = min(q_len, L)
        ks.append(k[L - n:L])
        if v is not None:
            vs.append(v[L - n:L])
        slots.append(W.token_slots(w, b, L - n, L))
    return (np.concatenate(ks), None if w.mla else np.concatenate(vs),
            np.concatenate(slots).astype(np.int32))


def _clone(c):
    kc, vc, ks, vs = c
    kc2, ks2 = kc.clone(), ks.clone()
    if vc is kc:
        return kc2, kc2, ks2, ks2
    return kc2, vc.clone(), ks2, vs.clone()


@pytest.mark.parametrize("idx,q_len", [(1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (1, 3), (5, 2), (2, 4), (3, 2)])
def test_decode_step_equals_append_then_attention(F, idx, q_len):
    from gpu_util import DEV, check_close, gpu_cache, oracle_cache, oracle_attention, \
        oracle_multiquery, to_dev_bf16
    w = W.make_workload(idx, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    base = gpu_cache(w, F, kvs, step=False, back=q_len)
    kn, vn, slots = _chunk(w, kvs, q_len)
    kn_d = to_dev_bf16(kn)
    vn_d = None if vn is None else to_dev_bf16(vn)
    slots_d = torch.from_numpy(slots).to(DEV)
    q = W.queries(w) if q_len == 1 else W.chunk_queries(w, q_len)
    q_d = to_dev_bf16(q)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    kw = dict(fmt=w.fmt, scale_mode=w.scale_mode, group_size=w.group_size,
              head_dim_v=w.head_dim_v, out_dtype=torch.float32)
    # two calls
    a = _clone(base)
    F.kv_append_quant(kn_d, vn_d, slots_d, a[0], None if w.mla else a[1], a[2],
                      None if w.mla else a[3], fmt=w.fmt, scale_mode=w.scale_mode,
                      group_size=w.group_size)
    attend = F.paged_decode_attention if q_len == 1 else F.paged_multiquery_attention
    out_a = attend(q_d, *a, bt, sl, w.n_kv_heads, w.sm_scale, **kw)
    # one call
    b = _clone(base)
    out_b = F.decode_step(kn_d, vn_d, slots_d, q_d, *b, bt, sl, w.n_kv_heads, w.sm_scale, **kw)
    short = bool((w.seq_lens < q_len).any())
    assert F.get_device_error() == (4 if short else 0)
    for x, y, name in zip(a, b, ("k codes", "v codes", "k scales", "v scales")):
        assert torch.equal(x, y), name
    assert torch.equal(out_a, out_b), "outputs differ"
    # and against the oracle
    o = oracle_cache(w, kvs)
    ref = oracle_attention(w, q, o) if q_len == 1 else oracle_multiquery(w, q, o, q_len)
    check_close(out_b.cpu().numpy().astype(np.float64), ref, bf16_out=False,
                what=f"cfg{idx} q_len={q_len}")


def test_decode_step_with_nothing_to_append(F):
    """num_new_tokens = 0: the step is the attention alone."""
    from gpu_util import DEV, gpu_cache, to_dev_bf16
    w = W.make_workload(1, "small")
    c = gpu_cache(w, F)
    q_d = to_dev_bf16(W.queries(w))
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    empty = torch.zeros((0, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16, device=DEV)
    kw = dict(fmt=w.fmt, scale_mode=w.scale_mode, out_dtype=torch.float32)
    ref = F.paged_decode_attention(q_d, *c, bt, sl, w.n_kv_heads, w.sm_scale, **kw)
    got = F.decode_step(empty, empty, torch.zeros(0, dtype=torch.int32, device=DEV), q_d, *c,
                        bt, sl, w.n_kv_heads, w.sm_scale, **kw)
    assert torch.equal(ref, got)
    assert F.get_device_error() == 0


def test_decode_step_replays_from_a_cuda_graph(F):
    """The step captured once in a CUDA graph (with its host-to-device input
    copy and device-to-host output copy) and replayed: the output equals an
    eager call's bit for bit, and replays pick up new inputs."""
    from gpu_util import DEV, gpu_cache, to_dev_bf16
    w = W.make_workload(2, "small")
    kvs = [W.request_kv(w, b) for b in range(w.batch)]
    c = gpu_cache(w, F, kvs, step=False)
    kn = np.stack([k[-1] for k, _ in kvs])
    vn = np.stack([v[-1] for _, v in kvs])
    q = W.queries(w)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    slots = torch.from_numpy(W.step_slots(w)).to(DEV)
    kw = dict(fmt=w.fmt, scale_mode=w.scale_mode, out_dtype=torch.float32)
    ws = torch.empty(F.decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                              w.head_dim, w.block_size, w.max_blocks),
                     dtype=torch.uint8, device=DEV)
    # eager reference (on a copy of the cache)
    ce = tuple(t.clone() for t in c)
    ref = F.decode_step(to_dev_bf16(kn), to_dev_bf16(vn), slots, to_dev_bf16(q), *ce, bt, sl,
                        w.n_kv_heads, w.sm_scale, workspace=ws, **kw)
    # graph: pinned inputs -> device, step, device -> pinned output
    q_h = torch.from_numpy(q.view(np.int16)).pin_memory()
    q_d = torch.empty(q_h.shape, dtype=torch.int16, device=DEV)
    kn_d, vn_d = to_dev_bf16(kn), to_dev_bf16(vn)
    out = torch.empty_like(ref)
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()

    def body():
        q_d.copy_(q_h, non_blocking=True)
        F.decode_step(kn_d, vn_d, slots, q_d.view(torch.bfloat16), *c, bt, sl, w.n_kv_heads,
                      w.sm_scale, out=out, workspace=ws, **kw)
        out_h.copy_(out, non_blocking=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref.cpu())
    assert F.get_device_error() == 0
    # new query values through the same pinned buffer
    q_h.copy_(torch.from_numpy((q ^ np.uint16(0x8000)).view(np.int16)))   # q -> -q
    g.replay()
    torch.cuda.synchronize()
    ce2 = tuple(t.clone() for t in c)
    ref2 = F.decode_step(to_dev_bf16(kn), to_dev_bf16(vn), slots,
                         to_dev_bf16(q ^ np.uint16(0x8000)), *ce2, bt, sl, w.n_kv_heads,
                         w.sm_scale, workspace=ws, **kw)
    assert torch.equal(out_h, ref2.cpu())
    assert not torch.equal(ref2, ref)
