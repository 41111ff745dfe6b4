"""GPU parity of the latent (MLA) decode over every FP8 code value.

The caches are written directly, not through the append: codes are drawn
from all finite E4M3 / E5M2 bytes, or only from the subnormal and smallest
normal ones, with a free-ranging fp32 scale per (token, 64-dim group).  The
decode's conversion of each code (sign, exponent, mantissa, subnormals) and
its scaling are checked against the oracle's format definitions
("DeepSeek V4 950: whole-network FP8 dataflow", 2kiu.com/news/4508674,
sec. 2.2: one cached latent per token, one scale per latent group)."""
import numpy as np
import pytest
import torch

from fp8_quantised_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4, E5, TG = W.E4M3, W.E5M2, W.SCALE_TOKEN_GROUP


def finite_codes(fmt):
    b = np.arange(256, dtype=np.uint8)
    keep = (b & 0x7F) != 0x7F if fmt == E4 else (b & 0x7C) != 0x7C
    return b[keep]


def small_codes(fmt):
    """Codes with exponent field 0 (subnormal) or 1 (smallest normal)."""
    b = finite_codes(fmt)
    e = (b >> 3) & 0xF if fmt == E4 else (b >> 2) & 0x1F
    return b[e <= 1]


# fmt, query heads, code set
CASES = [(E4, 64, "all"), (E4, 128, "small"), (E5, 128, "all"), (E5, 64, "small")]


@pytest.fixture(scope="module")
def F():
    import fp8_quantised_paged_gb300 as F
    F.get_device_error()
    F.set_decode_workers(0)
    yield F
    F.set_decode_workers(0)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{'e4m3' if c[0] == E4 else 'e5m2'}"
                                                       f"_{c[1]}_heads_{c[2]}_codes")
def test_latent_decode_over_every_code(F, case):
    from gpu_util import DEV, check_close, oracle_attention, to_dev_bf16
    fmt, hq, which = case
    w = W.make_shape_case(f"codes_{which}", [300, 129, 64], hq, 1, 576, 64, fmt, TG,
                          seed=7100 + CASES.index(case))
    rng = np.random.default_rng(7200 + CASES.index(case))
    pool = finite_codes(fmt) if which == "all" else small_codes(fmt)
    kc = rng.choice(pool, size=(w.num_blocks, 1, 64, 576)).astype(np.uint8)
    # scales 2^U(-2, 2) (a full 24-bit mantissa) over the largest code of the
    # set, so that the values, and the outputs, are of order one
    top = np.abs(torch.from_numpy(pool).view(
        torch.float8_e4m3fn if fmt == E4 else torch.float8_e5m2).float().numpy()).max()
    ks = (np.exp2(rng.uniform(-2.0, 2.0, size=(w.num_blocks, 1, 64, 9))) / top
          ).astype(np.float32)
    q = W.queries(w)
    ref = oracle_attention(w, q, (kc, kc, ks, ks))
    kd = torch.from_numpy(kc).to(DEV)
    sd = torch.from_numpy(ks).to(DEV)
    try:
        for workers in (1, 0):
            F.set_decode_workers(workers)
            out = F.paged_decode_attention(to_dev_bf16(q), kd, kd, sd, sd,
                                           torch.from_numpy(w.block_tables).to(DEV),
                                           torch.from_numpy(w.seq_lens).to(DEV), 1, w.sm_scale,
                                           fmt=fmt, scale_mode=TG, group_size=64, head_dim_v=512,
                                           out_dtype=torch.float32)
            got = out.cpu().numpy().astype(np.float64)
            check_close(got, ref, bf16_out=False, what=f"{w.name} workers={workers}")
    finally:
        F.set_decode_workers(0)
    assert F.get_device_error() == 0
