"""The Python example in README.md runs as written (prefill append, then one
fused decode step) and its output matches the oracle on the same cache."""
import os
import re

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example_source() -> str:
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1, "README.md should hold exactly one Python example"
    return blocks[0]


def test_readme_example_runs_and_matches_the_oracle():
    import fp8_quantised_paged_gb300 as F
    from fp8_quantised_paged_gb300 import workloads as W
    from gpu_util import check_close
    torch.manual_seed(0)
    ns = {}
    exec(compile(_example_source(), "README.md example", "exec"), ns)
    out = ns["out"]
    assert out.shape == (ns["B"], ns["Hq"], ns["D"]) and out.dtype == torch.bfloat16
    assert F.get_device_error() == 0
    # the oracle on the cache the example built
    kc, vc = ns["k_cache"].cpu().numpy(), ns["v_cache"].cpu().numpy()
    ks, vs = ns["k_scale"].cpu().numpy(), ns["v_scale"].cpu().numpy()
    q = ns["q"].cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.paged_decode_attention(
        q, kc, vc, ks, vs, ns["block_tables"].cpu().numpy(), ns["seq_lens"].cpu().numpy(),
        ns["bs"], ns["Hkv"], ns["D"], W.E4M3, W.SCALE_TOKEN_HEAD, ns["D"], ns["D"] ** -0.5)
    check_close(out.float().cpu().numpy().astype(np.float64), ref, bf16_out=True,
                what="README example")
