"""The wide GEMMs' mixed item order (GPU).

In prefill-sized launches the single-CTA GEMMs take the items of experts
with one 128-row chunk spread evenly among the items of experts with
several chunks, instead of in expert order (gemm_common.cuh, mix_item; the
scatter kernel writes the reordered tables).  Every output tile is still
computed by one item with the same reduction order, so the layer's output
must be bit-identical with MOE_MIX_ITEMS=0, and both must match the oracle.
Zipf routing over many experts gives both kinds: a few experts with many
chunks, most with one, some with none.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

# (spec, overrides, expected kinds: experts with one chunk, with several)
CASES = [
    ("nvfp4_zipf_small", dict(T=1200, E=96, K=4), (True, True)),
    ("nvfp4_zipf_small", dict(T=1537, E=160, K=6, clamp=0.0), (True, True)),
    ("nvfp4_zipf_small", dict(T=1100, E=8, K=2, logits="normal"), (False, True)),
    ("nvfp4_zipf_small", dict(T=1030, E=256, K=1, logits="normal"), (True, False)),
    ("bf16_small", dict(T=1300, E=64, K=4, logits="zipf1.1"), (True, True)),
]


def _chunks(logits, E, K):
    ids = torch.topk(logits, K, dim=1).indices
    c = torch.bincount(ids.flatten(), minlength=E).numpy()
    return (c + 127) // 128


@pytest.mark.parametrize("name,over,kinds", CASES,
                         ids=["nvfp4-mixed", "nvfp4-K6", "nvfp4-all-multi", "nvfp4-all-single",
                              "bf16-mixed"])
def test_mixed_order_output_is_bit_identical_and_matches_oracle(name, over, kinds, monkeypatch):
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=17)
    ch = _chunks(case["logits"], s["E"], s["K"])
    assert ((ch == 1).sum() > 0, (ch >= 2).sum() > 0) == kinds
    outs = []
    for mix in ("1", "0"):
        monkeypatch.setenv("MOE_MIX_ITEMS", mix)
        layer = make_layer(s, weights=case["weights"])
        outs.append(run_gpu(layer, case["hidden"], case["logits"]).cpu())
        assert layer.status() == 0
        layer.close()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = run_oracle(s, case)
    assert rel_l2(outs[0].float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
