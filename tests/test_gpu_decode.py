"""The single-launch decode layer (GPU).

For T <= 16 one persistent kernel runs the routing, the expert tables, the
GEMM1 input quantisation, both GEMMs and the combine.  Its CTAs claim work
from counters in order, so a launch with fewer CTAs than SMs (or CTAs that
are not all resident) still completes.  Checked against the oracle and
against the three-launch path (MOE_SINGLE_LAUNCH=0) bit for bit (the same
MMAs, epilogues and combine order), across repeated forwards of varying T
(the counters are reset by the kernel), with a launch cap of a few CTAs, for
every format and both activations; plus the bounded waits of the kernel.
"""
import time

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("nvfp4_small", dict(T=16, E=40, K=8)),
    ("nvfp4_small", dict(T=1, E=300, K=8)),
    ("mxfp8_small", dict(T=9, E=20, K=4)),
    ("bf16_small", dict(T=12)),
    ("tiny_bf16", dict()),
    ("nvfp4_small", dict(T=7, act="relu2")),
    ("mxfp8_small", dict(T=5, E=6, K=2, act="relu2")),
]


@pytest.mark.parametrize("name,over", CASES,
                         ids=["nvfp4-T16", "nvfp4-T1", "mxfp8", "bf16", "tiny", "nvfp4-relu2",
                              "mxfp8-relu2"])
def test_single_launch_matches_oracle_and_three_launch_path(name, over, monkeypatch):
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=83)
    ref = run_oracle(s, case, intermediates=True)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    from moe_expert_layer_histogram_gb300 import moe_last_launch_count
    assert moe_last_launch_count(layer.handle) == 1
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert layer.status() == 0
    assert np.array_equal(ids, ref["ids"]) and np.array_equal(off, ref["offsets"])
    assert np.array_equal(perm, ref["perm"])
    assert np.max(np.abs(w - ref["w"])) <= 1e-6
    if s["fmt"] != "bf16":
        codes, sf = (t.cpu().numpy() for t in layer.act_quant())
        assert np.array_equal(sf, ref["xq_sf"]) and np.array_equal(codes, ref["xq_codes"])
    h, y = (t.cpu().numpy() for t in layer.intermediates())
    assert rel_l2(h, ref["h"]) <= TOL[s["fmt"]], "GEMM2 input"
    assert rel_l2(y, ref["y"]) <= TOL[s["fmt"]], "GEMM2 output"
    got = out.cpu()
    assert rel_l2(got.float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
    layer.close()
    monkeypatch.setenv("MOE_SINGLE_LAUNCH", "0")
    layer = make_layer(s, weights=case["weights"])
    out3 = run_gpu(layer, case["hidden"], case["logits"]).cpu()
    assert moe_last_launch_count(layer.handle) == 3
    assert layer.status() == 0
    layer.close()
    assert torch.equal(got, out3)


def test_repeated_forwards_of_varying_size_reset_the_counters():
    s = workloads.spec("nvfp4_small", T=40, E=24, K=6)
    case = workloads.make_case(s, seed=89)
    layer = make_layer(s, max_tokens=40, weights=case["weights"])
    from moe_expert_layer_histogram_gb300 import moe_last_launch_count
    for T in (1, 16, 7, 40, 3, 16, 16):
        c = dict(case, hidden=case["hidden"][:T], logits=case["logits"][:T])
        ref = run_oracle(s, c)
        out = run_gpu(layer, c["hidden"], c["logits"])
        assert moe_last_launch_count(layer.handle) == (1 if T <= 16 else 6)
        assert layer.status() == 0
        assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"], T
    layer.close()


@pytest.mark.parametrize("ctas", [1, 3, 37])
def test_single_launch_with_few_ctas(ctas):
    # the work is claimed in order, so any number of CTAs completes it
    s = workloads.spec("nvfp4_small", T=13, E=30, K=8)
    case = workloads.make_case(s, seed=97)
    ref = run_oracle(s, case)
    layer = make_layer(s, weights=case["weights"], max_ctas=ctas)
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    layer.close()


def test_single_launch_in_place_and_graph_replay():
    from moe_expert_layer_histogram_gb300 import moe_forward
    s = workloads.spec("mxfp8_small", T=10)
    case = workloads.make_case(s, seed=101)
    layer = make_layer(s, weights=case["weights"])
    ref = run_gpu(layer, case["hidden"], case["logits"]).clone()
    # the output may overwrite the input: every input row is quantised before
    # the first GEMM reads it, and the combine writes after the last GEMM
    buf = case["hidden"].cuda().clone()
    moe_forward(layer.handle, buf, case["logits"].cuda(), buf, s["T"],
                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)
    hid, lg = case["hidden"].cuda(), case["logits"].cuda()
    out = torch.empty_like(hid)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe_forward(layer.handle, hid, lg, out, s["T"], torch.cuda.current_stream().cuda_stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert layer.status() == 0
    layer.close()


def test_single_launch_wait_runs_out_and_is_reported():
    s = workloads.spec("nvfp4_small", T=8)
    case = workloads.make_case(s, seed=103)
    layer = make_layer(s, weights=case["weights"], test_stall_gemm=1)
    t0 = time.perf_counter()
    run_gpu(layer, case["hidden"], case["logits"])
    waited = time.perf_counter() - t0
    assert layer.status() == 6                         # MOE_ERR_DEVICE_TIMEOUT
    assert layer.status() == 0
    assert 1.5 < waited < 60.0, waited
    layer.close()
    # the context is intact and a layer without the fault injection is right
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    ref = run_oracle(s, case)
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    layer.close()
