"""NVFP4 prefill GEMMs on CTA pairs (GPU).

Wide NVFP4 launches can run on clusters of two CTAs sharing one 256 x 256
MMA (tcgen05 cta_group::2; MOE_PAIR_CTAS=1): CTA r of a pair loads token chunk 2c + r and weight
tile 2n + r.  These cases check the pair kernels against the oracle and
against the single-CTA wide kernels (MOE_PAIR_CTAS=0) on the same inputs:
experts with an odd number of chunks (the second CTA of the last pair has
no rows), one-row and empty experts, many chunks per expert, the squared
ReLU, the in-kernel reduce and the batched-expert format.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, cfg_of, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _forward(s, case, monkeypatch, pairs, logits=None):
    monkeypatch.setenv("MOE_WIDE_TILES", "1")
    monkeypatch.setenv("MOE_PAIR_CTAS", "1" if pairs else "0")
    layer = make_layer(s, weights=case["weights"])
    lg = case["logits"] if logits is None else logits
    out = run_gpu(layer, case["hidden"], lg).cpu()
    h, y = (t.cpu() for t in layer.intermediates())
    assert layer.status() == 0
    layer.close()
    return out, h, y


CASES = [
    ("nvfp4_small", dict(T=200, E=3, K=2)),                 # 2-3 chunks per expert
    ("nvfp4_small", dict(T=700, E=4, K=2)),                 # 2-3 chunks, odd counts
    ("nvfp4_zipf_small", dict(T=1100, E=24, K=4)),          # skewed: 1..20 chunks
    ("nvfp4_small", dict(T=90, E=12, K=4, act="relu2")),    # one chunk each
    ("nvfp4_small", dict(T=384, E=2, K=1, clamp=3.0)),      # even chunk counts, clamp
]


@pytest.mark.parametrize("name,over", CASES,
                         ids=["chunks", "odd-chunks", "zipf", "relu2", "even-clamp"])
def test_pair_kernels_match_oracle_and_single_cta(name, over, monkeypatch):
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=61)
    ref = run_oracle(s, case, intermediates=True)
    out_p, h_p, y_p = _forward(s, case, monkeypatch, pairs=True)
    out_1, h_1, y_1 = _forward(s, case, monkeypatch, pairs=False)
    assert rel_l2(h_p.numpy(), ref["h"]) <= TOL["nvfp4"], "GEMM2 input"
    assert rel_l2(y_p.numpy(), ref["y"]) <= TOL["nvfp4"], "GEMM2 output"
    assert rel_l2(out_p.float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    # same operands, same K order per output element: the pair MMA and the
    # single-CTA MMA agree with each other much more closely than with the oracle
    assert rel_l2(y_p.numpy(), y_1.numpy()) <= 1e-3
    assert rel_l2(out_p.float().numpy(), out_1.float().numpy()) <= 1e-3


def test_pair_kernels_forced_empty_and_single_row_experts(monkeypatch):
    s = workloads.spec("nvfp4_small", T=600, E=10, K=3)
    case = workloads.make_case(s, seed=67)
    lg = case["logits"].clone()
    lg[:, [0, 4]] = -1.0e4                     # empty
    lg[:, 7] = -1.0e4
    lg[13, 7] = 1.0e4                          # one row
    ref = run_oracle(s, case, logits=lg.numpy())
    out, _, _ = _forward(s, case, monkeypatch, pairs=True, logits=lg)
    assert rel_l2(out.float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]


def test_pair_kernels_in_kernel_reduce(monkeypatch):
    s = workloads.spec("nvfp4_small", T=300, E=4, K=2, combine="reduce")
    case = workloads.make_case(s, seed=71)
    ref = run_oracle(s, case)
    out, _, _ = _forward(s, case, monkeypatch, pairs=True)
    assert rel_l2(out.float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]


def test_pair_kernels_batched_format(monkeypatch):
    monkeypatch.setenv("MOE_WIDE_TILES", "1")
    monkeypatch.setenv("MOE_PAIR_CTAS", "1")
    s = workloads.spec("nvfp4_small", E=5)
    M = 300
    case = workloads.make_case(s, T=1, seed=73)
    hid, counts = workloads.draw_batched(s, M, seed=73)
    hb = hid.view(torch.int16).numpy().view("uint16")
    ref = oracle.forward_batched(cfg_of(s), workloads.to_numpy_case(case)["weights"], hb,
                                 counts.numpy(), want_y=True)
    layer = make_layer(s, max_tokens=s["E"] * 384 // s["K"], weights=case["weights"])
    out = layer.forward_batched(hid.cuda(), counts.cuda())
    torch.cuda.synchronize()
    assert layer.status() == 0
    cn = counts.numpy()
    got = out.float().cpu().numpy()
    mask = np.zeros(got.shape[:2], bool)
    for e in range(s["E"]):
        mask[e, :cn[e]] = True
    assert rel_l2(got[mask], ref["y"][mask]) <= TOL["nvfp4"]
    layer.close()


def test_pair_kernels_with_few_ctas(monkeypatch):
    # a launch limited to 4 CTAs (2 pairs) walks every item in turn
    s = workloads.spec("nvfp4_zipf_small", T=1100, E=24, K=4)
    case = workloads.make_case(s, seed=79)
    ref = run_oracle(s, case)
    monkeypatch.setenv("MOE_WIDE_TILES", "1")
    monkeypatch.setenv("MOE_PAIR_CTAS", "1")
    layer = make_layer(s, weights=case["weights"], max_ctas=4)
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    layer.close()
