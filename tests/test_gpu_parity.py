"""CUDA layer vs the CPU oracle on the same seeded inputs (GPU).

Bit-exact: top-k ids, per-expert offsets, the permutation, and the GEMM1
activation quantisation (codes and scales).  Within tolerance: routing
weights (1e-6), GEMM2 input and output, and the layer output (relative L2
<= 5e-3 for BF16 weights, <= 2e-2 for MXFP8/NVFP4).  Sizes span several GEMM
tiles and leave ragged expert tails; edge cases: one token, forced-empty
experts, an expert with a single row, T = max_tokens, T = 0.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_helpers import (TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu,
                               run_oracle)

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny_bf16", {}),
    ("bf16_small", {}),
    ("mxfp8_small", {}),
    ("nvfp4_small", {}),
    ("nvfp4_zipf_small", {}),
    ("bf16_small", dict(T=300, E=4, K=2)),          # >128 rows per expert: several chunks
    ("nvfp4_small", dict(T=200, E=3, K=2)),
    ("mxfp8_small", dict(T=180, E=3, K=1)),
    # T <= 16: the one-block front end (routing .. GEMM1 input in one kernel)
    ("nvfp4_small", dict(T=5, E=300, K=8)),
    ("mxfp8_small", dict(T=16, E=200, K=6)),
    ("bf16_small", dict(T=9, E=40, K=3)),
]


def _ids(c):
    return c[0] + "-" + "-".join("%s%s" % kv for kv in sorted(c[1].items()))


@pytest.mark.parametrize("name,over", CASES, ids=[_ids(c) for c in CASES])
def test_layer_matches_oracle(name, over):
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=0)
    ref = run_oracle(s, case, intermediates=True)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(ids, ref["ids"])
    assert np.array_equal(off, ref["offsets"])
    assert np.array_equal(perm, ref["perm"])
    assert np.max(np.abs(w - ref["w"])) <= 1e-6
    if s["fmt"] != "bf16":
        codes, sf = (t.cpu().numpy() for t in layer.act_quant())
        assert np.array_equal(sf, ref["xq_sf"]), "activation scales differ"
        assert np.array_equal(codes, ref["xq_codes"]), "activation codes differ"
    h, y = (t.cpu().numpy() for t in layer.intermediates())
    assert rel_l2(h, ref["h"]) <= TOL[s["fmt"]], "GEMM2 input"
    assert rel_l2(y, ref["y"]) <= TOL[s["fmt"]], "GEMM2 output"
    got = out.float().cpu().numpy()
    assert rel_l2(got, bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
    layer.close()


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_edge_cases_single_token_empty_and_single_row_experts(fmt):
    name = {"bf16": "bf16_small", "mxfp8": "mxfp8_small", "nvfp4": "nvfp4_small"}[fmt]
    s = workloads.spec(name, T=40, E=10, K=3)
    case = workloads.make_case(s, seed=5)
    layer = make_layer(s, weights=case["weights"])
    # one token
    c1 = dict(case, hidden=case["hidden"][:1], logits=case["logits"][:1])
    ref = run_oracle(s, c1)
    out = run_gpu(layer, c1["hidden"], c1["logits"])
    assert np.array_equal(layer.routing()[0].cpu().numpy(), ref["ids"])
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[fmt]
    # forced-empty experts 0, 4, 9 and expert 7 with exactly one row
    lg = case["logits"].clone()
    lg[:, [0, 4, 9]] = -1.0e4
    lg[:, 7] = -1.0e4
    lg[13, 7] = 1.0e4
    ref = run_oracle(s, case, logits=lg.numpy())
    off_ref = ref["offsets"]
    assert off_ref[1] == off_ref[0] and off_ref[8] - off_ref[7] == 1
    out = run_gpu(layer, case["hidden"], lg)
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert np.array_equal(off, off_ref) and np.array_equal(perm, ref["perm"])
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[fmt]
    assert layer.status() == 0
    layer.close()


def test_max_tokens_and_reuse_across_sizes():
    s = workloads.spec("nvfp4_small", T=130, E=6, K=2)
    case = workloads.make_case(s, seed=9)
    layer = make_layer(s, max_tokens=130, weights=case["weights"])
    for T in (130, 7, 64, 130):
        c = dict(case, hidden=case["hidden"][:T], logits=case["logits"][:T])
        ref = run_oracle(s, c)
        out = run_gpu(layer, c["hidden"], c["logits"])
        assert out.shape == (T, s["H"])
        assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    layer.close()


def test_out_written_in_place_and_deterministic():
    s = workloads.spec("bf16_small")
    case = workloads.make_case(s, seed=1)
    layer = make_layer(s, weights=case["weights"])
    out = torch.full((s["T"], s["H"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    ptr = out.data_ptr()
    results = []
    for _ in range(3):
        layer.forward(case["hidden"].cuda(), case["logits"].cuda(), out=out)
        torch.cuda.synchronize()
        assert out.data_ptr() == ptr
        results.append(out.clone())
    assert not torch.isnan(out.float()).any()
    assert all(torch.equal(results[0], r) for r in results[1:])
    layer.close()


@pytest.mark.parametrize("T", [80, 7])
def test_forward_host_matches_device_forward(T, monkeypatch):
    # pinned host buffers: the kernels read and write them in place; pageable
    # buffers (and MOE_HOST_ZERO_COPY=0) go through device copies
    from moe_expert_layer_histogram_gb300 import moe_forward_host
    s = workloads.spec("mxfp8_small", T=T)
    case = workloads.make_case(s, seed=2)
    stream = torch.cuda.current_stream().cuda_stream
    layer = make_layer(s, weights=case["weights"])
    dev_out = run_gpu(layer, case["hidden"], case["logits"]).cpu()
    hid = case["hidden"].contiguous().pin_memory()
    lg = case["logits"].contiguous().pin_memory()
    host_out = torch.empty_like(hid).pin_memory()
    moe_forward_host(layer.handle, hid, lg, host_out, s["T"], stream)
    assert torch.equal(host_out, dev_out)
    pageable_out = torch.empty_like(case["hidden"])
    moe_forward_host(layer.handle, case["hidden"].contiguous(), case["logits"].contiguous(),
                     pageable_out, s["T"], stream)
    assert torch.equal(pageable_out, dev_out)
    layer.close()
    monkeypatch.setenv("MOE_HOST_ZERO_COPY", "0")
    layer = make_layer(s, weights=case["weights"])
    host_out.zero_()
    moe_forward_host(layer.handle, hid, lg, host_out, s["T"], stream)
    assert torch.equal(host_out, dev_out)
    assert layer.status() == 0
    layer.close()


def test_forward_host_with_unaligned_pinned_buffers():
    # pinned but not 16-byte aligned: the host entry point copies instead of
    # letting the kernels access the buffers in place
    from moe_expert_layer_histogram_gb300 import moe_forward_host
    s = workloads.spec("nvfp4_small", T=9)
    case = workloads.make_case(s, seed=5)
    stream = torch.cuda.current_stream().cuda_stream
    layer = make_layer(s, weights=case["weights"])
    dev_out = run_gpu(layer, case["hidden"], case["logits"]).cpu()
    n = case["hidden"].numel()
    hbuf = torch.empty(n + 1, dtype=torch.bfloat16).pin_memory()
    hbuf[1:] = case["hidden"].reshape(-1)
    obuf = torch.zeros(n + 1, dtype=torch.bfloat16).pin_memory()
    lg = case["logits"].contiguous().pin_memory()
    moe_forward_host(layer.handle, hbuf[1:], lg, obuf[1:], s["T"], stream)
    assert torch.equal(obuf[1:].view_as(dev_out), dev_out)
    assert layer.status() == 0
    layer.close()


def test_error_codes():
    from moe_expert_layer_histogram_gb300 import (MoEError, moe_create, moe_destroy,
                                                  moe_forward)
    with pytest.raises(MoEError) as e:
        moe_create(16, 200, 128, 8, 2, "bf16")          # H not a multiple of 128
    assert e.value.code == 2
    with pytest.raises(MoEError) as e:
        moe_create(16, 256, 128, 8, 9, "bf16")          # K > E
    assert e.value.code == 2
    with pytest.raises(MoEError) as e:
        moe_create(0, 256, 128, 8, 2, "bf16")
    assert e.value.code == 1
    h = moe_create(16, 256, 128, 8, 2, "bf16")
    x = torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(16, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(MoEError) as e:
        moe_forward(h, x, lg, x, 16)                    # no weights yet
    assert e.value.code == 3
    with pytest.raises(MoEError) as e:
        moe_forward(h, x, lg, x, 17)                    # T > max_tokens
    assert e.value.code == 1
    moe_forward(h, x, lg, x, 0)                         # T == 0: no-op
    # the kernels move activations in 16-byte vectors and read fp32 logits:
    # misaligned buffers are refused before anything is launched
    for args in ((x.view(-1)[1:], lg, x), (x, lg, x.view(-1)[4:]),
                 (x, lg.view(torch.uint8).view(-1)[2:], x)):
        with pytest.raises(MoEError) as e:
            moe_forward(h, *args, 16)
        assert e.value.code == 1
    moe_destroy(h)


def test_allocation_failure_reports_oom_and_frees(monkeypatch):
    from moe_expert_layer_histogram_gb300 import MoEError, moe_create, moe_destroy
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for n in (1, 5, 12):
        with pytest.raises(MoEError) as e:
            moe_create(512, 1024, 512, 16, 4, "nvfp4", test_fail_alloc_at=n)
        assert e.value.code == 5
    # the environment does not inject faults: only the config field does
    monkeypatch.setenv("MOE_TEST_FAIL_ALLOC_AT", "1")
    h = moe_create(512, 1024, 512, 16, 4, "nvfp4")
    moe_destroy(h)
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) < (64 << 20)


def test_forward_replays_from_a_cuda_graph():
    # the forward allocates nothing and never syncs the host, so it can be
    # captured once and replayed on new inputs written into the same buffers
    from moe_expert_layer_histogram_gb300 import moe_forward
    s = workloads.spec("nvfp4_small")
    case = workloads.make_case(s, seed=4)
    case2 = workloads.make_case(s, seed=6, weights=False)
    layer = make_layer(s, weights=case["weights"])
    hid, lg = case["hidden"].cuda(), case["logits"].cuda()
    ref1 = run_gpu(layer, hid, lg).clone()
    ref2 = run_gpu(layer, case2["hidden"].cuda(), case2["logits"].cuda()).clone()
    out = torch.empty_like(hid)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe_forward(layer.handle, hid, lg, out, s["T"], torch.cuda.current_stream().cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref1)
    hid.copy_(case2["hidden"])
    lg.copy_(case2["logits"])
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2)
    assert layer.status() == 0
    layer.close()


def test_mma_rate_measurement():
    import json
    import os
    from moe_expert_layer_histogram_gb300 import moe_measure_mma_rate
    bf16 = moe_measure_mma_rate("bf16", 256, iters=4000)
    peaks = os.path.join(os.path.dirname(os.path.dirname(__file__)), "MEASURED_PEAKS.json")
    ref = 2250.0
    if os.path.exists(peaks):
        ref = json.load(open(peaks)).get("bf16_tflops", ref) or ref
    # the tensor pipe's BF16 rate is of the order of a large cuBLAS GEMM's
    assert 0.5 * ref < bf16 < 1.6 * ref, (bf16, ref)
    fp8 = moe_measure_mma_rate("mxfp8", 256, iters=4000)
    fp4 = moe_measure_mma_rate("nvfp4", 256, iters=4000)
    assert fp8 > 1.5 * bf16 and fp4 > 1.5 * fp8, (bf16, fp8, fp4)
    with_copies = moe_measure_mma_rate("nvfp4", 128, copy_scales=True, iters=4000)
    assert 0 < with_copies


# ---- the non-gated ReLU^2 activation ---------------------------------------
@pytest.mark.parametrize("name,over", [
    ("bf16_small", dict(clamp=0.0, act="relu2")),
    ("mxfp8_small", dict(act="relu2")),
    ("nvfp4_small", dict(act="relu2")),
    ("nvfp4_small", dict(T=200, E=3, K=2, act="relu2")),
], ids=["bf16", "mxfp8", "nvfp4", "nvfp4-chunks"])
def test_relu2_layer_matches_oracle(name, over):
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=3)
    ref = run_oracle(s, case, intermediates=True)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert np.array_equal(ids, ref["ids"]) and np.array_equal(perm, ref["perm"])
    h, y = (t.cpu().numpy() for t in layer.intermediates())
    assert rel_l2(h, ref["h"]) <= TOL[s["fmt"]], "GEMM2 input"
    assert rel_l2(y, ref["y"]) <= TOL[s["fmt"]], "GEMM2 output"
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
    assert layer.status() == 0
    layer.close()


def test_relu2_with_clamp_is_unsupported():
    from moe_expert_layer_histogram_gb300 import MoEError, moe_create
    with pytest.raises(MoEError) as e:
        moe_create(16, 256, 128, 8, 2, "bf16", 7.0, "relu2")
    assert e.value.code == 2


# ---- the batched-expert format ----------------------------------------------
BATCHED = [
    ("bf16_small", dict(clamp=0.5), 20),
    ("mxfp8_small", dict(), 40),
    ("nvfp4_small", dict(), 9),
    ("nvfp4_small", dict(E=5), 300),          # several 128-row chunks per expert
    ("nvfp4_small", dict(act="relu2"), 24),
    ("mxfp8_small", dict(act="relu2", E=6), 130),
]


@pytest.mark.parametrize("name,over,M", BATCHED,
                         ids=["%s-%d-M%d" % (b[0], i, b[2]) for i, b in enumerate(BATCHED)])
def test_batched_format_matches_oracle(name, over, M):
    import oracle
    from tests.gpu_helpers import cfg_of
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, T=1, seed=11)
    hid, counts = workloads.draw_batched(s, M, seed=11)
    npw = workloads.to_numpy_case(case)["weights"]
    hb = hid.view(torch.int16).numpy().view("uint16")
    ref = oracle.forward_batched(cfg_of(s), npw, hb, counts.numpy(), want_y=True)
    layer = make_layer(s, max_tokens=max(1, (s["E"] * ((M + 127) // 128) * 128) // s["K"]),
                       weights=case["weights"])
    sentinel = torch.full((s["E"], M, s["H"]), 3.0, dtype=torch.bfloat16, device="cuda")
    out = layer.forward_batched(hid.cuda(), counts.cuda(), out=sentinel)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = out.float().cpu().numpy()
    cn = counts.numpy()
    for e in range(s["E"]):
        assert (got[e, cn[e]:] == 3.0).all(), "rows past the count were written"
    mask = np.zeros(got.shape[:2], bool)
    for e in range(s["E"]):
        mask[e, :cn[e]] = True
    assert rel_l2(got[mask], ref["y"][mask]) <= TOL[s["fmt"]]
    # a row-by-row bound too: no single expert far off
    for e in range(s["E"]):
        if cn[e]:
            assert rel_l2(got[e, :cn[e]], ref["y"][e, :cn[e]]) <= 2 * TOL[s["fmt"]], e
    layer.close()


def test_batched_counts_out_of_range_are_clamped_and_reported():
    s = workloads.spec("nvfp4_small")
    case = workloads.make_case(s, T=1, seed=2)
    M = 16
    hid, counts = workloads.draw_batched(s, M, seed=2)
    layer = make_layer(s, max_tokens=s["E"] * 128 // s["K"], weights=case["weights"])
    good = layer.forward_batched(hid.cuda(), counts.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    bad = counts.clone()
    bad[1] = M + 5                                  # clamps to M (expert 1 is already full)
    out = layer.forward_batched(hid.cuda(), bad.cuda())
    assert layer.status() == 1                      # MOE_ERR_INVALID_ARG, then cleared
    assert layer.status() == 0
    assert torch.equal(out, good)
    layer.close()


def test_batched_capacity_and_arguments():
    from moe_expert_layer_histogram_gb300 import MoEError, moe_forward_batched
    s = workloads.spec("bf16_small")
    case = workloads.make_case(s, T=1, seed=2)
    layer = make_layer(s, max_tokens=8, weights=case["weights"])   # capacity: 8*4 rows + pads
    hid = torch.zeros(s["E"], 600, s["H"], dtype=torch.bfloat16, device="cuda")
    cnt = torch.zeros(s["E"], dtype=torch.int32, device="cuda")
    with pytest.raises(MoEError) as e:
        moe_forward_batched(layer.handle, hid, cnt, 600, hid)
    assert e.value.code == 2
    moe_forward_batched(layer.handle, hid, cnt, 0, hid)            # M == 0: no-op
    with pytest.raises(MoEError) as e:
        moe_forward_batched(layer.handle, hid, cnt, -1, hid)
    assert e.value.code == 1
    layer.close()


# ---- GEMM items of two weight tiles (N = 256), used for prefill-sized T -------
@pytest.mark.parametrize("name,over,force", [
    ("bf16_small", dict(), True),
    ("mxfp8_small", dict(), True),
    ("nvfp4_small", dict(), True),
    ("nvfp4_small", dict(T=200, E=3, K=2), True),
    ("nvfp4_small", dict(act="relu2"), True),
    ("mxfp8_small", dict(act="relu2", T=150, E=4, K=2), True),
    ("nvfp4_zipf_small", dict(T=1100, E=24, K=4), False),   # T > 1024 selects them itself
    ("nvfp4_zipf_small", dict(T=2100, E=24, K=4), False),   # and the two-pass expert scan
], ids=["bf16", "mxfp8", "nvfp4", "nvfp4-chunks", "nvfp4-relu2", "mxfp8-relu2", "nvfp4-T1100",
        "nvfp4-T2100"])
def test_wide_items_match_oracle(name, over, force, monkeypatch):
    if force:
        monkeypatch.setenv("MOE_WIDE_TILES", "1")
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=12)
    ref = run_oracle(s, case, intermediates=True)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    h, y = (t.cpu().numpy() for t in layer.intermediates())
    assert rel_l2(h, ref["h"]) <= TOL[s["fmt"]], "GEMM2 input"
    assert rel_l2(y, ref["y"]) <= TOL[s["fmt"]], "GEMM2 output"
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
    layer.close()


def test_wide_nvfp4_scale_stagers_and_copies_agree(monkeypatch):
    # wide NVFP4 GEMM1 items get their scales written into TMEM by four
    # stager warps (tcgen05.st) or, with MOE_SCALE_STAGER=0, broadcast by the
    # MMA thread (tcgen05.cp): the same scale values reach the same MMAs, so
    # the outputs agree bit for bit, and both match the oracle
    s = workloads.spec("nvfp4_zipf_small", T=1100, E=24, K=4)
    case = workloads.make_case(s, seed=23)
    ref = run_oracle(s, case)
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_SCALE_STAGER", flag)
        layer = make_layer(s, weights=case["weights"])
        outs.append(run_gpu(layer, case["hidden"], case["logits"]).cpu())
        assert layer.status() == 0
        layer.close()
    assert torch.equal(outs[0], outs[1])
    assert rel_l2(outs[0].float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]


def test_batched_output_with_16_byte_alignment(monkeypatch):
    # GEMM2 stores whole 32-byte sectors when the output rows allow it and
    # 16-byte pieces otherwise: both give the same bytes
    monkeypatch.setenv("MOE_WIDE_TILES", "1")
    s = workloads.spec("nvfp4_small", E=3, K=2)
    M = 40
    case = workloads.make_case(s, T=1, seed=29)
    hid, counts = workloads.draw_batched(s, M, seed=29)
    layer = make_layer(s, max_tokens=s["E"] * 256 // s["K"], weights=case["weights"])
    ref = layer.forward_batched(hid.cuda(), counts.cuda())
    buf = torch.zeros(ref.numel() + 8, dtype=torch.bfloat16, device="cuda")
    off = buf[8:].view_as(ref)                           # 16 bytes past a 256-byte boundary
    assert off.data_ptr() % 32 == 16
    layer.forward_batched(hid.cuda(), counts.cuda(), out=off)
    torch.cuda.synchronize()
    assert layer.status() == 0
    cn = counts.numpy()
    for e in range(s["E"]):
        assert torch.equal(off[e, :cn[e]], ref[e, :cn[e]])
    layer.close()


def test_wide_items_batched_format(monkeypatch):
    import oracle
    from tests.gpu_helpers import cfg_of
    monkeypatch.setenv("MOE_WIDE_TILES", "1")
    s = workloads.spec("nvfp4_small", E=5)
    M = 260
    case = workloads.make_case(s, T=1, seed=13)
    hid, counts = workloads.draw_batched(s, M, seed=13)
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


# ---- the in-kernel reduce (GEMM2's epilogue sums the K outputs) ------------
@pytest.mark.parametrize("name,over,wide", [
    ("bf16_small", dict(combine="reduce"), False),
    ("mxfp8_small", dict(combine="reduce"), False),
    ("nvfp4_small", dict(combine="reduce"), False),
    ("nvfp4_small", dict(T=7, E=300, K=8, combine="reduce"), False),    # one-kernel front end
    ("nvfp4_small", dict(combine="reduce", act="relu2"), True),
    ("bf16_small", dict(T=300, E=4, K=2, combine="reduce"), True),
], ids=["bf16", "mxfp8", "nvfp4", "nvfp4-T7", "nvfp4-relu2-wide", "bf16-chunks-wide"])
def test_in_kernel_reduce_matches_oracle(name, over, wide, monkeypatch):
    if wide:
        monkeypatch.setenv("MOE_WIDE_TILES", "1")
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=17)
    ref = run_oracle(s, case)
    layer = make_layer(s, weights=case["weights"])
    outs = []
    for _ in range(3):                   # the accumulator is left at zero between forwards
        outs.append(run_gpu(layer, case["hidden"], case["logits"]).float().cpu().numpy())
    assert layer.status() == 0
    for o in outs:
        assert rel_l2(o, bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
    # only the summation order differs between runs: last-bit differences at most
    assert max(np.max(np.abs(o - outs[0])) for o in outs) <= 1e-2 * np.max(np.abs(outs[0]))
    layer.close()


@pytest.mark.parametrize("T", [9, 40])
def test_top16_routing_matches_oracle(T):
    # K = 16, the largest top-k the library accepts (one-kernel front end for
    # T <= 16, the three-kernel one above)
    s = workloads.spec("nvfp4_small", T=T, E=40, K=16)
    case = workloads.make_case(s, seed=29)
    ref = run_oracle(s, case)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert np.array_equal(ids, ref["ids"]) and np.array_equal(off, ref["offsets"])
    assert np.array_equal(perm, ref["perm"])
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    assert layer.status() == 0
    layer.close()


def test_forward_on_a_side_stream():
    # work is enqueued on the caller's stream only; results match the default
    # stream's bit for bit
    s = workloads.spec("mxfp8_small")
    case = workloads.make_case(s, seed=31)
    layer = make_layer(s, weights=case["weights"])
    ref = run_gpu(layer, case["hidden"], case["logits"]).clone()
    side = torch.cuda.Stream()
    hid, lg = case["hidden"].cuda(), case["logits"].cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        out = layer.forward(hid, lg)
        side.synchronize()
    assert torch.equal(out, ref)
    assert layer.status() == 0
    layer.close()


# ---- the combine fused into GEMM2's epilogue ---------------------------------
@pytest.mark.parametrize("name,over,env", [
    ("bf16_small", dict(), {}),                                           # narrow: combine kernel
    ("nvfp4_zipf_small", dict(T=1100, E=24, K=4), {}),                    # wide items
    ("nvfp4_zipf_small", dict(T=1100, E=24, K=4), {"MOE_PAIR_CTAS": "1"}),  # CTA pairs
    ("mxfp8_small", dict(act="relu2"), {}),
    ("nvfp4_small", dict(T=12, E=40, K=8), {}),                            # single-launch decode
    ("nvfp4_small", dict(T=12, E=40, K=8), {"MOE_SINGLE_LAUNCH": "0"}),    # fused decode GEMMs
    ("nvfp4_small", dict(T=300, E=40, K=16), {}),                          # top-16
], ids=["bf16", "nvfp4-wide", "nvfp4-pairs", "mxfp8-relu2", "decode", "decode-3-launch", "top16"])
def test_fused_combine_is_bit_identical_to_the_combine_kernel(name, over, env, monkeypatch):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=107)
    ref = run_oracle(s, case)
    outs = {}
    for mode in ("gather", "fused"):
        layer = make_layer(dict(s, combine=mode), weights=case["weights"])
        got = [run_gpu(layer, case["hidden"], case["logits"]).cpu() for _ in range(2)]
        assert layer.status() == 0
        assert torch.equal(got[0], got[1])          # the counters are back at zero
        outs[mode] = got[0]
        layer.close()
    assert torch.equal(outs["gather"], outs["fused"])
    assert rel_l2(outs["fused"].float().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[s["fmt"]]
