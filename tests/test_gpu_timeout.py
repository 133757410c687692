"""Bounded device waits (GPU): a GEMM whose data never arrives gives up.

The fault-injection field moe_config.test_stall_gemm = 1 makes one
CTA of every GEMM1 launch leave one stage of its shared-memory ring unloaded,
so the barrier waits on that stage are never satisfied (in the narrow kernel,
the 16-warp wide NVFP4 kernel and its CTA-pair form).  Each wait gives up
after 2 s: the kernel records MOE_ERR_DEVICE_TIMEOUT, drains its own copies,
frees its tensor memory and returns.  No fault, trap or hang is involved, and
the CUDA context stays usable, which the second half checks.
"""
import time

import numpy as np
import pytest

import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 6


@pytest.mark.parametrize("wide,cluster", [(False, None), (True, None), (True, "pairs")],
                         ids=["narrow", "wide", "wide-pairs"])
def test_gemm_wait_runs_out_and_is_reported(wide, cluster, monkeypatch):
    # wide: the 16-warp NVFP4 kernel, whose MMA thread waits on the stage
    # that never lands and whose stager warps then wait for a TMEM scale slot
    # that is never freed; pairs: the CTA-pair kernel, where the stalled
    # CTA's peer gives up its own waits on the shared MMA too
    if wide:
        monkeypatch.setenv("MOE_WIDE_TILES", "1")
        monkeypatch.setenv("MOE_PAIR_CTAS", "1" if cluster == "pairs" else "0")
    s = workloads.spec("nvfp4_small")
    case = workloads.make_case(s, seed=21)
    layer = make_layer(s, weights=case["weights"], test_stall_gemm=1)
    t0 = time.perf_counter()
    run_gpu(layer, case["hidden"], case["logits"])
    waited = time.perf_counter() - t0
    assert layer.status() == MOE_ERR_DEVICE_TIMEOUT
    assert layer.status() == 0                      # read once, then cleared
    assert 1.5 < waited < 60.0, waited
    layer.close()

    # the context is intact: a layer without the fault injection computes correctly
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    ref = run_oracle(s, case)
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    assert np.isfinite(out.float().cpu().numpy()).all()
    layer.close()
