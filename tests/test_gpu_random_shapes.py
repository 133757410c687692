"""Seeded random layer shapes against the oracle (GPU).

Each case draws a format, activation, combine mode and shape (H, I, E, K, T)
from a fixed seed, within the limits the library accepts: H and I multiples
of 128 (256 for NVFP4), 1 <= K <= min(E, 8), E up to 40, T up to 300.  Ids,
offsets and the permutation must match bit for bit, the output within the
format's tolerance.  Shapes the fixed cases do not reach (E = 1, K = E, odd
T, I != H/2, tiny hidden sizes) show up here.
"""
import random

import numpy as np
import pytest

import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

BASE = {"bf16": "bf16_small", "mxfp8": "mxfp8_small", "nvfp4": "nvfp4_small"}


def _draw(i):
    r = random.Random(1000 + i)
    fmt = r.choice(["bf16", "mxfp8", "nvfp4"])
    q = 256 if fmt == "nvfp4" else 128
    H = q * r.randint(1, 4)
    I = q * r.randint(1, 3)
    E = r.choice([1, 2, 3, 5, 8, 13, 24, 40])
    K = r.randint(1, min(E, 8))
    T = r.choice([1, 2, 5, 16, 17, 33, 100, 300])
    act = r.choice(["swiglu", "swiglu", "relu2"])
    clamp = 0.0 if act == "relu2" else r.choice([0.0, 0.0, 3.0])
    combine = r.choice(["gather", "gather", "reduce"])
    return dict(fmt=fmt, H=H, I=I, E=E, K=K, T=T, act=act, clamp=clamp, combine=combine)


CASES = [_draw(i) for i in range(12)] + [
    # a single expert (every token routed to it)
    dict(fmt="nvfp4", H=256, I=256, E=1, K=1, T=33, act="swiglu", clamp=0.0, combine="gather"),
]


@pytest.mark.parametrize("c", CASES, ids=["%(fmt)s-H%(H)d-I%(I)d-E%(E)d-K%(K)d-T%(T)d-%(act)s-%(combine)s" % c
                                          for c in CASES])
def test_random_shape_matches_oracle(c):
    s = workloads.spec(BASE[c["fmt"]], **c)
    case = workloads.make_case(s, seed=7)
    ref = run_oracle(s, case)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], case["logits"])
    assert layer.status() == 0
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert np.array_equal(ids, ref["ids"])
    assert np.array_equal(off, ref["offsets"])
    assert np.array_equal(perm, ref["perm"])
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[c["fmt"]]
    layer.close()
