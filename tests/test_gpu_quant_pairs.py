"""NVFP4 activation quantisation over every (scale, value) pair (GPU).

Each 16-element block of the hidden rows holds +-6 sf at its first position,
which fixes the block's e4m3 scale at sf exactly (6 sf / 6 = sf), and 15
bf16 values of magnitude at most 6 sf.  Over the rows, every positive e4m3
scale meets every bf16 value that can give a nonzero e2m1 code under it
(|x| >= sf / 16, both signs), plus a sample of smaller ones, signed zeros and
bf16 subnormals.  The kernels' codes and scales must equal the oracle's
(correctly rounded quotient x / sf, then e2m1 round-to-nearest-even) bit for
bit: through the scatter kernel (T > 16), the one-block front end and the
single-launch decode kernel (T <= 16, a sample of the pairs).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import bf16_bits_to_f64, make_layer, run_gpu

pytestmark = pytest.mark.gpu


def _bf16_values():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    return (bits << 16).view(np.float32)            # +0 .. largest finite, ascending


def _pairs(rng, per_scale=None):
    """[(sf, values)]: values of |x| <= 6 sf with both signs."""
    mags = _bf16_values()
    scales = oracle.decode("e4m3", np.arange(1, 0x7F, dtype=np.uint8))
    out = []
    for s in scales:
        s = np.float32(s)
        big = mags[(mags >= s / 16) & (mags <= 6 * s)]
        small = mags[mags < s / 16]
        small = np.concatenate([small[:4], rng.choice(small, 60, replace=False)])  # 0, subnormals
        v = np.concatenate([big, small])
        v = np.concatenate([v, -v])
        if per_scale is not None:
            v = rng.choice(v, per_scale, replace=False)
        out.append((s, rng.permutation(v)))
    return out


def _hidden(pairs, H):
    blocks = []
    for s, v in pairs:
        n = -(-v.size // 15)
        v = np.concatenate([v, np.zeros(n * 15 - v.size, np.float32)]).reshape(n, 15)
        lead = np.where(np.arange(n) % 2, -6 * s, 6 * s).astype(np.float32)[:, None]
        blocks.append(np.concatenate([lead, v], axis=1))
    b = np.concatenate(blocks)
    per_row = H // 16
    rows = -(-b.shape[0] // per_row)
    pad = np.tile(b[:1], (rows * per_row - b.shape[0], 1))
    x = np.concatenate([b, pad]).reshape(rows, H)
    return torch.from_numpy(x).to(torch.bfloat16).contiguous()


def _check(layer, hid):
    codes, sf = (t.cpu().numpy() for t in layer.act_quant())
    assert layer.status() == 0
    x = bf16_bits_to_f64(hid.view(torch.int16).numpy().view(np.uint16)).astype(np.float32)
    rc, rs = oracle.quant_row("nvfp4", x)
    assert np.array_equal(sf, rs), "scales differ"
    bad = np.nonzero(codes != rc)
    assert bad[0].size == 0, f"{bad[0].size} code bytes differ, first at {bad[0][0]}, {bad[1][0]}"


def test_scatter_quantises_every_scale_value_pair_like_the_oracle():
    rng = np.random.default_rng(5)
    pairs = _pairs(rng)
    s0 = workloads.spec("nvfp4_small")
    hid = _hidden(pairs, s0["H"])
    T = hid.shape[0]
    assert T > 16 and sum(v.size for _, v in pairs) > 200_000
    s = workloads.spec("nvfp4_small", T=T)
    case = workloads.make_case(s, seed=7)
    layer = make_layer(s, weights=case["weights"])
    run_gpu(layer, hid, case["logits"])
    _check(layer, hid)
    layer.close()


@pytest.mark.parametrize("single", ["1", "0"], ids=["decode-kernel", "one-block-front"])
def test_small_batches_quantise_sampled_pairs_like_the_oracle(single, monkeypatch):
    monkeypatch.setenv("MOE_SINGLE_LAUNCH", single)
    rng = np.random.default_rng(11)
    s0 = workloads.spec("nvfp4_small")
    pairs = _pairs(rng, per_scale=90)
    hid = _hidden(pairs, s0["H"])[:16].contiguous()
    s = workloads.spec("nvfp4_small", T=16)
    case = workloads.make_case(s, seed=9)
    layer = make_layer(s, weights=case["weights"])
    run_gpu(layer, hid, case["logits"])
    from moe_expert_layer_histogram_gb300 import moe_last_launch_count
    assert (moe_last_launch_count(layer.handle) == 1) == (single == "1")
    _check(layer, hid)
    layer.close()
