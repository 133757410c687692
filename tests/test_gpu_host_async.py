"""Pipelined host-buffer forward, moe_forward_host_async (GPU).

Each call enqueues the input copy, the layer and the output copy on a copy
stream and a compute stream of the layer's own and returns at once; the
caller's stream completes once the output is in host memory.  Consecutive
calls overlap (step i+1's input copy after step i's front end, step i's
output copy during step i+1), so these cases run several steps back to back
on different inputs and different output buffers and compare every output
bit for bit with the device-buffer forward of the same input: a copy that
overwrote the device input or output buffer too early would change a
result.  Covered: the six-launch path, the single-launch decode kernel, a
prefill-sized launch (wide items, plain stream order), BF16, varying T
between steps, and device forwards on the caller's stream between
pipelined steps.
"""
import pytest
import torch

import workloads
from tests.gpu_helpers import make_layer, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    ("nvfp4_small", dict(T=40, E=24, K=6)),              # six launches
    ("nvfp4_small", dict(T=9)),                          # single-launch decode
    ("nvfp4_zipf_small", dict(T=1100, E=24, K=4)),       # prefill-sized: wide items
    ("bf16_small", dict(T=96)),
]


def _inputs(s, n, T=None):
    out = []
    for i in range(n):
        c = workloads.make_case(s, T=T, seed=300 + i, weights=False)
        out.append((c["hidden"].contiguous().pin_memory(), c["logits"].contiguous().pin_memory()))
    return out


@pytest.mark.parametrize("name,over", CASES, ids=["six-launch", "decode", "prefill", "bf16"])
def test_pipelined_steps_match_device_forwards(name, over):
    from moe_expert_layer_histogram_gb300 import moe_forward_host_async
    s = workloads.spec(name, **over)
    wcase = workloads.make_case(s, seed=299)
    layer = make_layer(s, weights=wcase["weights"])
    ins = _inputs(s, 4)
    refs = [run_gpu(layer, h.cuda(), l.cuda()).cpu() for h, l in ins]
    outs = [torch.empty_like(h).pin_memory() for h, _ in ins]
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        for (h, l), o in zip(ins, outs):
            moe_forward_host_async(layer.handle, h, l, o, s["T"], stream)
    torch.cuda.synchronize()
    assert layer.status() == 0
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)
    layer.close()


def test_pipelined_steps_of_varying_size_and_device_forwards_between():
    import moe_expert_layer_histogram_gb300 as moe
    s = workloads.spec("nvfp4_small", T=48, E=24, K=6)
    wcase = workloads.make_case(s, seed=311)
    layer = make_layer(s, weights=wcase["weights"])
    sizes = [1, 48, 7, 33, 16, 48, 2]
    full = _inputs(s, len(sizes))
    steps = []
    for T, (h, l) in zip(sizes, full):
        h, l = h[:T].contiguous().pin_memory(), l[:T].contiguous().pin_memory()
        ref = run_gpu(layer, h.cuda(), l.cuda()).cpu()
        steps.append((T, h, l, ref, torch.empty_like(h).pin_memory()))
    stream = torch.cuda.current_stream().cuda_stream
    dev_h, dev_l = full[0][0].cuda(), full[0][1].cuda()
    dev_ref = run_gpu(layer, dev_h, dev_l).cpu()
    dev_out = torch.empty_like(dev_h)
    for i, (T, h, l, _, o) in enumerate(steps):
        moe.moe_forward_host_async(layer.handle, h, l, o, T, stream)
        if i % 3 == 1:
            # a device forward on the caller's stream, ordered after the step
            moe.moe_forward(layer.handle, dev_h, dev_l, dev_out, s["T"], stream)
    torch.cuda.synchronize()
    assert layer.status() == 0
    for T, _, _, ref, o in steps:
        assert torch.equal(o, ref), T
    assert torch.equal(dev_out.cpu(), dev_ref)
    layer.close()
