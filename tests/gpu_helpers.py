"""Shared helpers for the GPU tests: run the CUDA layer and the oracle on the
same seeded inputs and compare."""
import numpy as np

import oracle
import workloads

TOL = {"bf16": 5e-3, "mxfp8": 2e-2, "nvfp4": 2e-2}


def cfg_of(s):
    return dict(H=s["H"], I=s["I"], E=s["E"], K=s["K"], fmt=s["fmt"], clamp=s["clamp"],
                act=s.get("act", "swiglu"))


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / n) if n > 0 else float(np.linalg.norm(a - b))


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def make_layer(s, max_tokens=None, weights=None, device="cuda:0", **config):
    """config: further moe_config fields (max_ctas, test_stall_gemm, ...)."""
    import torch
    from moe_expert_layer_histogram_gb300 import MoELayer
    layer = MoELayer(max_tokens or s["T"], s["H"], s["I"], s["E"], s["K"], s["fmt"], s["clamp"],
                     s.get("act", "swiglu"), s.get("combine", "gather"), **config)
    if weights is not None:
        layer.prepare_weights({k: v.to(device).contiguous() for k, v in weights.items()})
    torch.cuda.synchronize()
    return layer


def run_gpu(layer, hidden, logits):
    import torch
    out = layer.forward(hidden.cuda().contiguous(), logits.cuda().contiguous())
    torch.cuda.synchronize()
    return out


def run_oracle(s, case, logits=None, intermediates=False):
    npc = workloads.to_numpy_case(case)
    lg = npc["logits"] if logits is None else logits
    return oracle.forward(cfg_of(s), npc["weights"], npc["hidden"], lg,
                          want_intermediates=intermediates)
