"""Independent torch restatements used to pin the oracle (tests only).

Written from the format definitions and the layer's definition with library
primitives (torch float8/bfloat16 casts, einsum, softmax, silu); shares no
code with the oracle or the CUDA path.
"""
import numpy as np
import torch

E2M1_MAG = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def e2m1_value(codes):
    c = codes.to(torch.int64)
    mag = E2M1_MAG[c & 7]
    return torch.where((c & 8) != 0, -mag, mag)


def e2m1_code(v):
    a = v.abs()
    idx = ((a > 0.25).int() + (a >= 0.75).int() + (a > 1.25).int() + (a >= 1.75).int()
           + (a > 2.5).int() + (a >= 3.5).int() + (a > 5.0).int())
    return idx | (torch.signbit(v).int() << 3)


def e4m3_value(bits):
    return bits.view(torch.float8_e4m3fn).to(torch.float64)


def e4m3_bits(x32):
    return x32.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


def unpack_nibbles(codes):
    c = torch.as_tensor(codes).to(torch.int64)
    out = torch.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=torch.int64)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def quant_dequant(fmt, x32):
    """Quantise fp32 rows per block with activation global scale 1 and
    return the dequantised values (float64)."""
    x32 = x32.to(torch.float32)
    n = x32.shape[-1]
    if fmt == "bf16":
        return x32.to(torch.bfloat16).to(torch.float64)
    if fmt == "nvfp4":
        b = x32.reshape(-1, 16)
        amax = b.abs().amax(-1)
        sf = e4m3_bits(amax / 6.0)
        sv = e4m3_value(sf).to(torch.float32).unsqueeze(-1)
        q = e2m1_code(b / torch.where(sv == 0, torch.ones_like(sv), sv))
        deq = e2m1_value(q) * sv.to(torch.float64)
        deq = torch.where(sv == 0, torch.zeros_like(deq), deq)
        return deq.reshape(x32.shape)
    b = x32.reshape(-1, 32)
    amax = b.abs().amax(-1).to(torch.float64)
    X = torch.floor(torch.log2(torch.where(amax == 0, torch.ones_like(amax), amax))) - 8
    scaled = (b.to(torch.float64) * torch.pow(2.0, -X).unsqueeze(-1)).to(torch.float32)
    deq = e4m3_value(e4m3_bits(scaled)) * torch.pow(2.0, X).unsqueeze(-1)
    deq = torch.where(amax.unsqueeze(-1) == 0, torch.zeros_like(deq), deq)
    return deq.reshape(x32.shape)


def dequant_weights(fmt, w, sf=None, gs=None):
    """Canonical weights [E, N, K(bytes)] -> float64 [E, N, K]."""
    w = torch.as_tensor(np.asarray(w))
    if fmt == "bf16":
        return w.view(torch.int16).view(torch.bfloat16).to(torch.float64) if w.dtype != torch.bfloat16 \
            else w.to(torch.float64)
    sf = torch.as_tensor(np.asarray(sf))
    if fmt == "mxfp8":
        v = e4m3_value(w)
        s = torch.pow(2.0, sf.to(torch.float64) - 127)
        return v * s.repeat_interleave(32, dim=-1)
    gs = torch.as_tensor(np.asarray(gs)).to(torch.float32)
    folded = e4m3_bits(e4m3_value(sf).to(torch.float32) * gs.view(-1, 1, 1))
    v = e2m1_value(unpack_nibbles(w))
    return v * e4m3_value(folded).repeat_interleave(16, dim=-1)


def expert_mlp_f64(fmt, clamp, a, W13e, W2e, act="swiglu"):
    """One expert on one dequantised GEMM1 input row ``a`` (float64 [H]).
    fp32 roundings mirror the layer's: the GEMM results and h are rounded
    to fp32 before the GEMM2-input quantisation.  Returns float64 [H] (the
    fp32 GEMM2 output)."""
    G = (W13e @ a).to(torch.float32)
    if act == "relu2":
        h = (torch.relu(G.to(torch.float64)) ** 2).to(torch.float32)
    else:
        I = G.shape[0] // 2
        g, u = G[:I], G[I:]
        if clamp and clamp > 0:
            g = g.clamp(-clamp, clamp)
            u = u.clamp(-clamp, clamp)
        h = (torch.nn.functional.silu(g.to(torch.float64)) * u.to(torch.float64)).to(torch.float32)
    hq = quant_dequant(fmt, h.unsqueeze(0))[0]
    return (W2e @ hq).to(torch.float32).to(torch.float64)


def gemm1_input_f64(fmt, hidden_bits):
    x = torch.as_tensor(np.asarray(hidden_bits)).view(torch.int16).view(torch.bfloat16).to(torch.float32)
    return quant_dequant(fmt, x) if fmt != "bf16" else x.to(torch.float64)


def dense_layer_f64(fmt, clamp, hidden_bits, logits, W13, W2, weights_k, act="swiglu"):
    """Top-k routed layer written densely: for each token, every selected
    expert's output weighted by the renormalised softmax.  Returns float64
    [T, H] (before bf16)."""
    a = gemm1_input_f64(fmt, hidden_bits)
    lg = torch.as_tensor(np.asarray(logits)).to(torch.float64)
    T = a.shape[0]
    top = torch.topk(lg, weights_k, dim=-1)
    p = torch.softmax(top.values, -1)
    out = torch.zeros(T, W2.shape[1], dtype=torch.float64)
    for t in range(T):
        for j in range(weights_k):
            e = int(top.indices[t, j])
            out[t] += p[t, j] * expert_mlp_f64(fmt, clamp, a[t], W13[e], W2[e], act)
    return out


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.linalg.norm(a - b)
    n = np.linalg.norm(b)
    return float(d / n) if n > 0 else float(d)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
