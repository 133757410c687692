"""Seeded synthetic workloads for the fused MoE expert layer.

This module only *draws inputs*: router logits, bf16 hidden states and the
layer's weights in their canonical (already quantised) form.  It holds none
of the layer's own arithmetic (routing, permutation, activation quantisation,
GEMMs, SwiGLU, combine, scale folding); both the CUDA path and the CPU oracle
consume what it produces, and it imports neither.

Quantised weights are produced the way an offline quantiser (modelopt
convention) produces a checkpoint, *before* the layer ever sees them:
  NVFP4: per expert global scale gs = amax_e / (6 * 448); per 16-block scale
         sf = e4m3(amax_b / (6 * gs)); codes q = e2m1(x / (sf * gs)).
         (the block scale is the block's largest magnitude times the global
         quantisation scale over the largest e2m1 value, the vLLM convention
         restated in PR #40082 report, sec. 关键源码片段.)
  MXFP8: per 32-block shared exponent X = floor(log2 amax) - 8, e8m0 scale
         X + 127, codes e4m3(x * 2^-X) (OCP MX v1.0 conversion rule).
The element roundings use torch's float8_e4m3fn cast (round to nearest even)
and a tie-to-even threshold table for e2m1.

Workloads (sizes, distributions) follow the five layer configurations of this
project: a tiny BF16 layer, a BF16 layer with clamp, an MXFP8 decode layer,
an NVFP4 decode sweep and an NVFP4 prefill layer with Zipf(1.1) expert
popularity; plus a 32K-token NVFP4 prefill with uniform routing, where the
tensor pipe rather than the weight bytes sets the pace.  Nothing here reads a dataset; every tensor is synthetic.
"""
import math

import torch

# name -> layer shape, format and input recipe
CONFIGS = {
    "tiny_bf16": dict(T=16, H=256, I=128, E=8, K=2, fmt="bf16", clamp=0.0,
                      wdist="fan_in", logits="normal"),
    "bf16": dict(T=512, H=2048, I=1024, E=64, K=6, fmt="bf16", clamp=7.0,
                 wdist="fan_in", logits="normal"),
    "mxfp8_decode": dict(T=64, H=7168, I=2048, E=256, K=8, fmt="mxfp8",
                         clamp=0.0, wdist=0.02, logits="normal"),
    "nvfp4_decode": dict(T=128, H=7168, I=2048, E=384, K=8, fmt="nvfp4",
                         clamp=0.0, wdist=0.02, logits="normal",
                         sweep=(1, 8, 32, 128)),
    "nvfp4_prefill": dict(T=8192, H=7168, I=2048, E=384, K=8, fmt="nvfp4",
                          clamp=0.0, wdist=0.02, logits="zipf1.1"),
    # a prefill large enough that the FP4 tensor pipe, not the weight bytes,
    # sets the pace: 262,144 routed rows over all 384 experts (~680 each)
    "nvfp4_prefill_32k": dict(T=32768, H=7168, I=2048, E=384, K=8, fmt="nvfp4",
                              clamp=0.0, wdist=0.02, logits="normal"),
}

# Reduced shapes of the same recipes for parity tests the oracle finishes in
# seconds; they still span several GEMM tiles and leave ragged expert tails.
SMALL = {
    "bf16_small": dict(T=96, H=512, I=256, E=16, K=4, fmt="bf16", clamp=7.0,
                       wdist="fan_in", logits="normal"),
    "mxfp8_small": dict(T=80, H=512, I=256, E=16, K=4, fmt="mxfp8", clamp=0.0,
                        wdist=0.02, logits="normal"),
    "nvfp4_small": dict(T=72, H=768, I=256, E=12, K=4, fmt="nvfp4", clamp=0.0,
                        wdist=0.02, logits="normal"),
    "nvfp4_zipf_small": dict(T=300, H=512, I=256, E=24, K=4, fmt="nvfp4",
                             clamp=5.0, wdist=0.02, logits="zipf1.1"),
}


def spec(name, **over):
    """Layer shape and input recipe.  ``act`` is the expert activation:
    "swiglu" (gated; W13 holds gate and up, 2I rows) unless overridden with
    "relu2" (non-gated squared ReLU; W13 holds the I rows of one projection)."""
    d = dict(CONFIGS.get(name) or SMALL[name])
    d.setdefault("act", "swiglu")
    d.update(over)
    d["name"] = name
    return d


def w13_rows(s):
    return s["I"] if s.get("act", "swiglu") == "relu2" else 2 * s["I"]


# ---------------------------------------------------------------------------
# element helpers (input synthesis only)
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _e4m3_bits(x):
    """fp32 -> e4m3fn bits (uint8), nearest even, saturating at +-448."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _e4m3_value(bits):
    return bits.view(torch.float8_e4m3fn).to(torch.float32)


def _e2m1_bits(v):
    """fp32 -> e2m1 code (uint8, low nibble), nearest with ties to the even
    code, saturating at +-6.  Magnitudes by code: 0 .5 1 1.5 2 3 4 6."""
    a = v.abs()
    idx = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
           + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
           + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    return idx | (torch.signbit(v).to(torch.uint8) << 3)


def quantize_weight_nvfp4(w):
    """w: float tensor [N, K] of one expert (bf16 values).  Returns
    (codes uint8 [N, K/2] low nibble = even element, sf uint8 [N, K/16]
    e4m3 bits, gs float32 scalar tensor)."""
    w = w.to(torch.float32)
    N, K = w.shape
    amax_e = w.abs().amax()
    gs = (amax_e / (E2M1_MAX * E4M3_MAX)).to(torch.float32)
    if float(gs) == 0.0:
        gs = torch.tensor(1.0, dtype=torch.float32, device=w.device)
    blk = w.view(N, K // 16, 16)
    amax_b = blk.abs().amax(dim=-1)
    sf = _e4m3_bits(amax_b / (E2M1_MAX * gs))
    denom = (_e4m3_value(sf) * gs).unsqueeze(-1)
    safe = torch.where(denom == 0, torch.ones_like(denom), denom)
    q = _e2m1_bits(blk / safe)
    q = torch.where(denom == 0, torch.zeros_like(q), q).view(N, K)
    codes = q[:, 0::2] | (q[:, 1::2] << 4)
    return codes.contiguous(), sf.contiguous(), gs


def quantize_weight_mxfp8(w):
    """w: float tensor [N, K].  Returns (codes uint8 [N, K] e4m3 bits,
    sf uint8 [N, K/32] e8m0)."""
    w = w.to(torch.float32)
    N, K = w.shape
    blk = w.view(N, K // 32, 32)
    amax = blk.abs().amax(dim=-1)
    _, e = torch.frexp(amax)                       # amax = m * 2^e, m in [.5,1)
    X = (e.to(torch.int32) - 1 - 8).clamp(-127, 127)
    X = torch.where(amax == 0, torch.zeros_like(X), X)
    scaled = torch.ldexp(blk, (-X).unsqueeze(-1).to(torch.float32))
    codes = _e4m3_bits(scaled).view(N, K)
    sf = (X + 127).to(torch.uint8)
    return codes.contiguous(), sf.contiguous()


# ---------------------------------------------------------------------------
# drawing
# ---------------------------------------------------------------------------
def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_logits(s, T, g, device):
    E = s["E"]
    lg = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if s["logits"].startswith("zipf"):
        # popularity p_e ~ rank_e^-s over a seeded random ranking of experts,
        # added as log-probabilities to N(0,1) logits
        sexp = float(s["logits"][4:])
        ranks = torch.randperm(E, generator=g, device=device).to(torch.float32) + 1.0
        logp = -sexp * torch.log(ranks)
        logp = logp - torch.logsumexp(logp, 0)
        lg = lg + logp.unsqueeze(0)
    return lg.contiguous()


def draw_hidden(s, T, g, device):
    return torch.randn(T, s["H"], generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16).contiguous()


def _expert_gen(seed, which, e, device):
    # every expert matrix has its own generator, so any subset of experts can
    # be drawn (or re-drawn) without drawing the others
    return _gen(seed * 1000003 + 2 * e + (1 if which == "w13" else 2), device)


def draw_expert(s, which, e, seed, device):
    """One expert's canonical matrix: W13_e [2I, H] (or [I, H] for ReLU^2)
    or W2_e [H, I] (bf16), or its quantised codes, block scales and (NVFP4)
    global scale."""
    H, I, fmt = s["H"], s["I"], s["fmt"]
    rows_in, cols_out = (H, w13_rows(s)) if which == "w13" else (I, H)
    std = (1.0 / math.sqrt(rows_in)) if s["wdist"] == "fan_in" else float(s["wdist"])
    g = _expert_gen(seed, which, e, device)
    x = (torch.randn(rows_in, cols_out, generator=g, device=device,
                     dtype=torch.float32) * std).to(torch.bfloat16)
    x = x.t().contiguous()                         # [N = cols_out, K = rows_in]
    if fmt == "bf16":
        return {which: x}
    if fmt == "nvfp4":
        c, f, gsc = quantize_weight_nvfp4(x)
        return {which: c, which + "_sf": f, which + "_gs": gsc}
    c, f = quantize_weight_mxfp8(x)
    return {which: c, which + "_sf": f}


def weight_shapes(s):
    """name -> (shape, torch dtype) of the canonical weight arrays."""
    E, H, I, fmt = s["E"], s["H"], s["I"], s["fmt"]
    out = {}
    for which, (N, K) in (("w13", (w13_rows(s), H)), ("w2", (H, I))):
        if fmt == "bf16":
            out[which] = ((E, N, K), torch.bfloat16)
        elif fmt == "nvfp4":
            out[which] = ((E, N, K // 2), torch.uint8)
            out[which + "_sf"] = ((E, N, K // 16), torch.uint8)
            out[which + "_gs"] = ((E,), torch.float32)
        else:
            out[which] = ((E, N, K), torch.uint8)
            out[which + "_sf"] = ((E, N, K // 32), torch.uint8)
    return out


def draw_weights(s, seed, device):
    """Canonical weights of all experts: W13 [E, 2I, H] (rows 0..I-1 gate,
    I..2I-1 up; [E, I, H] for ReLU^2) and W2 [E, H, I], reduction dim
    contiguous.  Each expert
    matrix is drawn in the input-major shape ([H, 2I] / [I, H]), transposed
    and, for MXFP8/NVFP4, quantised."""
    out = {k: torch.empty(shape, dtype=dt, device=device)
           for k, (shape, dt) in weight_shapes(s).items()}
    for which in ("w13", "w2"):
        for e in range(s["E"]):
            for k, v in draw_expert(s, which, e, seed, device).items():
                out[k][e] = v
    return out


def host_weights(s, experts, seed=0, source=None, device="cpu"):
    """numpy weights of full shape for the oracle in which only `experts` are
    filled (the other experts' pages are never touched, so a full-size layer
    costs host memory only for the experts a sampled check needs).  Copies
    from `source` (device weights of the same seed) or draws them on
    `device` and copies them to the host."""
    import numpy as np
    out = {}
    for k, (shape, dt) in weight_shapes(s).items():
        npdt = {torch.bfloat16: np.uint16, torch.uint8: np.uint8, torch.float32: np.float32}[dt]
        out[k] = np.zeros(shape, npdt)
    for e in sorted(set(int(x) for x in experts)):
        for which in ("w13", "w2"):
            if source is not None:
                part = {k: source[k][e] for k in source if k.startswith(which)}
            else:
                part = draw_expert(s, which, e, seed, device)
            for k, v in part.items():
                v = v.detach().cpu()
                if v.dtype == torch.bfloat16:
                    v = v.view(torch.int16)
                out[k][e] = v.numpy().view(out[k].dtype) if v.dim() else v.item()
    return out


def make_case(s, T=None, seed=0, device="cpu", weights=True):
    """Draw one workload: logits then hidden from one generator, and the
    weights from per-expert generators."""
    T = s["T"] if T is None else T
    g = _gen(seed, device)
    case = {"spec": s, "T": T}
    case["logits"] = draw_logits(s, T, g, device)
    case["hidden"] = draw_hidden(s, T, g, device)
    if weights:
        case["weights"] = draw_weights(s, seed, device)
    return case


def draw_batched(s, M, seed=0, device="cpu"):
    """Batched-expert input: bf16 hidden [E, M, H] N(0,1) and int32 counts
    [E] with rows 0..counts[e]-1 of block e valid.  Counts are uniform in
    [0, M], with expert 0 empty, expert 1 full (M rows) and expert 2 holding
    one row whenever E > 2; rows past a count hold N(0,1) values too (they
    must be ignored)."""
    g = _gen(seed * 7919 + 17, device)
    E, H = s["E"], s["H"]
    counts = torch.randint(0, M + 1, (E,), generator=g, device=device, dtype=torch.int32)
    if E > 2 and M > 0:
        counts[0], counts[1], counts[2] = 0, M, 1
    hidden = torch.randn(E, M, H, generator=g, device=device,
                         dtype=torch.float32).to(torch.bfloat16).contiguous()
    return hidden, counts


def forced_empty_logits(logits, experts):
    """Force the given experts to be chosen by no token (logit -1e4)."""
    lg = logits.clone()
    lg[:, experts] = -1.0e4
    return lg


def to_numpy_case(case):
    """CPU numpy view for the oracle: bf16 as uint16 bits."""
    out = {"logits": case["logits"].detach().cpu().numpy(),
           "hidden": case["hidden"].detach().cpu().view(torch.int16).numpy().view("uint16")}
    if "weights" in case:
        w = {}
        for k, v in case["weights"].items():
            v = v.detach().cpu()
            if v.dtype == torch.bfloat16:
                w[k] = v.view(torch.int16).numpy().view("uint16")
            else:
                w[k] = v.numpy()
        out["weights"] = w
    return out
