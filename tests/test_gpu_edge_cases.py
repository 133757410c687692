"""The method's edge cases on the GPU, bit-exact against the oracle.

- Tied router logits: rows of equal values, -0.0 beside +0.0, equal maxima
  in lanes 32 apart, ties across the top-k boundary, and rows drawn on a
  coarse grid so that ties are everywhere.  The order is value descending
  with the lower expert index first and -0.0 equal to +0.0; ids, offsets and
  the permutation must match the oracle bit for bit, through the one-kernel
  front end (T <= 16), the three-kernel one and the no-allocation entry point.
- GEMM1 input quantisation of crafted blocks: all-zero and signed-zero
  blocks, NVFP4 scales in the e4m3 subnormals, scales that round to zero (a
  tie at half the smallest subnormal included), scales that saturate at 448,
  exact e2m1 rounding ties, single outliers, bf16 subnormal inputs; for
  MXFP8 zero and subnormal block maxima, huge and tiny exponents and e4m3
  saturation after scaling.  Codes and scales must equal the oracle's.
- The prepared weight tiles: codes un-swizzled and scales read back from the
  tile layout equal the canonical codes and, for NVFP4, the oracle's folded
  scales e4m3(float(sf) * gs), byte for byte, on full-size expert matrices.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import TOL, bf16_bits_to_f64, make_layer, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- tied logits
def tied_logits(T, E, K, seed):
    """Router logits full of ties (fp32 [T, E])."""
    rng = np.random.default_rng(seed)
    lg = np.round(rng.standard_normal((T, E)) * 2.0) / 2.0      # coarse grid: ties everywhere
    lg = lg.astype(np.float32)
    lg[0, :] = 0.25                                            # all equal
    lg[1, :] = -1.0                                            # signed zeros tied at the top
    for e, v in ((2, -0.0), (5, 0.0), (37, -0.0), (69, 0.0)):
        if e < E:
            lg[1, e] = v
    lg[2, :] = -3.0                                            # equal maxima 32 lanes apart
    for e in (3, 35, 67, 99):
        if e < E:
            lg[2, e] = 3.0
    for e in (1, 33, 65):
        if e < E:
            lg[2, e] = 2.0
    base = np.sort(rng.standard_normal(E).astype(np.float32))[::-1].copy()
    lg[3, :] = base                                            # tie across the top-k boundary
    lg[3, K - 1] = lg[3, K] = base[K - 1]
    lg[4, :] = -2.0                                            # one lane, several j, all equal
    for e in range(7, E, 32):
        lg[4, e] = 1.5
    lg[5, :] = np.where(np.arange(E) % 2 == 0, 0.0, -0.0).astype(np.float32)
    return lg


def _check_routing(ids, w, off, perm, lg, K, E):
    ids_ref, w_ref = oracle.route(lg, K)
    off_ref, perm_ref, _ = oracle.permute(ids_ref, E)
    assert np.array_equal(ids, ids_ref)
    assert np.array_equal(off, off_ref)
    assert np.array_equal(perm, perm_ref)
    assert np.max(np.abs(w - w_ref)) <= 1e-6


@pytest.mark.parametrize("T,E,K", [(12, 96, 6), (16, 300, 8), (64, 96, 6), (200, 300, 8),
                                   (40, 512, 16)])
def test_tied_logits_route_bit_exact(T, E, K):
    # T <= 16 runs the one-kernel front end, larger T the three-kernel one
    s = workloads.spec("nvfp4_small", T=T, E=E, K=K)
    case = workloads.make_case(s, seed=41)
    lg = tied_logits(T, E, K, seed=T * 1000 + E)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, case["hidden"], torch.from_numpy(lg))
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    assert layer.status() == 0
    _check_routing(ids, w, off, perm, lg, K, E)
    ref = run_oracle(s, case, logits=lg)
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL["nvfp4"]
    layer.close()
    # the no-allocation entry point on the same logits
    from moe_expert_layer_histogram_gb300 import moe_route_permute_static
    dev = torch.device("cuda")
    sids = torch.empty(T, K, dtype=torch.int32, device=dev)
    sw = torch.empty(T, K, dtype=torch.float32, device=dev)
    soff = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sperm = torch.empty(T * K, dtype=torch.int32, device=dev)
    moe_route_permute_static(torch.from_numpy(lg).cuda(), T, E, K, sids, sw, soff, sperm,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    _check_routing(sids.cpu().numpy(), sw.cpu().numpy(), soff.cpu().numpy(),
                   sperm.cpu().numpy(), lg, K, E)


# ---------------------------------------------------------------- activation quantisation
def _nvfp4_blocks(rng):
    """Crafted 16-element blocks (fp32 values that are exact in bf16)."""
    b = []
    b.append(np.zeros(16))                                             # all zero
    b.append(np.where(np.arange(16) % 2, -0.0, 0.0))                   # signed zeros
    b.append(rng.standard_normal(16) * 0.004)                          # amax/6 subnormal in e4m3
    b.append(rng.standard_normal(16) * 0.0005)                         # scale rounds to 0
    t = rng.standard_normal(16) * 0.001
    t[3] = 6 * 2.0 ** -10                                              # amax/6 = 2^-10: tie -> 0
    b.append(t)
    t = rng.standard_normal(16) * 0.001
    t[9] = -6 * 2.0 ** -10 * 1.0078125                                 # just above the tie
    b.append(t)
    b.append(rng.standard_normal(16) * 3000.0)                         # scale saturates at 448
    t = np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75, -2.5, -3.5,
                  -5, -6])                                             # e2m1 ties (sf = 1)
    b.append(t)
    b.append(t * 2.0 ** -7)                                            # the same ties, subnormal sf
    t = rng.standard_normal(16) * 1e-3
    t[0] = 100.0                                                       # one outlier
    b.append(t)
    b.append(np.full(16, 1e-39) * np.sign(rng.standard_normal(16)))    # bf16 subnormal inputs
    b.append(rng.standard_normal(16))                                  # ordinary
    return b


def _mxfp8_blocks(rng):
    """Crafted 32-element blocks."""
    b = []
    b.append(np.zeros(32))
    b.append(np.where(np.arange(32) % 3 == 0, -0.0, 0.0))
    b.append(np.full(32, 1e-39) * np.sign(rng.standard_normal(32)))    # subnormal amax
    t = np.zeros(32)
    t[5] = 3e-40                                                       # one subnormal, rest zero
    b.append(t)
    b.append(rng.standard_normal(32) * 1e-30)                          # tiny exponent
    b.append(rng.standard_normal(32) * 1e37)                           # huge exponent
    t = rng.standard_normal(32) * 0.3
    t[0] = 1.9375                                                      # scaled to 496: saturates
    b.append(t)
    t = rng.standard_normal(32) * 0.1
    t[7] = 1.0625                                                      # scaled to 272: tie -> 256
    t[8] = -1.1875                                                     # scaled to 304: tie -> 320
    t[9] = 1.96875                                                     # block maximum, X = -8
    b.append(t)
    t = rng.standard_normal(32) * 1e-4
    t[1] = -50.0                                                       # one outlier
    b.append(t)
    b.append(rng.standard_normal(32))
    return b


def edge_hidden(fmt, T, H, seed):
    """bf16 hidden [T, H] whose rows cycle through the crafted blocks."""
    rng = np.random.default_rng(seed)
    blocks = _nvfp4_blocks(rng) if fmt == "nvfp4" else _mxfp8_blocks(rng)
    n = 16 if fmt == "nvfp4" else 32
    rows = []
    for t in range(T):
        row = [blocks[(t + j) % len(blocks)] for j in range(H // n)]
        rows.append(np.concatenate(row))
    x = torch.from_numpy(np.stack(rows).astype(np.float32)).to(torch.bfloat16)
    return x.contiguous()


@pytest.mark.parametrize("fmt,T", [("nvfp4", 11), ("nvfp4", 50), ("mxfp8", 13), ("mxfp8", 45)])
def test_activation_quantisation_edge_blocks_bit_exact(fmt, T):
    # T <= 16: the one-kernel front end quantises; larger T: the scatter
    name = {"nvfp4": "nvfp4_small", "mxfp8": "mxfp8_small"}[fmt]
    s = workloads.spec(name, T=T)
    case = workloads.make_case(s, seed=43)
    hid = edge_hidden(fmt, T, s["H"], seed=T)
    layer = make_layer(s, weights=case["weights"])
    run_gpu(layer, hid, case["logits"])
    codes, sf = (t.cpu().numpy() for t in layer.act_quant())
    assert layer.status() == 0
    x = bf16_bits_to_f64(hid.view(torch.int16).numpy().view(np.uint16)).astype(np.float32)
    rc, rs = oracle.quant_row(fmt, x)
    assert np.array_equal(sf, rs), "scales differ"
    assert np.array_equal(codes, rc), "codes differ"
    # the crafted blocks exercise every branch the oracle takes
    if fmt == "nvfp4":
        assert (rs == 0).any() and (rs == 0x7E).any() and (rs[(rs > 0) & (rs < 8)]).size
    else:
        assert (rs == 127).any() and (rs < 127 - 100).any() and (rs > 127 + 100).any()
    layer.close()


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_layer_output_on_edge_blocks(fmt):
    # moderate edge blocks (no overflow downstream) through the whole layer
    name = {"nvfp4": "nvfp4_small", "mxfp8": "mxfp8_small"}[fmt]
    s = workloads.spec(name, T=30)
    case = workloads.make_case(s, seed=47)
    hid = edge_hidden(fmt, 30, s["H"], seed=5)
    big = hid.float().abs() > 64.0
    hid = torch.where(big, torch.sign(hid.float()) * 4.0, hid.float()).to(torch.bfloat16)
    c2 = dict(case, hidden=hid)
    ref = run_oracle(s, c2)
    layer = make_layer(s, weights=case["weights"])
    out = run_gpu(layer, hid, case["logits"])
    assert layer.status() == 0
    assert rel_l2(out.float().cpu().numpy(), bf16_bits_to_f64(ref["out"])) <= TOL[fmt]
    layer.close()


# ---------------------------------------------------------------- prepared weight tiles
def untile(tiles, N, row_bytes, sf_tiles, interleave_half):
    """Inverse of the tile layout (see moe_debug_weight_tiles in moe.h):
    canonical codes [N, row_bytes] and scales [N, row_bytes/128 * 4 * sf_tiles]."""
    nblk, nkb = N // 128, row_bytes // 128
    tb = 16384 + 512 * sf_tiles
    t = tiles.reshape(nblk, nkb, tb)
    code = t[:, :, :16384].reshape(nblk, nkb, 128, 8, 16)
    r = np.arange(128)
    c = np.arange(8)
    pos = c[None, :] ^ (r[:, None] % 8)                        # [128, 8] stored position
    code = code[:, :, r[:, None], pos, :]                      # [nblk, nkb, 128, 8, 16]
    code = code.transpose(0, 2, 1, 3, 4).reshape(nblk * 128, row_bytes)
    sfs = None
    if sf_tiles:
        s = t[:, :, 16384:].reshape(nblk, nkb, sf_tiles, 512)
        j = np.arange(4)
        idx = (r[:, None] % 32) * 16 + (r[:, None] // 32) * 4 + j[None, :]   # [128, 4]
        s = s[:, :, :, idx]                                    # [nblk, nkb, sft, 128, 4]
        sfs = s.transpose(0, 3, 1, 2, 4).reshape(nblk * 128, nkb * sf_tiles * 4)
    if interleave_half:
        prow = np.arange(N)
        g, rr = prow // 128, prow % 128
        src = np.where(rr < 64, g * 64 + rr, interleave_half + g * 64 + rr - 64)
        out_c = np.empty_like(code)
        out_c[src] = code
        code = out_c
        if sfs is not None:
            out_s = np.empty_like(sfs)
            out_s[src] = sfs
            sfs = out_s
    return code, sfs


@pytest.mark.parametrize("name,over", [
    ("nvfp4_decode", dict(T=16, E=3, K=2)),          # full-size expert matrices
    ("mxfp8_decode", dict(T=16, E=2, K=2)),
    ("bf16_small", dict()),
    ("nvfp4_small", dict(act="relu2")),
], ids=["nvfp4-full", "mxfp8-full", "bf16", "nvfp4-relu2"])
def test_prepared_weight_tiles_equal_canonical_and_folded(name, over):
    from moe_expert_layer_histogram_gb300 import moe_debug_weight_tiles
    s = workloads.spec(name, **over)
    case = workloads.make_case(s, seed=53, device="cuda", weights=True)
    layer = make_layer(s, weights=case["weights"])
    H, I, E, fmt = s["H"], s["I"], s["E"], s["fmt"]
    sft = {"nvfp4": 4, "mxfp8": 1, "bf16": 0}[fmt]
    bpe = {"nvfp4": 0.5, "mxfp8": 1, "bf16": 2}[fmt]
    n13 = workloads.w13_rows(s)
    swiglu = s.get("act", "swiglu") == "swiglu"
    w = {k: v.cpu() for k, v in case["weights"].items()}
    for e in range(E):
        for which, N, Kd, half in ((13, n13, H, I if swiglu else 0), (2, H, I, 0)):
            rb = int(Kd * bpe)
            size = (N // 128) * (rb // 128) * (16384 + 512 * sft)
            dst = torch.empty(size, dtype=torch.uint8, device="cuda")
            moe_debug_weight_tiles(layer.handle, which, e, dst,
                                   torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            code, sfs = untile(dst.cpu().numpy(), N, rb, sft, half)
            key = "w13" if which == 13 else "w2"
            canon = w[key][e]
            if canon.dtype == torch.bfloat16:
                canon = canon.view(torch.int16)
            canon = canon.numpy().view(np.uint8).reshape(N, rb)
            assert np.array_equal(code, canon), (e, which, "codes")
            if fmt == "nvfp4":
                folded = oracle.fold_scales(w[key + "_sf"][e].numpy(), float(w[key + "_gs"][e]))
                assert np.array_equal(sfs, folded), (e, which, "folded scales")
            elif fmt == "mxfp8":
                assert np.array_equal(sfs, w[key + "_sf"][e].numpy()), (e, which, "scales")
    from moe_expert_layer_histogram_gb300 import MoEError
    with pytest.raises(MoEError) as err:                       # wrong size is refused
        moe_debug_weight_tiles(layer.handle, 13, 0, torch.empty(16, dtype=torch.uint8,
                                                               device="cuda"))
    assert err.value.code == 1
    layer.close()
