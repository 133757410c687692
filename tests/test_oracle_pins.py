"""Pins for the CPU oracle: it is checked against things other than itself --
closed-form format definitions, library casts (torch float8/bfloat16),
hand-derived golden blocks, brute force and invariants.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.txt")


# ---------------------------------------------------------------------------
# element codecs against their closed-form definitions and library casts
# ---------------------------------------------------------------------------
def test_e2m1_decode_table():
    # OCP MX v1.0 FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 sign.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.array(mags + [-m for m in mags], np.float32)
    got = oracle.decode("e2m1", np.arange(16, dtype=np.uint8))
    assert np.array_equal(got, want)
    assert np.signbit(got[8])          # code 0x8 is negative zero


def _e4m3_closed_form(c):
    s = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 7
    if e == 0xF and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode("e4m3", codes)
    want = np.array([_e4m3_closed_form(int(c)) for c in codes], np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(got[ok], lib[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_e8m0_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode("e8m0", codes)
    want = np.array([2.0 ** (c - 127) for c in range(255)], np.float64)
    assert np.array_equal(got[:255].astype(np.float64), want)
    assert np.isnan(got[255])
    if hasattr(torch, "float8_e8m0fnu"):
        lib = torch.from_numpy(codes[:255].copy()).view(torch.float8_e8m0fnu).float().numpy()
        assert np.array_equal(got[:255], lib)


def test_encode_decode_identity_on_finite_codes():
    e4 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.encode("e4m3", oracle.decode("e4m3", e4)), e4)
    e2 = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.encode("e2m1", oracle.decode("e2m1", e2)), e2)


def _e4m3_probe_values():
    pos = np.array([_e4m3_closed_form(c) for c in range(0x7F)], np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    vals = [pos, mids]
    for m in mids:                                   # one fp32 ulp either side
        f = np.float32(m)
        vals.append(np.array([np.nextafter(f, np.float32(0)),
                              np.nextafter(f, np.float32(1e9))], np.float64))
    rng = np.random.default_rng(1)
    vals.append(np.exp(rng.uniform(math.log(1e-4), math.log(600.0), 20000)))
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v, np.float32([0.0, -0.0, 447.9, 448.0, 460.0,
                                              465.0, 1e6, -1e6])])


def test_e4m3_encode_matches_library_cast():
    x = _e4m3_probe_values()
    got = oracle.encode("e4m3", x)
    # torch's cast rounds to nearest even but does not saturate: clamp first
    lib = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
    (5.0, 0x6), (7.0, 0x7), (100.0, 0x7), (0.2, 0x0), (0.26, 0x1), (-0.3, 0x9),
    (-0.2, 0x8), (2.6, 0x5), (4.9, 0x6), (5.1, 0x7), (-6.0, 0xF), (0.0, 0x0)])
def test_e2m1_encode_hand_cases(x, code):
    # ties to the even code, saturation at 6 (OCP MX v1.0 FP4 E2M1)
    assert int(oracle.encode("e2m1", np.float32([x]))[0]) == code


def test_e2m1_encode_matches_threshold_table():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-8, 8, 50000),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])]).astype(np.float32)
    x = np.concatenate([x, -x])
    got = oracle.encode("e2m1", x)
    a = np.abs(x)
    idx = ((a > 0.25).astype(int) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
           + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    want = (idx | (np.signbit(x).astype(int) << 3)).astype(np.uint8)
    assert np.array_equal(got, want)


def test_bf16_encode_matches_library_cast():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000)).astype(np.float32)
    bits = x.view(np.uint32)
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)    # exact half-way
    x = np.concatenate([x, ties, np.float32([3.4e38, -3.4e38, 0.0, -0.0])])
    got = oracle.encode("bf16", x)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, lib)


# ---------------------------------------------------------------------------
# block quantisers and the scale fold: hand-derived golden cases
# ---------------------------------------------------------------------------
def _expand(field, conv):
    out = []
    for tok in field.split(","):
        tok = tok.strip()
        if "*" in tok:
            v, n = tok.split("*")
            out += [conv(v)] * int(n)
        else:
            out.append(conv(tok))
    return out


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            rows.append([f.strip() for f in line.split("|")])
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0] + ":" + r[1][:24])
def test_golden_blocks(row):
    kind = row[0]
    if kind == "fold":
        sf = np.uint8(int(row[1], 16))
        gs = np.float32(row[2])
        got = oracle.fold_scales(np.array([sf]), gs)[0]
        assert int(got) == int(row[3], 16)
        return
    x = np.array(_expand(row[1], float), np.float32)
    want_sf = int(row[2], 16)
    want = np.array(_expand(row[3], lambda s: int(s, 16)), np.uint8)
    codes, sf = oracle.quant_row(kind, x[None])
    assert int(sf[0, 0]) == want_sf
    if kind == "nvfp4":
        unpacked = np.empty(16, np.uint8)
        unpacked[0::2] = codes[0] & 0xF
        unpacked[1::2] = codes[0] >> 4
        assert np.array_equal(unpacked, want)
    else:
        assert np.array_equal(codes[0], want)


def test_nvfp4_round_trip_exact_on_grid():
    # blocks whose values sit on the e2m1 grid times an e4m3-exact scale
    # 2^k must dequantise to themselves
    grid = np.float32([6, -3, 0.5, 1, 1.5, 2, 4, -6, 0, 0.5, -0.5, 1, 3, -4, 2, 1.5])
    for k in range(-6, 7):
        x = (grid * np.float32(2.0 ** k))[None]
        codes, sf = oracle.quant_row("nvfp4", x)
        back = oracle.dequant_row("nvfp4", codes, sf, 16)
        assert np.array_equal(back, x), k


def test_mxfp8_round_trip_exact_on_grid():
    rng = np.random.default_rng(4)
    for X in (-20, -8, 0, 5):
        codes = rng.integers(0, 0x7E, 32).astype(np.uint8) | (rng.integers(0, 2, 32) << 7).astype(np.uint8)
        codes[0] = 0x7E                              # amax = 448 * 2^X
        x = (oracle.decode("e4m3", codes) * np.float32(2.0 ** X))[None]
        c, sf = oracle.quant_row("mxfp8", x)
        assert int(sf[0, 0]) == X + 127
        assert np.array_equal(oracle.dequant_row("mxfp8", c, sf, 32), x)


def test_nvfp4_packing_low_nibble_first():
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1] = 6.0, 0.5                      # codes 0x7 and 0x1
    codes, sf = oracle.quant_row("nvfp4", x)
    assert int(codes[0, 0]) == 0x17 and int(sf[0, 0]) == 0x38


def _ref_nvfp4_quant(x):
    """Independent restatement: scale by torch's e4m3 cast, elements by the
    threshold table; for cross-checking the oracle on random data."""
    t = torch.from_numpy(x.astype(np.float32)).view(-1, 16)
    amax = t.abs().amax(-1)
    sf = (amax / 6.0).clamp(max=448).to(torch.float8_e4m3fn)
    sv = sf.float().unsqueeze(-1)
    q = torch.where(sv == 0, torch.zeros_like(t), t / torch.where(sv == 0, torch.ones_like(sv), sv))
    a = q.abs()
    idx = ((a > 0.25).int() + (a >= 0.75).int() + (a > 1.25).int() + (a >= 1.75).int()
           + (a > 2.5).int() + (a >= 3.5).int() + (a > 5.0).int())
    code = idx | (torch.signbit(q).int() << 3)
    code = torch.where(sv == 0, torch.zeros_like(code), code)
    return code.numpy().astype(np.uint8), sf.view(torch.uint8).numpy()


def test_nvfp4_quant_random_vs_independent_restatement():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((200, 64)) * 10.0 ** rng.uniform(-4, 2, (200, 1))).astype(np.float32)
    codes, sf = oracle.quant_row("nvfp4", x)
    unpacked = np.empty((200, 64), np.uint8)
    unpacked[:, 0::2] = codes & 0xF
    unpacked[:, 1::2] = codes >> 4
    rc, rsf = _ref_nvfp4_quant(x)
    assert np.array_equal(sf.reshape(-1), rsf)
    assert np.array_equal(unpacked.reshape(-1, 16), rc)


def test_mxfp8_quant_random_vs_independent_restatement():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((100, 64)) * 10.0 ** rng.uniform(-6, 3, (100, 1))).astype(np.float32)
    codes, sf = oracle.quant_row("mxfp8", x)
    xb = x.reshape(-1, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    X = np.floor(np.log2(amax)).astype(int) - 8
    assert np.array_equal(sf.reshape(-1), (X + 127).astype(np.uint8))
    scaled = np.clip(xb * 2.0 ** (-X[:, None]), -448, 448).astype(np.float32)
    lib = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes.reshape(-1, 32), lib)


def test_fold_matches_library_cast():
    rng = np.random.default_rng(7)
    sf = rng.integers(0, 0x7E, 5000).astype(np.uint8)
    for gs in (np.float32(0.5), np.float32(3.7e-5), np.float32(1.0 / 3.0), np.float32(2.0)):
        got = oracle.fold_scales(sf, gs)
        prod = torch.from_numpy(oracle.decode("e4m3", sf)) * torch.tensor(gs)
        lib = prod.clamp(max=448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got, lib)


# ---------------------------------------------------------------------------
# routing and permutation: brute force and invariants
# ---------------------------------------------------------------------------
def _brute_topk(logits, K):
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        ids[t] = order[:K]
    return ids


@pytest.mark.parametrize("T,E,K", [(37, 8, 2), (20, 64, 6), (9, 384, 8), (5, 3, 3)])
def test_route_vs_brute_force(T, E, K):
    rng = np.random.default_rng(T * E + K)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, :] = 0.5                                  # all tied: lowest indices win
    lg[1, : E // 2] = np.float32(-0.0)
    lg[1, E // 2:] = np.float32(0.0)                # -0.0 == +0.0: index order
    ids, w = oracle.route(lg, K)
    assert np.array_equal(ids, _brute_topk(lg, K))
    assert list(ids[0]) == list(range(K))
    assert list(ids[1]) == list(range(K))
    for t in range(T):
        assert len(set(ids[t].tolist())) == K
        sel = lg[t, ids[t]].astype(np.float64)
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w[t], ref, rtol=0, atol=1e-7)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) <= 4 * 2.0 ** -24 * K
        assert np.all(np.diff(w[t]) <= 0)           # rank order: weights descend


def test_route_softmax_equals_renormalised_full_softmax():
    rng = np.random.default_rng(11)
    lg = rng.standard_normal((16, 32)).astype(np.float32)
    ids, w = oracle.route(lg, 5)
    full = torch.softmax(torch.from_numpy(lg).double(), -1).numpy()
    for t in range(16):
        p = full[t, ids[t]]
        assert np.allclose(w[t], p / p.sum(), rtol=0, atol=1e-7)


@pytest.mark.parametrize("T,E,K", [(50, 8, 2), (33, 24, 4), (1, 384, 8), (64, 5, 5)])
def test_permutation_invariants(T, E, K):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 1] = -1e4                                 # forced-empty expert
    ids, _ = oracle.route(lg, K)
    off, perm, inv = oracle.permute(ids, E)
    R = T * K
    assert off[0] == 0 and off[-1] == R and np.all(np.diff(off) >= 0)
    assert off[2] - off[1] == 0 or K == E
    assert np.array_equal(np.sort(perm), np.arange(R))       # each slot once
    assert np.array_equal(inv[perm], np.arange(R))           # inv o perm = id
    flat = ids.reshape(-1)
    ref = np.argsort(flat, kind="stable")                    # library stable sort
    assert np.array_equal(perm, ref)
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(np.diff(off), counts)
