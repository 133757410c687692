"""Layer-level pins for the oracle (CPU only).

- The permuted, expert-by-expert forward equals a brute-force per-token
  evaluation that never permutes (bit-exact).
- With top-k = E the layer is a dense softmax-weighted sum over all experts;
  an independent torch restatement on library primitives agrees.
- Top-k < E against the same restatement with torch.topk; clamp on and off;
  forced-empty experts and a one-row expert.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import refs


def _case(name, seed=0, **over):
    s = workloads.spec(name, **over)
    c = workloads.make_case(s, seed=seed)
    return s, workloads.to_numpy_case(c)


def _cfg(s):
    return dict(H=s["H"], I=s["I"], E=s["E"], K=s["K"], fmt=s["fmt"], clamp=s["clamp"],
                act=s.get("act", "swiglu"))


TINY = [
    ("tiny_bf16", dict()),
    ("bf16_small", dict(T=12, H=128, I=64, E=6, K=3)),
    ("mxfp8_small", dict(T=10, H=128, I=64, E=5, K=2)),
    ("nvfp4_small", dict(T=11, H=128, I=64, E=7, K=3)),
    ("nvfp4_zipf_small", dict(T=9, H=64, I=32, E=9, K=4)),
]


@pytest.mark.parametrize("name,over", TINY, ids=[t[0] for t in TINY])
def test_permuted_forward_equals_per_token_brute_force(name, over):
    s, c = _case(name, **over)
    cfg = _cfg(s)
    res = oracle.forward(cfg, c["weights"], c["hidden"], c["logits"])
    for t in range(c["hidden"].shape[0]):
        _, ob = oracle.token_forward(cfg, c["weights"], c["hidden"][t], c["logits"][t])
        assert np.array_equal(ob, res["out"][t]), t


def _dequant(s, w):
    fmt = s["fmt"]
    W13 = refs.dequant_weights(fmt, w["w13"], w.get("w13_sf"), w.get("w13_gs"))
    W2 = refs.dequant_weights(fmt, w["w2"], w.get("w2_sf"), w.get("w2_gs"))
    return W13, W2


@pytest.mark.parametrize("fmt,clamp", [("bf16", 0.0), ("bf16", 0.4), ("mxfp8", 0.0),
                                       ("nvfp4", 0.0), ("nvfp4", 0.05)])
def test_dense_special_case_k_equals_e(fmt, clamp):
    name = {"bf16": "bf16_small", "mxfp8": "mxfp8_small", "nvfp4": "nvfp4_small"}[fmt]
    s, c = _case(name, T=6, H=64 if fmt != "mxfp8" else 64, I=32, E=4, K=4, clamp=clamp)
    cfg = _cfg(s)
    W13, W2 = _dequant(s, c["weights"])
    ref = refs.dense_layer_f64(fmt, clamp, c["hidden"], c["logits"], W13, W2, s["E"])
    for t in range(6):
        of, _ = oracle.token_forward(cfg, c["weights"], c["hidden"][t], c["logits"][t])
        assert refs.rel_l2(of, ref[t].numpy()) < 2e-6, t


@pytest.mark.parametrize("name,over", TINY[1:], ids=[t[0] for t in TINY[1:]])
def test_topk_layer_vs_restatement(name, over):
    s, c = _case(name, seed=3, **over)
    cfg = _cfg(s)
    W13, W2 = _dequant(s, c["weights"])
    ref = refs.dense_layer_f64(s["fmt"], s["clamp"], c["hidden"], c["logits"], W13, W2, s["K"])
    res = oracle.forward(cfg, c["weights"], c["hidden"], c["logits"])
    out = refs.bf16_bits_to_f32(res["out"])
    # the only differences left are bf16 rounding of the output
    assert refs.rel_l2(out, ref.numpy()) < 4e-3
    # and before the final rounding they agree to fp32 precision
    for t in range(min(4, c["hidden"].shape[0])):
        of, _ = oracle.token_forward(cfg, c["weights"], c["hidden"][t], c["logits"][t])
        assert refs.rel_l2(of, ref[t].numpy()) < 2e-6


def test_clamp_changes_result_and_is_symmetric():
    # a plausible mistake is clamping only the gate, or only one side
    s, c = _case("bf16_small", T=4, H=64, I=32, E=3, K=2, clamp=0.0)
    W13, W2 = _dequant(s, c["weights"])
    base = oracle.forward(_cfg(s), c["weights"], c["hidden"], c["logits"])["out"]
    s2 = dict(s, clamp=0.05)
    clamped = oracle.forward(_cfg(s2), c["weights"], c["hidden"], c["logits"])["out"]
    assert not np.array_equal(base, clamped)
    ref = refs.dense_layer_f64("bf16", 0.05, c["hidden"], c["logits"], W13, W2, 2)
    assert refs.rel_l2(refs.bf16_bits_to_f32(clamped), ref.numpy()) < 4e-3


def test_forced_empty_and_single_row_experts():
    s, c = _case("nvfp4_small", T=9, H=64, I=32, E=8, K=2)
    lg = c["logits"].copy()
    lg[:, [2, 5]] = -1.0e4                          # experts 2, 5 chosen by nobody
    lg[:, 7] = -1.0e4
    lg[4, 7] = 1.0e4                                # expert 7 gets exactly one row
    res = oracle.forward(_cfg(s), c["weights"], c["hidden"], lg)
    off = res["offsets"]
    assert off[3] - off[2] == 0 and off[6] - off[5] == 0
    assert off[8] - off[7] == 1
    for t in range(9):
        _, ob = oracle.token_forward(_cfg(s), c["weights"], c["hidden"][t], lg[t])
        assert np.array_equal(ob, res["out"][t])


def test_zero_tokens():
    s, c = _case("tiny_bf16")
    res = oracle.forward(_cfg(s), c["weights"], c["hidden"][:0], c["logits"][:0])
    assert res["out"].shape == (0, s["H"])


def test_intermediates_shapes_and_activation_codes():
    s, c = _case("nvfp4_small", T=5, H=64, I=32, E=4, K=2)
    res = oracle.forward(_cfg(s), c["weights"], c["hidden"], c["logits"],
                         want_intermediates=True)
    x = refs.bf16_bits_to_f32(c["hidden"])
    codes, sf = oracle.quant_row("nvfp4", x)
    assert np.array_equal(res["xq_codes"], codes) and np.array_equal(res["xq_sf"], sf)
    assert res["h"].shape == (10, 32) and res["y"].shape == (10, 64)


# ---- the non-gated ReLU^2 activation ---------------------------------------
RELU2 = [
    ("bf16_small", dict(T=10, H=128, I=64, E=5, K=2, clamp=0.0, act="relu2")),
    ("mxfp8_small", dict(T=9, H=128, I=64, E=4, K=2, act="relu2")),
    ("nvfp4_small", dict(T=11, H=128, I=64, E=6, K=3, act="relu2")),
]


@pytest.mark.parametrize("name,over", RELU2, ids=[t[0] for t in RELU2])
def test_relu2_layer_vs_restatement_and_brute_force(name, over):
    s, c = _case(name, seed=8, **over)
    cfg = _cfg(s)
    assert c["weights"]["w13"].shape[1] == s["I"]          # one projection, I rows
    W13, W2 = _dequant(s, c["weights"])
    ref = refs.dense_layer_f64(s["fmt"], 0.0, c["hidden"], c["logits"], W13, W2, s["K"],
                               act="relu2")
    res = oracle.forward(cfg, c["weights"], c["hidden"], c["logits"])
    assert refs.rel_l2(refs.bf16_bits_to_f32(res["out"]), ref.numpy()) < 4e-3
    for t in range(c["hidden"].shape[0]):
        of, ob = oracle.token_forward(cfg, c["weights"], c["hidden"][t], c["logits"][t])
        assert np.array_equal(ob, res["out"][t]), t
        assert refs.rel_l2(of, ref[t].numpy()) < 2e-6, t


def test_relu2_is_not_swiglu_and_is_nonnegative_before_gemm2():
    # h = max(G, 0)^2 >= 0 (a sign or gating mistake shows up here)
    s, c = _case("bf16_small", seed=2, T=6, H=64, I=32, E=3, K=2, clamp=0.0, act="relu2")
    res = oracle.forward(_cfg(s), c["weights"], c["hidden"], c["logits"],
                         want_intermediates=True)
    assert (res["h"] >= 0).all() and (res["h"] == 0).any() and (res["h"] > 0).any()


def test_relu2_rejects_clamp():
    s, c = _case("bf16_small", T=4, H=64, I=32, E=3, K=2, clamp=0.0, act="relu2")
    cfg = dict(_cfg(s), clamp=3.0)
    with pytest.raises(AssertionError):
        oracle.forward(cfg, c["weights"], c["hidden"], c["logits"])


# ---- the batched-expert format ----------------------------------------------
BATCHED = [
    ("bf16_small", dict(H=128, I=64, E=4, clamp=0.5), 5),
    ("mxfp8_small", dict(H=128, I=64, E=4), 6),
    ("nvfp4_small", dict(H=128, I=64, E=5), 7),
    ("nvfp4_small", dict(H=128, I=64, E=4, act="relu2"), 3),
]


@pytest.mark.parametrize("name,over,M", BATCHED, ids=["%s-%d" % (b[0], i) for i, b in enumerate(BATCHED)])
def test_batched_format_vs_restatement(name, over, M):
    import torch
    s = workloads.spec(name, **over)
    w = workloads.to_numpy_case(workloads.make_case(s, T=1, seed=4))["weights"]
    hid, counts = workloads.draw_batched(s, M, seed=4)
    hb = hid.view(torch.int16).numpy().view("uint16")
    cn = counts.numpy()
    assert cn[0] == 0 and cn[1] == M and cn[2] == 1
    res = oracle.forward_batched(_cfg(s), w, hb, cn, want_y=True)
    W13, W2 = _dequant(s, w)
    for e in range(s["E"]):
        for r in range(M):
            if r >= cn[e]:
                assert not res["out"][e, r].any()        # rows past the count untouched
                continue
            a = refs.gemm1_input_f64(s["fmt"], hb[e, r:r + 1])[0]
            y = refs.expert_mlp_f64(s["fmt"], s["clamp"], a, W13[e], W2[e], s["act"])
            assert refs.rel_l2(res["y"][e, r], y.numpy()) < 2e-6, (e, r)
    # the output is the bf16 rounding of y
    y32 = torch.from_numpy(res["y"])
    assert np.array_equal(y32.to(torch.bfloat16).view(torch.int16).numpy().view("uint16"),
                          res["out"])


def test_batched_rows_match_the_routed_layer_rows():
    # a batched call whose rows are the routed layer's permuted rows gives
    # that layer's GEMM2 output row for row
    s, c = _case("mxfp8_small", seed=5, T=7, H=128, I=64, E=4, K=2)
    cfg = _cfg(s)
    res = oracle.forward(cfg, c["weights"], c["hidden"], c["logits"], want_intermediates=True)
    off, perm = res["offsets"], res["perm"]
    counts = np.diff(off).astype(np.int32)
    M = int(counts.max())
    hid = np.zeros((s["E"], M, s["H"]), np.uint16)
    for e in range(s["E"]):
        for r in range(counts[e]):
            hid[e, r] = c["hidden"][perm[off[e] + r] // s["K"]]
    b = oracle.forward_batched(cfg, c["weights"], hid, counts, want_y=True)
    for e in range(s["E"]):
        assert np.array_equal(b["y"][e, :counts[e]], res["y"][off[e]:off[e + 1]])
