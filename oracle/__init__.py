"""CPU oracle for the fused MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library under
``moe_expert_layer_histogram_gb300`` and its binding) never does, and shares
no code with it.  The arithmetic lives in ``moe_oracle.c`` (plain C); this
module only marshals numpy arrays through ctypes.

What each function follows is documented in ``moe_oracle.h``.
"""
import ctypes
import numpy as np

from . import build as _build

FMT_BF16, FMT_MXFP8, FMT_NVFP4 = 0, 1, 2
FMT = {"bf16": FMT_BF16, "mxfp8": FMT_MXFP8, "nvfp4": FMT_NVFP4}
ACT = {"swiglu": 0, "relu2": 1}

_lib = None


class _Cfg(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("K", ctypes.c_int), ("fmt", ctypes.c_int),
                ("clamp", ctypes.c_float), ("act", ctypes.c_int)]


class _Weights(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_sf", ctypes.c_void_p),
                ("w13_gs", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_sf", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.orc_encode_n.argtypes = [ci, vp, i64, vp]
        L.orc_decode_n.argtypes = [ci, vp, i64, vp]
        L.orc_quant_row.argtypes = [ci, vp, ci, vp, vp]
        L.orc_dequant_row.argtypes = [ci, vp, vp, ci, vp]
        L.orc_fold_scales.argtypes = [vp, i64, ctypes.c_float, vp]
        L.orc_route.argtypes = [vp, ci, ci, ci, vp, vp]
        L.orc_permute.argtypes = [vp, ci, ci, ci, vp, vp, vp]
        L.orc_forward.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Weights),
                                  vp, vp, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.orc_token_forward.argtypes = [ctypes.POINTER(_Cfg),
                                        ctypes.POINTER(_Weights), vp, vp, vp, vp]
        L.orc_forward_batched.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Weights),
                                          vp, vp, ci, vp, vp]
        L.orc_num_threads.restype = ci
        L.orc_set_num_threads.argtypes = [ci]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- codecs ---------------------------------------------------------------
_KIND = {"bf16": 0, "e4m3": 1, "e2m1": 2, "e8m0": 3}


def encode(kind, x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16 if kind == "bf16" else np.uint8)
    assert lib().orc_encode_n(_KIND[kind], _p(x), x.size, _p(out)) == 0
    return out


def decode(kind, codes):
    codes = _c(codes, np.uint16 if kind == "bf16" else np.uint8)
    out = np.empty(codes.shape, np.float32)
    assert lib().orc_decode_n(_KIND[kind], _p(codes), codes.size, _p(out)) == 0
    return out


def quant_row(fmt, x):
    """Quantise rows of ``x`` (float32 [..., n]) -> (codes, scales), canonical
    packed layout (NVFP4: element 2j in the low nibble)."""
    f = FMT[fmt] if isinstance(fmt, str) else fmt
    x = _c(x, np.float32)
    n = x.shape[-1]
    rows = x.reshape(-1, n)
    cb = n // 2 if f == FMT_NVFP4 else n
    sb = n // 16 if f == FMT_NVFP4 else n // 32
    codes = np.empty((rows.shape[0], cb), np.uint8)
    sf = np.empty((rows.shape[0], sb), np.uint8)
    for r in range(rows.shape[0]):
        assert lib().orc_quant_row(f, _p(rows[r]), n, _p(codes[r]), _p(sf[r])) == 0
    return codes.reshape(x.shape[:-1] + (cb,)), sf.reshape(x.shape[:-1] + (sb,))


def dequant_row(fmt, codes, sf, n):
    f = FMT[fmt] if isinstance(fmt, str) else fmt
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    c2 = codes.reshape(-1, codes.shape[-1])
    s2 = sf.reshape(-1, sf.shape[-1])
    out = np.empty((c2.shape[0], n), np.float32)
    for r in range(c2.shape[0]):
        assert lib().orc_dequant_row(f, _p(c2[r]), _p(s2[r]), n, _p(out[r])) == 0
    return out.reshape(codes.shape[:-1] + (n,))


def fold_scales(sf, gs):
    sf = _c(sf, np.uint8)
    out = np.empty_like(sf)
    lib().orc_fold_scales(_p(sf), sf.size, float(gs), _p(out))
    return out


# ---- routing / permutation -----------------------------------------------
def route(logits, K):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    lib().orc_route(_p(logits), T, E, K, _p(ids), _p(w))
    return ids, w


def permute(ids, E):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    off = np.empty(E + 1, np.int32)
    perm = np.empty(T * K, np.int32)
    inv = np.empty(T * K, np.int32)
    lib().orc_permute(_p(ids), T, K, E, _p(off), _p(perm), _p(inv))
    return off, perm, inv


# ---- the layer --------------------------------------------------------------
def _pack(cfg, weights):
    c = _Cfg(cfg["H"], cfg["I"], cfg["E"], cfg["K"], FMT[cfg["fmt"]],
             float(cfg.get("clamp", 0.0) or 0.0), ACT[cfg.get("act", "swiglu")])
    keep = {}
    ptrs = []
    for name in ("w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs"):
        a = weights.get(name)
        if a is not None:
            a = np.ascontiguousarray(a)
            keep[name] = a
        ptrs.append(_p(a))
    return c, _Weights(*ptrs), keep


def forward(cfg, weights, hidden, logits, want_intermediates=False):
    """Whole layer.  ``hidden``: uint16 bf16 bits [T,H]; ``logits``: f32
    [T,E]; ``weights``: dict of canonical numpy arrays.  Returns a dict with
    ``out`` (uint16 bf16 bits [T,H]) and, on request, ids, w, offsets, perm,
    xq_codes, xq_sf, h [T*K,I], y [T*K,H]."""
    c, W, keep = _pack(cfg, weights)
    hidden = _c(hidden, np.uint16)
    logits = _c(logits, np.float32)
    T, H = hidden.shape
    I, E, K = cfg["I"], cfg["E"], cfg["K"]
    f = FMT[cfg["fmt"]]
    R = T * K
    res = {"out": np.empty((T, H), np.uint16),
           "ids": np.empty((T, K), np.int32), "w": np.empty((T, K), np.float32),
           "offsets": np.empty(E + 1, np.int32), "perm": np.empty(R, np.int32)}
    if want_intermediates:
        if f != FMT_BF16:
            res["xq_codes"] = np.empty((T, H // 2 if f == FMT_NVFP4 else H), np.uint8)
            res["xq_sf"] = np.empty((T, H // 16 if f == FMT_NVFP4 else H // 32), np.uint8)
        res["h"] = np.empty((R, I), np.float32)
        res["y"] = np.empty((R, H), np.float32)
    rc = lib().orc_forward(ctypes.byref(c), ctypes.byref(W), _p(hidden), _p(logits), T,
                           _p(res["out"]), _p(res["ids"]), _p(res["w"]),
                           _p(res["offsets"]), _p(res["perm"]),
                           _p(res.get("xq_codes")), _p(res.get("xq_sf")),
                           _p(res.get("h")), _p(res.get("y")))
    assert rc == 0, rc
    del keep
    return res


def token_forward(cfg, weights, hidden_row, logits_row):
    """Brute-force single-token evaluation (no permutation).  Returns
    (out_f32 [H], out_bf16_bits [H])."""
    c, W, keep = _pack(cfg, weights)
    hidden_row = _c(hidden_row, np.uint16)
    logits_row = _c(logits_row, np.float32)
    H = cfg["H"]
    of = np.empty(H, np.float32)
    ob = np.empty(H, np.uint16)
    assert lib().orc_token_forward(ctypes.byref(c), ctypes.byref(W), _p(hidden_row),
                                   _p(logits_row), _p(of), _p(ob)) == 0
    del keep
    return of, ob


def forward_batched(cfg, weights, hidden, counts, want_y=False):
    """Batched-expert format.  ``hidden``: uint16 bf16 bits [E,M,H];
    ``counts``: int32 [E] (rows 0..counts[e]-1 of block e are expert e's).
    Returns ``out`` uint16 [E,M,H] (rows past counts[e] zero) and, on
    request, ``y`` float32 [E,M,H]."""
    c, W, keep = _pack(cfg, weights)
    hidden = _c(hidden, np.uint16)
    counts = _c(counts, np.int32)
    E, M, H = hidden.shape
    res = {"out": np.zeros((E, M, H), np.uint16)}
    if want_y:
        res["y"] = np.zeros((E, M, H), np.float32)
    rc = lib().orc_forward_batched(ctypes.byref(c), ctypes.byref(W), _p(hidden), _p(counts),
                                   M, _p(res["out"]), _p(res.get("y")))
    assert rc == 0, rc
    del keep
    return res


def num_threads():
    return lib().orc_num_threads()


def set_num_threads(n):
    lib().orc_set_num_threads(int(n))
