"""GB300 fused Mixture-of-Experts expert layer -- Python binding.

A thin ctypes binding of the C ABI declared in ``include/moe.h`` with the same
entry-point names (``moe_create``, ``moe_prepare_weights``, ``moe_forward``,
``moe_destroy`` ...).  It only marshals arguments: every step of the layer
(routing, permutation, activation quantisation, both grouped GEMMs, SwiGLU,
re-quantisation, combine) runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  There is no CPU fallback: if the CUDA
library is missing, loading fails with an error.
"""
import ctypes
import os

from . import _build

LIB_PATH = _build.LIB

MOE_FMT = {"bf16": 0, "mxfp8": 1, "nvfp4": 2}
MOE_ACT = {"swiglu": 0, "relu2": 1}
MOE_COMBINE = {"gather": 0, "reduce": 1, "fused": 2}
MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_NO_WEIGHTS", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_OOM",
                6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_NO_DEVICE"}


class MoEConfig(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int), ("hidden", ctypes.c_int),
                ("inter", ctypes.c_int), ("num_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("format", ctypes.c_int),
                ("clamp_limit", ctypes.c_float), ("activation", ctypes.c_int),
                ("combine", ctypes.c_int), ("max_ctas", ctypes.c_int),
                ("test_fail_alloc_at", ctypes.c_int), ("test_stall_gemm", ctypes.c_int)]


class MoEError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(code, code),
                                           moe_status_string(code)))


EXPORTS = ("moe_create", "moe_prepare_weights", "moe_forward", "moe_forward_batched",
           "moe_forward_host", "moe_forward_host_async",
           "moe_debug_routing", "moe_debug_act_quant", "moe_debug_intermediates",
           "moe_debug_weight_tiles",
           "moe_get_status", "moe_timing_start", "moe_timing_stop", "moe_last_launch_count",
           "moe_gemm_ctas",
           "moe_route_permute_static", "moe_measure_mma_rate", "moe_status_string",
           "moe_destroy")

_lib = None


def lib():
    """Load the CUDA library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, ci = ctypes.c_void_p, ctypes.c_int
    L.moe_create.argtypes = [ctypes.POINTER(MoEConfig), ctypes.POINTER(vp)]
    L.moe_prepare_weights.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_forward.argtypes = [vp, vp, vp, vp, ci, vp]
    L.moe_forward_host.argtypes = [vp, vp, vp, vp, ci, vp]
    L.moe_forward_host_async.argtypes = [vp, vp, vp, vp, ci, vp]
    L.moe_forward_batched.argtypes = [vp, vp, vp, ci, vp, vp]
    L.moe_debug_routing.argtypes = [vp, vp, vp, vp, vp, vp]
    L.moe_debug_act_quant.argtypes = [vp, vp, vp, vp]
    L.moe_debug_intermediates.argtypes = [vp, vp, vp, vp]
    L.moe_debug_weight_tiles.argtypes = [vp, ci, ci, vp, ctypes.c_size_t, vp]
    L.moe_get_status.argtypes = [vp]
    L.moe_timing_start.argtypes = [vp, ci]
    L.moe_timing_stop.argtypes = [vp, vp, vp]
    L.moe_last_launch_count.argtypes = [vp]
    L.moe_gemm_ctas.argtypes = [vp, ci]
    L.moe_route_permute_static.argtypes = [vp, ci, ci, ci, vp, vp, vp, vp, vp]
    L.moe_measure_mma_rate.argtypes = [ci, ci, ci, ci, ctypes.POINTER(ctypes.c_double), vp]
    L.moe_status_string.argtypes = [ci]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_destroy.argtypes = [vp]
    L.moe_destroy.restype = None
    for name in EXPORTS:
        if name not in ("moe_status_string", "moe_destroy"):
            getattr(L, name).restype = ci
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(code, where):
    if code != MOE_OK:
        raise MoEError(code, where)


# ---- the C entry points, same names -------------------------------------------
def moe_status_string(code):
    return lib().moe_status_string(int(code)).decode()


def moe_create(max_tokens, hidden, inter, num_experts, top_k, fmt, clamp_limit=0.0,
               activation="swiglu", combine="gather", max_ctas=0, test_fail_alloc_at=0,
               test_stall_gemm=0):
    cfg = MoEConfig(int(max_tokens), int(hidden), int(inter), int(num_experts), int(top_k),
                    MOE_FMT[fmt] if isinstance(fmt, str) else int(fmt), float(clamp_limit or 0.0),
                    MOE_ACT[activation] if isinstance(activation, str) else int(activation),
                    MOE_COMBINE[combine] if isinstance(combine, str) else int(combine),
                    int(max_ctas), int(test_fail_alloc_at), int(test_stall_gemm))
    h = ctypes.c_void_p()
    _check(lib().moe_create(ctypes.byref(cfg), ctypes.byref(h)), "moe_create")
    return h.value


def moe_prepare_weights(handle, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, stream=None):
    _check(lib().moe_prepare_weights(handle, _ptr(w13), _ptr(w13_sf), _ptr(w13_gs), _ptr(w2),
                                     _ptr(w2_sf), _ptr(w2_gs), stream),
           "moe_prepare_weights")


def moe_forward(handle, hidden, router_logits, out, T, stream=None):
    _check(lib().moe_forward(handle, _ptr(hidden), _ptr(router_logits), _ptr(out), int(T), stream),
           "moe_forward")


def moe_forward_batched(handle, hidden, counts, M, out, stream=None):
    _check(lib().moe_forward_batched(handle, _ptr(hidden), _ptr(counts), int(M), _ptr(out),
                                     stream), "moe_forward_batched")


def moe_forward_host(handle, hidden_host, router_logits_host, out_host, T, stream=None):
    _check(lib().moe_forward_host(handle, _ptr(hidden_host), _ptr(router_logits_host),
                                  _ptr(out_host), int(T), stream), "moe_forward_host")


def moe_forward_host_async(handle, hidden_host, router_logits_host, out_host, T, stream=None):
    """Pipelined host-buffer forward: returns at once; `stream` completes
    once out_host holds the result (keep the host buffers until then)."""
    _check(lib().moe_forward_host_async(handle, _ptr(hidden_host), _ptr(router_logits_host),
                                        _ptr(out_host), int(T), stream), "moe_forward_host_async")


def moe_debug_routing(handle, topk_ids=None, topk_w=None, offsets=None, perm=None, stream=None):
    _check(lib().moe_debug_routing(handle, _ptr(topk_ids), _ptr(topk_w), _ptr(offsets),
                                   _ptr(perm), stream), "moe_debug_routing")


def moe_debug_act_quant(handle, codes, scales, stream=None):
    _check(lib().moe_debug_act_quant(handle, _ptr(codes), _ptr(scales), stream),
           "moe_debug_act_quant")


def moe_debug_intermediates(handle, h=None, y=None, stream=None):
    _check(lib().moe_debug_intermediates(handle, _ptr(h), _ptr(y), stream),
           "moe_debug_intermediates")


def moe_debug_weight_tiles(handle, which, expert, dst, stream=None):
    """Copy expert `expert`'s prepared W13 (which=13) or W2 (which=2) tiles
    into `dst` (a uint8 tensor of exactly the tiles' size)."""
    _check(lib().moe_debug_weight_tiles(handle, int(which), int(expert), _ptr(dst),
                                        dst.numel() * dst.element_size(), stream),
           "moe_debug_weight_tiles")


def moe_get_status(handle):
    return lib().moe_get_status(handle)


KERNELS = ("route_hist", "scan", "scatter_quant", "gemm1_swiglu", "gemm2", "combine")


def moe_timing_start(handle, max_forwards):
    _check(lib().moe_timing_start(handle, int(max_forwards)), "moe_timing_start")


def moe_timing_stop(handle):
    """Returns ({kernel name: summed ms}, number of recorded forwards)."""
    ms = (ctypes.c_float * 6)()
    n = ctypes.c_int()
    _check(lib().moe_timing_stop(handle, ms, ctypes.byref(n)), "moe_timing_stop")
    return dict(zip(KERNELS, list(ms))), n.value


def moe_last_launch_count(handle):
    return lib().moe_last_launch_count(handle)


def moe_gemm_ctas(handle, wide):
    return lib().moe_gemm_ctas(handle, int(bool(wide)))


def moe_route_permute_static(router_logits, T, E, K, topk_ids, topk_w, offsets, perm,
                             stream=None):
    """Routing + expert permutation with no device allocation (for callers
    that cannot allocate; scratch is a fixed array inside the library, so
    T <= 4096 and concurrent calls on the GPU must not overlap)."""
    _check(lib().moe_route_permute_static(_ptr(router_logits), int(T), int(E), int(K),
                                          _ptr(topk_ids), _ptr(topk_w), _ptr(offsets),
                                          _ptr(perm), stream), "moe_route_permute_static")


def moe_measure_mma_rate(fmt, n_cols=128, copy_scales=False, iters=20000, stream=None):
    """Dense TFLOP/s of the layer's MMA kind for `fmt` on the current GPU
    (tcgen05.mma on shared-memory-resident operands, one CTA per SM)."""
    out = ctypes.c_double()
    _check(lib().moe_measure_mma_rate(MOE_FMT[fmt] if isinstance(fmt, str) else int(fmt),
                                      int(n_cols), int(bool(copy_scales)), int(iters),
                                      ctypes.byref(out), stream), "moe_measure_mma_rate")
    return out.value


def moe_destroy(handle):
    if handle:
        lib().moe_destroy(handle)


# ---- torch convenience wrapper -------------------------------------------------
class MoELayer:
    """One layer on the current CUDA device; tensors are torch CUDA tensors,
    work goes on torch's current stream."""

    def __init__(self, max_tokens, hidden, inter, num_experts, top_k, fmt, clamp_limit=0.0,
                 activation="swiglu", combine="gather", **config):
        import torch
        self.torch = torch
        self.H, self.I, self.E, self.K = hidden, inter, num_experts, top_k
        self.fmt = fmt
        self.max_tokens = max_tokens
        self.handle = moe_create(max_tokens, hidden, inter, num_experts, top_k, fmt, clamp_limit,
                                 activation, combine, **config)
        self.T = 0

    def _stream(self):
        return self.torch.cuda.current_stream().cuda_stream

    def prepare_weights(self, w):
        for v in w.values():
            assert v.is_cuda and v.is_contiguous()
        moe_prepare_weights(self.handle, w["w13"], w.get("w13_sf"), w.get("w13_gs"), w["w2"],
                            w.get("w2_sf"), w.get("w2_gs"), self._stream())

    def forward(self, hidden, router_logits, out=None):
        torch = self.torch
        T = hidden.shape[0]
        assert hidden.is_cuda and hidden.dtype == torch.bfloat16 and hidden.is_contiguous()
        assert router_logits.dtype == torch.float32 and router_logits.is_contiguous()
        if out is None:
            out = torch.empty_like(hidden)
        moe_forward(self.handle, hidden, router_logits, out, T, self._stream())
        self.T = T
        return out

    def forward_batched(self, hidden, counts, out=None):
        """hidden bf16 [E, M, H], counts int32 [E] (device) -> out bf16
        [E, M, H] (rows past a count are left as they are)."""
        torch = self.torch
        E, M, H = hidden.shape
        assert E == self.E and H == self.H and hidden.dtype == torch.bfloat16
        assert hidden.is_cuda and hidden.is_contiguous() and counts.dtype == torch.int32
        if out is None:
            out = torch.zeros_like(hidden)
        moe_forward_batched(self.handle, hidden, counts, M, out, self._stream())
        return out

    def routing(self):
        torch = self.torch
        T, K, E = self.T, self.K, self.E
        dev = torch.device("cuda")
        ids = torch.empty(T, K, dtype=torch.int32, device=dev)
        w = torch.empty(T, K, dtype=torch.float32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        moe_debug_routing(self.handle, ids, w, off, perm, self._stream())
        return ids, w, off, perm

    def act_quant(self):
        torch = self.torch
        T, H = self.T, self.H
        cb = H // 2 if self.fmt == "nvfp4" else H
        nsf = H // 16 if self.fmt == "nvfp4" else H // 32
        codes = torch.empty(T, cb, dtype=torch.uint8, device="cuda")
        sf = torch.empty(T, nsf, dtype=torch.uint8, device="cuda")
        moe_debug_act_quant(self.handle, codes, sf, self._stream())
        return codes, sf

    def intermediates(self):
        torch = self.torch
        R = self.T * self.K
        h = torch.empty(R, self.I, dtype=torch.float32, device="cuda")
        y = torch.empty(R, self.H, dtype=torch.float32, device="cuda")
        moe_debug_intermediates(self.handle, h, y, self._stream())
        return h, y

    def status(self):
        return moe_get_status(self.handle)

    def close(self):
        if self.handle:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
