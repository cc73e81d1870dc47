"""Python binding of libmoe, the GB300 (sm_103a) MoE expert-layer library.

Argument marshalling only: every step of the layer runs in libmoe's CUDA
kernels; this module turns torch tensors into device pointers and the current
torch stream into a cudaStream_t, and raises on error codes.  PyTorch supplies
device memory and streams.  Importing fails loudly when libmoe.so has not
been built (run ``python moe_expert_layer_ep_gb300/build.py`` or
``__graft_entry__.build()``); there is no
fallback implementation.

The C functions and their contracts are declared in include/moe.h; the
functions here carry the same names.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_DTYPE_FP8 = 0
MOE_DTYPE_BF16 = 1
MOE_DTYPE_MXFP8 = 2
MOE_DTYPE_MXFP4 = 3
MOE_LAYOUT_AUTO = 0
MOE_LAYOUT_COMPACT = 1
MOE_LAYOUT_MASKED = 2

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_BUFFER_TOO_SMALL",
    4: "MOE_ERR_MISALIGNED", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_EXPERT_ID", 7: "MOE_ERR_MASKED_OVERFLOW",
    8: "MOE_ERR_TIMEOUT", 9: "MOE_ERR_DTYPE_MISMATCH",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}


class MoeError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({_lib.moe_strerror(code).decode()})")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("K", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E_global", ctypes.c_int32), ("E_local", ctypes.c_int32), ("expert_start", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("block_e", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32), ("max_m", ctypes.c_int64)]


_WS_FIELDS = ["total_bytes", "status", "meta", "counts", "padded", "start", "masked_m", "m_indices", "src2dst",
              "block_info", "chunk_hist", "chunk_rank", "a", "a_sf", "h", "h_sf", "y"]


class MoePlanOutputs(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in ("status", "meta", "counts", "padded", "start", "masked_m",
                                               "m_indices", "src2dst", "block_info")]


class MoeWsLayout(ctypes.Structure):
    _fields_ = [(f, ctypes.c_uint64) for f in _WS_FIELDS] + [
        ("rows", ctypes.c_int64), ("all_tokens", ctypes.c_int64), ("blocks", ctypes.c_int64),
        ("layout", ctypes.c_int32), ("chunks", ctypes.c_int32),
        ("block_vrow", ctypes.c_uint64), ("partial", ctypes.c_uint64),
        ("partial_rows", ctypes.c_int64), ("k_splits1", ctypes.c_int32), ("k_splits2", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run python moe_expert_layer_ep_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "moe_compact_all_tokens": (I64, [I64, I32, I32]),
        "moe_choose_layout": (I32, [I32, I32]),
        "moe_ctx_create": (I32, [P(MoeShape), VP, VP, VP, VP, P(VP)]),
        "moe_ctx_destroy": (None, [VP]),
        "moe_workspace_layout": (I32, [VP, P(MoeWsLayout)]),
        "moe_workspace_size": (I32, [VP, P(ctypes.c_size_t)]),
        "moe_plan_layout": (I32, [VP, VP, VP, VP]),
        "moe_quant_scatter": (I32, [VP, VP, VP, VP]),
        "moe_grouped_gemm_w13_act": (I32, [VP, VP, VP]),
        "moe_grouped_gemm_w2": (I32, [VP, VP, VP]),
        "moe_combine": (I32, [VP, VP, VP, VP, VP]),
        "moe_forward": (I32, [VP, VP, VP, VP, VP, VP, VP]),
        "moe_forward_launches": (I32, [VP]),
        "moe_read_device_status": (I32, [VP, VP, P(I32)]),
        "moe_clear_device_status": (I32, [VP, VP]),
        "moe_selftest_wait_timeout": (I32, [VP, I64, VP]),
        "moe_sf_offset": (I64, [I64, I64, I64, I32]),
        "moe_strerror": (ctypes.c_char_p, [I32]),
        "moe_plan_layout_noalloc": (I32, [P(MoeShape), VP, P(MoePlanOutputs), VP]),
        "moe_requant_weights_ue8m0": (I32, [VP, VP, VP, VP, I64, I64, I64, VP]),
        "moe_route": (I32, [VP, VP, I64, I64, I32, I32, VP, VP, VP, VP, I64, VP]),
        "moe_route_workspace_size": (I64, [I64, I64, I32]),
        "moe_router_prepare": (I32, [VP, VP, I64, I64, VP]),
        "moe_pack_mx_scales": (I32, [VP, I64, VP, I64, I64, I64, VP]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("moe_compact_all_tokens", "moe_choose_layout", "moe_ctx_create", "moe_ctx_destroy",
            "moe_workspace_layout", "moe_workspace_size", "moe_plan_layout", "moe_quant_scatter",
            "moe_grouped_gemm_w13_act", "moe_grouped_gemm_w2", "moe_combine", "moe_forward",
            "moe_forward_launches", "moe_read_device_status", "moe_clear_device_status",
            "moe_selftest_wait_timeout", "moe_sf_offset", "moe_strerror", "moe_plan_layout_noalloc",
            "moe_requant_weights_ue8m0", "moe_route", "moe_pack_mx_scales", "moe_route_workspace_size",
            "moe_router_prepare")


def _check(code, what):
    if code != 0:
        raise MoeError(code, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _require_cuda(name, t, dtype=None, numel=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def moe_compact_all_tokens(num_assignments, num_experts, block_e=128):
    return int(_lib.moe_compact_all_tokens(num_assignments, num_experts, block_e))


def moe_choose_layout(E_global, E_local):
    return int(_lib.moe_choose_layout(E_global, E_local))


class MoeContext:
    """Owns one moe_ctx (shape + weights); see moe_ctx_create in include/moe.h."""

    def __init__(self, handle, shape, weights):
        self.handle = handle
        self.shape = shape
        self._weights = weights   # keep the weight tensors alive with the context
        lay = MoeWsLayout()
        _check(_lib.moe_workspace_layout(handle, ctypes.byref(lay)), "moe_workspace_layout")
        self.ws_layout = lay

    @property
    def fp8(self):
        """FP8 operands (1x128 / 128x128 or MXFP8 1x32 scales)."""
        return self.shape.dtype in (MOE_DTYPE_FP8, MOE_DTYPE_MXFP8, MOE_DTYPE_MXFP4)

    @property
    def mx(self):
        """1x32 scales on activations and h (MXFP8 and MXFP4)."""
        return self.shape.dtype in (MOE_DTYPE_MXFP8, MOE_DTYPE_MXFP4)

    @property
    def masked(self):
        return self.ws_layout.layout == MOE_LAYOUT_MASKED

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.moe_ctx_destroy(h)


def make_shape(T, K, I, E_global, E_local, topk, dtype, layout=MOE_LAYOUT_AUTO, expert_start=0, max_m=0,
               block_e=128):
    if isinstance(dtype, str):
        dtype = {"fp8": MOE_DTYPE_FP8, "bf16": MOE_DTYPE_BF16, "mxfp8": MOE_DTYPE_MXFP8, "mxfp4": MOE_DTYPE_MXFP4}[dtype]
    if isinstance(layout, str):
        layout = {"auto": MOE_LAYOUT_AUTO, "compact": MOE_LAYOUT_COMPACT, "masked": MOE_LAYOUT_MASKED}[layout]
    return MoeShape(T=T, K=K, I=I, E_global=E_global, E_local=E_local, expert_start=expert_start, topk=topk,
                    block_e=block_e, dtype=dtype, layout=layout, reserved=0, max_m=max_m)


def moe_ctx_create(shape, w13, w13_sf, w2, w2_sf):
    """shape: MoeShape; weights as in include/moe.h (CUDA tensors)."""
    fp4 = shape.dtype == MOE_DTYPE_MXFP4
    mx = shape.dtype == MOE_DTYPE_MXFP8 or fp4
    fp8 = shape.dtype == MOE_DTYPE_FP8 or mx
    E, K, I = shape.E_local, shape.K, shape.I
    wdt = torch.uint8 if fp8 else torch.bfloat16
    wd = 2 if fp4 else 1      # two FP4 codes per byte
    _require_cuda("w13", w13, wdt, E * 2 * I * K // wd)
    _require_cuda("w2", w2, wdt, E * K * I // wd)
    if w13_sf is not None:
        _require_cuda("w13_sf", w13_sf, torch.uint8, E * 2 * I * K // 32 if mx else E * (2 * I // 128) * (K // 128))
    if w2_sf is not None:
        _require_cuda("w2_sf", w2_sf, torch.uint8, E * K * I // 32 if mx else E * (K // 128) * (I // 128))
    h = ctypes.c_void_p()
    _check(_lib.moe_ctx_create(ctypes.byref(shape), _ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf),
                               ctypes.byref(h)), "moe_ctx_create")
    return MoeContext(h, shape, (w13, w13_sf, w2, w2_sf))


def moe_workspace_size(ctx):
    return int(ctx.ws_layout.total_bytes)


def alloc_workspace(ctx, device=None):
    """Device workspace of moe_workspace_size bytes (torch allocation)."""
    return torch.empty(max(1, moe_workspace_size(ctx)), dtype=torch.uint8, device=device or "cuda")


def moe_plan_layout(ctx, topk_ids, ws, stream=None):
    _require_cuda("topk_ids", topk_ids, torch.int32, ctx.shape.T * ctx.shape.topk)
    _check(_lib.moe_plan_layout(ctx.handle, _ptr(topk_ids), _ptr(ws), _stream(stream)), "moe_plan_layout")


def moe_quant_scatter(ctx, x, ws, stream=None):
    _require_cuda("x", x, torch.bfloat16, ctx.shape.T * ctx.shape.K)
    _check(_lib.moe_quant_scatter(ctx.handle, _ptr(x), _ptr(ws), _stream(stream)), "moe_quant_scatter")


def moe_grouped_gemm_w13_act(ctx, ws, stream=None):
    _check(_lib.moe_grouped_gemm_w13_act(ctx.handle, _ptr(ws), _stream(stream)), "moe_grouped_gemm_w13_act")


def moe_grouped_gemm_w2(ctx, ws, stream=None):
    _check(_lib.moe_grouped_gemm_w2(ctx.handle, _ptr(ws), _stream(stream)), "moe_grouped_gemm_w2")


def moe_combine(ctx, topk_weights, ws, out, stream=None):
    _require_cuda("topk_weights", topk_weights, torch.float32, ctx.shape.T * ctx.shape.topk)
    _require_cuda("out", out, torch.bfloat16, ctx.shape.T * ctx.shape.K)
    _check(_lib.moe_combine(ctx.handle, _ptr(topk_weights), _ptr(ws), _ptr(out), _stream(stream)), "moe_combine")


def moe_forward(ctx, x, topk_ids, topk_weights, ws, out, stream=None):
    s = ctx.shape
    _require_cuda("x", x, torch.bfloat16, s.T * s.K)
    _require_cuda("topk_ids", topk_ids, torch.int32, s.T * s.topk)
    _require_cuda("topk_weights", topk_weights, torch.float32, s.T * s.topk)
    _require_cuda("out", out, torch.bfloat16, s.T * s.K)
    _check(_lib.moe_forward(ctx.handle, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(ws), _ptr(out),
                            _stream(stream)), "moe_forward")


def moe_forward_launches(ctx):
    return int(_lib.moe_forward_launches(ctx.handle))


def moe_read_device_status(ws, stream=None):
    v = ctypes.c_int32()
    _check(_lib.moe_read_device_status(_ptr(ws), _stream(stream), ctypes.byref(v)), "moe_read_device_status")
    return int(v.value)


def moe_clear_device_status(ws, stream=None):
    _check(_lib.moe_clear_device_status(_ptr(ws), _stream(stream)), "moe_clear_device_status")


def moe_selftest_wait_timeout(ws, timeout_ns, stream=None):
    _check(_lib.moe_selftest_wait_timeout(_ptr(ws), int(timeout_ns), _stream(stream)), "moe_selftest_wait_timeout")


def moe_sf_offset(block, group, n_groups, row):
    return int(_lib.moe_sf_offset(block, group, n_groups, row))


def moe_plan_layout_noalloc(shape, topk_ids, outputs, stream=None):
    """outputs: dict of int32 CUDA tensors keyed like MoePlanOutputs's fields
    (missing keys are passed as NULL)."""
    if topk_ids is not None:
        _require_cuda("topk_ids", topk_ids, torch.int32, shape.T * shape.topk)
    o = MoePlanOutputs(**{k: _ptr(v) for k, v in outputs.items()})
    _check(_lib.moe_plan_layout_noalloc(ctypes.byref(shape), _ptr(topk_ids), ctypes.byref(o), _stream(stream)),
           "moe_plan_layout_noalloc")


def moe_requant_weights_ue8m0(w_in, scale_in, w_out=None, scale_out=None, stream=None):
    """w_in uint8 [E, N, C] e4m3; scale_in float32 [E, N/128, C/128].  Returns
    (w_out, scale_out) with UE8M0 block scales (see include/moe.h)."""
    E, N, C = w_in.shape
    _require_cuda("w_in", w_in, torch.uint8)
    _require_cuda("scale_in", scale_in, torch.float32, E * (N // 128) * (C // 128))
    if w_out is None:
        w_out = torch.empty_like(w_in)
    if scale_out is None:
        scale_out = torch.empty((E, N // 128, C // 128), dtype=torch.uint8, device=w_in.device)
    _require_cuda("w_out", w_out, torch.uint8, w_in.numel())
    _require_cuda("scale_out", scale_out, torch.uint8, E * (N // 128) * (C // 128))
    _check(_lib.moe_requant_weights_ue8m0(_ptr(w_in), _ptr(scale_in), _ptr(w_out), _ptr(scale_out), E, N, C,
                                          _stream(stream)), "moe_requant_weights_ue8m0")
    return w_out, scale_out


def moe_router_prepare(w_router, out=None, stream=None):
    """fp32 router weights [E, K] -> bf16 planes [3, E, K] (hi + mid + lo == w);
    see include/moe.h."""
    E, K = w_router.shape
    _require_cuda("w_router", w_router, torch.float32)
    if out is None:
        out = torch.empty((3, E, K), dtype=torch.bfloat16, device=w_router.device)
    _require_cuda("out", out, torch.bfloat16, 3 * E * K)
    _check(_lib.moe_router_prepare(_ptr(w_router), _ptr(out), E, K, _stream(stream)), "moe_router_prepare")
    return out


def moe_route_workspace_size(T, K, E):
    return int(_lib.moe_route_workspace_size(T, K, E))


def moe_route(x, w_planes, topk, logits=None, topk_ids=None, topk_weights=None, ws=None, stream=None):
    """x bf16 [T, K], w_planes bf16 [3, E, K] (moe_router_prepare) ->
    (topk_ids int32 [T, k], topk_weights fp32 [T, k], logits fp32 [T, E]);
    see include/moe.h.  ws: uint8 device scratch (allocated here if None)."""
    T, K = x.shape
    E = w_planes.shape[1]
    _require_cuda("x", x, torch.bfloat16)
    _require_cuda("w_planes", w_planes, torch.bfloat16, 3 * E * K)
    dev = x.device
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(max(16, moe_route_workspace_size(T, K, E)), dtype=torch.uint8, device=dev)
    _require_cuda("logits", logits, torch.float32, T * E)
    _require_cuda("topk_ids", topk_ids, torch.int32, T * topk)
    _require_cuda("topk_weights", topk_weights, torch.float32, T * topk)
    _require_cuda("ws", ws, torch.uint8)
    _check(_lib.moe_route(_ptr(x), _ptr(w_planes), T, K, E, topk, _ptr(logits), _ptr(topk_ids), _ptr(topk_weights),
                          _ptr(ws), ws.numel(), _stream(stream)), "moe_route")
    return topk_ids, topk_weights, logits


def moe_pack_mx_scales(sf, out=None, stream=None, C=None):
    """MXFP8 weight scales uint8 [E, N, ld] (natural layout; ld = C/32, or
    more when the scale rows are padded, in which case pass C) -> the packed
    order moe_ctx_create takes for MOE_DTYPE_MXFP8 (see include/moe.h)."""
    E, N, ld = sf.shape
    C = ld * 32 if C is None else C
    _require_cuda("sf", sf, torch.uint8)
    if out is None:
        out = torch.empty((E, N, C // 32), dtype=torch.uint8, device=sf.device)
    _require_cuda("out", out, torch.uint8, E * N * (C // 32))
    _check(_lib.moe_pack_mx_scales(_ptr(sf), ld, _ptr(out), E, N, C, _stream(stream)), "moe_pack_mx_scales")
    return out


def ws_view(ctx, ws, name):
    """A typed torch view of one workspace intermediate (test and debug use)."""
    L, s = ctx.ws_layout, ctx.shape
    off = getattr(L, name)
    i32 = {"status": 4, "meta": 8, "counts": s.E_local, "padded": s.E_local, "start": s.E_local,
           "masked_m": s.E_local, "m_indices": L.all_tokens, "src2dst": s.T * s.topk,
           "block_info": 4 * L.blocks}
    if name in i32:
        n = i32[name]
        return ws[off:off + 4 * n].view(torch.int32)
    esz = 1 if ctx.fp8 else 2
    if name in ("a", "h", "y"):
        cols = s.I if name == "h" else s.K
        nbytes = L.rows * cols * (2 if name == "y" else esz)
        v = ws[off:off + nbytes]
        if name == "y" or not ctx.fp8:
            v = v.view(torch.bfloat16)
        return v.view(L.rows, cols)
    if name in ("a_sf", "h_sf"):
        groups = (s.K if name == "a_sf" else s.I) // 128
        return ws[off:off + L.blocks * groups * 512]
    raise KeyError(name)
