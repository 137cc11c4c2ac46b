"""Python binding of libmoe.so (the sm_103a MoE expert layer).

Argument marshalling only: every function forwards to the C entry point of
the same name in ``include/moe.h``; all of the layer's work runs in the
library's CUDA kernels.  Tensors are passed by device pointer
(``tensor.data_ptr()``) and must already live on the GPU; the stream defaults
to PyTorch's current stream.  There is no fallback: if ``libmoe.so`` has not
been built (``python -m bit_grouped_expert_gb300.build``) the import of the
library raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARGUMENT = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_TOO_MANY_TOKENS = 5
MOE_ERR_CUDA = 6
MOE_ERR_DEVICE_TIMEOUT = 7
MOE_ERR_NONFINITE = 8
MOE_ERR_DEVICE_BOUNDS = 9

MOE_FLAG_DEBUG_CHECKS = 0x1
MOE_FLAG_FORCE_GROUPED = 0x2
MOE_FLAG_SIMT_EXPERTS = 0x4
MOE_FLAG_TILE_ROWS_64 = 0x8
MOE_FLAG_PRENORM = 0x10
MOE_FLAG_TRACE = 0x20
MOE_FLAG_TEST_WITHHOLD = 0x40
MOE_TRACE_CTAS = 256
MOE_TRACE_SLOTS = 32

EXPORTS = ("moe_plan", "moe_plan_destroy", "moe_workspace_bytes", "moe_workspace_init", "moe_route",
           "moe_route_from_logits", "moe_route_from_ids", "moe_forward", "moe_prefill_stack", "moe_router_split_bytes",
           "moe_router_split", "moe_route_view", "moe_rmsnorm", "moe_dequant",
           "moe_device_status", "moe_last_launch_count", "moe_status_str", "moe_profile_events", "moe_profile_stride",
           "moe_last_cuda_error",
           "moe_decode_static", "moe_decode_stack", "gdn_scan", "attn_decode_workspace_bytes", "attn_decode")

MOE_DECODE_STATIC_SCRATCH_BYTES = 65536

MOE_KERNEL_ROUTER = 1
MOE_KERNEL_TOPK = 2
MOE_KERNEL_SCATTER = 3
MOE_KERNEL_GATEUP = 4
MOE_KERNEL_DOWN = 5
MOE_KERNEL_COMBINE = 6
MOE_KERNEL_DECODE_LAYER = 7
MOE_KERNEL_RMSNORM = 10
MOE_KERNEL_GATHER = 11
MOE_KERNEL_GDN_SCAN = 12
MOE_KERNEL_ATTN_DECODE = 13


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: {status_str(status)} ({status})"
        if status == MOE_ERR_CUDA:
            msg += ": " + lib().moe_last_cuda_error().decode()
        super().__init__(msg)


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "n_experts", "top_k", "inter", "n_shared", "group_size")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_d", "gate_q_d", "up_q_d", "gate_s_d", "gate_b_d", "up_s_d",
                                               "up_b_d", "down_q_d", "down_s_d", "down_b_d", "shared_gate_d",
                                               "router_split_d")]


class moe_route_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("keys_d", "topk_id_d", "topk_w_d", "counts_d", "offsets_d", "perm_d",
                                               "inv_d", "blockmap_d", "n_tiles_d", "h_d", "y_d", "status_d",
                                               "trace_d")] + \
               [("max_tiles", ctypes.c_int32), ("block_rows", ctypes.c_int32), ("blockmap2_d", ctypes.c_void_p),
                ("n_tiles2_d", ctypes.c_void_p), ("max_tiles2", ctypes.c_int32), ("block_rows2", ctypes.c_int32)]


_lib = None


def lib():
    """Load libmoe.so (raises OSError if it is missing: no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"libmoe.so not built at {LIB_PATH}; run bit_grouped_expert_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t, ctypes.c_float
        L.moe_plan.restype = i32
        L.moe_plan.argtypes = [ctypes.POINTER(moe_config), i32, u32, ctypes.POINTER(vp)]
        L.moe_plan_destroy.restype = None
        L.moe_plan_destroy.argtypes = [vp]
        L.moe_workspace_bytes.restype = sz
        L.moe_workspace_bytes.argtypes = [vp]
        L.moe_workspace_init.restype = i32
        L.moe_workspace_init.argtypes = [vp, vp, sz, vp]
        L.moe_route.restype = i32
        L.moe_route.argtypes = [vp, vp, i32, vp, vp, vp, sz, vp]
        L.moe_route_from_logits.restype = i32
        L.moe_route_from_logits.argtypes = [vp, vp, i32, vp, sz, vp]
        L.moe_route_from_ids.restype = i32
        L.moe_route_from_ids.argtypes = [vp, vp, vp, i32, vp, sz, vp]
        L.moe_forward.restype = i32
        L.moe_forward.argtypes = [vp, vp, vp, i32, ctypes.POINTER(moe_weights), vp, vp, vp, sz, vp]
        L.moe_prefill_stack.restype = i32
        L.moe_prefill_stack.argtypes = [vp, vp, i32, i32, ctypes.POINTER(moe_weights), ctypes.POINTER(vp), vp, sz,
                                        vp]
        L.moe_router_split_bytes.restype = sz
        L.moe_router_split_bytes.argtypes = [i32, i32]
        L.moe_router_split.restype = i32
        L.moe_router_split.argtypes = [vp, i32, i32, vp, sz, vp]
        L.moe_route_view.restype = i32
        L.moe_route_view.argtypes = [vp, vp, i32, ctypes.POINTER(moe_route_ptrs)]
        L.moe_rmsnorm.restype = i32
        L.moe_rmsnorm.argtypes = [vp, i32, i32, f32, vp, vp]
        L.moe_dequant.restype = i32
        L.moe_dequant.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.moe_device_status.restype = i32
        L.moe_device_status.argtypes = [vp, vp, vp, ctypes.POINTER(i32), i32]
        L.moe_last_launch_count.restype = i32
        L.moe_last_launch_count.argtypes = []
        L.moe_profile_events.restype = i32
        L.moe_profile_events.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32]
        L.moe_profile_stride.restype = i32
        L.moe_profile_stride.argtypes = [i32, i32]
        L.moe_last_cuda_error.restype = ctypes.c_char_p
        L.moe_last_cuda_error.argtypes = []
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_status_str.argtypes = [i32]
        L.moe_decode_stack.restype = i32
        L.moe_decode_stack.argtypes = [vp, vp, i32, ctypes.POINTER(moe_weights), ctypes.POINTER(vp), vp, sz, vp]
        L.moe_decode_static.restype = i32
        L.moe_decode_static.argtypes = [ctypes.POINTER(moe_config), vp, vp, ctypes.POINTER(moe_weights), vp, vp, vp,
                                        u32, vp]
        L.gdn_scan.restype = i32
        L.gdn_scan.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        L.attn_decode_workspace_bytes.restype = sz
        L.attn_decode_workspace_bytes.argtypes = [i32, i32, i32]
        L.attn_decode.restype = i32
        L.attn_decode.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, vp, sz, vp, vp]
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().moe_status_str(int(status)).decode()


def _ptr(t):
    """Device pointer of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t):
    return t.numel() * t.element_size()


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)


class Plan:
    """Owns a moe_plan_t (host memory only)."""

    def __init__(self, handle: int, cfg: moe_config, max_tokens: int, flags: int):
        self.handle = handle
        self.cfg = cfg
        self.max_tokens = max_tokens
        self.flags = flags

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.moe_plan_destroy(self.handle)
            self.handle = None


def make_config(hidden=2048, n_experts=256, top_k=8, inter=512, n_shared=1, group_size=64) -> moe_config:
    return moe_config(hidden, n_experts, top_k, inter, n_shared, group_size)


def moe_plan(cfg: moe_config, max_tokens: int, flags: int = 0) -> Plan:
    h = ctypes.c_void_p()
    _check("moe_plan", lib().moe_plan(ctypes.byref(cfg), int(max_tokens), int(flags), ctypes.byref(h)))
    return Plan(h.value, cfg, max_tokens, flags)


def moe_workspace_bytes(plan: Plan) -> int:
    return int(lib().moe_workspace_bytes(plan.handle))


def moe_workspace_init(plan: Plan, ws, stream=None):
    _check("moe_workspace_init", lib().moe_workspace_init(plan.handle, _ptr(ws), _nbytes(ws), _stream(stream)))


def make_weights(w: dict) -> moe_weights:
    """moe_weights from a dict of device tensors (keys: router, gate_q, ...;
    shared_gate and router_split optional).  The caller keeps the tensors
    alive."""
    return moe_weights(*[_ptr(w.get(n[:-2])) for n, _ in moe_weights._fields_])


def moe_route(plan: Plan, x, T: int, router, logit_bias, ws, stream=None):
    _check("moe_route", lib().moe_route(plan.handle, _ptr(x), int(T), _ptr(router), _ptr(logit_bias), _ptr(ws),
                                        _nbytes(ws), _stream(stream)))


def moe_route_from_logits(plan: Plan, keys, T: int, ws, stream=None):
    _check("moe_route_from_logits", lib().moe_route_from_logits(plan.handle, _ptr(keys), int(T), _ptr(ws),
                                                                _nbytes(ws), _stream(stream)))


def moe_route_from_ids(plan: Plan, ids, w, T: int, ws, stream=None):
    _check("moe_route_from_ids", lib().moe_route_from_ids(plan.handle, _ptr(ids), _ptr(w), int(T), _ptr(ws),
                                                          _nbytes(ws), _stream(stream)))


def moe_router_split_bytes(E: int, H: int) -> int:
    return int(lib().moe_router_split_bytes(int(E), int(H)))


def moe_router_split(router, E: int, H: int, split, stream=None):
    """The router's three bf16 parts into ``split`` (a device tensor of
    moe_router_split_bytes(E, H) bytes), for the ``router_split`` weight."""
    _check("moe_router_split", lib().moe_router_split(_ptr(router), int(E), int(H), _ptr(split), _nbytes(split),
                                                      _stream(stream)))


def _weights_array(weights):
    n = len(weights)
    return (moe_weights * max(n, 1))(*[w if isinstance(w, moe_weights) else make_weights(w) for w in weights])


def _bias_array(logit_bias, n):
    if logit_bias is None:
        return None
    if len(logit_bias) != n:
        raise ValueError("one logit bias (or None) per layer")
    return (ctypes.c_void_p * max(n, 1))(*[_ptr(b) for b in logit_bias])


def moe_prefill_stack(plan: Plan, r, T: int, weights, logit_bias=None, ws=None, stream=None):
    """T tokens of the residual stream ``r`` through len(weights) pre-norm
    layers in chunks of the plan's max_tokens (chunk-major), in place."""
    n = len(weights)
    _check("moe_prefill_stack", lib().moe_prefill_stack(plan.handle, _ptr(r), int(T), n, _weights_array(weights),
                                                        _bias_array(logit_bias, n), _ptr(ws), _nbytes(ws),
                                                        _stream(stream)))


def moe_forward(plan: Plan, x, residual, T: int, weights, logit_bias, out, ws, stream=None):
    cw = weights if isinstance(weights, moe_weights) else make_weights(weights)
    _check("moe_forward", lib().moe_forward(plan.handle, _ptr(x), _ptr(residual), int(T), ctypes.byref(cw),
                                            _ptr(logit_bias), _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_decode_stack(plan: Plan, r, weights, logit_bias=None, ws=None, stream=None):
    """Single-token decode through len(weights) pre-norm layers, r updated in
    place.  ``weights``: list of weight dicts (or moe_weights); ``logit_bias``:
    None or a list of per-layer bias tensors (entries may be None)."""
    n = len(weights)
    _check("moe_decode_stack", lib().moe_decode_stack(plan.handle, _ptr(r), n, _weights_array(weights),
                                                      _bias_array(logit_bias, n), _ptr(ws), _nbytes(ws),
                                                      _stream(stream)))


def moe_decode_static(cfg: moe_config, x, residual, weights, logit_bias, out, status=None, flags: int = 0,
                      stream=None):
    """One token through the layer with no device allocation (library-owned
    static scratch; see the header).  ``status``: optional device int32."""
    cw = weights if isinstance(weights, moe_weights) else make_weights(weights)
    _check("moe_decode_static", lib().moe_decode_static(ctypes.byref(cfg), _ptr(x), _ptr(residual), ctypes.byref(cw),
                                                        _ptr(logit_bias), _ptr(out), _ptr(status), int(flags),
                                                        _stream(stream)))


def gdn_scan(q, k, v, alpha, beta, state, o, T: int, Hk: int, Hv: int, dk: int = 128, dv: int = 128, stream=None):
    """Gated DeltaNet scan of one sequence (gdn.h): q, k [T, Hk, dk] and v
    [T, Hv, dv] bf16, alpha, beta [T, Hv] fp32, state [Hv, dk, dv] fp32
    (updated in place), o [T, Hv, dv] bf16 (written)."""
    _check("gdn_scan", lib().gdn_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(state), _ptr(o),
                                      int(T), int(Hk), int(Hv), int(dk), int(dv), _stream(stream)))


def attn_decode_workspace_bytes(L: int, Hq: int = 16, D: int = 256) -> int:
    return int(lib().attn_decode_workspace_bytes(int(L), int(Hq), int(D)))


def attn_decode(q, k, v, L: int, Hq: int, Hkv: int, D: int, ws, o, scale: float = 0.0, stream=None):
    """One query token against a KV cache (attn.h): q [Hq, D], k, v [L, Hkv, D]
    bf16, ws a uint8 device tensor of attn_decode_workspace_bytes(L, Hq, D)
    bytes or more, o [Hq, D] bf16 (written)."""
    _check("attn_decode", lib().attn_decode(_ptr(q), _ptr(k), _ptr(v), int(L), int(Hq), int(Hkv), int(D),
                                            float(scale), _ptr(ws), _nbytes(ws) if not isinstance(ws, int) else 0,
                                            _ptr(o), _stream(stream)))


def moe_route_view(plan: Plan, ws, T: int) -> moe_route_ptrs:
    r = moe_route_ptrs()
    _check("moe_route_view", lib().moe_route_view(plan.handle, _ptr(ws), int(T), ctypes.byref(r)))
    return r


def workspace_tensor(ws, ptr: int, numel: int, dtype):
    """A typed view of ``numel`` elements of the workspace tensor ``ws`` (a
    uint8 tensor) starting at device address ``ptr`` (from moe_route_view)."""
    off = int(ptr) - ws.data_ptr()
    nbytes = numel * _itemsize(dtype)
    if off < 0 or off + nbytes > _nbytes(ws):
        raise ValueError("pointer range outside the workspace")
    return ws[off:off + nbytes].view(dtype)


def _itemsize(dtype):
    import torch
    return torch.empty((), dtype=dtype).element_size()


def moe_rmsnorm(r, T: int, H: int, eps: float, x, stream=None):
    _check("moe_rmsnorm", lib().moe_rmsnorm(_ptr(r), int(T), int(H), float(eps), _ptr(x), _stream(stream)))


def moe_dequant(q, s, b, rows: int, K: int, G: int, w, stream=None):
    _check("moe_dequant", lib().moe_dequant(_ptr(q), _ptr(s), _ptr(b), int(rows), int(K), int(G), _ptr(w),
                                            _stream(stream)))


def moe_device_status(plan: Plan, ws, stream=None, reset: bool = True) -> int:
    st = ctypes.c_int32(-1)
    _check("moe_device_status", lib().moe_device_status(plan.handle, _ptr(ws), _stream(stream), ctypes.byref(st),
                                                        int(bool(reset))))
    return int(st.value)


def moe_last_launch_count() -> int:
    return int(lib().moe_last_launch_count())


def moe_profile_events(kernel: int, start_events=(), stop_events=()):
    """Bracket the i-th later launch of ``kernel`` on this thread with
    ``start_events[i % n]`` / ``stop_events[i % n]`` (torch.cuda.Event objects
    created with enable_timing=True); empty lists turn the hook off."""
    n = len(start_events)
    if n != len(stop_events):
        raise ValueError("start and stop event lists differ in length")
    for e in list(start_events) + list(stop_events):
        if not e.cuda_event:  # torch creates the CUDA event lazily, on its first record
            e.record()
    arr = ctypes.c_void_p * max(n, 1)
    a = arr(*[e.cuda_event for e in start_events]) if n else None
    b = arr(*[e.cuda_event for e in stop_events]) if n else None
    _check("moe_profile_events", lib().moe_profile_events(int(kernel), a, b, n))


def moe_profile_stride(kernel: int, stride: int):
    """Bracket only every ``stride``-th launch of ``kernel`` from now on."""
    _check("moe_profile_stride", lib().moe_profile_stride(int(kernel), int(stride)))
