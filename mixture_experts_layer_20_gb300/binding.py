"""Thin Python binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch supplies device memory and the current stream.  Importing this
module fails loudly when the library has not been built (run
``python -m mixture_experts_layer_20_gb300.build`` or
``__graft_entry__.build()``); there is no fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python -m mixture_experts_layer_20_gb300.build)")
_lib = ctypes.CDLL(LIB_PATH)

_vp, _i, _sz, _st = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "router_logits", "topk_ids", "topk_gates", "expert_counts", "expert_offsets", "perm",
        "slot_pos", "chunk_table", "x_perm", "h", "h_shared", "y", "y_shared", "x_stage",
        "out_stage", "act_x", "act_x_scales", "act_h", "act_h_scales", "total")]


class ForwardExt(ctypes.Structure):
    _fields_ = [("router_bias", _vp), ("w_gate_up_shared", _vp), ("w_down_shared", _vp),
                ("I_shared", _i), ("bias_selection_only", _i), ("single_launch", _i),
                ("y_fp32", _i), ("act_mxfp8", _i)]


_SIGS = {
    "moe_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_workspace_init": (_st, [_vp, _sz, _vp]),
    "moe_route": (_st, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_ex": (_st, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "moe_forward_graph": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp, _i,
                                ctypes.POINTER(ctypes.c_void_p)]),
    "moe_graph_launch": (_st, [_vp, _vp]),
    "moe_mxfp8_quantize": (_st, [_vp, ctypes.c_longlong, _i, _vp, _vp, _vp]),
    "moe_forward_mxfp8": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz,
                                _vp, _vp]),
    "moe_nvfp4_quantize": (_st, [_vp, _i, ctypes.c_longlong, _i, _vp, _vp, _vp, _vp]),
    "moe_forward_nvfp4": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                _vp, _sz, _vp, _vp]),
    "moe_graph_destroy": (_st, [_vp]),
    "moe_permute": (_st, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_permute_static_scratch": (_st, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp]),
    "moe_expert_ffn": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "moe_combine": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "moe_forward": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "moe_forward_ex": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp,
                             ctypes.POINTER(ForwardExt)]),
    "moe_forward_host": (_st, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp,
                               ctypes.POINTER(ForwardExt)]),
    "moe_workspace_layout": (_st, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(WorkspaceLayout)]),
    "moe_workspace_size_ex": (_sz, [_i, _i, _i, _i, _i, ctypes.POINTER(ForwardExt)]),
    "moe_workspace_layout_ex": (_st, [_i, _i, _i, _i, _i, ctypes.POINTER(ForwardExt),
                                      ctypes.POINTER(WorkspaceLayout)]),
    "moe_get_device_status": (_st, [_vp, _sz, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_st]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_set_wait_timeout_ns": (_st, [ctypes.c_ulonglong]),
    "moe_launch_count": (ctypes.c_ulonglong, []),
    "moe_profiler_enable": (_st, [_i]),
    "moe_profiler_only": (_st, [ctypes.c_char_p]),
    "moe_profiler_collect": (_st, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_double), _i, ctypes.POINTER(ctypes.c_int)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK, MOE_ERR_RANGE = range(8)


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _lib.moe_status_string(status).decode()
        detail = _lib.moe_last_error().decode()
        super().__init__(f"{what}: {name}: {detail}")


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _want(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


# ---------------------------------------------------------------- workspace

def moe_workspace_size(T, d, E, I, top_k, I_shared=0, y_fp32=False, act_mxfp8=False) -> int:
    if not y_fp32 and not act_mxfp8:
        return int(_lib.moe_workspace_size(T, d, E, I, top_k, I_shared))
    ext = ForwardExt(None, None, None, I_shared, 0, 0, int(y_fp32), int(act_mxfp8))
    return int(_lib.moe_workspace_size_ex(T, d, E, I, top_k, ctypes.byref(ext)))


def moe_workspace_layout(T, d, E, I, top_k, I_shared=0, y_fp32=False, act_mxfp8=False) -> dict:
    lay = WorkspaceLayout()
    if not y_fp32 and not act_mxfp8:
        _check(_lib.moe_workspace_layout(T, d, E, I, top_k, I_shared, ctypes.byref(lay)),
               "moe_workspace_layout")
    else:
        ext = ForwardExt(None, None, None, I_shared, 0, 0, int(y_fp32), int(act_mxfp8))
        _check(_lib.moe_workspace_layout_ex(T, d, E, I, top_k, ctypes.byref(ext),
                                            ctypes.byref(lay)), "moe_workspace_layout_ex")
    return {n: getattr(lay, n) for n, _ in WorkspaceLayout._fields_}


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(_lib.moe_workspace_init(_p(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def new_workspace(T, d, E, I, top_k, I_shared=0, device="cuda", y_fp32=False,
                  act_mxfp8=False) -> torch.Tensor:
    """A zeroed uint8 device workspace for these shapes (and fp32 y, MXFP8 tokens)."""
    n = max(moe_workspace_size(T, d, E, I, top_k, I_shared, y_fp32, act_mxfp8), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_get_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the workspace's device status (MOE_OK,
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK or MOE_ERR_RANGE)."""
    return int(_lib.moe_get_device_status(_p(ws), ws.numel(), _stream(stream)))


def moe_set_wait_timeout_ns(ns: int):
    _check(_lib.moe_set_wait_timeout_ns(ns), "moe_set_wait_timeout_ns")


def moe_launch_count() -> int:
    return int(_lib.moe_launch_count())


def moe_profiler_enable(on: bool):
    _check(_lib.moe_profiler_enable(1 if on else 0), "moe_profiler_enable")


def moe_profiler_only(name):
    """Trace only launches of kernel `name` (None: every launch)."""
    _check(_lib.moe_profiler_only(name.encode() if name else None), "moe_profiler_only")


def moe_profiler_collect(n_max: int = 64) -> dict:
    """{kernel name: (launches, total ms)} since the last collect."""
    names = ctypes.create_string_buffer(64 * n_max)
    launches = (ctypes.c_int * n_max)()
    total = (ctypes.c_double * n_max)()
    n = ctypes.c_int(0)
    _check(_lib.moe_profiler_collect(names, launches, total, n_max, ctypes.byref(n)),
           "moe_profiler_collect")
    out = {}
    for i in range(n.value):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0", 1)[0].decode()
        out[nm] = (launches[i], total[i])
    return out


# ---------------------------------------------------------------- the four steps

def moe_route(x, w_router, top_k, router_bias=None, topk_ids=None, topk_gates=None, ws=None,
              stream=None, bias_selection_only=False):
    _want(x, torch.bfloat16, "x"); _want(w_router, torch.bfloat16, "w_router")
    _want(router_bias, torch.float32, "router_bias")
    T, d = x.shape
    E = w_router.shape[0]
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if topk_gates is None:
        topk_gates = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    _want(topk_ids, torch.int32, "topk_ids"); _want(topk_gates, torch.float32, "topk_gates")
    if ws is None:
        ws = new_workspace(T, d, E, 64, top_k, device=x.device)
    _check(_lib.moe_route_ex(_p(x), _p(w_router), _p(router_bias), 1 if bias_selection_only else 0,
                             T, d, E, top_k, _p(topk_ids), _p(topk_gates), _p(ws), ws.numel(),
                             _stream(stream)), "moe_route")
    return topk_ids, topk_gates


def moe_permute(topk_ids, E, x=None, ws=None, stream=None):
    """Returns (counts [E], offsets [E+1], perm [T*k], slot_pos [T,k], x_perm or None)."""
    _want(topk_ids, torch.int32, "topk_ids"); _want(x, torch.bfloat16, "x")
    T, k = topk_ids.shape
    d = x.shape[1] if x is not None else 64
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    slot_pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=dev) if x is not None else None
    if ws is None:
        ws = new_workspace(T, d, E, 64, k, device=dev)
    _check(_lib.moe_permute(_p(topk_ids), _p(x), T, d, E, k, _p(counts), _p(offsets), _p(perm),
                            _p(slot_pos), _p(x_perm), _p(ws), ws.numel(), _stream(stream)),
           "moe_permute")
    return counts, offsets, perm, slot_pos, x_perm


def moe_permute_static_scratch(topk_ids, E, x=None, device_status=None, stream=None):
    """moe_permute without a workspace: the scratch table lives in the
    library's own fixed device array (for callers that cannot allocate)."""
    _want(topk_ids, torch.int32, "topk_ids"); _want(x, torch.bfloat16, "x")
    _want(device_status, torch.int32, "device_status")
    T, k = topk_ids.shape
    d = x.shape[1] if x is not None else 64
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    slot_pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=dev) if x is not None else None
    _check(_lib.moe_permute_static_scratch(_p(topk_ids), _p(x), T, d, E, k, _p(counts),
                                           _p(offsets), _p(perm), _p(slot_pos), _p(x_perm),
                                           _p(device_status), _stream(stream)),
           "moe_permute_static_scratch")
    return counts, offsets, perm, slot_pos, x_perm


def moe_expert_ffn(x_perm, expert_offsets, w_gate_up, w_down, y=None, ws=None, stream=None):
    _want(x_perm, torch.bfloat16, "x_perm"); _want(expert_offsets, torch.int32, "expert_offsets")
    _want(w_gate_up, torch.bfloat16, "w_gate_up"); _want(w_down, torch.bfloat16, "w_down")
    rows, d = x_perm.shape
    E, I2, _ = w_gate_up.shape
    I = I2 // 2
    if y is None:
        y = torch.empty((rows, d), dtype=torch.float16, device=x_perm.device)
    _want(y, torch.float16, "y")
    if ws is None:
        ws = new_workspace(rows, d, E, I, 1, device=x_perm.device)
    _check(_lib.moe_expert_ffn(_p(x_perm), _p(expert_offsets), _p(w_gate_up), _p(w_down), rows, d,
                               E, I, _p(y), _p(ws), ws.numel(), _stream(stream)), "moe_expert_ffn")
    return y


def moe_combine(y, slot_pos, topk_gates, y_shared=None, out=None, ws=None, stream=None):
    _want(y, torch.float16, "y"); _want(slot_pos, torch.int32, "slot_pos")
    _want(topk_gates, torch.float32, "topk_gates"); _want(y_shared, torch.float16, "y_shared")
    T, k = slot_pos.shape
    d = y.shape[1]
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=y.device)
    _want(out, torch.bfloat16, "out")
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=y.device)
    _check(_lib.moe_combine(_p(y), _p(slot_pos), _p(topk_gates), _p(y_shared), T, d, k, _p(out),
                            _p(ws), ws.numel(), _stream(stream)), "moe_combine")
    return out


def moe_forward(x, w_router, w_gate_up, w_down, top_k, out=None, ws=None, router_bias=None,
                w_gate_up_shared=None, w_down_shared=None, stream=None, bias_selection_only=False,
                single_launch=False, y_fp32=False):
    """The whole layer.  Returns out [T, d] bf16.  single_launch: one kernel
    launch for the whole layer (decode-sized batches, see moe_forward_ext_t);
    y_fp32: expert outputs kept in fp32 (needs new_workspace(..., y_fp32=True))."""
    for t, n in ((x, "x"), (w_router, "w_router"), (w_gate_up, "w_gate_up"), (w_down, "w_down"),
                 (w_gate_up_shared, "w_gate_up_shared"), (w_down_shared, "w_down_shared")):
        _want(t, torch.bfloat16, n)
    _want(router_bias, torch.float32, "router_bias")
    T, d = x.shape
    E, I2, _ = w_gate_up.shape
    I = I2 // 2
    I_s = w_down_shared.shape[1] if w_down_shared is not None else 0
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    _want(out, torch.bfloat16, "out")
    if ws is None:
        ws = new_workspace(T, d, E, I, top_k, I_s, device=x.device, y_fp32=y_fp32)
    s = _stream(stream)
    if router_bias is None and I_s == 0 and not single_launch and not y_fp32:
        st = _lib.moe_forward(_p(x), _p(w_router), _p(w_gate_up), _p(w_down), T, d, E, I, top_k,
                              _p(out), _p(ws), ws.numel(), s)
    else:
        ext = ForwardExt(router_bias.data_ptr() if router_bias is not None else None,
                         w_gate_up_shared.data_ptr() if I_s else None,
                         w_down_shared.data_ptr() if I_s else None, I_s,
                         1 if bias_selection_only else 0, 1 if single_launch else 0,
                         1 if y_fp32 else 0)
        st = _lib.moe_forward_ex(_p(x), _p(w_router), _p(w_gate_up), _p(w_down), T, d, E, I,
                                 top_k, _p(out), _p(ws), ws.numel(), s, ctypes.byref(ext))
    _check(st, "moe_forward")
    return out


def moe_forward_host(x_host, w_router, w_gate_up, w_down, top_k, out_host, ws,
                     router_bias=None, w_gate_up_shared=None, w_down_shared=None, stream=None,
                     single_launch=False):
    """The whole layer on host tensors (pinned for async copies); queued on
    the stream, not synchronised."""
    if x_host.is_cuda or out_host.is_cuda or x_host.dtype != torch.bfloat16 \
            or out_host.dtype != torch.bfloat16:
        raise ValueError("x_host and out_host must be bf16 host tensors")
    for t, n in ((w_router, "w_router"), (w_gate_up, "w_gate_up"), (w_down, "w_down"),
                 (w_gate_up_shared, "w_gate_up_shared"), (w_down_shared, "w_down_shared")):
        _want(t, torch.bfloat16, n)
    T, d = x_host.shape
    E, I2, _ = w_gate_up.shape
    I_s = w_down_shared.shape[1] if w_down_shared is not None else 0
    ext = ForwardExt(router_bias.data_ptr() if router_bias is not None else None,
                     w_gate_up_shared.data_ptr() if I_s else None,
                     w_down_shared.data_ptr() if I_s else None, I_s, 0,
                     1 if single_launch else 0)
    _check(_lib.moe_forward_host(_p(x_host), _p(w_router), _p(w_gate_up), _p(w_down), T, d, E,
                                 I2 // 2, top_k, _p(out_host), _p(ws), ws.numel(), _stream(stream),
                                 ctypes.byref(ext)), "moe_forward_host")
    return out_host


def moe_mxfp8_quantize(w, stream=None):
    """bf16 [..., K] weights -> (codes uint8 [..., K], scales uint8 [K/128, rows, 4]) on the
    device, rows = the product of the leading dimensions."""
    _want(w, torch.bfloat16, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    scales = torch.empty((K // 128, rows, 4), dtype=torch.uint8, device=w.device)
    _check(_lib.moe_mxfp8_quantize(_p(w), rows, K, _p(codes), _p(scales), _stream(stream)),
           "moe_mxfp8_quantize")
    return codes, scales


def moe_nvfp4_quantize(w, stream=None):
    """bf16 [G, rows, K] weights (G matrices, one per expert) -> (codes uint8
    [G*rows, K/2], scales uint8 [K/256, G*rows, 16], tensor scales float32 [G])
    on the device."""
    _want(w, torch.bfloat16, "w")
    G, rows, K = w.shape
    codes = torch.empty((G * rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((K // 256, G * rows, 16), dtype=torch.uint8, device=w.device)
    tscale = torch.empty((G,), dtype=torch.float32, device=w.device)
    _check(_lib.moe_nvfp4_quantize(_p(w), G, rows, K, _p(codes), _p(scales), _p(tscale),
                                   _stream(stream)), "moe_nvfp4_quantize")
    return codes, scales, tscale


def moe_forward_nvfp4(x, w_router, nv_gate_up, nv_down, top_k, out=None, ws=None,
                      router_bias=None, w_gate_up_shared=None, w_down_shared=None, stream=None,
                      bias_selection_only=False, y_fp32=False):
    """The whole layer with NVFP4 expert weights: nv_gate_up / nv_down are the
    (codes, scales, tensor scales) of moe_nvfp4_quantize for W_gate_up
    [E,2I,d] and W_down [E,d,I].  Returns out [T, d] bf16."""
    for t, n in ((x, "x"), (w_router, "w_router"), (w_gate_up_shared, "w_gate_up_shared"),
                 (w_down_shared, "w_down_shared")):
        _want(t, torch.bfloat16, n)
    _want(router_bias, torch.float32, "router_bias")
    cgu, sgu, tgu = nv_gate_up
    cd, sd, td = nv_down
    for t, n in ((cgu, "codes_gate_up"), (sgu, "scales_gate_up"), (cd, "codes_down"),
                 (sd, "scales_down")):
        _want(t, torch.uint8, n)
    _want(tgu, torch.float32, "tscale_gate_up"); _want(td, torch.float32, "tscale_down")
    T, d = x.shape
    E = tgu.shape[0]
    I = cgu.shape[0] // (2 * E)
    I_s = w_down_shared.shape[1] if w_down_shared is not None else 0
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = new_workspace(T, d, E, I, top_k, I_s, device=x.device, y_fp32=y_fp32)
    ext = ForwardExt(router_bias.data_ptr() if router_bias is not None else None,
                     w_gate_up_shared.data_ptr() if I_s else None,
                     w_down_shared.data_ptr() if I_s else None, I_s,
                     1 if bias_selection_only else 0, 0, 1 if y_fp32 else 0)
    _check(_lib.moe_forward_nvfp4(_p(x), _p(w_router), _p(cgu), _p(sgu), _p(tgu), _p(cd), _p(sd),
                                  _p(td), T, d, E, I, top_k, _p(out), _p(ws), ws.numel(),
                                  _stream(stream), ctypes.byref(ext)), "moe_forward_nvfp4")
    return out


def moe_forward_mxfp8(x, w_router, mx_gate_up, mx_down, top_k, out=None, ws=None,
                      router_bias=None, w_gate_up_shared=None, w_down_shared=None, stream=None,
                      bias_selection_only=False, y_fp32=False, act_mxfp8=False):
    """The whole layer with MXFP8 expert weights: mx_gate_up / mx_down are the
    (codes, scales) pairs of moe_mxfp8_quantize for W_gate_up [E,2I,d] and
    W_down [E,d,I].  act_mxfp8: the tokens micro-scaled too (W8A8, decode
    sizes; needs new_workspace(..., act_mxfp8=True)).  Returns out [T, d] bf16."""
    for t, n in ((x, "x"), (w_router, "w_router"), (w_gate_up_shared, "w_gate_up_shared"),
                 (w_down_shared, "w_down_shared")):
        _want(t, torch.bfloat16, n)
    _want(router_bias, torch.float32, "router_bias")
    cgu, sgu = mx_gate_up
    cd, sd = mx_down
    for t, n in ((cgu, "codes_gate_up"), (sgu, "scales_gate_up"), (cd, "codes_down"),
                 (sd, "scales_down")):
        _want(t, torch.uint8, n)
    T, d = x.shape
    E, I2, _ = cgu.shape
    I = I2 // 2
    I_s = w_down_shared.shape[1] if w_down_shared is not None else 0
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = new_workspace(T, d, E, I, top_k, I_s, device=x.device, y_fp32=y_fp32,
                           act_mxfp8=act_mxfp8)
    ext = ForwardExt(router_bias.data_ptr() if router_bias is not None else None,
                     w_gate_up_shared.data_ptr() if I_s else None,
                     w_down_shared.data_ptr() if I_s else None, I_s,
                     1 if bias_selection_only else 0, 0, 1 if y_fp32 else 0,
                     1 if act_mxfp8 else 0)
    _check(_lib.moe_forward_mxfp8(_p(x), _p(w_router), _p(cgu), _p(sgu), _p(cd), _p(sd), T, d, E,
                                  I, top_k, _p(out), _p(ws), ws.numel(), _stream(stream),
                                  ctypes.byref(ext)), "moe_forward_mxfp8")
    return out


class ForwardGraph:
    """The whole layer captured once as a CUDA graph (moe_forward_graph) and
    replayed with launch(): x and out are device tensors, or bf16 host tensors
    (pinned) whose copies are captured too.  Change x's contents between
    replays, not the tensor; every buffer is kept alive by this object."""

    def __init__(self, x, w_router, w_gate_up, w_down, top_k, out, ws, router_bias=None,
                 w_gate_up_shared=None, w_down_shared=None, bias_selection_only=False,
                 single_launch=False):
        host = not x.is_cuda
        if x.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or out.is_cuda == host:
            raise ValueError("x and out must be bf16 tensors on the same side (device or host)")
        for t, n in ((w_router, "w_router"), (w_gate_up, "w_gate_up"), (w_down, "w_down"),
                     (w_gate_up_shared, "w_gate_up_shared"), (w_down_shared, "w_down_shared")):
            _want(t, torch.bfloat16, n)
        _want(router_bias, torch.float32, "router_bias")
        T, d = x.shape
        E, I2, _ = w_gate_up.shape
        I_s = w_down_shared.shape[1] if w_down_shared is not None else 0
        self._ext = ForwardExt(router_bias.data_ptr() if router_bias is not None else None,
                               w_gate_up_shared.data_ptr() if I_s else None,
                               w_down_shared.data_ptr() if I_s else None, I_s,
                               1 if bias_selection_only else 0, 1 if single_launch else 0)
        self._keep = (x, w_router, w_gate_up, w_down, out, ws, router_bias, w_gate_up_shared,
                      w_down_shared)
        self._h = ctypes.c_void_p()
        _check(_lib.moe_forward_graph(x.data_ptr(), _p(w_router), _p(w_gate_up), _p(w_down), T, d,
                                      E, I2 // 2, top_k, out.data_ptr(), _p(ws), ws.numel(),
                                      ctypes.byref(self._ext), 1 if host else 0,
                                      ctypes.byref(self._h)), "moe_forward_graph")

    def launch(self, stream=None):
        _check(_lib.moe_graph_launch(self._h, _stream(stream)), "moe_graph_launch")

    def close(self):
        if self._h:
            _lib.moe_graph_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def workspace_views(ws: torch.Tensor, T, d, E, I, top_k, I_shared=0, y_fp32=False,
                    act_mxfp8=False) -> dict:
    """Typed views of moe_forward's intermediates inside its workspace."""
    L = moe_workspace_layout(T, d, E, I, top_k, I_shared, y_fp32, act_mxfp8)
    n = T * top_k

    def view(off, count, dtype, shape):
        b = torch.empty((), dtype=dtype).element_size()
        return ws[off:off + count * b].view(dtype).view(shape)

    return {
        "topk_ids": view(L["topk_ids"], n, torch.int32, (T, top_k)),
        "topk_gates": view(L["topk_gates"], n, torch.float32, (T, top_k)),
        "expert_counts": view(L["expert_counts"], E, torch.int32, (E,)),
        "expert_offsets": view(L["expert_offsets"], E + 1, torch.int32, (E + 1,)),
        "perm": view(L["perm"], n, torch.int32, (n,)),
        "slot_pos": view(L["slot_pos"], n, torch.int32, (T, top_k)),
        "x_perm": view(L["x_perm"], n * d, torch.bfloat16, (n, d)),
        "h": view(L["h"], n * I, torch.bfloat16, (n, I)),
        "y": view(L["y"], n * d, torch.float32 if y_fp32 else torch.float16, (n, d)),
        # MXFP8 tokens of act_mxfp8 (codes in the GEMMs' order within each 256-wide chunk)
        "act_x": view(L["act_x"], T * d if act_mxfp8 else 0, torch.uint8,
                      (T, d) if act_mxfp8 else (0,)),
        "act_x_scales": view(L["act_x_scales"], T * d // 32 if act_mxfp8 else 0, torch.uint8,
                             (T, d // 32) if act_mxfp8 else (0,)),
        "act_h": view(L["act_h"], n * I if act_mxfp8 else 0, torch.uint8,
                      (n, I) if act_mxfp8 else (0,)),
        "act_h_scales": view(L["act_h_scales"], n * I // 32 if act_mxfp8 else 0, torch.uint8,
                             (n, I // 32) if act_mxfp8 else (0,)),
    }
