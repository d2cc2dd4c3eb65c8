"""ctypes binding of ``libmoe_w4a8.so`` (C ABI in ``include/moe_w4a8.h``).

Argument marshalling only: torch tensors are checked for dtype, shape,
contiguity and device, and their ``data_ptr()`` is passed with the current
CUDA stream.  Every step of the layer runs in the library's CUDA kernels;
there is no CPU fallback -- if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_w4a8.so")
ABI_VERSION = 4
ENGINE_AUTO, ENGINE_GROUPED, ENGINE_DECODE, ENGINE_TCGEN05 = -1, 0, 1, 2
NOALLOC_SCRATCH_BYTES = 16 << 20
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = _load()
        msg = f"{fn} failed with status {status}: {lib.moe_w4a8_status_string(status).decode()}"
        if status == 4:
            msg += f" [{lib.moe_w4a8_last_error().decode()}]"
        super().__init__(msg)
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("T", "H", "I", "E", "n_shared", "top_k", "group")]

    def __repr__(self):
        return "Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    dp = ctypes.POINTER(Dims)
    lib.moe_w4a8_version.restype = ctypes.c_int
    lib.moe_w4a8_status_string.argtypes = [ctypes.c_int]
    lib.moe_w4a8_status_string.restype = ctypes.c_char_p
    lib.moe_w4a8_last_error.restype = ctypes.c_char_p
    lib.moe_w4a8_workspace_size.argtypes = [dp]
    lib.moe_w4a8_workspace_size.restype = sz
    lib.moe_w4a8_partials_workspace_size.argtypes = [dp, i64]
    lib.moe_w4a8_partials_workspace_size.restype = sz
    lib.moe_w4a8_forward.argtypes = [p, p, p, p, p, p, p, dp, p, p, sz, p]
    ci = ctypes.c_int
    lib.moe_w4a8_forward_debug.argtypes = [p, p, p, p, p, p, p, dp, p, p, p, p, ci, p, sz, p]
    lib.moe_w4a8_route.argtypes = [p, dp, p, p, p, p, p, p, p, sz, p]
    lib.moe_w4a8_debug_routing.argtypes = [dp, p, sz, p, p, p, p, p]
    lib.moe_w4a8_forward_routed.argtypes = [p, p, p, p, p, p, p, p, dp, p, p, sz, p]
    lib.moe_w4a8_gemm1_partials.argtypes = [p, p, dp, p, p, i64, p, ci, p, sz, p]
    lib.moe_w4a8_gemm2_partials.argtypes = [p, p, dp, p, i64, p, ci, p, sz, p]
    lib.moe_w4a8_device_status.argtypes = [p, sz, p]
    lib.moe_w4a8_engine_for.argtypes = [dp]
    lib.moe_w4a8_engine_for.restype = ctypes.c_int
    lib.moe_w4a8_selftest_barrier_timeout.argtypes = [p, sz, p]
    lib.moe_w4a8_forward_noalloc.argtypes = [p, p, p, p, p, p, p, dp, p, p]
    lib.moe_w4a8_forward_host_workspace_size.argtypes = [dp]
    lib.moe_w4a8_forward_host_workspace_size.restype = sz
    lib.moe_w4a8_forward_host.argtypes = [p, p, p, p, p, p, p, dp, p, p, sz, p]
    lib.moe_w4a8_forward_bf16_workspace_size.argtypes = [dp]
    lib.moe_w4a8_forward_bf16_workspace_size.restype = sz
    lib.moe_w4a8_forward_bf16.argtypes = [p, p, p, p, p, p, dp, p, p, sz, p]
    lib.moe_w4a8_forward_w2w4.argtypes = [p, p, p, p, p, p, p, p, dp, p, p, sz, p]
    lib.moe_w4a8_mixed_bank_layout.argtypes = [p, dp, p, p, p, p]
    lib.moe_w4a8_forward_w2w4_compact.argtypes = [p, p, p, p, p, p, p, p, p, p, dp, p, p, sz, p]
    for name in ("moe_w4a8_forward", "moe_w4a8_forward_debug", "moe_w4a8_route", "moe_w4a8_gemm1_partials",
                 "moe_w4a8_gemm2_partials", "moe_w4a8_forward_noalloc", "moe_w4a8_device_status",
                 "moe_w4a8_selftest_barrier_timeout", "moe_w4a8_forward_host", "moe_w4a8_forward_bf16",
                 "moe_w4a8_forward_w2w4", "moe_w4a8_debug_routing", "moe_w4a8_forward_routed",
                 "moe_w4a8_mixed_bank_layout", "moe_w4a8_forward_w2w4_compact"):
        getattr(lib, name).restype = ctypes.c_int
    if lib.moe_w4a8_version() != ABI_VERSION:
        raise RuntimeError(f"{LIB_PATH}: ABI version {lib.moe_w4a8_version()} != {ABI_VERSION}")
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise MoeError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _one_device(fn: str, tensors):
    """The one CUDA device all of `tensors` (None entries skipped) live on."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"{fn}: the device tensors must share one device, got {sorted(map(str, devs))}")
    return devs.pop()


def _call(fn: str, tensors, *args):
    """Calls entry point `fn` with `args` followed by the current stream of the
    device `tensors` share, with that device current for the launches."""
    dev = _one_device(fn, tensors)
    if dev.index == torch.cuda.current_device():
        _check(fn, getattr(_load(), fn)(*args, _stream(dev)))
        return
    with torch.cuda.device(dev):
        _check(fn, getattr(_load(), fn)(*args, _stream(dev)))


def _need(t, name, dtype, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def dims_of(T, H, I, E, n_shared, top_k, group) -> Dims:
    return Dims(T, H, I, E, n_shared, top_k, group)


def moe_w4a8_version() -> int:
    return _load().moe_w4a8_version()


def moe_w4a8_status_string(status: int) -> str:
    return _load().moe_w4a8_status_string(status).decode()


def moe_w4a8_engine_for(d: Dims) -> int:
    """ENGINE_DECODE, ENGINE_TCGEN05 or ENGINE_GROUPED: what moe_w4a8_forward runs for these sizes on the current device."""
    return _load().moe_w4a8_engine_for(ctypes.byref(d))


def moe_w4a8_workspace_size(d: Dims) -> int:
    n = _load().moe_w4a8_workspace_size(ctypes.byref(d))
    if n == 0:
        raise MoeError("moe_w4a8_workspace_size", 1)
    return n


def moe_w4a8_partials_workspace_size(d: Dims, n_pairs: int) -> int:
    """Workspace of moe_w4a8_gemm{1,2}_partials for n_pairs pairs."""
    n = _load().moe_w4a8_partials_workspace_size(ctypes.byref(d), n_pairs)
    if n == 0:
        raise MoeError("moe_w4a8_partials_workspace_size", 1)
    return n


partials_workspace_size = moe_w4a8_partials_workspace_size


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(nbytes + 256, dtype=torch.uint8, device=device)


def _ws_view(ws: torch.Tensor):
    """(pointer, bytes) of the 256-byte aligned part of a uint8 workspace tensor."""
    _need(ws, "workspace", torch.uint8)
    base = ws.data_ptr()
    aligned = (base + 255) & ~255
    return ctypes.c_void_p(aligned), ws.numel() - (aligned - base)


def _bank_shapes(d: Dims):
    slots = d.E + d.n_shared
    return ((slots, 2 * d.I, d.H // 2), (slots, 2 * d.I, d.H // d.group), (slots, d.H, d.I // 2),
            (slots, d.H, d.I // d.group))


def _check_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out):
    s13, s13s, s2, s2s = _bank_shapes(d)
    _need(x_q, "x_q", torch.int8, (d.T, d.H))
    _need(x_scale, "x_scale", torch.float32, (d.T,))
    _need(router_logits, "router_logits", torch.float32, (d.T, d.E))
    _need(w13_packed, "w13_packed", torch.uint8, s13)
    _need(w13_scale, "w13_scale", torch.float32, s13s)
    _need(w2_packed, "w2_packed", torch.uint8, s2)
    _need(w2_scale, "w2_scale", torch.float32, s2s)
    _need(out, "out", torch.float32, (d.T, d.H))


def moe_w4a8_forward(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims, out,
                     workspace: torch.Tensor):
    _check_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out)
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward", (x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, out,
                               workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_forward_host_workspace_size(d: Dims) -> int:
    """Workspace of moe_w4a8_forward_host (the layer's plus the staged inputs and output)."""
    n = _load().moe_w4a8_forward_host_workspace_size(ctypes.byref(d))
    if n == 0:
        raise MoeError("moe_w4a8_forward_host_workspace_size", 1)
    return n


def _need_host(t, name, dtype, shape):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous CPU tensor of shape {tuple(shape)}")


def moe_w4a8_forward_host(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims, out,
                          workspace: torch.Tensor):
    """The layer with x_q, x_scale, router_logits and out in host memory (CPU tensors).

    Pinned tensors are read and written in place by the kernels (no copy
    engine transfers); pageable ones go through asynchronous copies.  The
    call is asynchronous on the current stream of the workspace's device:
    synchronise it before reading `out` or reusing the inputs.
    """
    s13, s13s, s2, s2s = _bank_shapes(d)
    _need_host(x_q, "x_q", torch.int8, (d.T, d.H))
    _need_host(x_scale, "x_scale", torch.float32, (d.T,))
    _need_host(router_logits, "router_logits", torch.float32, (d.T, d.E))
    _need_host(out, "out", torch.float32, (d.T, d.H))
    _need(w13_packed, "w13_packed", torch.uint8, s13)
    _need(w13_scale, "w13_scale", torch.float32, s13s)
    _need(w2_packed, "w2_packed", torch.uint8, s2)
    _need(w2_scale, "w2_scale", torch.float32, s2s)
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_host", (w13_packed, w13_scale, w2_packed, w2_scale, workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_forward_bf16_workspace_size(d: Dims) -> int:
    """Workspace of moe_w4a8_forward_bf16 (the layer's plus the quantised activations)."""
    n = _load().moe_w4a8_forward_bf16_workspace_size(ctypes.byref(d))
    if n == 0:
        raise MoeError("moe_w4a8_forward_bf16_workspace_size", 1)
    return n


def moe_w4a8_forward_bf16(x_bf16, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims, out,
                          workspace: torch.Tensor):
    """The layer from bf16 activations [T, H]: the per-token int8 quantisation runs on the device."""
    s13, s13s, s2, s2s = _bank_shapes(d)
    _need(x_bf16, "x_bf16", torch.bfloat16, (d.T, d.H))
    _need(router_logits, "router_logits", torch.float32, (d.T, d.E))
    _need(w13_packed, "w13_packed", torch.uint8, s13)
    _need(w13_scale, "w13_scale", torch.float32, s13s)
    _need(w2_packed, "w2_packed", torch.uint8, s2)
    _need(w2_scale, "w2_scale", torch.float32, s2s)
    _need(out, "out", torch.float32, (d.T, d.H))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_bf16", (x_bf16, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, out,
                                    workspace),
          _ptr(x_bf16), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed), _ptr(w2_scale),
          ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_forward_w2w4(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, slot_bits,
                          d: Dims, out, workspace: torch.Tensor):
    """The layer on a mixed 2/4-bit bank: slot_bits (uint8 CUDA tensor [E+S], 2 or 4) gives each slot's width.

    2-bit slots hold four codes per byte in the first half of each row (see the header).  Decode-engine
    sizes only.
    """
    _check_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out)
    _need(slot_bits, "slot_bits", torch.uint8, (d.E + d.n_shared,))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_w2w4", (x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale,
                                    slot_bits, out, workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), _ptr(slot_bits), ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_mixed_bank_layout(slot_bits, d: Dims):
    """The compact layout of a mixed 2/4-bit bank, computed on the host.

    slot_bits: uint8 CPU tensor [E+S] (2 or 4).  Returns (w13_off, w2_off, w13_bytes, w2_bytes): each slot's
    byte offset in the gate/up and the down bank (int64 CPU tensors [E+S]) and the two banks' sizes.
    """
    _need_host(slot_bits, "slot_bits", torch.uint8, (d.E + d.n_shared,))
    n = d.E + d.n_shared
    o13 = torch.empty(n, dtype=torch.int64)
    o2 = torch.empty(n, dtype=torch.int64)
    b13, b2 = ctypes.c_int64(0), ctypes.c_int64(0)
    _check("moe_w4a8_mixed_bank_layout",
           _load().moe_w4a8_mixed_bank_layout(_ptr(slot_bits), ctypes.byref(d), _ptr(o13), _ptr(o2),
                                               ctypes.byref(b13), ctypes.byref(b2)))
    return o13, o2, b13.value, b2.value


def moe_w4a8_forward_w2w4_compact(x_q, x_scale, router_logits, w13_packed, w13_off, w13_scale, w2_packed, w2_off,
                                  w2_scale, slot_bits, d: Dims, out, workspace: torch.Tensor):
    """The layer on a mixed 2/4-bit bank in compact storage (see moe_w4a8_mixed_bank_layout).

    w13_packed, w2_packed: uint8 CUDA tensors holding every slot's rows at the slot's own width; w13_off,
    w2_off: int64 CUDA tensors [E+S], each slot's byte offset (multiples of 16).  Scales and slot_bits as
    for moe_w4a8_forward_w2w4.
    """
    s13, s13s, s2, s2s = _bank_shapes(d)
    n = d.E + d.n_shared
    _need(x_q, "x_q", torch.int8, (d.T, d.H))
    _need(x_scale, "x_scale", torch.float32, (d.T,))
    _need(router_logits, "router_logits", torch.float32, (d.T, d.E))
    _need(w13_packed, "w13_packed", torch.uint8)
    _need(w13_off, "w13_off", torch.int64, (n,))
    _need(w13_scale, "w13_scale", torch.float32, s13s)
    _need(w2_packed, "w2_packed", torch.uint8)
    _need(w2_off, "w2_off", torch.int64, (n,))
    _need(w2_scale, "w2_scale", torch.float32, s2s)
    _need(slot_bits, "slot_bits", torch.uint8, (n,))
    _need(out, "out", torch.float32, (d.T, d.H))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_w2w4_compact", (x_q, x_scale, router_logits, w13_packed, w13_off, w13_scale, w2_packed,
                                            w2_off, w2_scale, slot_bits, out, workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_off), _ptr(w13_scale),
          _ptr(w2_packed), _ptr(w2_off), _ptr(w2_scale), _ptr(slot_bits), ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_forward_noalloc(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims,
                             out):
    """The layer using the library's built-in scratch array instead of a workspace.

    For callers that cannot allocate device memory when they run the layer
    (runtimes that own all device memory, or hot paths where cudaMalloc is
    not allowed).  Calls on one device share the array, so calls that may
    overlap on the GPU must be serialised; layers needing more than
    NOALLOC_SCRATCH_BYTES of intermediates are rejected.
    """
    _check_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out)
    _call("moe_w4a8_forward_noalloc", (x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, out),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), ctypes.byref(d), _ptr(out))
    return out


def moe_w4a8_forward_debug(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims, out,
                           workspace, h_q=None, s_h=None, y=None, engine: int = ENGINE_AUTO):
    _check_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out)
    P = d.T * (d.top_k + d.n_shared)
    if h_q is not None:
        _need(h_q, "h_q", torch.int8, (P, d.I))
    if s_h is not None:
        _need(s_h, "s_h", torch.float32, (P,))
    if y is not None:
        _need(y, "y", torch.float32, (P, d.H))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_debug", (x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, out,
                                     h_q, s_h, y, workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(router_logits), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), ctypes.byref(d), _ptr(out), _ptr(h_q), _ptr(s_h), _ptr(y), engine, wp, wb)
    return out


def moe_w4a8_route(router_logits, d: Dims, topk_ids, topk_w, counts, offsets, perm, inv, workspace):
    _need(router_logits, "router_logits", torch.float32, (d.T, d.E))
    _need(topk_ids, "topk_ids", torch.int32, (d.T, d.top_k))
    _need(topk_w, "topk_w", torch.float32, (d.T, d.top_k))
    _need(counts, "counts", torch.int32, (d.E,))
    _need(offsets, "offsets", torch.int32, (d.E + 1,))
    _need(perm, "perm", torch.int32, (d.T * d.top_k,))
    _need(inv, "inv", torch.int32, (d.T * d.top_k,))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_route", (router_logits, topk_ids, topk_w, counts, offsets, perm, inv, workspace),
          _ptr(router_logits), ctypes.byref(d), _ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets),
          _ptr(perm), _ptr(inv), wp, wb)


def moe_w4a8_forward_routed(x_q, x_scale, topk_ids, topk_w, w13_packed, w13_scale, w2_packed, w2_scale, d: Dims,
                            out, workspace):
    """The layer with the routing supplied by the caller (see the header)."""
    _need(x_q, "x_q", torch.int8, (d.T, d.H))
    _need(x_scale, "x_scale", torch.float32, (d.T,))
    _need(topk_ids, "topk_ids", torch.int32, (d.T, d.top_k))
    _need(topk_w, "topk_w", torch.float32, (d.T, d.top_k))
    w13s, s13s, w2s, s2s = _bank_shapes(d)
    _need(w13_packed, "w13_packed", torch.uint8, w13s)
    _need(w13_scale, "w13_scale", torch.float32, s13s)
    _need(w2_packed, "w2_packed", torch.uint8, w2s)
    _need(w2_scale, "w2_scale", torch.float32, s2s)
    _need(out, "out", torch.float32, (d.T, d.H))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_forward_routed", (x_q, x_scale, topk_ids, topk_w, w13_packed, w13_scale, w2_packed, w2_scale, out,
                                      workspace),
          _ptr(x_q), _ptr(x_scale), _ptr(topk_ids), _ptr(topk_w), _ptr(w13_packed), _ptr(w13_scale), _ptr(w2_packed),
          _ptr(w2_scale), ctypes.byref(d), _ptr(out), wp, wb)
    return out


def moe_w4a8_debug_routing(d: Dims, workspace, topk_ids, topk_w, perm, inv):
    """The routing of the last moe_w4a8_forward_debug call on `workspace` (see the header)."""
    _need(topk_ids, "topk_ids", torch.int32, (d.T, d.top_k))
    _need(topk_w, "topk_w", torch.float32, (d.T, d.top_k))
    _need(perm, "perm", torch.int32, (d.T * d.top_k,))
    _need(inv, "inv", torch.int32, (d.T * d.top_k,))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_debug_routing", (workspace, topk_ids, topk_w, perm, inv), ctypes.byref(d), wp, wb,
          _ptr(topk_ids), _ptr(topk_w), _ptr(perm), _ptr(inv))


def moe_w4a8_gemm1_partials(x_q, w13_packed, d: Dims, pair_token, pair_slot, p1, workspace,
                            engine: int = ENGINE_GROUPED):
    n = pair_slot.shape[0]
    _need(x_q, "x_q", torch.int8, (d.T, d.H))
    _need(w13_packed, "w13_packed", torch.uint8, _bank_shapes(d)[0])
    _need(pair_token, "pair_token", torch.int32, (n,))
    _need(pair_slot, "pair_slot", torch.int32, (n,))
    _need(p1, "p1", torch.int32, (n, 2 * d.I, d.H // d.group))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_gemm1_partials", (x_q, w13_packed, pair_token, pair_slot, p1, workspace),
          _ptr(x_q), _ptr(w13_packed), ctypes.byref(d), _ptr(pair_token), _ptr(pair_slot), n, _ptr(p1), engine, wp,
          wb)


def moe_w4a8_gemm2_partials(h_q, w2_packed, d: Dims, pair_slot, p2, workspace, engine: int = ENGINE_GROUPED):
    n = pair_slot.shape[0]
    _need(h_q, "h_q", torch.int8, (n, d.I))
    _need(w2_packed, "w2_packed", torch.uint8, _bank_shapes(d)[2])
    _need(pair_slot, "pair_slot", torch.int32, (n,))
    _need(p2, "p2", torch.int32, (n, d.H, d.I // d.group))
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_gemm2_partials", (h_q, w2_packed, pair_slot, p2, workspace),
          _ptr(h_q), _ptr(w2_packed), ctypes.byref(d), _ptr(pair_slot), n, _ptr(p2), engine, wp, wb)


def moe_w4a8_selftest_barrier_timeout(workspace: torch.Tensor):
    """Enqueue the bounded-wait self-test (see the C header); read the result with moe_w4a8_device_status."""
    wp, wb = _ws_view(workspace)
    _call("moe_w4a8_selftest_barrier_timeout", (workspace,), wp, wb)


def moe_w4a8_device_status(workspace: torch.Tensor | None, device=None) -> int:
    """Synchronises the current stream and returns the status word of the last call (0 = ok, 5 = timeout).

    workspace None: the status of the last moe_w4a8_forward_noalloc call on `device` (default: current device).
    """
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(dev):
            return _load().moe_w4a8_device_status(None, 0, _stream(dev))
    wp, wb = _ws_view(workspace)
    with torch.cuda.device(workspace.device):
        return _load().moe_w4a8_device_status(wp, wb, _stream(workspace.device))


class Layer:
    """A device-resident expert bank with its dims and a workspace; forward() runs the layer."""

    def __init__(self, d: Dims, w13, s13, w2, s2, device):
        self.d, self.device = d, torch.device(device)
        self.w13, self.s13, self.w2, self.s2 = w13, s13, w2, s2
        self.workspace = alloc_workspace(moe_w4a8_workspace_size(d), self.device)

    @classmethod
    def from_numpy(cls, w, bank, device, T=None):
        d = Dims(w.T if T is None else T, w.H, w.I, w.E, w.S, w.top_k, w.group)
        dev = torch.device(device)
        t = lambda a: torch.from_numpy(a).to(dev)  # noqa: E731
        return cls(d, t(bank.w13), t(bank.s13), t(bank.w2), t(bank.s2), dev)

    def forward(self, x_q, x_scale, router_logits, out=None):
        if out is None:
            out = torch.empty((self.d.T, self.d.H), dtype=torch.float32, device=self.device)
        return moe_w4a8_forward(x_q, x_scale, router_logits, self.w13, self.s13, self.w2, self.s2, self.d, out,
                                self.workspace)

    def forward_numpy(self, tokens):
        t = lambda a: torch.from_numpy(a).to(self.device)  # noqa: E731
        out = self.forward(t(tokens.x_q), t(tokens.x_scale), t(tokens.logits))
        torch.cuda.synchronize(self.device)
        return out
