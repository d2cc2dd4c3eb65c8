"""CPU oracle of the routed-expert W4A8 MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline/reference
legs of ``bench.py`` may import this package.  It wraps ``liboracle.so``
(plain C, fp64, built from ``oracle.c`` by ``__graft_entry__.build()``) with
numpy arrays; it shares no code with the CUDA path.  The definitions and
their sources are in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_ORACLE_LIB: another build of oracle.c (the planted-mistake tests load mutated copies)
LIB_PATH = os.environ.get("MOE_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")
_lib = None


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("T", "H", "I", "E", "n_shared", "top_k", "group")]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.orc_unpack.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.orc_unpack2.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.orc_partials_bits.argtypes = [p, i64, p, i64, i64, ctypes.c_int, p]
    lib.orc_partials_bits.restype = None
    lib.orc_route.argtypes = [i64, i64, i64, p, p, p]
    lib.orc_permute.argtypes = [i64, i64, i64, p, p, p, p, p]
    lib.orc_partials.argtypes = [p, i64, p, i64, i64, p]
    lib.orc_partials.restype = None
    lib.orc_silu.argtypes = [ctypes.c_double]
    lib.orc_silu.restype = ctypes.c_double
    lib.orc_hidden.argtypes = [p, ctypes.c_float, p, p, i64, i64, i64, p, p, p]
    lib.orc_hidden.restype = None
    lib.orc_requant.argtypes = [p, i64, p, p]
    lib.orc_requant.restype = None
    lib.orc_quantize_bf16.argtypes = [p, i64, i64, p, p]
    lib.orc_quantize_bf16.restype = None
    lib.orc_down.argtypes = [p, ctypes.c_float, p, p, i64, i64, i64, p, p]
    lib.orc_down.restype = None
    lib.orc_pair_output.argtypes = [ctypes.POINTER(Dims), p, p, p, p, p, p, i64, i64, p, p, p]
    lib.orc_pair_output.restype = None
    lib.orc_forward_tokens.argtypes = [ctypes.POINTER(Dims), p, p, p, p, p, p, p, i64, p, p]
    lib.orc_forward_tokens_mixed.argtypes = [ctypes.POINTER(Dims), p, p, p, p, p, p, p, p, i64, p, p]
    _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def dims(T, H, I, E, n_shared, top_k, group) -> Dims:
    return Dims(T, H, I, E, n_shared, top_k, group)


def unpack(byte: int, high: int) -> int:
    return _load().orc_unpack(byte, high)


def route(logits: np.ndarray, top_k: int):
    """-> (ids int32 [T,k], w float64 [T,k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float64)
    if _load().orc_route(T, E, top_k, _p(logits), _p(ids), _p(w)):
        raise ValueError("orc_route: invalid arguments")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """-> (counts [E], offsets [E+1], perm [T*k], inv [T*k]), all int32."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    if _load().orc_permute(T, E, k, _p(ids), _p(counts), _p(offsets), _p(perm), _p(inv)):
        raise ValueError("orc_permute: expert id out of range")
    return counts, offsets, perm, inv


def partials(a: np.ndarray, W: np.ndarray, group: int, bits: int = 4) -> np.ndarray:
    """int32 [rows, K/g] partials of int8 row a (K) against packed rows W [rows, K/2] of `bits`-bit codes."""
    a = _c(a, np.int8)
    W = _c(W, np.uint8)
    K = a.shape[0]
    rows = W.shape[0]
    P = np.empty((rows, K // group), np.int32)
    _load().orc_partials_bits(_p(a), K, _p(W), rows, group, bits, _p(P))
    return P


def unpack2(byte: int, pos: int) -> int:
    """The 2-bit code at position pos (0..3) of a packed byte."""
    return _load().orc_unpack2(byte, pos)


def silu(z: float) -> float:
    return _load().orc_silu(z)


def hidden(x_row, x_scale, w13e, s13e, group):
    """One pair's gemm1 + act: -> (P1 int32 [2I, H/g], G f64 [2I], h f64 [I])."""
    x_row = _c(x_row, np.int8)
    w13e = _c(w13e, np.uint8)
    s13e = _c(s13e, np.float32)
    H = x_row.shape[0]
    I = w13e.shape[0] // 2
    P1 = np.empty((2 * I, H // group), np.int32)
    G = np.empty(2 * I, np.float64)
    h = np.empty(I, np.float64)
    _load().orc_hidden(_p(x_row), float(x_scale), _p(w13e), _p(s13e), H, I, group, _p(P1), _p(G), _p(h))
    return P1, G, h


def requant(h: np.ndarray):
    """-> (h_q int8 [I], s_h float)."""
    h = _c(h, np.float64)
    hq = np.empty(h.shape[0], np.int8)
    sh = np.empty(1, np.float32)
    _load().orc_requant(_p(h), h.shape[0], _p(hq), _p(sh))
    return hq, float(sh[0])


def quantize_bf16(x_bits: np.ndarray):
    """S0 of bf16 activations (uint16 bit patterns [T][H]) -> (x_q int8 [T][H], x_scale float32 [T])."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    x_q = np.empty((T, H), np.int8)
    x_scale = np.empty(T, np.float32)
    _load().orc_quantize_bf16(_p(x_bits), T, H, _p(x_q), _p(x_scale))
    return x_q, x_scale


def down(hq, sh, w2e, s2e, group):
    """One pair's gemm2: -> (P2 int32 [H, I/g], Y f64 [H])."""
    hq = _c(hq, np.int8)
    w2e = _c(w2e, np.uint8)
    s2e = _c(s2e, np.float32)
    I = hq.shape[0]
    H = w2e.shape[0]
    P2 = np.empty((H, I // group), np.int32)
    y = np.empty(H, np.float64)
    _load().orc_down(_p(hq), float(sh), _p(w2e), _p(s2e), H, I, group, _p(P2), _p(y))
    return P2, y


def _layer_args(x_q, x_scale, w13, s13, w2, s2):
    return (_c(x_q, np.int8), _c(x_scale, np.float32), _c(w13, np.uint8), _c(s13, np.float32),
            _c(w2, np.uint8), _c(s2, np.float32))


def pair_output(d: Dims, x_q, x_scale, w13, s13, w2, s2, t: int, slot: int):
    """Y of one (token, bank slot) pair: -> (h_q int8 [I], s_h, Y f64 [H])."""
    x_q, x_scale, w13, s13, w2, s2 = _layer_args(x_q, x_scale, w13, s13, w2, s2)
    hq = np.empty(d.I, np.int8)
    sh = np.empty(1, np.float32)
    y = np.empty(d.H, np.float64)
    _load().orc_pair_output(ctypes.byref(d), _p(x_q), _p(x_scale), _p(w13), _p(s13), _p(w2), _p(s2),
                            t, slot, _p(hq), _p(sh), _p(y))
    return hq, float(sh[0]), y


def forward_tokens(d: Dims, x_q, x_scale, logits, w13, s13, w2, s2, tokens=None, slot_bits=None) -> np.ndarray:
    """Layer output (f64 [len(tokens), H]) for the listed tokens (all tokens if None).

    slot_bits (optional uint8 [E+S], 2 or 4): each slot's code width (default: all 4).
    """
    x_q, x_scale, w13, s13, w2, s2 = _layer_args(x_q, x_scale, w13, s13, w2, s2)
    logits = _c(logits, np.float32)
    tokens = np.arange(d.T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    bits = None if slot_bits is None else _c(slot_bits, np.uint8)
    out = np.empty((tokens.shape[0], d.H), np.float64)
    if _load().orc_forward_tokens_mixed(ctypes.byref(d), _p(x_q), _p(x_scale), _p(logits), _p(w13), _p(s13),
                                        _p(w2), _p(s2), _p(bits) if bits is not None else None, tokens.shape[0],
                                        _p(tokens), _p(out)):
        raise ValueError("orc_forward_tokens: invalid arguments")
    return out


def forward_workload(w, tokens_data, bank, tokens=None) -> np.ndarray:
    """forward_tokens for a synth Workload with its Tokens and Bank."""
    d = dims(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)
    return forward_tokens(d, tokens_data.x_q, tokens_data.x_scale, tokens_data.logits,
                          bank.w13, bank.s13, bank.w2, bank.s2, tokens, getattr(bank, "slot_bits", None))
