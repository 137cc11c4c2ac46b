"""CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
library (``bit_grouped_expert_gb300``) never imports or links it and shares no
code with it.

``moe_oracle.c`` is the oracle proper: plain fp64 loops that state the layer as
the source pages describe it (see the header of ``moe_oracle.h`` for the
passages and readings).  ``brute.py`` is a second, independent numpy
statement for tiny shapes that cross-checks the C code.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked dequant examples, closed forms, invariants, brute force and a
library-routine special case).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_SRC = [os.path.join(_HERE, "moe_oracle.c")]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe_oracle.so with gcc + OpenMP (no FP contraction, so x86
    and Arm hosts give the same bits)."""
    with _lock:
        srcs = _SRC + [os.path.join(_HERE, "moe_oracle.h")]
        stale = force or not os.path.exists(_LIB_PATH) or any(
            os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in srcs)
        if stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-ffp-contract=off",
                   "-fno-fast-math", "-o", tmp] + _SRC + ["-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("H", "E", "k", "I", "n_shared", "G")]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router", "gate_q", "up_q", "gate_s", "gate_b", "up_s", "up_b", "down_q", "down_s", "down_b", "shared_gate")]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.orc_bf16_to_double.restype = dbl
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_round_bf16.argtypes = [dbl, dbl]
        lib.orc_expert_bytes.restype = ctypes.c_size_t
        lib.orc_expert_bytes.argtypes = [i32, i32, i32]
        lib.orc_dequant.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        lib.orc_logits.argtypes = [vp, i32, i32, vp, i32, vp, vp]
        lib.orc_select.argtypes = [vp, i32, i32, i32, vp, vp]
        lib.orc_route_maps.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_rmsnorm.argtypes = [vp, i32, i32, dbl, vp]
        lib.orc_moe_layer.restype = i32
        lib.orc_moe_layer.argtypes = [ctypes.POINTER(_Dims), vp, vp, i32, ctypes.POINTER(_Weights),
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_num_threads.restype = i32
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous numpy arrays"
    return a.ctypes.data


@dataclass(frozen=True)
class Dims:
    H: int = 2048
    E: int = 256
    k: int = 8
    I: int = 512
    n_shared: int = 1
    G: int = 64


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(hi: float, lo: float = 0.0) -> int:
    return int(_load().orc_round_bf16(float(hi), float(lo)))


def expert_bytes(H: int, I: int, G: int = 64) -> int:
    return int(_load().orc_expert_bytes(H, I, G))


def dequant(q: np.ndarray, s: np.ndarray, b: np.ndarray, G: int = 64) -> np.ndarray:
    """bf16 [rows, K] = bf16_rne(scale * code + bias), codes unpacked low nibble first."""
    rows, kw = q.shape
    K = kw * 8
    w = np.empty((rows, K), np.uint16)
    _load().orc_dequant(_p(np.ascontiguousarray(q, np.uint32)), _p(np.ascontiguousarray(s, np.uint16)),
                        _p(np.ascontiguousarray(b, np.uint16)), rows, K, G, _p(w))
    return w


def logits(x: np.ndarray, router: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    T, H = x.shape
    E = router.shape[0]
    keys = np.empty((T, E), np.float32)
    if T:
        _load().orc_logits(_p(np.ascontiguousarray(x)), T, H, _p(np.ascontiguousarray(router, np.float32)), E,
                           _p(None if bias is None else np.ascontiguousarray(bias, np.float32)), _p(keys))
    return keys


def select(keys: np.ndarray, k: int):
    keys = np.ascontiguousarray(keys, np.float32)
    T, E = keys.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if T:
        _load().orc_select(_p(keys), T, E, k, _p(ids), _p(w))
    return ids, w


def route_maps(ids: np.ndarray, E: int, n_shared: int = 1, BN: int = 128) -> dict:
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    P = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(P, np.int32)
    inv = np.empty(P, np.int32)
    max_tiles = P // BN + E + (T + BN - 1) // BN + 1
    bm = np.zeros((max_tiles, 4), np.int32)
    nt = np.zeros(1, np.int32)
    _load().orc_route_maps(_p(ids), T, E, k, n_shared, BN, _p(counts), _p(offsets), _p(perm), _p(inv),
                           _p(bm), _p(nt))
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv,
            "blockmap": bm[: int(nt[0])].copy(), "n_tiles": int(nt[0])}


def rmsnorm(r: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    T, H = r.shape
    x = np.empty_like(r, dtype=np.uint16)
    if T:
        _load().orc_rmsnorm(_p(np.ascontiguousarray(r, np.uint16)), T, H, eps, _p(x))
    return x


def moe_layer(dims: Dims, x: np.ndarray, W: dict, res: np.ndarray | None = None, bias: np.ndarray | None = None,
              keys: np.ndarray | None = None, intermediates: bool = False) -> dict:
    """Run the whole layer on the CPU.  ``W`` holds the packed arrays (see
    ``synthetic.experts``) stacked over E + n_shared experts plus ``router``.
    ``keys`` (optional) replaces the oracle's own router output with given
    fp32 selection keys.  ``W["shared_gate"]`` (optional, fp32 [H]) scales the
    shared expert's output by sigmoid(x . gate).  Returns out (bf16 bits), out_exact (fp64 before the
    final rounding) and, with ``intermediates``, keys/ids/w/h/y."""
    T = x.shape[0]
    H, E, k, I, S = dims.H, dims.E, dims.k, dims.I, dims.n_shared
    x = np.ascontiguousarray(x, np.uint16)
    out = np.empty((T, H), np.uint16)
    out_exact = np.empty((T, H), np.float64)
    keep = {}
    arrs = {n: np.ascontiguousarray(W[n]) for n in
            ("router", "gate_q", "up_q", "gate_s", "gate_b", "up_s", "up_b", "down_q", "down_s", "down_b")}
    sg = W.get("shared_gate")
    arrs["shared_gate"] = None if sg is None else np.ascontiguousarray(sg, np.float32)
    cw = _Weights(*[_p(arrs[f[0]]) for f in _Weights._fields_])
    cd = _Dims(H, E, k, I, S, dims.G)
    if intermediates:
        keep = {"keys": np.empty((T, E), np.float32), "ids": np.empty((T, k), np.int32),
                "w": np.empty((T, k), np.float64), "h": np.empty(((k + S) * T, I), np.uint16),
                "y": np.empty(((k + S) * T, H), np.uint16)}
    kin = None if keys is None else np.ascontiguousarray(keys, np.float32)
    rc = _load().orc_moe_layer(ctypes.byref(cd), _p(x), _p(None if res is None else np.ascontiguousarray(res, np.uint16)),
                               T, ctypes.byref(cw), _p(None if bias is None else np.ascontiguousarray(bias, np.float32)),
                               _p(kin), _p(out), _p(out_exact),
                               _p(keep.get("keys")), _p(keep.get("ids")), _p(keep.get("w")), _p(keep.get("h")),
                               _p(keep.get("y")))
    if rc != 0:
        raise RuntimeError(f"oracle layer failed: {rc}")
    return {"out": out, "out_exact": out_exact, **keep}


def num_threads() -> int:
    return int(_load().orc_num_threads())
