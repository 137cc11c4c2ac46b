"""Seeded synthetic inputs for the MoE expert layer (host side, numpy arrays).

The generator is the C code in ``gen.c`` (SplitMix64 counter streams, see
``gen.h``); this wrapper builds it on first use and returns numpy arrays.
bf16 tensors are returned as ``np.uint16`` bit patterns.  Nothing here
computes any part of the layer: it only draws the inputs that the oracle and
the CUDA path both consume.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_SRC = [os.path.join(_HERE, "gen.c")]
_lock = threading.Lock()
_lib = None

T_X, T_ROUTER, T_RESID, T_SHGATE = 1, 2, 13, 14
T_GDN_Q, T_GDN_K, T_GDN_V, T_GDN_ALPHA, T_GDN_BETA, T_GDN_STATE = 15, 16, 17, 18, 19, 20
T_ATT_Q, T_ATT_K, T_ATT_V = 21, 22, 23


def build(force: bool = False) -> str:
    """Compile libsynth.so (gcc, OpenMP) if missing or older than its sources."""
    with _lock:
        stale = force or not os.path.exists(_LIB_PATH) or any(
            os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC + [os.path.join(_HERE, "gen.h")])
        if stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-ffp-contract=off", "-o", tmp] + _SRC + ["-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, u32, i32, dbl, sz = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        vp = ctypes.c_void_p
        lib.syn_key.restype = u64
        lib.syn_key.argtypes = [u64, u32, u32, u32]
        lib.syn_draw.restype = u64
        lib.syn_draw.argtypes = [u64, u64]
        lib.syn_normal.restype = dbl
        lib.syn_normal.argtypes = [u64, u64]
        lib.syn_uniform.restype = dbl
        lib.syn_uniform.argtypes = [u64, u64]
        lib.syn_fill_normal_bf16.argtypes = [u64, dbl, dbl, vp, sz]
        lib.syn_fill_normal_f32.argtypes = [u64, dbl, dbl, vp, sz]
        lib.syn_fill_uniform_bf16.argtypes = [u64, dbl, dbl, vp, sz]
        lib.syn_fill_uniform_f32.argtypes = [u64, dbl, dbl, vp, sz]
        lib.syn_fill_words.argtypes = [u64, vp, sz]
        lib.syn_expert.argtypes = [u64, u32, u32, i32, i32, i32] + [vp] * 9
        lib.syn_layer_experts.argtypes = [u64, u32, i32, i32, i32, i32] + [vp] * 9
        lib.syn_zipf_bias.argtypes = [u64, u32, i32, dbl, vp]
        lib.syn_num_threads.restype = i32
        _lib = lib
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def key(seed: int, tensor: int, layer: int = 0, expert: int = 0) -> int:
    return _load().syn_key(seed, tensor, layer, expert)


def activations(seed: int, T: int, H: int, layer: int = 0, tensor: int = T_X) -> np.ndarray:
    """x [T, H] bf16 ~ N(0, 1)."""
    out = np.empty((T, H), dtype=np.uint16)
    if out.size:
        _load().syn_fill_normal_bf16(key(seed, tensor, layer), 0.0, 1.0, _p(out), out.size)
    return out


def router(seed: int, E: int, H: int, layer: int = 0, std: float = 0.02) -> np.ndarray:
    """Router weight [E, H] fp32 ~ N(0, std)."""
    out = np.empty((E, H), dtype=np.float32)
    _load().syn_fill_normal_f32(key(seed, T_ROUTER, layer), 0.0, std, _p(out), out.size)
    return out


def shared_gate(seed: int, H: int, layer: int = 0, std: float = 0.02) -> np.ndarray:
    """Shared-expert gate vector [H] fp32 ~ N(0, std)."""
    out = np.empty(H, dtype=np.float32)
    _load().syn_fill_normal_f32(key(seed, T_SHGATE, layer), 0.0, std, _p(out), out.size)
    return out


def gdn_inputs(seed: int, T: int, Hk: int, Hv: int, dk: int = 128, dv: int = 128, layer: int = 0,
               state_std: float = 0.0, alpha=(0.85, 1.0), beta=(0.05, 0.95)) -> dict:
    """Inputs of one Gated DeltaNet scan (one sequence):
    q, k [T, Hk, dk] bf16 ~ N(0, 1/dk) (so |k| is near 1, as after the
    model's L2 normalisation), v [T, Hv, dv] bf16 ~ N(0, 1), decay alpha
    [T, Hv] fp32 ~ U(alpha), write strength beta [T, Hv] fp32 ~ U(beta), and
    an initial state [Hv, dk, dv] fp32 ~ N(0, state_std) (zeros when 0)."""
    lib = _load()
    out = {"q": np.empty((T, Hk, dk), np.uint16), "k": np.empty((T, Hk, dk), np.uint16),
           "v": np.empty((T, Hv, dv), np.uint16), "alpha": np.empty((T, Hv), np.float32),
           "beta": np.empty((T, Hv), np.float32), "state": np.zeros((Hv, dk, dv), np.float32)}
    sd = 1.0 / np.sqrt(dk)
    if T:
        lib.syn_fill_normal_bf16(key(seed, T_GDN_Q, layer), 0.0, sd, _p(out["q"]), out["q"].size)
        lib.syn_fill_normal_bf16(key(seed, T_GDN_K, layer), 0.0, sd, _p(out["k"]), out["k"].size)
        lib.syn_fill_normal_bf16(key(seed, T_GDN_V, layer), 0.0, 1.0, _p(out["v"]), out["v"].size)
        lib.syn_fill_uniform_f32(key(seed, T_GDN_ALPHA, layer), alpha[0], alpha[1], _p(out["alpha"]),
                                 out["alpha"].size)
        lib.syn_fill_uniform_f32(key(seed, T_GDN_BETA, layer), beta[0], beta[1], _p(out["beta"]), out["beta"].size)
    if state_std > 0:
        lib.syn_fill_normal_f32(key(seed, T_GDN_STATE, layer), 0.0, state_std, _p(out["state"]), out["state"].size)
    return out


def attn_inputs(seed: int, L: int, Hq: int = 16, Hkv: int = 2, D: int = 256, layer: int = 0) -> dict:
    """One decode-attention call: query q [Hq, D] and the cache k, v [L, Hkv, D],
    all bf16 ~ N(0, 1)."""
    lib = _load()
    out = {"q": np.empty((Hq, D), np.uint16), "k": np.empty((L, Hkv, D), np.uint16),
           "v": np.empty((L, Hkv, D), np.uint16)}
    for name, t in (("q", T_ATT_Q), ("k", T_ATT_K), ("v", T_ATT_V)):
        if out[name].size:
            lib.syn_fill_normal_bf16(key(seed, t, layer), 0.0, 1.0, _p(out[name]), out[name].size)
    return out


WEIGHT_NAMES = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")


def empty_experts(n_exp: int, H: int, I: int) -> dict:
    """Uninitialised stacked expert arrays with the packed layout's shapes."""
    return {
        "gate_q": np.empty((n_exp, I, H // 8), np.uint32),
        "gate_s": np.empty((n_exp, I, H // 64), np.uint16),
        "gate_b": np.empty((n_exp, I, H // 64), np.uint16),
        "up_q": np.empty((n_exp, I, H // 8), np.uint32),
        "up_s": np.empty((n_exp, I, H // 64), np.uint16),
        "up_b": np.empty((n_exp, I, H // 64), np.uint16),
        "down_q": np.empty((n_exp, H, I // 8), np.uint32),
        "down_s": np.empty((n_exp, H, I // 64), np.uint16),
        "down_b": np.empty((n_exp, H, I // 64), np.uint16),
    }


def experts(seed: int, n_exp: int, H: int, I: int, layer: int = 0, centred: bool = False) -> dict:
    """Packed int4 groupwise-affine experts 0..n_exp-1 of one layer.

    q ~ U{0..15}, scale ~ U(0.005, 0.02) -> bf16, bias ~ N(0, 0.01) -> bf16
    (``centred``: bias - 7.5 * scale, keeping the mean weight near zero).
    """
    w = empty_experts(n_exp, H, I)
    _load().syn_layer_experts(seed, layer, n_exp, H, I, int(centred), *[_p(w[n]) for n in WEIGHT_NAMES])
    return w


def zipf_bias(seed: int, E: int, s: float = 1.1, layer: int = 0) -> np.ndarray:
    """Per-expert logit bias -s*ln(rank) over a seeded ranking of the experts."""
    out = np.empty(E, np.float32)
    _load().syn_zipf_bias(seed, layer, E, s, _p(out))
    return out


def words(seed: int, tensor: int, n: int, layer: int = 0, expert: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint32)
    _load().syn_fill_words(key(seed, tensor, layer, expert), _p(out), n)
    return out


def num_threads() -> int:
    return _load().syn_num_threads()
