"""KDA oracle -- test infrastructure only.

A plain fp64 CPU recurrence (``kda_oracle.c``) behind ctypes. Only the
tests, the smoke check and the benchmark's CPU-baseline leg may import this
package; the CUDA library never does, and the two share no code.

The recurrence, per (sequence, head), is the token-by-token KDA update
("K3 vs DSV4 architecture divergence", locsic.com, KDA section:
forget -> correct -> write; "Kimi K3: The Manos, The Mythos, The Legendos",
SemiAnalysis, sections "DeltaNet" / "Gated DeltaNet" / "FlashKDA 算法"):

    S <- Diag(exp(clamp(g_t, -5, 0))) S
    u  = beta_t (v_t - S^T k_t)
    S <- S + k_t u^T
    o_t = scale * S^T q_t

Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, reductions to DeltaNet / gated linear attention / a hand-worked
example); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    f = lib.kda_oracle_prefill
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, P, P, ctypes.c_double, P, P, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int32]
    f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def _f32(x):
    a = np.asarray(x, dtype=np.float32)
    return np.ascontiguousarray(a)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def prefill(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, nthreads=None, _lib_path=None):
    """fp64 token recurrence over packed sequences.

    q, k, g: [T_total, H, Dk]; v: [T_total, H, Dv]; beta: [T_total, H]
    (any float array-likes; they are taken at their exact float32 values,
    which holds every bf16 and fp32 input exactly).
    init_state: [N, H, Dk, Dv] (float64 kept as is) or None for zeros.
    cu_seqlens: int [N+1] or None for one sequence of length T_total.
    Returns (out [T_total, H, Dv] float64, final_state [N, H, Dk, Dv] float64).
    """
    q, k, v, g = _f32(q), _f32(k), _f32(v), _f32(g)
    beta = _f32(beta)
    T, H, Dk = q.shape
    Dv = v.shape[2]
    assert k.shape == (T, H, Dk) and g.shape == (T, H, Dk)
    assert v.shape == (T, H, Dv) and beta.shape == (T, H)
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int32)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    assert cu[-1] == T, "cu_seqlens[-1] must equal T_total"
    init = None
    if init_state is not None:
        init = np.ascontiguousarray(np.asarray(init_state, dtype=np.float64))
        assert init.shape == (N, H, Dk, Dv)
    out = np.zeros((T, H, Dv), dtype=np.float64)
    fin = np.zeros((N, H, Dk, Dv), dtype=np.float64)
    nt = nthreads or default_threads()
    lib = _load() if _lib_path is None else _bind(_lib_path)
    rc = lib.kda_oracle_prefill(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                                beta.ctypes.data, float(scale),
                                None if init is None else init.ctypes.data, cu.ctypes.data,
                                N, H, Dk, Dv, out.ctypes.data, fin.ctypes.data, nt)
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    return out, fin


def decode_step(q, k, v, g, beta, scale, state):
    """One decode step for B sequences: q, k, g [B, H, Dk]; v [B, H, Dv];
    beta [B, H]; state [B, H, Dk, Dv]. It is the same recurrence run for one
    token per sequence. Returns (out [B, H, Dv], new_state), both float64."""
    B = np.asarray(q).shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return prefill(q, k, v, g, beta, scale, init_state=state, cu_seqlens=cu)
