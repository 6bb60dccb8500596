"""KDA (Kimi Delta Attention) operator for NVIDIA GB300, behind a C ABI.

The compute runs in ``libkda.so`` (hand-written CUDA for sm_103a, declared
in ``include/kda.h``). This package is a thin ctypes binding with the same
entry-point names; PyTorch only supplies device memory and streams. There is
no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4
KDA_ERR_DEVICE = 5
KDA_ERR_TOO_LARGE = 6
KDA_ERR_RANGE = 7
KDA_BF16 = 0
KDA_F32 = 1
KDA_SCHEDULE_SPLIT = 0
KDA_SCHEDULE_FUSED = 1
KDA_SCHEDULE_DIRECT = 2

EXPORTED = ("kda_status_string", "kda_abi_version", "kda_prefill_workspace_size", "kda_prefill",
            "kda_decode_step", "kda_workspace_status", "kda_check_cu_seqlens",
            "kda_prefill_schedule", "kda_decode", "kda_prefill_ex", "kda_layer_prologue",
            "kda_layer_epilogue", "kda_prefill_set_schedule", "kda_prefill_noalloc",
            "kda_noalloc_status", "kda_layer_prologue_decode", "kda_prefill_workspace_size_ring",
            "kda_prefill_workspace_size_min", "kda_prefill_plan")


class PrefillPlanInfo(ctypes.Structure):
    """kda_prefill_plan_info: the plan that kda_prefill runs."""
    _fields_ = [("schedule", ctypes.c_int32), ("groups", ctypes.c_int32),
                ("group_chains", ctypes.c_int32), ("ring", ctypes.c_int32),
                ("bytes", ctypes.c_size_t), ("lead_items", ctypes.c_int64)]

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, status_string(code), code))


def load() -> ctypes.CDLL:
    """Load libkda.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkda.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_abi_version.argtypes = []
        lib.kda_abi_version.restype = ctypes.c_int
        lib.kda_prefill_workspace_size.argtypes = [I32] * 7
        lib.kda_prefill_workspace_size.restype = SZ
        lib.kda_prefill_workspace_size_ring.argtypes = [I32] * 7
        lib.kda_prefill_workspace_size_ring.restype = SZ
        lib.kda_prefill_workspace_size_min.argtypes = [I32] * 7
        lib.kda_prefill_workspace_size_min.restype = SZ
        lib.kda_prefill_plan.argtypes = [I32] * 7 + [SZ, ctypes.POINTER(PrefillPlanInfo)]
        lib.kda_prefill_plan.restype = ctypes.c_int
        lib.kda_prefill.argtypes = [P, P, P, P, P, F32, P, P, I32, I32, I32, I32, I32, I32, P, P,
                                    P, SZ, P]
        lib.kda_prefill.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [P, P, P, P, P, F32, I32, I32, I32, I32, P, P, P]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_workspace_status.argtypes = [P, P]
        lib.kda_workspace_status.restype = ctypes.c_int
        lib.kda_check_cu_seqlens.argtypes = [P, I32, I32]
        lib.kda_check_cu_seqlens.restype = ctypes.c_int
        lib.kda_prefill_schedule.argtypes = [I32] * 7
        lib.kda_prefill_schedule.restype = ctypes.c_int
        lib.kda_decode.argtypes = [P, P, P, P, P, F32, I32, I32, I32, I32, I32, I32, P, I32, P, P,
                                   P]
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_prefill_ex.argtypes = [P, P, P, P, P, F32, P, P, I32, I32, I32, I32, I32, I32, I32,
                                       I32, I32, P, P, P, P, SZ, P]
        lib.kda_prefill_ex.restype = ctypes.c_int
        lib.kda_layer_prologue.argtypes = [P] * 8 + [I32, P, I32, I32, I32, I32, I32] + [P] * 6
        lib.kda_layer_prologue.restype = ctypes.c_int
        lib.kda_layer_epilogue.argtypes = [P, P, P, I32, I32, I32, I32, P, P]
        lib.kda_layer_epilogue.restype = ctypes.c_int
        lib.kda_layer_prologue_decode.argtypes = [P] * 8 + [I32] * 6 + [P, I32, P] + [P] * 6
        lib.kda_layer_prologue_decode.restype = ctypes.c_int
        lib.kda_prefill_set_schedule.argtypes = [ctypes.c_int]
        lib.kda_prefill_set_schedule.restype = ctypes.c_int
        lib.kda_prefill_noalloc.argtypes = [P, P, P, P, P, F32, P, P, I32, I32, I32, I32, I32, I32,
                                            P, P, P]
        lib.kda_prefill_noalloc.restype = ctypes.c_int
        lib.kda_noalloc_status.argtypes = [P]
        lib.kda_noalloc_status.restype = ctypes.c_int
        # test-only entry point (include/kda_testing.h)
        lib.kda_testing_prefill_chain_timeout.argtypes = [P, P, P, P, P, F32, P, P, I32, I32, I32,
                                                          I32, I32, I32, P, P, P, SZ, I32, P]
        lib.kda_testing_prefill_chain_timeout.restype = ctypes.c_int
        lib.kda_testing_prefill_plan.argtypes = [I32] * 8 + [SZ, ctypes.POINTER(PrefillPlanInfo)]
        lib.kda_testing_prefill_plan.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def kda_status_string(code: int) -> str:
    return status_string(code)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _io_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return KDA_BF16
    if dt == torch.float32:
        return KDA_F32
    raise KDAError(KDA_ERR_UNSUPPORTED, "dtype %s" % dt)


def _check_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("KDA tensors must be CUDA tensors")
            if not t.is_contiguous():
                raise ValueError("KDA tensors must be contiguous")


def kda_prefill_workspace_size(N: int, T: int, H: int, D: int, chunk: int, io: int,
                               varlen: bool = False) -> int:
    return int(load().kda_prefill_workspace_size(N, T, H, D, chunk, io, int(bool(varlen))))


def kda_prefill_workspace_size_ring(N: int, T: int, H: int, D: int, chunk: int, io: int,
                                    varlen: bool = False) -> int:
    return int(load().kda_prefill_workspace_size_ring(N, T, H, D, chunk, io, int(bool(varlen))))


def kda_prefill_workspace_size_min(N: int, T: int, H: int, D: int, chunk: int, io: int,
                                   varlen: bool = False) -> int:
    return int(load().kda_prefill_workspace_size_min(N, T, H, D, chunk, io, int(bool(varlen))))


def kda_prefill_plan(N: int, T: int, H: int, D: int, chunk: int, io: int, varlen: bool,
                     workspace_bytes: int) -> PrefillPlanInfo:
    """The plan kda_prefill runs for these sizes and workspace size (C entry
    point ``kda_prefill_plan``); raises on invalid sizes or a workspace below
    the minimum."""
    info = PrefillPlanInfo()
    rc = int(load().kda_prefill_plan(N, T, H, D, chunk, io, int(bool(varlen)),
                                     int(workspace_bytes), ctypes.byref(info)))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_prefill_plan")
    return info


def kda_prefill_schedule(N: int, T: int, H: int, D: int, chunk: int, io: int,
                         varlen: bool = False) -> int:
    """KDA_SCHEDULE_* that kda_prefill uses for these sizes on the current
    device (C entry point ``kda_prefill_schedule``); raises on invalid sizes."""
    s = int(load().kda_prefill_schedule(N, T, H, D, chunk, io, int(bool(varlen))))
    if s < 0:
        raise KDAError(-s, "kda_prefill_schedule")
    return s


def kda_prefill_set_schedule(schedule: int) -> int:
    """Process-wide override of the bf16 prefill schedule (C entry point
    ``kda_prefill_set_schedule``): -1 = automatic, KDA_SCHEDULE_SPLIT or
    KDA_SCHEDULE_FUSED. Returns the previous value."""
    prev = int(load().kda_prefill_set_schedule(int(schedule)))
    if prev < -1:
        raise KDAError(-prev, "kda_prefill_set_schedule")
    return prev


_WS_SIZE = {"fast": kda_prefill_workspace_size, "ring": kda_prefill_workspace_size_ring,
            "min": kda_prefill_workspace_size_min}


def prefill_workspace(q, cu_seqlens=None, N=None, T=None, chunk=64, kind="fast"):
    """A device workspace for these inputs (torch allocates it; the library
    never does): kind "fast" = kda_prefill_workspace_size() bytes (the fastest
    plan), "ring" = kda_prefill_workspace_size_ring() (bounded: blocks in
    per-chain rings), "min" = kda_prefill_workspace_size_min()."""
    T_total, H, D = q.shape
    if cu_seqlens is not None:
        N, T = cu_seqlens.numel() - 1, T_total
    else:
        N = 1 if N is None else N
        T = T_total // N if T is None else T
    nbytes = _WS_SIZE[kind](N, T, H, D, chunk, _io_code(q.dtype), cu_seqlens is not None)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)


def kda_prefill(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, chunk=64, out=None,
                final_state=None, workspace=None, stream=None, N=None, T=None,
                output_final_state=True, snapshot_interval=0, snapshots=None):
    """Chunked KDA prefill (C entry points ``kda_prefill`` / ``kda_prefill_ex``).

    q, k, v: [T_total, H, D] (bf16 or fp32); g: fp32 [T_total, H, D], or
    [T_total, H] for one decay per token and head; beta: [T_total, H];
    init_state: fp32 [N, H, D, D] or None; cu_seqlens: device int32 [N+1] or
    None (then N sequences of length T, default N=1). With snapshot_interval
    > 0, snapshots: fp32 [N, S, H, D, D] receives the state after every
    snapshot_interval tokens of each sequence (S entries at most).
    Returns (out, final_state)."""
    lib = load()
    io = _io_code(q.dtype)
    T_total, H, D = q.shape
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
        T = T_total
    else:
        N = 1 if N is None else N
        T = T_total // N if T is None else T
    g_per_channel = 0 if g.dim() == 2 else 1
    _check_cuda(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, workspace, snapshots)
    if out is None:
        out = torch.empty_like(q)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = prefill_workspace(q, cu_seqlens, N, T, chunk)
    max_snaps = 0 if snapshots is None else snapshots.shape[1]
    if g_per_channel == 1 and not snapshot_interval:
        rc = lib.kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                             _ptr(init_state), _ptr(cu_seqlens), N, T, H, D, chunk, io, _ptr(out),
                             _ptr(final_state), _ptr(workspace), workspace.numel(),
                             _stream_ptr(stream))
    else:
        rc = lib.kda_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                _ptr(init_state), _ptr(cu_seqlens), N, T, H, D, chunk, io,
                                g_per_channel, int(snapshot_interval), max_snaps, _ptr(snapshots),
                                _ptr(out), _ptr(final_state), _ptr(workspace), workspace.numel(),
                                _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_prefill")
    return out, final_state


def kda_decode_step(q, k, v, g, beta, scale, state, out=None, stream=None):
    """One decode step (C entry point ``kda_decode_step``): q, k, v, g
    [B, H, D]; beta [B, H]; state fp32 [B, H, D, D] updated in place.
    Returns out [B, H, D]."""
    lib = load()
    io = _io_code(q.dtype)
    B, H, D = q.shape
    _check_cuda(q, k, v, g, beta, state, out)
    if out is None:
        out = torch.empty_like(q)
    rc = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), B, H,
                             D, io, _ptr(state), _ptr(out), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_decode_step")
    return out


def kda_decode(q, k, v, g, beta, scale, state_pool, state_indices=None, out=None, stream=None):
    """Decode of T tokens per sequence (C entry point ``kda_decode``):
    q, k, v [B, T, H, D]; g [B, T, H, D] (per channel) or [B, T, H] (one
    decay per token and head); beta [B, T, H]; state_pool fp32
    [P, H, D, D] updated in place; state_indices device int32 [B] or None
    (sequence b uses pool entry b). Returns out [B, T, H, D]."""
    lib = load()
    io = _io_code(q.dtype)
    B, T, H, D = q.shape
    g_per_channel = 1 if g.dim() == 4 else 0
    _check_cuda(q, k, v, g, beta, state_pool, state_indices, out)
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise ValueError("state_indices must be int32")
    if out is None:
        out = torch.empty_like(q)
    rc = lib.kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), B, T, H, D,
                        io, g_per_channel, _ptr(state_pool), state_pool.shape[0],
                        _ptr(state_indices), _ptr(out), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_decode")
    return out


def kda_layer_prologue(q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q, conv_k, conv_v,
                       cu_seqlens=None, stream=None):
    """The layer steps before the operator (C entry point ``kda_layer_prologue``):
    rows [T_total, H, D] of projected q, k, v, alpha and beta [T_total, H];
    depthwise causal convolutions conv_* fp32 [H, D, W]. Returns
    (q, k, v, g, beta) ready for ``kda_prefill``."""
    lib = load()
    io = _io_code(q_raw.dtype)
    T_total, H, D = q_raw.shape
    W = conv_q.shape[2]
    N = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check_cuda(q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q, conv_k, conv_v, cu_seqlens)
    q, k, v = (torch.empty_like(q_raw) for _ in range(3))
    g = torch.empty((T_total, H, D), dtype=torch.float32, device=q_raw.device)
    beta = torch.empty_like(beta_raw)
    rc = lib.kda_layer_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(alpha_raw),
                                _ptr(beta_raw), _ptr(conv_q), _ptr(conv_k), _ptr(conv_v), W,
                                _ptr(cu_seqlens), N, T_total, H, D, io, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(g), _ptr(beta), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_layer_prologue")
    return q, k, v, g, beta


def kda_layer_prologue_decode(q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q, conv_k, conv_v,
                              conv_state, state_indices=None, stream=None):
    """The layer steps before the operator for T new tokens per sequence (C entry
    point ``kda_layer_prologue_decode``): rows [B, T, H, D] of projected q, k, v,
    alpha and beta [B, T, H]; conv_* fp32 [H, D, W]; conv_state [P, 3, W - 1,
    H, D] in the rows' dtype (updated in place; None when W = 1); state_indices
    device int32 [B] or None. Returns (q, k, v, g, beta) for ``kda_decode``."""
    lib = load()
    io = _io_code(q_raw.dtype)
    B, T, H, D = q_raw.shape
    W = conv_q.shape[2]
    _check_cuda(q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q, conv_k, conv_v, conv_state,
                state_indices)
    if conv_state is not None and conv_state.dtype != q_raw.dtype:
        raise ValueError("conv_state must have the rows' dtype")
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise ValueError("state_indices must be int32")
    P = conv_state.shape[0] if conv_state is not None else B
    q, k, v = (torch.empty_like(q_raw) for _ in range(3))
    g = torch.empty((B, T, H, D), dtype=torch.float32, device=q_raw.device)
    beta = torch.empty_like(beta_raw)
    rc = lib.kda_layer_prologue_decode(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(alpha_raw),
                                       _ptr(beta_raw), _ptr(conv_q), _ptr(conv_k), _ptr(conv_v),
                                       W, B, T, H, D, io, _ptr(conv_state), P,
                                       _ptr(state_indices), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_layer_prologue_decode")
    return q, k, v, g, beta


def kda_layer_epilogue(o, gate_raw, norm_weight, y=None, stream=None):
    """Per-head RMS norm of the operator output times sigmoid(gate_raw)
    (C entry point ``kda_layer_epilogue``). Returns y [T_total, H, D]."""
    lib = load()
    io = _io_code(o.dtype)
    T_total, H, D = o.shape
    _check_cuda(o, gate_raw, norm_weight, y)
    if y is None:
        y = torch.empty_like(o)
    rc = lib.kda_layer_epilogue(_ptr(o), _ptr(gate_raw), _ptr(norm_weight), T_total, H, D, io,
                                _ptr(y), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_layer_epilogue")
    return y


def kda_workspace_status(workspace, stream=None) -> int:
    return int(load().kda_workspace_status(_ptr(workspace), _stream_ptr(stream)))


def kda_prefill_noalloc(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, chunk=64,
                        out=None, final_state=None, stream=None, N=None, T=None):
    """kda_prefill without a workspace (C entry point ``kda_prefill_noalloc``):
    its scratch is the library's static device array. Returns (out,
    final_state); device-side errors are read with kda_noalloc_status()."""
    lib = load()
    io = _io_code(q.dtype)
    T_total, H, D = q.shape
    if cu_seqlens is not None:
        N, T = cu_seqlens.numel() - 1, T_total
    else:
        N = 1 if N is None else N
        T = T_total // N if T is None else T
    _check_cuda(q, k, v, g, beta, init_state, cu_seqlens, out, final_state)
    if out is None:
        out = torch.empty_like(q)
    if final_state is None:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    rc = lib.kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                 _ptr(init_state), _ptr(cu_seqlens), N, T, H, D, chunk, io,
                                 _ptr(out), _ptr(final_state), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KDAError(rc, "kda_prefill_noalloc")
    return out, final_state


def kda_noalloc_status(stream=None) -> int:
    """Reads and clears the device status word of kda_prefill_noalloc's static
    array on the current device (C entry point ``kda_noalloc_status``)."""
    return int(load().kda_noalloc_status(_stream_ptr(stream)))


def kda_check_cu_seqlens(cu_host, T_total: int) -> int:
    import numpy as np
    a = np.ascontiguousarray(np.asarray(cu_host, dtype=np.int32))
    return int(load().kda_check_cu_seqlens(a.ctypes.data, a.shape[0] - 1, int(T_total)))
