"""Python binding of libkda, the GB300 (sm_103a) Kimi Delta Attention core.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libkda.so`` behind the C ABI declared in ``include/kda.h``.
PyTorch provides device memory and the stream.  There is no fallback: if
the library is missing, every call raises.

Entry points (same names as the C ABI):
  kda_chunk_fwd        chunked prefill over packed (varlen) sequences
  kda_recurrent_step   one decode token per sequence on a pooled state
  kda_chunk_workspace_bytes, kda_workspace_status, kda_status_string
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

(KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA,
 KDA_ERR_DEVICE_TIMEOUT) = range(6)
# bits of the chunk workspace's status word (kda_workspace_status)
KDA_WS_BAD_SEQLENS, KDA_WS_BAD_SLOT, KDA_WS_TIMEOUT, KDA_WS_EXACT_DECAY, KDA_WS_STRONG_DECAY = (
    1, 2, 4, 8, 16)
KDA_F32, KDA_BF16 = 0, 1
KDA_CHUNK_PRECISE = 1
KDA_CHUNK_SCAN_WIDE = 2
KDA_CHUNK_SCAN_SPLIT = 4
KDA_CHUNK_GATED = 8
KDA_CONV_NONE = 0
KDA_CONV_SILU = 1
_CONV_ACT = {"silu": KDA_CONV_SILU, "none": KDA_CONV_NONE, None: KDA_CONV_NONE}
_SCAN_FLAGS = {"auto": 0, "wide": KDA_CHUNK_SCAN_WIDE, "split": KDA_CHUNK_SCAN_SPLIT}
CHUNK = 64

EXPORTS = ("kda_status_string", "kda_version", "kda_chunk_workspace_bytes", "kda_chunk_fwd",
           "kda_chunk_intra", "kda_chunk_scan", "kda_workspace_status", "kda_recurrent_step",
           "kda_chunk_fwd_noalloc", "kda_chunk_fwd_gated", "kda_recurrent_step_gated",
           "kda_output_gate_norm", "kda_recurrent_multi_step", "kda_short_conv_fwd",
           "kda_short_conv_update", "kda_short_conv_multi_update", "kda_recurrent_multi_step_gated",
           "kda_status_from_workspace_flags")
NOALLOC_WORKSPACE_BYTES = 64 * 1024 * 1024

_lib = None
_lock = threading.Lock()


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {kda_status_string(status)}")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libkda (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"libkda is not built ({path} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_size_t)
        L.kda_status_string.argtypes = [i32]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_version.restype = i32
        L.kda_status_from_workspace_flags.argtypes = [i32]
        L.kda_status_from_workspace_flags.restype = i32
        L.kda_chunk_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32, i32]
        L.kda_chunk_workspace_bytes.restype = sz
        for name in ("kda_chunk_fwd", "kda_chunk_intra", "kda_chunk_scan"):
            fn = getattr(L, name)
            fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i64, i32, i32, i32,
                           f32, i32, i32, vp, sz, vp]
            fn.restype = i32
        L.kda_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i64,
                                            i32, i32, i32, f32, i32, i32, vp]
        L.kda_chunk_fwd_noalloc.restype = i32
        L.kda_workspace_status.argtypes = [vp, ctypes.POINTER(i32), vp]
        L.kda_workspace_status.restype = i32
        L.kda_recurrent_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, i32, i32, i32, i32,
                                         f32, i32, vp]
        L.kda_recurrent_step.restype = i32
        L.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, i32, vp, vp, f32, vp, vp,
                                          vp, i64, vp, vp, i32, i64, i32, i32, i32, f32, i32, i32,
                                          vp, sz, vp]
        L.kda_chunk_fwd_gated.restype = i32
        L.kda_recurrent_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, i32, vp, vp, f32, vp,
                                               vp, i64, vp, i32, i32, i32, i32, f32, i32, vp]
        L.kda_recurrent_step_gated.restype = i32
        L.kda_output_gate_norm.argtypes = [vp, vp, vp, f32, i64, i32, i32, vp]
        L.kda_output_gate_norm.restype = i32
        L.kda_recurrent_multi_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, i32, i32,
                                               i32, i32, i32, f32, i32, vp]
        L.kda_recurrent_multi_step.restype = i32
        L.kda_recurrent_multi_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, i32, vp, vp, f32,
                                                     vp, vp, vp, i64, vp, i32, i32, i32, i32, i32, f32,
                                                     i32, vp]
        L.kda_recurrent_multi_step_gated.restype = i32
        L.kda_short_conv_fwd.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, vp, vp, i64,
                                         i32, vp]
        L.kda_short_conv_fwd.restype = i32
        L.kda_short_conv_update.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, vp]
        L.kda_short_conv_update.restype = i32
        L.kda_short_conv_multi_update.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32,
                                                  i32, vp]
        L.kda_short_conv_multi_update.restype = i32
        _lib = L
        return L


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bf16 or fp32, got {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} shape {tuple(t.shape)} != {tuple(shape)}")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def kda_chunk_workspace_bytes(total_tokens: int, n_seqs: int, H: int, K: int = 128,
                              V: int = 128, dtype: int = KDA_BF16, flags: int = 0) -> int:
    return int(load().kda_chunk_workspace_bytes(total_tokens, n_seqs, H, K, V, dtype, flags))


def _chunk_args(q, k, v, g, beta, cu_seqlens, n_seqs, initial_state, final_state,
                state_indices, n_slots, o, gate_dtype):
    """Shape, dtype and pool checks shared by the chunked entry points.
    Returns (T, H, K, V, N, dtype code, slots)."""
    T, H, K = q.shape
    V = v.shape[-1]
    dt = _dtype_code(q)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be int32 [N+1] with N >= 1")
        N = cu_seqlens.numel() - 1
    else:
        N = 1 if n_seqs is None else int(n_seqs)
    for name, t, dtype_, shape in (("q", q, q.dtype, (T, H, K)), ("k", k, q.dtype, (T, H, K)),
                                   ("v", v, q.dtype, (T, H, V)),
                                   ("g", g, gate_dtype, (T, H, K)),
                                   ("beta", beta, gate_dtype, (T, H)),
                                   ("state_indices", state_indices, torch.int32, (N,)),
                                   ("o", o, q.dtype, (T, H, V))):
        _check(t, name, dtype_, shape)
    _check(initial_state, "initial_state", torch.float32)
    _check(final_state, "final_state", torch.float32)
    if state_indices is None:
        slots = 0
        for name, t in (("initial_state", initial_state), ("final_state", final_state)):
            if t is not None and tuple(t.shape) != (N, H, V, K):
                raise ValueError(f"{name} must be [{N}, {H}, {V}, {K}]")
    else:
        if final_state is None:
            raise ValueError("with state_indices, final_state must be the destination pool")
        slots = final_state.shape[0] if n_slots is None else int(n_slots)
        for name, t in (("initial_state", initial_state), ("final_state", final_state)):
            if t is None:
                continue
            if t.dim() != 4 or tuple(t.shape[1:]) != (H, V, K):
                raise ValueError(f"{name} pool must be [slots, {H}, {V}, {K}]")
            if t.shape[0] < slots:
                raise ValueError(f"{name} pool has {t.shape[0]} slots, fewer than n_slots = {slots}")
    return T, H, K, V, N, dt, slots


def kda_chunk_fwd(q, k, v, g, beta, *, cu_seqlens=None, n_seqs=None, initial_state=None,
                  final_state=None, state_indices=None, n_slots=None, scale=None,
                  precise=False, output_final_state=True, o=None, workspace=None, stream=None,
                  phase="fwd", scan="auto", _gate=None):
    """Chunked KDA forward.

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H] (all CUDA, contiguous).
    cu_seqlens: int32 [N+1] or None (then n_seqs equal-length sequences,
    default 1).  Without state_indices, initial_state / final_state are
    [N, H, V, K]; with state_indices (int32 [N]) they are slot pools
    [slots, H, V, K] and final_state may be the same tensor as
    initial_state (in-place hand-off).  scan: "auto", "wide" or "split"
    selects the tensor-core state-scan layout (see KDA_CHUNK_SCAN_*).
    Returns (o, final_state).
    """
    gdt = q.dtype if _gate is not None else torch.float32  # raw gates come in the q dtype
    T, H, K, V, N, dt, slots = _chunk_args(q, k, v, g, beta, cu_seqlens, n_seqs, initial_state,
                                           final_state, state_indices, n_slots, o, gdt)
    if state_indices is None and final_state is None and output_final_state:
        final_state = torch.empty((N, H, V, K), dtype=torch.float32, device=q.device)
    if o is None:
        o = torch.empty((T, H, V), dtype=q.dtype, device=q.device)
    flags = (KDA_CHUNK_PRECISE if precise else 0) | _SCAN_FLAGS[scan]
    if _gate is not None:
        flags |= KDA_CHUNK_GATED
    need = kda_chunk_workspace_bytes(T, N, H, K, V, dt, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    if scale is None:
        scale = K ** -0.5
    if _gate is not None:
        if phase != "fwd":
            raise ValueError("the gated forward runs as one call (phase='fwd')")
        a_log, dt_bias, lower_bound, out_gate, norm_weight, norm_eps = _gate
        name = "kda_chunk_fwd_gated"
        st = load().kda_chunk_fwd_gated(
            _p(q), _p(k), _p(v), _p(g), _p(beta), _p(a_log), _p(dt_bias),
            float(0.0 if lower_bound is None else lower_bound), int(lower_bound is not None),
            _p(out_gate), _p(norm_weight), float(norm_eps), _p(initial_state), _p(final_state), _p(state_indices), slots, _p(o), _p(cu_seqlens),
            N, T, H, K, V, float(scale), dt, flags, _p(workspace), workspace.numel(),
            _stream(stream))
    else:
        name = {"fwd": "kda_chunk_fwd", "intra": "kda_chunk_intra", "scan": "kda_chunk_scan"}[phase]
        st = getattr(load(), name)(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(initial_state),
                                   _p(final_state), _p(state_indices), slots, _p(o),
                                   _p(cu_seqlens), N, T, H, K, V, float(scale), dt, flags,
                                   _p(workspace), workspace.numel(), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, name)
    return o, final_state


def _check_gate(a_log, dt_bias, H, K):
    _check(a_log, "a_log", torch.float32, (H,))
    _check(dt_bias, "dt_bias", torch.float32, (H, K))


def _check_epilogue(out_gate, norm_weight, shape, dtype):
    if out_gate is None:
        return
    _check(out_gate, "out_gate", dtype, shape)
    _check(norm_weight, "norm_weight", torch.float32, (shape[-1],))


def kda_chunk_fwd_gated(q, k, v, raw_gate, raw_beta, a_log, dt_bias, *, lower_bound=None,
                        out_gate=None, norm_weight=None, norm_eps=1e-6, **kw):
    """Chunked KDA forward from the model's raw gates, activated in-kernel:
    g = lower_bound * sigmoid(exp(a_log[h]) (raw_gate + dt_bias[h])) (or
    -exp(a_log[h]) softplus(raw_gate + dt_bias[h]) without a lower bound),
    beta = sigmoid(raw_beta).  raw_gate [T, H, K] and raw_beta [T, H] in the
    q dtype; a_log [H] and dt_bias [H, K] fp32.  With out_gate ([T, H, V], q
    dtype) and norm_weight ([V] fp32), each output row becomes
    o / sqrt(mean(o^2) + norm_eps) * norm_weight * sigmoid(out_gate).  Other
    arguments as for kda_chunk_fwd.  Returns (o, final_state)."""
    T, H, K = q.shape
    _check_gate(a_log, dt_bias, H, K)
    _check_epilogue(out_gate, norm_weight, tuple(v.shape), q.dtype)
    return kda_chunk_fwd(q, k, v, raw_gate, raw_beta,
                         _gate=(a_log, dt_bias, lower_bound, out_gate, norm_weight, norm_eps), **kw)


def kda_output_gate_norm(o, gate, weight, eps=1e-6, *, stream=None):
    """In place on o [.., V]: o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)."""
    _check(o, "o")
    _check(gate, "gate", o.dtype, tuple(o.shape))
    _check(weight, "weight", torch.float32, (o.shape[-1],))
    st = load().kda_output_gate_norm(_p(o), _p(gate), _p(weight), float(eps),
                                     o.numel() // o.shape[-1], o.shape[-1], _dtype_code(o),
                                     _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_output_gate_norm")
    return o


def kda_recurrent_step_gated(q, k, v, raw_gate, raw_beta, a_log, dt_bias, state_pool, *,
                             lower_bound=None, out_gate=None, norm_weight=None, norm_eps=1e-6,
                             state_indices=None, scale=None, o=None, stream=None):
    """kda_recurrent_step from the model's raw gates, with the optional output
    epilogue applied in the step (see kda_chunk_fwd_gated)."""
    N, H, K = q.shape
    V = v.shape[-1]
    dt = _dtype_code(q)
    for name, t, dtype_, shape in (("q", q, q.dtype, (N, H, K)), ("k", k, q.dtype, (N, H, K)),
                                   ("v", v, q.dtype, (N, H, V)),
                                   ("raw_gate", raw_gate, q.dtype, (N, H, K)),
                                   ("raw_beta", raw_beta, q.dtype, (N, H)),
                                   ("state_pool", state_pool, torch.float32, None),
                                   ("state_indices", state_indices, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    _check_gate(a_log, dt_bias, H, K)
    _check_epilogue(out_gate, norm_weight, (N, H, V), q.dtype)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, V, K):
        raise ValueError(f"state_pool must be [slots, {H}, {V}, {K}]")
    if o is None:
        o = torch.empty((N, H, V), dtype=q.dtype, device=q.device)
    _check(o, "o", q.dtype, (N, H, V))
    if scale is None:
        scale = K ** -0.5
    st = load().kda_recurrent_step_gated(
        _p(q), _p(k), _p(v), _p(raw_gate), _p(raw_beta), _p(a_log), _p(dt_bias),
        float(0.0 if lower_bound is None else lower_bound), int(lower_bound is not None),
        _p(out_gate), _p(norm_weight), float(norm_eps), _p(state_pool), _p(state_indices),
        state_pool.shape[0], _p(o), N, H, K, V, float(scale), dt, _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_step_gated")
    return o


def kda_status_from_workspace_flags(flags: int) -> int:
    """The kda_status a workspace status word stands for (pure host function)."""
    return int(load().kda_status_from_workspace_flags(int(flags)))


def kda_workspace_status(workspace, stream=None, check=False) -> int:
    """Status word (KDA_WS_* bits) of the last chunked forward that used this
    workspace; synchronises the stream.  With check=True a word that stands
    for an error (a bounded device wait that gave up, bad cu_seqlens or
    slots) raises KdaError with that status."""
    if workspace is None:
        raise ValueError("workspace is required")
    out = ctypes.c_int(0)
    st = load().kda_workspace_status(_p(workspace), ctypes.byref(out), _stream(stream))
    if st == KDA_ERR_CUDA:
        raise KdaError(st, "kda_workspace_status")
    if check and st != KDA_OK:
        raise KdaError(st, f"kda_workspace_status (flags {int(out.value):#x})")
    return int(out.value)


def kda_recurrent_step(q, k, v, g, beta, state_pool, *, state_indices=None, scale=None, o=None,
                       stream=None):
    """One decode token per sequence, updating ``state_pool`` [slots, H, V, K] in place.

    q, k, g: [N, H, K]; v: [N, H, V]; beta: [N, H]; state_indices int32 [N]
    or None (slot n).  Returns o [N, H, V].
    """
    N, H, K = q.shape
    V = v.shape[-1]
    dt = _dtype_code(q)
    for name, t, dtype_, shape in (("q", q, q.dtype, (N, H, K)), ("k", k, q.dtype, (N, H, K)),
                                   ("v", v, q.dtype, (N, H, V)),
                                   ("g", g, torch.float32, (N, H, K)),
                                   ("beta", beta, torch.float32, (N, H)),
                                   ("state_pool", state_pool, torch.float32, None),
                                   ("state_indices", state_indices, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, V, K):
        raise ValueError(f"state_pool must be [slots, {H}, {V}, {K}]")
    if o is None:
        o = torch.empty((N, H, V), dtype=q.dtype, device=q.device)
    _check(o, "o", q.dtype, (N, H, V))
    if scale is None:
        scale = K ** -0.5
    st = load().kda_recurrent_step(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(state_pool),
                                   _p(state_indices), state_pool.shape[0], _p(o), N, H, K, V,
                                   float(scale), dt, _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_step")
    return o


def kda_recurrent_multi_step(q, k, v, g, beta, state_pool, state_indices, *, num_accepted=None,
                             scale=None, o=None, stream=None):
    """Speculative decode: S tokens per sequence through the recurrence.

    q, k, g [N, S, H, K]; v [N, S, H, V]; beta [N, S, H]; state_indices int32
    [N, S] (the state after token t goes to slot state_indices[n, t]);
    num_accepted int32 [N] or None (start from slot state_indices[n, a - 1],
    else [n, 0]).  Updates state_pool in place; returns o [N, S, H, V].
    """
    N, S, H, K = q.shape
    V = v.shape[-1]
    dt = _dtype_code(q)
    for name, t, dtype_, shape in (("q", q, q.dtype, (N, S, H, K)), ("k", k, q.dtype, (N, S, H, K)),
                                   ("v", v, q.dtype, (N, S, H, V)),
                                   ("g", g, torch.float32, (N, S, H, K)),
                                   ("beta", beta, torch.float32, (N, S, H)),
                                   ("state_pool", state_pool, torch.float32, None),
                                   ("state_indices", state_indices, torch.int32, (N, S)),
                                   ("num_accepted", num_accepted, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, V, K):
        raise ValueError(f"state_pool must be [slots, {H}, {V}, {K}]")
    if o is None:
        o = torch.empty((N, S, H, V), dtype=q.dtype, device=q.device)
    _check(o, "o", q.dtype, (N, S, H, V))
    if scale is None:
        scale = K ** -0.5
    st = load().kda_recurrent_multi_step(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(state_pool),
                                         _p(state_indices), _p(num_accepted), state_pool.shape[0],
                                         _p(o), N, S, H, K, V, float(scale), dt, _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_multi_step")
    return o


def kda_recurrent_multi_step_gated(q, k, v, raw_gate, raw_beta, a_log, dt_bias, state_pool,
                                   state_indices, *, num_accepted=None, lower_bound=None,
                                   out_gate=None, norm_weight=None, norm_eps=1e-6, scale=None,
                                   o=None, stream=None):
    """kda_recurrent_multi_step from the model's raw gates (raw_gate
    [N, S, H, K], raw_beta [N, S, H], q dtype), with the optional output
    epilogue (out_gate [N, S, H, V]); see kda_recurrent_step_gated."""
    N, S, H, K = q.shape
    V = v.shape[-1]
    dt = _dtype_code(q)
    for name, t, dtype_, shape in (("q", q, q.dtype, (N, S, H, K)), ("k", k, q.dtype, (N, S, H, K)),
                                   ("v", v, q.dtype, (N, S, H, V)),
                                   ("raw_gate", raw_gate, q.dtype, (N, S, H, K)),
                                   ("raw_beta", raw_beta, q.dtype, (N, S, H)),
                                   ("state_pool", state_pool, torch.float32, None),
                                   ("state_indices", state_indices, torch.int32, (N, S)),
                                   ("num_accepted", num_accepted, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    _check_gate(a_log, dt_bias, H, K)
    _check_epilogue(out_gate, norm_weight, (N, S, H, V), q.dtype)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, V, K):
        raise ValueError(f"state_pool must be [slots, {H}, {V}, {K}]")
    if o is None:
        o = torch.empty((N, S, H, V), dtype=q.dtype, device=q.device)
    _check(o, "o", q.dtype, (N, S, H, V))
    if scale is None:
        scale = K ** -0.5
    st = load().kda_recurrent_multi_step_gated(
        _p(q), _p(k), _p(v), _p(raw_gate), _p(raw_beta), _p(a_log), _p(dt_bias),
        float(0.0 if lower_bound is None else lower_bound), int(lower_bound is not None),
        _p(out_gate), _p(norm_weight), float(norm_eps), _p(state_pool), _p(state_indices),
        _p(num_accepted), state_pool.shape[0], _p(o), N, S, H, K, V, float(scale), dt,
        _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_multi_step_gated")
    return o


def kda_short_conv_fwd(x, weight, *, cu_seqlens=None, n_seqs=None, activation="silu",
                       initial_states=None, final_states=None, state_indices=None, n_slots=None,
                       y=None, stream=None):
    """Short causal convolution over packed sequences (prefill).

    x [T, D]; weight [ks, D] (same dtype); cu_seqlens int32 [N+1] or None
    (n_seqs equal lengths, default 1); activation "silu" or "none".  Conv
    states are [N, ks-1, D] per sequence, or pools [slots, ks-1, D] picked by
    state_indices (int32 [N]); initial_states None = zeros; final_states None =
    not written (may be the initial pool, updated in place).  Returns
    (y [T, D], final_states).
    """
    T, D = x.shape
    ks = weight.shape[0]
    dt = _dtype_code(x)
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if n_seqs is None else int(n_seqs))
    for name, t, dtype_, shape in (("x", x, x.dtype, (T, D)), ("weight", weight, x.dtype, (ks, D)),
                                   ("cu_seqlens", cu_seqlens, torch.int32, (N + 1,)),
                                   ("state_indices", state_indices, torch.int32, (N,)),
                                   ("initial_states", initial_states, x.dtype, None),
                                   ("final_states", final_states, x.dtype, None)):
        _check(t, name, dtype_, shape)
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", x.dtype, (T, D))
    pool = final_states if final_states is not None else initial_states
    slots = 0
    if state_indices is not None:
        slots = pool.shape[0] if n_slots is None else int(n_slots)
    st = load().kda_short_conv_fwd(_p(x), _p(weight), _p(y), _p(cu_seqlens), N, T, D, ks,
                                   _CONV_ACT[activation], _p(initial_states), _p(final_states),
                                   _p(state_indices), slots, dt, _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_short_conv_fwd")
    return y, final_states


def kda_short_conv_update(x, weight, state_pool, *, state_indices=None, activation="silu", y=None,
                          stream=None):
    """One decode token per sequence: x [N, D]; state_pool [slots, ks-1, D]
    (slot n, or state_indices int32 [N]) shifted in place.  Returns y [N, D]."""
    N, D = x.shape
    ks = weight.shape[0]
    dt = _dtype_code(x)
    for name, t, dtype_, shape in (("x", x, x.dtype, (N, D)), ("weight", weight, x.dtype, (ks, D)),
                                   ("state_pool", state_pool, x.dtype, None),
                                   ("state_indices", state_indices, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    if state_pool.dim() != 3 or tuple(state_pool.shape[1:]) != (ks - 1, D):
        raise ValueError(f"state_pool must be [slots, {ks - 1}, {D}]")
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", x.dtype, (N, D))
    st = load().kda_short_conv_update(_p(x), _p(weight), _p(y), _p(state_pool), _p(state_indices),
                                      state_pool.shape[0], N, D, ks, _CONV_ACT[activation], dt,
                                      _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_short_conv_update")
    return y


def kda_short_conv_multi_update(x, weight, state_pool, state_indices, *, num_accepted=None,
                                activation="silu", y=None, stream=None):
    """S tokens per sequence through the conv: x [N, S, D]; state_pool
    [slots, ks-1, D]; state_indices int32 [N, S] (state after token t to
    slot [n][t]); num_accepted int32 [N] or None (start slot [n][a-1], else
    [n][0]).  Returns y [N, S, D]."""
    N, S, D = x.shape
    ks = weight.shape[0]
    dt = _dtype_code(x)
    for name, t, dtype_, shape in (("x", x, x.dtype, (N, S, D)), ("weight", weight, x.dtype, (ks, D)),
                                   ("state_pool", state_pool, x.dtype, None),
                                   ("state_indices", state_indices, torch.int32, (N, S)),
                                   ("num_accepted", num_accepted, torch.int32, (N,))):
        _check(t, name, dtype_, shape)
    if state_indices is None:
        raise ValueError("state_indices is required")
    if state_pool.dim() != 3 or tuple(state_pool.shape[1:]) != (ks - 1, D):
        raise ValueError(f"state_pool must be [slots, {ks - 1}, {D}]")
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", x.dtype, (N, S, D))
    st = load().kda_short_conv_multi_update(_p(x), _p(weight), _p(y), _p(state_pool),
                                            _p(state_indices), _p(num_accepted), state_pool.shape[0],
                                            N, S, D, ks, _CONV_ACT[activation], dt, _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_short_conv_multi_update")
    return y


def kda_chunk_fwd_noalloc(q, k, v, g, beta, *, o, final_state=None, cu_seqlens=None, n_seqs=None,
                          initial_state=None, state_indices=None, n_slots=None, scale=None,
                          precise=False, stream=None):
    """kda_chunk_fwd without a workspace argument, for hosts that cannot
    allocate device memory: the library serves the scratch space from a
    fixed 64 MiB array of its own (see include/kda.h).  This wrapper
    allocates nothing either, so ``o`` is required, and ``final_state`` is
    written only when given (it is required, as the destination pool, with
    state_indices).  Arguments are checked as for kda_chunk_fwd.  Returns
    (o, final_state)."""
    if o is None:
        raise ValueError("kda_chunk_fwd_noalloc allocates nothing: pass o")
    T, H, K, V, N, dt, slots = _chunk_args(q, k, v, g, beta, cu_seqlens, n_seqs, initial_state,
                                           final_state, state_indices, n_slots, o, torch.float32)
    flags = KDA_CHUNK_PRECISE if precise else 0
    if scale is None:
        scale = K ** -0.5
    st = load().kda_chunk_fwd_noalloc(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(initial_state),
                                      _p(final_state), _p(state_indices), slots, _p(o),
                                      _p(cu_seqlens), N, T, H, K, V, float(scale), dt, flags,
                                      _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_noalloc")
    return o, final_state
