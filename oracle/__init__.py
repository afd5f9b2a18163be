"""KDA oracle: slow, plain, fp64 CPU statements of what the KDA core computes.

TEST INFRASTRUCTURE ONLY.  The CUDA library never imports, links or calls
anything here, and nothing here imports the library.  Only ``tests/``, the
smoke check and the benchmark's CPU-baseline leg use this package.

Two independent statements of the same mathematics:

* ``recurrence`` -- the token-by-token recurrence (C, fp64, ``kda_oracle.c``),
  as defined on the nnterp "kimi_linear" page (paragraph on Kimi Delta
  Attention: channel-wise decay before each delta-rule update, L2 norm of q
  and k inside the kernel) with the L2 norm and scale of the Ascend model
  file's ``_l2_normalize`` / ``_torch_chunk_kda``.  This is THE oracle.
* ``chunked_form`` -- the chunk-parallel (WY/UT) form restated, step by step
  and in the same order, from ``_torch_chunk_kda`` in the Ascend model file
  (tail padding, per-chunk cumulative log-decay, strictly-lower interaction
  matrix, forward substitution, corrected keys/values, causal intra-chunk
  scores, inter-chunk state pass).  Pure numpy, fp64, exact pairwise
  exponentials; used only to cross-check the recurrence on tiny inputs.

``gate_activation`` is the model's gate activation (raw decay gate plus
per-channel bias, scaled by exp(A_log), through a lower-bounded sigmoid or a
softplus; raw beta through a sigmoid), as written in the Ascend model file's
``_prefill_torch_kda`` and decode branch; the gated entry points compute it
in-kernel and are compared against ``gate_activation`` followed by the
recurrence.

``output_gate_norm`` is the model's output epilogue (RMSNorm over the value
dim, its weight, times sigmoid of the output gate; ``_project_out``).

``multi_step`` is speculative decode with a verify width of S tokens per
sequence: per-token state slots, and the initial state picked by the number of
tokens accepted in the previous step.

``short_conv_prefill`` / ``short_conv_update`` are the model's depthwise causal
short convolution on the fused q/k/v projection (``KimiShortConvolution``),
over packed sequences and one decode token at a time, with its state cache.

``step`` is one decode token of the recurrence on rows of a state pool picked
by slot indices (the model file's ``_decode_gdr`` / ``_decode_fused_kda``
semantics: the pool is updated in place).

State orientation: the oracle works in the mathematical K x V orientation.
The library stores states as [.., V, K]; callers transpose when comparing.

Parity status of each function is recorded with its pins in
``tests/test_oracle_pins.py``; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C recurrence with the host gcc (portable flags, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_recurrence.argtypes = [
                dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64),
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                dp, dp, dp, ctypes.c_int]
            lib.kda_oracle_recurrence.restype = ctypes.c_int
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _f64(x) -> np.ndarray:
    """Widen to a contiguous fp64 numpy array (exact for bf16 and fp32 values)."""
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().cpu().float().numpy() if str(x.dtype) == "torch.bfloat16" else x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, g, beta, cu_seqlens=None, initial_state=None, scale=None,
               n_threads: int = 0):
    """Token recurrence in fp64.

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]  (T = all tokens, packed);
    cu_seqlens: [N+1] sequence offsets, or None for one sequence;
    initial_state: [N, H, K, V] (math orientation) or None for zeros.
    Returns (o [T, H, V], final_state [N, H, K, V]), both fp64.
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
    n = len(cu) - 1
    if scale is None:
        scale = K ** -0.5
    o = np.zeros((T, H, V), dtype=np.float64)
    sf = np.zeros((n, H, K, V), dtype=np.float64)
    s0 = None if initial_state is None else _f64(initial_state)
    if s0 is not None and s0.shape != (n, H, K, V):
        raise ValueError(f"initial_state shape {s0.shape} != {(n, H, K, V)}")
    rc = _load().kda_oracle_recurrence(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, H, K, V, float(scale),
        _ptr(s0) if s0 is not None else None, _ptr(o), _ptr(sf), int(n_threads))
    if rc != 0:
        raise RuntimeError("kda_oracle_recurrence failed (bad arguments or out of memory)")
    return o, sf


def step(q, k, v, g, beta, pool, state_indices=None, scale=None):
    """One decode token per sequence on a state pool, in fp64.

    q, k, g: [N, H, K]; v: [N, H, V]; beta: [N, H]; pool: [slots, H, K, V]
    (math orientation, NOT modified); state_indices: [N] slot per sequence or
    None for slot n.  Returns (o [N, H, V], new_pool) with the picked slots
    advanced by one token and every other slot unchanged.
    """
    q = _f64(q)
    N = q.shape[0]
    pool = _f64(pool).copy()
    idx = np.arange(N) if state_indices is None else np.asarray(
        state_indices.cpu().numpy() if hasattr(state_indices, "cpu") else state_indices, dtype=np.int64)
    cu = np.arange(N + 1, dtype=np.int64)
    o, sf = recurrence(q, k, v, g, beta, cu_seqlens=cu, initial_state=pool[idx], scale=scale)
    pool[idx] = sf
    return o, pool


def _l2_normalize(x: np.ndarray) -> np.ndarray:
    # eps 1e-6 added to the sum of squares, inside the root (model file, _l2_normalize)
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + 1e-6)


def chunked_form(q, k, v, g, beta, initial_state=None, chunk: int = 64, scale=None):
    """Chunk-parallel KDA for ONE sequence, in fp64 (model file, _torch_chunk_kda).

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]; initial_state: [H, K, V]
    or None.  Returns (o [T, H, V], final_state [H, K, V]).
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    S_all = np.zeros((H, K, V)) if initial_state is None else _f64(initial_state).copy()

    # 1. right-pad to a multiple of the chunk: zero q/k/v, zero log-decay (no
    #    decay) and zero beta (no write), so padded tokens leave the state alone.
    pad = (-T) % chunk
    if pad:
        zk = np.zeros((pad, H, K))
        q, k, g = (np.concatenate([t, zk]) for t in (q, k, g))
        v = np.concatenate([v, np.zeros((pad, H, V))])
        beta = np.concatenate([beta, np.zeros((pad, H))])
    n_chunks = q.shape[0] // chunk

    # 2. L2-normalise q and k over the key dim; fold the scale into q.
    qn = _l2_normalize(q) * scale
    kn = _l2_normalize(k)

    o = np.zeros((n_chunks * chunk, H, V))
    for h in range(H):
        S = S_all[h]
        for c in range(n_chunks):
            rows = slice(c * chunk, (c + 1) * chunk)
            Q, Kc, Vc = qn[rows, h], kn[rows, h], v[rows, h]
            b = beta[rows, h]
            # 3. cumulative log-decay inside the chunk
            G = np.cumsum(g[rows, h], axis=0)
            # 4. strictly-lower interaction matrix, rows scaled by beta:
            #    M[r, j] = beta_r * sum_d k_r,d k_j,d exp(G_r,d - G_j,d), j < r
            M = np.zeros((chunk, chunk))
            for r in range(chunk):
                for j in range(r):
                    M[r, j] = b[r] * np.sum(Kc[r] * Kc[j] * np.exp(G[r] - G[j]))
            # 5. forward substitution: X = (I + M)^-1 built row by row, then
            #    columns scaled by beta: Tm = (I + M)^-1 diag(beta)
            X = np.zeros((chunk, chunk))
            for r in range(chunk):
                X[r] = -(M[r, :r] @ X[:r]) if r else 0.0
                X[r, r] += 1.0
            Tm = X * b[None, :]
            # 6. corrected keys and values
            W = Tm @ (np.exp(G) * Kc)
            U = Tm @ Vc
            # 7. causal intra-chunk scores, diagonal kept
            A = np.zeros((chunk, chunk))
            for r in range(chunk):
                for j in range(r + 1):
                    A[r, j] = np.sum(Q[r] * np.exp(G[r] - G[j]) * Kc[j])
            # 8. inter-chunk pass: new values, output, state carried to the next chunk
            Vnew = U - W @ S
            o[rows, h] = (Q * np.exp(G)) @ S + A @ Vnew
            GC = G[-1]
            S = np.exp(GC)[:, None] * S + (np.exp(GC[None, :] - G) * Kc).T @ Vnew
        S_all[h] = S
    return o[:T], S_all


def _softplus(x: np.ndarray) -> np.ndarray:
    """max(x, 0) + log1p(exp(-|x|)): the model file's ``_softplus``, in fp64."""
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def _sigmoid(x: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-x)) without overflow for large |x| (fp64)."""
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def gate_activation(raw_gate, raw_beta, a_log, dt_bias, lower_bound=None):
    """The gate activation of the Ascend model file (``_prefill_torch_kda``; the
    same formulas in the decode branch of ``KimiDeltaAttention.forward``):

        x    = raw_gate + dt_bias[h, k]
        g    = lower_bound * sigmoid(exp(a_log[h]) * x)   with a lower bound
             = -exp(a_log[h]) * softplus(x)               without
        beta = sigmoid(raw_beta)

    raw_gate [T, H, K], raw_beta [T, H], a_log [H], dt_bias [H, K] (the model's
    flat [H*K] parameter viewed per head).  Returns (g, beta) in fp64."""
    x = _f64(raw_gate) + _f64(dt_bias)[None, :, :]
    scale = np.exp(_f64(a_log))[None, :, None]
    if lower_bound is None:
        g = -scale * _softplus(x)
    else:
        g = float(lower_bound) * _sigmoid(scale * x)
    return g, _sigmoid(_f64(raw_beta))



def output_gate_norm(o, gate, weight, eps):
    """The output epilogue of the model (Ascend model file,
    ``KimiDeltaAttention._project_out``): RMSNorm over the value dim of each
    (token, head) row, times its weight, times sigmoid of the output gate,

        out[t, h, v] = o[t, h, v] / sqrt(mean_v o[t, h, :]^2 + eps) * weight[v]
                       * sigmoid(gate[t, h, v])

    o, gate [.., H, V]; weight [V].  fp64."""
    x = _f64(o)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(eps))
    return x * r * _f64(weight) * _sigmoid(_f64(gate))


def multi_step(q, k, v, g, beta, pool, state_indices, num_accepted=None, scale=None):
    """Speculative (multi-token) decode on a state pool, as the model's
    ``_decode_fused_kda`` / ``_decode_gdr`` call it with a verify width S
    (``ssm_state_indices`` of batch x S entries, ``num_accepted_tokens``).
    Reading of the call: sequence n starts from slot
    state_indices[n, num_accepted[n] - 1] (from state_indices[n, 0] when
    num_accepted is None), runs its S tokens in order through the
    recurrence, and the state after token t is written to slot
    state_indices[n, t].

    q, k, g [N, S, H, K]; v [N, S, H, V]; beta [N, S, H]; pool [slots, H, K, V]
    (oracle orientation); state_indices [N, S]; num_accepted [N] or None.
    Returns (o [N, S, H, V], new pool), fp64."""
    q, k, v, g, b = (_f64(t) for t in (q, k, v, g, beta))
    idx = np.asarray(state_indices, dtype=np.int64)
    N, S = idx.shape
    out_pool = _f64(pool).copy()
    o = np.zeros(v.shape, dtype=np.float64)
    for n in range(N):
        a = 1 if num_accepted is None else int(num_accepted[n])
        state = out_pool[idx[n, a - 1]].copy()
        for t in range(S):
            o_t, s_t = recurrence(q[n, t:t + 1], k[n, t:t + 1], v[n, t:t + 1], g[n, t:t + 1],
                                  b[n, t:t + 1], initial_state=state[None], scale=scale)
            o[n, t] = o_t[0]
            state = s_t[0]
            out_pool[idx[n, t]] = state
    return o, out_pool


def _act(y: np.ndarray, activation: str) -> np.ndarray:
    if activation == "silu":
        return y * _sigmoid(y)
    if activation in (None, "none"):
        return y
    raise ValueError(activation)


def short_conv_prefill(x, weight, cu_seqlens, activation="silu", initial_states=None):
    """Depthwise causal convolution over packed sequences (Ascend model file,
    ``KimiShortConvolution``, prefill branch: ``causal_conv1d_fn``):

        y[t, d] = act( sum_{i<ks} weight[i, d] * x[t - (ks - 1) + i, d] )

    where positions before the sequence start read its initial state (the
    ks - 1 previous inputs; zeros when ``initial_states`` is None, as the model
    passes has_initial_state = 0).  x [T, D]; weight [ks, D] (the model's
    ``_conv_weight``); initial_states [N, ks - 1, D] or None.
    Returns y [T, D] and the final states [N, ks - 1, D] (each sequence's last
    ks - 1 inputs, reaching into its initial state when it is shorter), fp64."""
    x = _f64(x)
    w = _f64(weight)
    ks, D = w.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    y = np.zeros_like(x)
    finals = np.zeros((N, ks - 1, D))
    for n in range(N):
        s, e = cu[n], cu[n + 1]
        init = np.zeros((ks - 1, D)) if initial_states is None else _f64(initial_states)[n]
        ext = np.concatenate([init, x[s:e]], axis=0)  # rows: ks - 1 history, then the sequence
        for t in range(e - s):
            y[s + t] = _act(np.sum(w * ext[t:t + ks], axis=0), activation)
        finals[n] = ext[len(ext) - (ks - 1):]
    return y, finals


def short_conv_update(x, weight, state, activation="silu"):
    """One decode token per sequence (the update branch:
    ``causal_conv1d_update``): y[n, d] = act(sum_i weight[i, d] * window[i, d])
    with window = [state[n] ; x[n]], and the state shifts by one token.
    x [N, D]; weight [ks, D]; state [N, ks - 1, D].  Returns (y, new state)."""
    x = _f64(x)
    w = _f64(weight)
    st = _f64(state)
    win = np.concatenate([st, x[:, None, :]], axis=1)  # [N, ks, D]
    y = _act(np.sum(w[None] * win, axis=1), activation)
    return y, win[:, 1:].copy()


def short_conv_multi_update(x, weight, pool, state_indices, num_accepted=None, activation="silu"):
    """Speculative decode through the short conv: the model's update branch
    with a verify width S > 1 (the flattened [batch x S] tokens,
    ``conv_state_indices`` from the per-sequence state blocks and
    ``num_accepted_tokens``).  Reading of the call, the one taken for the
    core's multi-token decode: sequence n starts from the conv state in slot
    state_indices[n, num_accepted[n] - 1] (slot state_indices[n, 0] when
    num_accepted is None), runs its S tokens in order through the one-token
    update, and the state after token t is written to slot
    state_indices[n, t].

    x [N, S, D]; weight [ks, D]; pool [slots, ks - 1, D]; state_indices
    [N, S]; num_accepted [N] or None.  Returns (y [N, S, D], new pool), fp64."""
    x = _f64(x)
    idx = np.asarray(state_indices, dtype=np.int64)
    N, S = idx.shape
    out_pool = _f64(pool).copy()
    y = np.zeros(x.shape, dtype=np.float64)
    for n in range(N):
        a = 1 if num_accepted is None else int(num_accepted[n])
        state = out_pool[idx[n, a - 1]].copy()
        for t in range(S):
            yt, st = short_conv_update(x[n, t:t + 1], weight, state[None], activation=activation)
            y[n, t] = yt[0]
            state = st[0]
            out_pool[idx[n, t]] = state
    return y, out_pool
