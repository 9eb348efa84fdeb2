"""CPU oracle for the recurrent-cell unroll (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
CUDA library and its binding) never imports this package.

The C source ``oracle.c`` is compiled on first use with gcc (``-O2 -fopenmp``,
portable C, no target-specific flags) into ``oracle/_build/liboracle.so`` and
loaded with ctypes.  Every function takes numpy arrays and returns float64
results.  See ``oracle.c`` for the equations and the passages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

LSTM, GRU = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _LayerW(ctypes.Structure):
    _fields_ = [("w_ih", ctypes.c_void_p), ("w_hh", ctypes.c_void_p),
                ("b_ih", ctypes.c_void_p), ("b_hh", ctypes.c_void_p),
                ("w_hr", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_rnn_forward.restype = i
            lib.oracle_rnn_forward.argtypes = [i, i, i, i, i, i, i, i, i, P, P, P, P, P, P, P, P,
                                               P, i, i, P]
            lib.oracle_pack.restype = i
            lib.oracle_pack.argtypes = [i, i, P, P, P, P]
            lib.oracle_rssm_unroll.restype = i
            lib.oracle_rssm_unroll.argtypes = [i, i, i, i, i, i] + [P] * 14 + [P, P, P, P, P, i, i]
            lib.oracle_rssm_unroll2.restype = i
            lib.oracle_rssm_unroll2.argtypes = ([i, i, i, i, i, i] + [P] * 14 + [P, P, P, P, P, i, i]
                                                + [i, P, P, P, P, P])
            lib.oracle_rnn_backward.restype = i
            lib.oracle_rnn_backward.argtypes = [i] * 9 + [P] * 16 + [i, P]
            lib.oracle_rssm_backward.restype = i
            lib.oracle_rssm_backward.argtypes = [i] * 6 + [P] * 31
            lib.oracle_rssm_backward2.restype = i
            lib.oracle_rssm_backward2.argtypes = [i] * 6 + [P] * 31 + [i] + [P] * 8
            lib.oracle_bf16_round.restype = ctypes.c_double
            lib.oracle_bf16_round.argtypes = [ctypes.c_float]
            lib.oracle_num_threads_default.restype = i
            _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return int(_load().oracle_num_threads_default())


def bf16_round(values) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) -> value, as float64."""
    lib = _load()
    v = _f32(values).ravel()
    return np.array([lib.oracle_bf16_round(float(f)) for f in v], dtype=np.float64).reshape(
        np.shape(values))


def pack(lengths, T: int):
    """Length sort metadata: (sorted_idx, unsorted_idx, batch_sizes), int32."""
    lib = _load()
    ln = _i32(lengths)
    B = ln.shape[0]
    s = np.zeros(B, np.int32)
    u = np.zeros(B, np.int32)
    bs = np.zeros(T, np.int32)
    rc = lib.oracle_pack(B, T, _ptr(ln), _ptr(s), _ptr(u), _ptr(bs))
    if rc != 0:
        raise ValueError("lengths outside [1, T]")
    return s, u, bs


def rnn_forward(cell: int, x, weights, *, hidden: int, proj: int = 0, bidirectional: bool = False,
                lengths=None, h0=None, c0=None, bf16_weights: bool = False, rows=None,
                threads: int = 0, cell_clip=None, proj_clip=None):
    """Stacked LSTM / GRU (optionally bidirectional / projected) forward in fp64.

    cell_clip / proj_clip: None or (lo, hi).  The LSTM cell state is clamped
    to [lo, hi] as soon as it is updated (before tanh); the projected hidden
    state as soon as it is formed (cell-state and projection clipping named in
    "RNN Op Changes", apache/mxnet issue 9543).

    x: [T, B, in]; weights: list over layer*D + dir of dicts with keys
    w_ih, w_hh, b_ih, b_hh (None = zero) and w_hr (projection, LSTM only).
    rows: optional list of batch rows to compute (others are left zero).
    Returns (y [T,B,D*Hout], h_n [L*D,B,Hout], c_n [L*D,B,H] or None).
    """
    lib = _load()
    x = _f32(x)
    T, B, in_dim = x.shape
    D = 2 if bidirectional else 1
    L = len(weights) // D
    assert L * D == len(weights) and L >= 1
    Hout = proj if proj > 0 else hidden
    keep = []
    arr = (_LayerW * (L * D))()
    for i, w in enumerate(weights):
        vals = [_f32(w.get(k)) for k in ("w_ih", "w_hh", "b_ih", "b_hh", "w_hr")]
        keep.extend(vals)
        arr[i] = _LayerW(*[_ptr(v) for v in vals])
    ln = _i32(lengths)
    h0a, c0a = _f32(h0), _f32(c0)
    y = np.zeros((T, B, D * Hout), np.float64)
    hn = np.zeros((L * D, B, Hout), np.float64)
    cn = np.zeros((L * D, B, hidden), np.float64)
    rw = _i32(rows)
    clip = None
    if cell_clip is not None or proj_clip is not None:
        inf = float("inf")
        cl = cell_clip if cell_clip is not None else (-inf, inf)
        pl = proj_clip if proj_clip is not None else (-inf, inf)
        clip = np.array([cl[0], cl[1], pl[0], pl[1]], np.float64)
    rc = lib.oracle_rnn_forward(int(cell), int(bidirectional), L, in_dim, hidden, proj,
                                int(bool(bf16_weights)), T, B, _ptr(x), _ptr(ln), _ptr(h0a),
                                _ptr(c0a), ctypes.addressof(arr), _ptr(y), _ptr(hn), _ptr(cn),
                                _ptr(rw), 0 if rw is None else len(rw), int(threads), _ptr(clip))
    if rc != 0:
        raise ValueError("oracle_rnn_forward: invalid arguments")
    return y, hn, (cn if cell == LSTM else None)


def rnn_backward(cell: int, x, weights, dy, *, hidden: int, proj: int = 0,
                 bidirectional: bool = False, lengths=None, h0=None, c0=None, dh_n=None,
                 dc_n=None, bf16_weights: bool = False, threads: int = 0, cell_clip=None,
                 proj_clip=None):
    """Backward pass through time of a stacked LSTM / GRU, or LSTM with
    projection, optionally bidirectional, over padded or variable-length
    batches, in fp64:
    the gradients of a loss with dL/dy = dy [T,B,D*Ho] (and dL/dh_n
    [L*D,B,Ho], dL/dc_n [L*D,B,H], None = 0; Ho = proj or hidden).

    weights: list over layer*D + dir of dicts w_ih, w_hh, b_ih, b_hh (None =
    zero) and w_hr (projection).  Returns a dict: dx [T,B,in], dh0
    [L*D,B,Ho], dc0 [L*D,B,H] (LSTM, else None), and lists over layer*D + dir
    of dw_ih, dw_hh, db_ih, db_hh, dw_hr (None without projection) in the
    weights' shapes.  lengths: None or int32 [B] in [1, T]; row b runs its
    first len_b steps as in rnn_forward and its dx is 0 beyond them.
    bf16_weights: the weight matrices are rounded to bf16 first (biases stay
    fp32), as in rnn_forward.  cell_clip / proj_clip: None or (lo, hi), the
    LSTM clipping of rnn_forward; a clamp passes the gradient where its input
    lies in [lo, hi].
    """
    lib = _load()
    x = _f32(x)
    T, B, in_dim = x.shape
    D = 2 if bidirectional else 1
    LD = len(weights)
    L = LD // D
    assert L * D == LD and L >= 1
    H = hidden
    Ho = proj if proj > 0 else H
    nG = 4 if cell == LSTM else 3
    keep = []
    arr = (_LayerW * LD)()
    for i, w in enumerate(weights):
        vals = [_f32(w.get(k)) for k in ("w_ih", "w_hh", "b_ih", "b_hh")] + \
            [_f32(w.get("w_hr")) if proj > 0 else None]
        keep.extend(vals)
        arr[i] = _LayerW(*[_ptr(v) for v in vals])
    h0a, c0a, dya, dhn, dcn = _f32(h0), _f32(c0), _f32(dy), _f32(dh_n), _f32(dc_n)
    ln = _i32(lengths)  # kept alive across the call
    clip = None
    if cell_clip is not None or proj_clip is not None:
        inf = float("inf")
        cl = cell_clip if cell_clip is not None else (-inf, inf)
        pl = proj_clip if proj_clip is not None else (-inf, inf)
        clip = np.array([cl[0], cl[1], pl[0], pl[1]], np.float64)
    in_l = [in_dim if i // D == 0 else D * Ho for i in range(LD)]
    dx = np.zeros((T, B, in_dim))
    dh0 = np.zeros((LD, B, Ho))
    dc0 = np.zeros((LD, B, H))
    dwih = np.zeros(sum(nG * H * k for k in in_l))
    dwhh = np.zeros(LD * nG * H * Ho)
    dbih = np.zeros(LD * nG * H)
    dbhh = np.zeros(LD * nG * H)
    dwhr = np.zeros(max(1, LD * proj * H))
    rc = lib.oracle_rnn_backward(int(cell), int(bidirectional), L, in_dim, H, int(proj),
                                 int(bool(bf16_weights)), T, B,
                                 _ptr(x), _ptr(ln), _ptr(h0a), _ptr(c0a), ctypes.addressof(arr), _ptr(dya),
                                 _ptr(dhn), _ptr(dcn), _ptr(dx), _ptr(dh0), _ptr(dc0),
                                 _ptr(dwih), _ptr(dwhh), _ptr(dbih), _ptr(dbhh),
                                 _ptr(dwhr) if proj > 0 else None, int(threads), _ptr(clip))
    if rc != 0:
        raise ValueError("oracle_rnn_backward: invalid arguments")
    offs = np.cumsum([0] + [nG * H * k for k in in_l])
    return {"dx": dx, "dh0": dh0, "dc0": dc0 if cell == LSTM else None,
            "dw_ih": [dwih[offs[i]:offs[i + 1]].reshape(nG * H, in_l[i]) for i in range(LD)],
            "dw_hh": [dwhh[i * nG * H * Ho:(i + 1) * nG * H * Ho].reshape(nG * H, Ho)
                      for i in range(LD)],
            "db_ih": [dbih[i * nG * H:(i + 1) * nG * H] for i in range(LD)],
            "db_hh": [dbhh[i * nG * H:(i + 1) * nG * H] for i in range(LD)],
            "dw_hr": [dwhr[i * proj * H:(i + 1) * proj * H].reshape(proj, H) for i in range(LD)]
            if proj > 0 else None}


def rssm_unroll(weights, actions, eps, *, state0=None, belief0=None, rows=None, threads: int = 0):
    """RSSM prior unroll (actions given) in fp64.

    weights: dict W1,b1,W_ih,W_hh,b_ih,b_hh,W2,b2,W3,b3 (PyTorch Linear/GRUCell layout).
    actions [T,B,A], eps [T,B,S].  Returns (means, stds, states, beliefs).
    """
    lib = _load()
    a = _f32(actions)
    e = _f32(eps)
    T, B, A = a.shape
    S = e.shape[2]
    W = {k: _f32(v) for k, v in weights.items()}
    Hd = W["W1"].shape[0]
    RH = W["W_hh"].shape[1]
    means = np.zeros((T, B, S))
    stds = np.zeros((T, B, S))
    states = np.zeros((T, B, S))
    beliefs = np.zeros((T, B, RH))
    s0, b0 = _f32(state0), _f32(belief0)
    rw = _i32(rows)
    rc = lib.oracle_rssm_unroll(S, A, Hd, RH, T, B, *[_ptr(W[k]) for k in (
        "W1", "b1", "W_ih", "W_hh", "b_ih", "b_hh", "W2", "b2", "W3", "b3")],
        _ptr(s0), _ptr(b0), _ptr(a), _ptr(e), _ptr(means), _ptr(stds), _ptr(states),
        _ptr(beliefs), _ptr(rw), 0 if rw is None else len(rw), int(threads))
    if rc != 0:
        raise ValueError("oracle_rssm_unroll: invalid arguments")
    return means, stds, states, beliefs


RSSM_WEIGHTS = ("W1", "b1", "W_ih", "W_hh", "b_ih", "b_hh", "W2", "b2", "W3", "b3")


def rssm_backward(weights, actions, eps, *, state0=None, belief0=None, dmeans=None, dstds=None,
                  dstates=None, dbeliefs=None, actor=None):
    """Backward pass through time of the RSSM prior unroll in fp64: the
    gradients of a loss whose gradient with respect to the outputs is
    dmeans, dstds, dstates [T,B,S] and dbeliefs [T,B,RH] (None = 0).
    Returns a dict: dstate0 [B,S], dbelief0 [B,RH], dactions [T,B,A] and
    d<name> for every weight and bias of rssm_unroll's dict, in its shape.
    eps is an input (the noise), not differentiated.

    With actor (the dict of rssm_unroll_actor) the unroll is variant 2:
    actions is ignored (may be None), dactions is the gradient reaching each
    action the actor produced, and dWa1, dba1, dWa2, dba2 are added.
    """
    lib = _load()
    a = None if actor is not None else _f32(actions)
    e = _f32(eps)
    T, B, S = e.shape
    Ac = {k: _f32(v) for k, v in actor.items()} if actor is not None else None
    A = Ac["Wa2"].shape[0] if Ac is not None else (a.shape[2] if a is not None else 0)
    W = {k: _f32(weights.get(k)) for k in RSSM_WEIGHTS}
    Hd = W["W1"].shape[0]
    RH = W["W_hh"].shape[1]
    s0, b0 = _f32(state0), _f32(belief0)
    g_in = [_f32(v) for v in (dmeans, dstds, dstates, dbeliefs)]
    shapes = {"W1": (Hd, S + A), "b1": (Hd,), "W_ih": (3 * RH, Hd), "W_hh": (3 * RH, RH),
              "b_ih": (3 * RH,), "b_hh": (3 * RH,), "W2": (Hd, RH), "b2": (Hd,),
              "W3": (2 * S, Hd), "b3": (2 * S,)}
    out = {"dstate0": np.zeros((B, S)), "dbelief0": np.zeros((B, RH)),
           "dactions": np.zeros((T, B, A))}
    for k in RSSM_WEIGHTS:
        out["d" + k] = np.zeros(shapes[k])
    Ha = 0
    actor_args = [None] * 8
    if Ac is not None:
        Ha = Ac["Wa1"].shape[0]
        for k, shp in (("Wa1", (Ha, S + RH)), ("ba1", (Ha,)), ("Wa2", (A, Ha)), ("ba2", (A,))):
            out["d" + k] = np.zeros(shp)
        actor_args = [_ptr(Ac["Wa1"]), _ptr(Ac.get("ba1")), _ptr(Ac["Wa2"]), _ptr(Ac.get("ba2")),
                      _ptr(out["dWa1"]), _ptr(out["dba1"]), _ptr(out["dWa2"]), _ptr(out["dba2"])]
    rc = lib.oracle_rssm_backward2(
        S, A, Hd, RH, T, B, *[_ptr(W[k]) for k in RSSM_WEIGHTS], _ptr(s0), _ptr(b0), _ptr(a),
        _ptr(e), *[_ptr(v) for v in g_in], _ptr(out["dstate0"]), _ptr(out["dbelief0"]),
        _ptr(out["dactions"]), *[_ptr(out["d" + k]) for k in RSSM_WEIGHTS], Ha, *actor_args)
    if rc != 0:
        raise ValueError("oracle_rssm_backward: invalid arguments")
    return out


def rssm_unroll_actor(weights, actor, eps, *, state0=None, belief0=None, rows=None,
                      threads: int = 0):
    """RSSM prior unroll with the actor in the loop (unroll variant 2) in fp64.

    The action of step t is actor(state, belief) of the state and belief
    before the step; actor = dict Wa1 [Ha, S+RH] (state columns first), ba1
    [Ha], Wa2 [A, Ha], ba2 [A] (biases may be None), read as
    action = tanh(Wa2 ELU(Wa1 [state, belief] + ba1) + ba2).  eps [T,B,S].
    Returns (means, stds, states, beliefs, actions).
    """
    lib = _load()
    e = _f32(eps)
    T, B, S = e.shape
    W = {k: _f32(v) for k, v in weights.items()}
    Ac = {k: _f32(v) for k, v in actor.items()}
    Hd = W["W1"].shape[0]
    RH = W["W_hh"].shape[1]
    A = Ac["Wa2"].shape[0]
    Ha = Ac["Wa1"].shape[0]
    means = np.zeros((T, B, S))
    stds = np.zeros((T, B, S))
    states = np.zeros((T, B, S))
    beliefs = np.zeros((T, B, RH))
    actions = np.zeros((T, B, A))
    s0, b0 = _f32(state0), _f32(belief0)
    rw = _i32(rows)
    rc = lib.oracle_rssm_unroll2(S, A, Hd, RH, T, B, *[_ptr(W[k]) for k in (
        "W1", "b1", "W_ih", "W_hh", "b_ih", "b_hh", "W2", "b2", "W3", "b3")],
        _ptr(s0), _ptr(b0), None, _ptr(e), _ptr(means), _ptr(stds), _ptr(states),
        _ptr(beliefs), _ptr(rw), 0 if rw is None else len(rw), int(threads), Ha,
        _ptr(Ac["Wa1"]), _ptr(Ac.get("ba1")), _ptr(Ac["Wa2"]), _ptr(Ac.get("ba2")),
        _ptr(actions))
    if rc != 0:
        raise ValueError("oracle_rssm_unroll_actor: invalid arguments")
    return means, stds, states, beliefs, actions
