"""Thin ctypes binding of librcu.so (argument marshalling only).

Every function here has the name of the C entry point it calls (see
include/rcu.h) and only turns torch tensors into device pointers and CUDA
streams; every step of the computation runs in the library's kernels.  The
library must have been built (``recurrent_cell_unroll_gb300._build.build()``);
a missing library raises instead of falling back to anything else.

Inputs are re-materialised when their strides are not the C-canonical ones
(a tensor of shape [1, 4, 5] with strides (5, 5, 1) passes ``is_contiguous()``
but is not canonical; see "[Performance] LSTM/GRU scan: canonical strides +
cuDNN flat-storage clones + thread-local recurrent mode", pytorch/rl PR 3754).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

RCU_LSTM, RCU_GRU, RCU_BIDIR = 0, 1, 0x100
RCU_F32, RCU_BF16 = 0, 1
RCU_OK, RCU_ERR_INVALID, RCU_ERR_UNSUPPORTED, RCU_ERR_CUDA = 0, -1, -2, -3
RCU_ERR_TIMEOUT, RCU_ERR_LENGTHS, RCU_ERR_STATE = -4, -5, -6
RCU_ATTR_BARRIER_TIMEOUT_NS, RCU_ATTR_TEST_DROP_ARRIVAL, RCU_ATTR_FORCE_PATH = 1, 2, 3
RCU_ATTR_PROFILE, RCU_ATTR_TRACE, RCU_ATTR_TC_KSPLIT = 4, 5, 7
RCU_ATTR_LAYER_PIPELINE = 10
RCU_CLIP_CELL, RCU_CLIP_PROJ = 0, 1
RCU_ATTR_HOST_CHUNKS, RCU_MAX_HOST_CHUNKS = 8, 16

EXPORTED = (
    "rcu_last_error", "rcu_version", "rnn_create", "rnn_set_weights", "rnn_forward",
    "rnn_get_pack", "rnn_get_status", "rnn_set_attr", "rnn_set_clip", "rnn_last_launch_count",
    "rnn_destroy",
    "rnn_profile_entry", "rnn_profile_reset", "rnn_get_trace", "rnn_lstm_forward_noalloc",
    "rssm_create", "rssm_set_weights", "rssm_unroll", "rssm_get_status",
    "rssm_last_launch_count", "rssm_destroy", "rssm_set_attr", "rssm_get_trace",
    "rssm_set_actor", "rssm_unroll_actor", "rnn_forward_host", "rssm_unroll_host",
    "rssm_unroll_actor_host", "rnn_backward", "rnn_get_weight_grads", "rssm_backward",
    "rssm_get_weight_grads", "rssm_profile_entry", "rssm_profile_reset", "rssm_backward_actor",
    "rssm_get_actor_grads", "rnn_host_plan",
)

_lib = None
_lock = threading.Lock()


class RcuError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"rcu error {code}: {msg}")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def signatures() -> dict:
    """ctypes (restype, argtypes) of every entry point of include/rcu.h."""
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    return {
        "rcu_last_error": (ctypes.c_char_p, []),
        "rcu_version": (ctypes.c_char_p, []),
        "rnn_create": (I, [ctypes.POINTER(P), I, I, I, I, I, I]),
        "rnn_set_weights": (I, [P, I, I, P, P, P, P, P, P]),
        "rnn_forward": (I, [P, I, I, P, P, P, P, P, P, P, P, P]),
        "rnn_get_pack": (I, [P, P, P, P, P]),
        "rnn_get_status": (I, [P, P]),
        "rnn_set_attr": (I, [P, I, I64]),
        "rnn_set_clip": (I, [P, I, I, ctypes.c_double, ctypes.c_double]),
        "rnn_last_launch_count": (I, [P]),
        "rnn_host_plan": (I, [P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]),
        "rnn_destroy": (I, [P]),
        "rnn_profile_entry": (I, [P, I, ctypes.POINTER(ctypes.c_char_p),
                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)]),
        "rnn_profile_reset": (I, [P]),
        "rnn_get_trace": (I, [P, P, I, P]),
        "rnn_lstm_forward_noalloc": (I, [I, I, I, I] + [P] * 10 + [P]),
        "rssm_create": (I, [ctypes.POINTER(P), I, I, I, I]),
        "rssm_set_weights": (I, [P] + [P] * 10 + [P]),
        "rssm_unroll": (I, [P, I, I] + [P] * 8 + [P]),
        "rssm_get_status": (I, [P, P]),
        "rssm_last_launch_count": (I, [P]),
        "rssm_destroy": (I, [P]),
        "rssm_set_attr": (I, [P, I, I64]),
        "rssm_get_trace": (I, [P, P, I, P]),
        "rssm_set_actor": (I, [P, I, P, P, P, P, P]),
        "rssm_unroll_actor": (I, [P, I, I] + [P] * 8 + [P]),
        "rnn_forward_host": (I, [P, I, I] + [P] * 8),
        "rnn_backward": (I, [P, I, I] + [P] * 11),
        "rnn_get_weight_grads": (I, [P, I, I, P, P, P, P, P, P]),
        "rssm_unroll_host": (I, [P, I, I] + [P] * 8 + [P]),
        "rssm_unroll_actor_host": (I, [P, I, I] + [P] * 8 + [P]),
        "rssm_backward": (I, [P, I, I] + [P] * 12),
        "rssm_get_weight_grads": (I, [P] + [P] * 11),
        "rssm_backward_actor": (I, [P, I, I] + [P] * 11),
        "rssm_get_actor_grads": (I, [P] * 6),
        "rssm_profile_entry": (I, [P, I, ctypes.POINTER(ctypes.c_char_p),
                                   ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)]),
        "rssm_profile_reset": (I, [P]),
    }


def load(path: Optional[str] = None):
    """Load librcu.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"librcu.so not found at {p}: build it with "
                               "recurrent_cell_unroll_gb300._build.build()")
        lib = ctypes.CDLL(p)
        sig = signatures()
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int) -> int:
    if rc != RCU_OK:
        raise RcuError(rc, load().rcu_last_error().decode())
    return rc


def canonical_contiguous(t: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    """Return t if its strides are the C-canonical ones, else a canonical copy."""
    if t is None:
        return None
    expect, acc = [], 1
    for n in reversed(t.shape):
        expect.append(acc)
        acc *= n
    if tuple(reversed(expect)) == tuple(t.stride()) and t.storage_offset() >= 0:
        return t
    return t.clone(memory_format=torch.contiguous_format)


def _dev(t: Optional[torch.Tensor], dtype=torch.float32):
    if t is None:
        return None, None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    t = canonical_contiguous(t)
    return t, ctypes.c_void_p(t.data_ptr())


def _host(t: Optional[torch.Tensor], dtype=torch.float32, out=False):
    """Host tensor -> (kept tensor, pointer).  Pinned tensors (pin_memory) are
    used in place by the kernels; pageable ones are staged by the library."""
    if t is None:
        return None, None
    if t.is_cuda:
        raise ValueError("the *_host entry points take host tensors")
    if t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    if out:
        if canonical_contiguous(t) is not t:
            raise ValueError("outputs must be C-contiguous")
    else:
        t = canonical_contiguous(t)
    return t, ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# --------------------------------------------------------------------------- C names

def rcu_version() -> str:
    return load().rcu_version().decode()


def rnn_create(cell: int, layers: int, in_dim: int, hidden: int, proj: int = 0,
               dtype: int = RCU_F32) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load().rnn_create(ctypes.byref(h), cell, layers, in_dim, hidden, proj, dtype))
    return h


def rnn_set_weights(h, layer: int, direction: int, W_ih, W_hh, b_ih=None, b_hh=None, W_hr=None,
                    stream=None):
    keep = [_dev(t) for t in (W_ih, W_hh, b_ih, b_hh, W_hr)]
    _check(load().rnn_set_weights(h, layer, direction, *[k[1] for k in keep], _stream(stream)))


def rnn_forward(h, T: int, B: int, x, lengths, h0, c0, eps, y, h_n, c_n, stream=None):
    x_, xp = _dev(x)
    l_, lp = _dev(lengths, torch.int32)
    h0_, h0p = _dev(h0)
    c0_, c0p = _dev(c0)
    e_, ep = _dev(eps)
    for out in (y, h_n, c_n):
        if out is not None and not out.is_contiguous():
            raise ValueError("outputs must be contiguous")
    _, yp = _dev(y)
    _, hnp = _dev(h_n)
    _, cnp = _dev(c_n)
    _check(load().rnn_forward(h, T, B, xp, lp, h0p, c0p, ep, yp, hnp, cnp, _stream(stream)))


def rnn_get_pack(h, sorted_idx, unsorted_idx, batch_sizes, stream=None):
    _check(load().rnn_get_pack(h, *[_dev(t, torch.int32)[1] for t in
                                   (sorted_idx, unsorted_idx, batch_sizes)], _stream(stream)))


def rnn_get_status(h, stream=None) -> int:
    """Synchronise and return the device status code (0 = ok); does not raise."""
    return load().rnn_get_status(h, _stream(stream))


def rnn_set_attr(h, attr: int, value: int):
    _check(load().rnn_set_attr(h, attr, value))


def rnn_last_launch_count(h) -> int:
    return load().rnn_last_launch_count(h)


def rnn_profile_entry(h, i: int):
    """(name, total_ms, launches) of profile entry i, or None past the end."""
    name, ms, n = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int64()
    rc = load().rnn_profile_entry(h, i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(n))
    if rc != RCU_OK:
        return None
    return name.value.decode(), ms.value, n.value


def rnn_profile_reset(h):
    _check(load().rnn_profile_reset(h))


def rssm_profile_entry(h, i: int):
    """(name, total_ms, count) of RSSM profile entry i, or None past the end."""
    name, ms, n = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int64()
    rc = load().rssm_profile_entry(h, i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(n))
    if rc != RCU_OK:
        return None
    return name.value.decode(), ms.value, n.value


def rssm_profile_reset(h):
    _check(load().rssm_profile_reset(h))


def rnn_get_trace(h, n_steps: int, stream=None):
    """[n_steps, 16] int64 global-timer stamps of the first layer (see rcu.h)."""
    out = torch.zeros((n_steps, 16), dtype=torch.int64)
    _check(load().rnn_get_trace(h, ctypes.c_void_p(out.data_ptr()), n_steps, _stream(stream)))
    return out


def rnn_destroy(h):
    if h:
        load().rnn_destroy(h)


def rnn_lstm_forward_noalloc(T: int, B: int, in_dim: int, hidden: int, x, W_ih, W_hh,
                             b_ih=None, b_hh=None, h0=None, c0=None, y=None, h_n=None, c_n=None,
                             stream=None):
    """One-layer fp32 LSTM through the allocation-free entry point (see rcu.h)."""
    ins = [_dev(t) for t in (x, W_ih, W_hh, b_ih, b_hh, h0, c0)]
    outs = [_dev(t) for t in (y, h_n, c_n)]
    _check(load().rnn_lstm_forward_noalloc(T, B, in_dim, hidden, *[k[1] for k in ins],
                                           *[k[1] for k in outs], _stream(stream)))


def rnn_forward_host(h, T: int, B: int, x, lengths, h0, c0, y, h_n, c_n, stream=None):
    """rnn_forward on host tensors (see rcu.h); results are in y/h_n/c_n once
    the stream has passed the call."""
    ins = [_host(x), _host(lengths, torch.int32), _host(h0), _host(c0)]
    outs = [_host(t, out=True) for t in (y, h_n, c_n)]
    _check(load().rnn_forward_host(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                                   _stream(stream)))


def rnn_host_plan(h) -> dict:
    """How the last rnn_forward_host call moved x and y (see rcu.h)."""
    c, xi, yi = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().rnn_host_plan(h, ctypes.byref(c), ctypes.byref(xi), ctypes.byref(yi)))
    return {"chunks": c.value, "x_in_place": bool(xi.value), "y_in_place": bool(yi.value)}


def rnn_backward(h, T: int, B: int, x, lengths, h0, c0, dy, dh_n, dc_n, dx, dh0, dc0,
                 stream=None):
    """Backward pass through time (see rcu.h); device tensors."""
    ins = [_dev(x), _dev(lengths, torch.int32)] + [_dev(t) for t in (h0, c0, dy, dh_n, dc_n)]
    outs = [_dev(t) for t in (dx, dh0, dc0)]
    _check(load().rnn_backward(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                               _stream(stream)))


def rnn_get_weight_grads(h, layer: int, dW_ih, dW_hh, db_ih, db_hh, dW_hr=None, stream=None,
                         direction: int = 0):
    outs = [_dev(t) for t in (dW_ih, dW_hh, db_ih, db_hh, dW_hr)]
    _check(load().rnn_get_weight_grads(h, layer, direction, *[k[1] for k in outs],
                                       _stream(stream)))


def rssm_create(state_dim: int, action_dim: int, hidden: int, rnn_hidden: int):
    h = ctypes.c_void_p()
    _check(load().rssm_create(ctypes.byref(h), state_dim, action_dim, hidden, rnn_hidden))
    return h


def rssm_set_weights(h, W1, b1, W_ih, W_hh, b_ih, b_hh, W2, b2, W3, b3, stream=None):
    keep = [_dev(t) for t in (W1, b1, W_ih, W_hh, b_ih, b_hh, W2, b2, W3, b3)]
    _check(load().rssm_set_weights(h, *[k[1] for k in keep], _stream(stream)))


def rssm_unroll(h, T: int, B: int, state0, belief0, actions, eps, means, stds, states, beliefs,
                stream=None):
    ins = [_dev(t) for t in (state0, belief0, actions, eps)]
    outs = [_dev(t) for t in (means, stds, states, beliefs)]
    _check(load().rssm_unroll(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                              _stream(stream)))


def rssm_backward(h, T: int, B: int, state0, belief0, actions, eps, dmeans, dstds, dstates,
                  dbeliefs, dstate0, dbelief0, dactions, stream=None):
    """Backward pass through time of rssm_unroll (see rcu.h); device tensors."""
    ins = [_dev(t) for t in (state0, belief0, actions, eps, dmeans, dstds, dstates, dbeliefs)]
    outs = [_dev(t) for t in (dstate0, dbelief0, dactions)]
    _check(load().rssm_backward(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                                _stream(stream)))


def rssm_backward_actor(h, T: int, B: int, state0, belief0, eps, dmeans, dstds, dstates,
                        dbeliefs, dstate0, dbelief0, dactions, stream=None):
    """Backward pass through time of rssm_unroll_actor (see rcu.h); device tensors."""
    ins = [_dev(t) for t in (state0, belief0, eps, dmeans, dstds, dstates, dbeliefs)]
    outs = [_dev(t) for t in (dstate0, dbelief0, dactions)]
    _check(load().rssm_backward_actor(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                                      _stream(stream)))


RSSM_ACTOR_NAMES = ("Wa1", "ba1", "Wa2", "ba2")


def rssm_get_actor_grads(h, grads: dict, stream=None):
    """Copy the last rssm_backward_actor's actor gradients into the device
    tensors of grads (keys of RSSM_ACTOR_NAMES; missing or None are skipped)."""
    outs = [_dev(grads.get(k)) for k in RSSM_ACTOR_NAMES]
    _check(load().rssm_get_actor_grads(h, *[k[1] for k in outs], _stream(stream)))


RSSM_WEIGHT_NAMES = ("W1", "b1", "W_ih", "W_hh", "b_ih", "b_hh", "W2", "b2", "W3", "b3")


def rssm_weight_shapes(S: int, A: int, Hd: int, RH: int) -> dict:
    """Shapes of the prior's weights (rssm_set_weights' layouts) by name."""
    return {"W1": (Hd, S + A), "b1": (Hd,), "W_ih": (3 * RH, Hd), "W_hh": (3 * RH, RH),
            "b_ih": (3 * RH,), "b_hh": (3 * RH,), "W2": (Hd, RH), "b2": (Hd,),
            "W3": (2 * S, Hd), "b3": (2 * S,)}


def rssm_get_weight_grads(h, grads: dict, stream=None):
    """Copy the last rssm_backward's weight gradients into the device tensors
    of grads (keys of RSSM_WEIGHT_NAMES; missing or None are skipped)."""
    outs = [_dev(grads.get(k)) for k in RSSM_WEIGHT_NAMES]
    _check(load().rssm_get_weight_grads(h, *[k[1] for k in outs], _stream(stream)))


def rssm_set_actor(h, actor_hidden: int, Wa1, ba1, Wa2, ba2, stream=None):
    keep = [_dev(t) for t in (Wa1, ba1, Wa2, ba2)]
    _check(load().rssm_set_actor(h, actor_hidden, *[k[1] for k in keep], _stream(stream)))


def rssm_unroll_actor(h, T: int, B: int, state0, belief0, eps, means, stds, states, beliefs,
                      actions_out, stream=None):
    ins = [_dev(t) for t in (state0, belief0, eps)]
    outs = [_dev(t) for t in (means, stds, states, beliefs, actions_out)]
    _check(load().rssm_unroll_actor(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                                    _stream(stream)))


def rssm_unroll_host(h, T: int, B: int, state0, belief0, actions, eps, means, stds, states,
                     beliefs, stream=None):
    ins = [_host(t) for t in (state0, belief0, actions, eps)]
    outs = [_host(t, out=True) for t in (means, stds, states, beliefs)]
    _check(load().rssm_unroll_host(h, T, B, *[k[1] for k in ins], *[k[1] for k in outs],
                                   _stream(stream)))


def rssm_unroll_actor_host(h, T: int, B: int, state0, belief0, eps, means, stds, states, beliefs,
                           actions_out, stream=None):
    ins = [_host(t) for t in (state0, belief0, eps)]
    outs = [_host(t, out=True) for t in (means, stds, states, beliefs, actions_out)]
    _check(load().rssm_unroll_actor_host(h, T, B, *[k[1] for k in ins],
                                         *[k[1] for k in outs], _stream(stream)))


def rssm_get_status(h, stream=None) -> int:
    return load().rssm_get_status(h, _stream(stream))


def rssm_last_launch_count(h) -> int:
    return load().rssm_last_launch_count(h)


def rssm_set_attr(h, attr: int, value: int):
    _check(load().rssm_set_attr(h, attr, value))


def rssm_get_trace(h, n_steps: int, stream=None):
    """[n_steps, 16] int64 stamps of the last traced rssm_unroll (see rcu.h)."""
    out = torch.zeros((n_steps, 16), dtype=torch.int64)
    _check(load().rssm_get_trace(h, ctypes.c_void_p(out.data_ptr()), n_steps, _stream(stream)))
    return out


def rssm_destroy(h):
    if h:
        load().rssm_destroy(h)


# --------------------------------------------------------------------------- convenience wrappers

class RNN:
    """Owns an rnn handle; weights from the seeded-workload dict layout."""

    def __init__(self, cell: str, layers: int, in_dim: int, hidden: int, proj: int = 0,
                 bidirectional: bool = False, dtype: str = "f32"):
        c = RCU_LSTM if cell == "lstm" else RCU_GRU
        if bidirectional:
            c |= RCU_BIDIR
        self.cell, self.layers, self.hidden, self.proj = cell, layers, hidden, proj
        self.in_dim = in_dim
        self.D = 2 if bidirectional else 1
        self.Hout = proj if proj > 0 else hidden
        self.h = rnn_create(c, layers, in_dim, hidden, proj, RCU_BF16 if dtype == "bf16" else RCU_F32)

    @classmethod
    def from_spec(cls, spec):
        return cls(spec.cell, spec.layers, spec.in_dim, spec.hidden, spec.proj, spec.bidir, spec.dtype)

    def set_weights(self, weights, device="cuda", stream=None):
        for i, w in enumerate(weights):
            layer, d = divmod(i, self.D)
            t = {k: (None if v is None else v.to(device=device, dtype=torch.float32))
                 for k, v in w.items()}
            rnn_set_weights(self.h, layer, d, t["w_ih"], t["w_hh"], t.get("b_ih"), t.get("b_hh"),
                            t.get("w_hr"), stream)

    def _shapes(self, x, lengths=None, h0=None, c0=None, **seq):
        """The C ABI takes plain pointers and reads every tensor at the size
        the handle and (T, B) imply: a tensor of another shape is an error
        here, before any pointer crosses."""
        if x.dim() != 3 or x.shape[2] != self.in_dim:
            raise ValueError(f"x must be [T, B, {self.in_dim}], got {tuple(x.shape)}")
        T, B, _ = x.shape
        LD = self.layers * self.D
        want = {"lengths": (B,), "h0": (LD, B, self.Hout), "c0": (LD, B, self.hidden)}
        want.update({k: (T, B, self.D * self.Hout) if k in ("dy", "out") else
                     (LD, B, self.Hout if k == "dh_n" else self.hidden) for k in seq})
        for k, t in dict(lengths=lengths, h0=h0, c0=c0, **seq).items():
            if t is not None and tuple(t.shape) != want[k]:
                raise ValueError(f"{k} must be {list(want[k])}, got {list(t.shape)}")
        return T, B

    def forward(self, x, lengths=None, h0=None, c0=None, out=None, stream=None):
        T, B = self._shapes(x, lengths, h0, c0, out=out)
        dev = x.device
        y = out if out is not None else torch.empty((T, B, self.D * self.Hout), device=dev)
        hn = torch.empty((self.layers * self.D, B, self.Hout), device=dev)
        cn = torch.empty((self.layers * self.D, B, self.hidden), device=dev) \
            if self.cell == "lstm" else None
        rnn_forward(self.h, T, B, x, lengths, h0, c0, None, y, hn, cn, stream)
        return y, hn, cn

    def backward(self, x, dy, lengths=None, h0=None, c0=None, dh_n=None, dc_n=None, stream=None):
        """Gradients of a loss with dL/dy = dy (and dL/dh_n, dL/dc_n) through
        the forward on x (with lengths: int32 [B] on the device): returns (dx, dh0, dc0 or None, weight grads as a
        list over layers of dicts w_ih, w_hh, b_ih, b_hh)."""
        T, B = self._shapes(x, lengths, h0, c0, dy=dy, dh_n=dh_n, dc_n=dc_n)
        in_dim = x.shape[2]
        dev = x.device
        dx = torch.empty_like(x)
        LD = self.layers * self.D
        dh0 = torch.empty((LD, B, self.Hout), device=dev)
        dc0 = torch.empty((LD, B, self.hidden), device=dev) if self.cell == "lstm" else None
        rnn_backward(self.h, T, B, x, lengths, h0, c0, dy, dh_n, dc_n, dx, dh0, dc0, stream)
        nG = 4 if self.cell == "lstm" else 3
        grads = []  # over layer * D + direction, like the weights
        for i in range(LD):
            layer, d = divmod(i, self.D)
            k = in_dim if layer == 0 else self.D * self.Hout
            g = {"w_ih": torch.empty((nG * self.hidden, k), device=dev),
                 "w_hh": torch.empty((nG * self.hidden, self.Hout), device=dev),
                 "b_ih": torch.empty((nG * self.hidden,), device=dev),
                 "b_hh": torch.empty((nG * self.hidden,), device=dev),
                 "w_hr": torch.empty((self.proj, self.hidden), device=dev) if self.proj else None}
            rnn_get_weight_grads(self.h, layer, g["w_ih"], g["w_hh"], g["b_ih"], g["b_hh"],
                                 g["w_hr"], stream, direction=d)
            grads.append(g)
        return dx, dh0, dc0, grads

    def status(self, stream=None) -> int:
        return rnn_get_status(self.h, stream)

    def set_attr(self, attr, value):
        rnn_set_attr(self.h, attr, value)

    def set_clip(self, what: int, bounds=None):
        """Clamp the LSTM cell state (RCU_CLIP_CELL) or the projected hidden
        state (RCU_CLIP_PROJ) to bounds = (lo, hi); None turns it off."""
        if bounds is None:
            _check(load().rnn_set_clip(self.h, what, 0, 0.0, 0.0))
        else:
            _check(load().rnn_set_clip(self.h, what, 1, float(bounds[0]), float(bounds[1])))

    def launch_count(self) -> int:
        return rnn_last_launch_count(self.h)

    def profile(self) -> dict:
        """{kernel name: (total_ms, launches)} recorded while RCU_ATTR_PROFILE is on."""
        out, i = {}, 0
        while True:
            e = rnn_profile_entry(self.h, i)
            if e is None:
                return out
            out[e[0]] = (e[1], e[2])
            i += 1

    def close(self):
        if self.h:
            rnn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class RSSM:
    """Owns an rssm handle."""

    def __init__(self, state_dim: int, action_dim: int, hidden: int, rnn_hidden: int):
        self.S, self.A, self.Hd, self.RH = state_dim, action_dim, hidden, rnn_hidden
        self.Ha = 0  # actor width once set_actor has run
        self.h = rssm_create(state_dim, action_dim, hidden, rnn_hidden)

    def set_weights(self, w, device="cuda", stream=None):
        t = {k: (None if v is None else v.to(device=device, dtype=torch.float32))
             for k, v in w.items()}
        rssm_set_weights(self.h, t["W1"], t.get("b1"), t["W_ih"], t["W_hh"], t.get("b_ih"),
                         t.get("b_hh"), t["W2"], t.get("b2"), t["W3"], t.get("b3"), stream)

    def unroll(self, actions, eps, state0=None, belief0=None, stream=None):
        T, B, _ = eps.shape
        dev = eps.device
        means = torch.empty((T, B, self.S), device=dev)
        stds = torch.empty_like(means)
        states = torch.empty_like(means)
        beliefs = torch.empty((T, B, self.RH), device=dev)
        rssm_unroll(self.h, T, B, state0, belief0, actions, eps, means, stds, states, beliefs,
                    stream)
        return means, stds, states, beliefs

    def backward(self, actions, eps, state0=None, belief0=None, dmeans=None, dstds=None,
                 dstates=None, dbeliefs=None, stream=None):
        """Gradients of a loss with the given gradients with respect to the
        unroll's outputs (None = 0): returns (dstate0, dbelief0, dactions,
        dict of weight gradients keyed like set_weights)."""
        T, B, _ = eps.shape
        dev = eps.device
        dstate0 = torch.empty((B, self.S), device=dev)
        dbelief0 = torch.empty((B, self.RH), device=dev)
        dactions = torch.empty((T, B, self.A), device=dev) if self.A > 0 else None
        rssm_backward(self.h, T, B, state0, belief0, actions, eps, dmeans, dstds, dstates,
                      dbeliefs, dstate0, dbelief0, dactions, stream)
        S, A, Hd, RH = self.S, self.A, self.Hd, self.RH
        shapes = rssm_weight_shapes(S, A, Hd, RH)
        grads = {k: torch.empty(shapes[k], device=dev) for k in RSSM_WEIGHT_NAMES}
        rssm_get_weight_grads(self.h, grads, stream)
        return dstate0, dbelief0, dactions, grads

    def backward_actor(self, eps, state0=None, belief0=None, dmeans=None, dstds=None,
                       dstates=None, dbeliefs=None, stream=None):
        """Backward pass of unroll_actor: returns (dstate0, dbelief0, dactions
        (the gradient reaching each produced action), dict of the prior's
        weight gradients, dict of the actor's: Wa1, ba1, Wa2, ba2)."""
        T, B, _ = eps.shape
        dev = eps.device
        dstate0 = torch.empty((B, self.S), device=dev)
        dbelief0 = torch.empty((B, self.RH), device=dev)
        dactions = torch.empty((T, B, self.A), device=dev)
        rssm_backward_actor(self.h, T, B, state0, belief0, eps, dmeans, dstds, dstates, dbeliefs,
                            dstate0, dbelief0, dactions, stream)
        S, A, Hd, RH, Ha = self.S, self.A, self.Hd, self.RH, self.Ha
        shapes = rssm_weight_shapes(S, A, Hd, RH)
        grads = {k: torch.empty(shapes[k], device=dev) for k in RSSM_WEIGHT_NAMES}
        rssm_get_weight_grads(self.h, grads, stream)
        ashapes = {"Wa1": (Ha, S + RH), "ba1": (Ha,), "Wa2": (A, Ha), "ba2": (A,)}
        agrads = {k: torch.empty(ashapes[k], device=dev) for k in RSSM_ACTOR_NAMES}
        rssm_get_actor_grads(self.h, agrads, stream)
        return dstate0, dbelief0, dactions, grads, agrads

    def set_actor(self, a, device="cuda", stream=None):
        """Actor of the second unroll variant: dict Wa1 [Ha, S+RH], ba1 [Ha],
        Wa2 [A, Ha], ba2 [A] (biases may be None)."""
        t = {k: (None if v is None else v.to(device=device, dtype=torch.float32))
             for k, v in a.items()}
        rssm_set_actor(self.h, t["Wa1"].shape[0], t["Wa1"], t.get("ba1"), t["Wa2"],
                       t.get("ba2"), stream)
        self.Ha = t["Wa1"].shape[0]

    def unroll_actor(self, eps, state0=None, belief0=None, stream=None):
        """Unroll over eps' T steps with the actions computed by the actor;
        returns (means, stds, states, beliefs, actions)."""
        T, B, _ = eps.shape
        dev = eps.device
        means = torch.empty((T, B, self.S), device=dev)
        stds = torch.empty_like(means)
        states = torch.empty_like(means)
        beliefs = torch.empty((T, B, self.RH), device=dev)
        actions = torch.empty((T, B, self.A), device=dev)
        rssm_unroll_actor(self.h, T, B, state0, belief0, eps, means, stds, states, beliefs,
                          actions, stream)
        return means, stds, states, beliefs, actions

    def launch_count(self) -> int:
        return rssm_last_launch_count(self.h)

    def set_attr(self, attr, value):
        rssm_set_attr(self.h, attr, value)

    def profile(self) -> dict:
        """{phase name: (total_ms, count)} recorded while RCU_ATTR_PROFILE is on."""
        out, i = {}, 0
        while True:
            e = rssm_profile_entry(self.h, i)
            if e is None:
                return out
            out[e[0]] = (e[1], e[2])
            i += 1

    def close(self):
        if self.h:
            rssm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
