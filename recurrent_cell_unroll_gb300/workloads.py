"""Seeded synthetic workloads (shapes and value distributions only).

This module draws random inputs; it holds none of the recurrence's
arithmetic.  Both the tests (CUDA path and oracle alike) and the benchmark
take their inputs from here, so the two sides always see the same fp32 bits.

All draws come from one CPU ``torch.Generator`` seeded per workload, in this
order: for each layer, then direction: W_ih, W_hh, b_ih, b_hh, [W_hr]; then
x; then lengths; then h0, c0; then (RSSM) actions and eps; the training
workloads' output gradients come last, so every other draw stays that of the
forward workload.  Weights and biases
follow the PyTorch module default, U(-1/sqrt(hidden), 1/sqrt(hidden)); RSSM
Linear layers use U(-1/sqrt(fan_in), 1/sqrt(fan_in)).

The named workloads are the shapes the pages discuss: the TVM TE LSTM
benchmark shape (T=80, B=1, 512 -> 256), the dreamer/planet RSSM prior
(state 20, hidden 200; with given actions, and with an actor of width 200
computing them on the fly), a speech-style projected LSTM at T=1000, a
variable-length bidirectional LSTM, and a large stacked GRU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class RnnSpec:
    name: str
    cell: str              # "lstm" | "gru"
    layers: int
    in_dim: int
    hidden: int
    T: int
    B: int
    proj: int = 0
    bidir: bool = False
    dtype: str = "f32"     # "f32" | "bf16" (bf16 weights, fp32 state/accumulate)
    varlen: Optional[tuple] = None   # (min_len, max_len) inclusive, or None
    h0_std: float = 0.0    # > 0: h0 ~ N(0, h0_std^2); 0: h0 = c0 = zero (NULL)
    c0_std: float = 0.0
    train: bool = False    # a training pass: forward + backward through time given dy

    @property
    def D(self) -> int:
        return 2 if self.bidir else 1

    @property
    def nG(self) -> int:
        return 4 if self.cell == "lstm" else 3

    @property
    def Hout(self) -> int:
        return self.proj if self.proj > 0 else self.hidden

    def scaled(self, **kw) -> "RnnSpec":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class RssmSpec:
    name: str
    T: int
    B: int
    state_dim: int = 20
    action_dim: int = 6
    hidden: int = 200
    rnn_hidden: int = 200
    state0_std: float = 0.0
    belief0_std: float = 0.0
    # unroll variant 2: actions from an actor of this hidden width (0 = given)
    actor_hidden: int = 0
    # a training pass: the unroll and its backward pass through time given the
    # gradients of the four outputs
    train: bool = False

    def scaled(self, **kw) -> "RssmSpec":
        return dataclasses.replace(self, **kw)


LSTM_T80 = RnnSpec("lstm_f32_T80_B1_512x256", "lstm", 1, 512, 256, T=80, B=1)
RSSM_B50 = RssmSpec("rssm_f32_B50_T50_S20_A6_H200", T=50, B=50)
RSSM_ACTOR = RssmSpec("rssm_actor_f32_B50_T50_S20_A6_H200_X200", T=50, B=50, actor_hidden=200)
# forward + backward through time of the given-actions unroll; the output
# gradients dmeans, dstds, dstates, dbeliefs ~ N(0, 1)
RSSM_TRAIN = RSSM_B50.scaled(name="rssm_train_f32_B50_T50_S20_A6_H200", train=True)
LSTMP_2L = RnnSpec("lstmp_bf16_2L_T1000_B32_80x1024p256", "lstm", 2, 80, 1024, T=1000, B=32,
                   proj=256, dtype="bf16")
BILSTM_VAR = RnnSpec("bilstm_f32_varlen_B64_T500_256x512", "lstm", 1, 256, 512, T=500, B=64,
                     bidir=True, varlen=(50, 500))
GRU_3L = RnnSpec("gru_bf16_3L_T512_B256_1024", "gru", 3, 1024, 1024, T=512, B=256, dtype="bf16",
                 h0_std=0.1)
# forward + backward through time of the unidirectional form of the varlen
# shape (256 -> 512, B = 64, T = 500); dy ~ N(0, 1)
LSTM_TRAIN = RnnSpec("lstm_train_f32_T500_B64_256x512", "lstm", 1, 256, 512, T=500, B=64,
                     train=True)
# forward + backward through time of the variable-length bidirectional shape
# itself (the same x, lengths and weights as BILSTM_VAR; dy ~ N(0, 1))
BILSTM_TRAIN = BILSTM_VAR.scaled(name="bilstm_train_f32_varlen_B64_T500_256x512", train=True)

# forward + backward through time of the 3-layer GRU itself (its x, h0 and
# weights; dy ~ N(0, 1)): the bf16 forward, the fp32 gradient of the model
# with the bf16-rounded weights
GRU_TRAIN = GRU_3L.scaled(name="gru_train_bf16_3L_T512_B256_1024", train=True)

WORKLOADS = {s.name: s for s in (LSTM_T80, RSSM_B50, LSTMP_2L, BILSTM_VAR, GRU_3L,
                                  RSSM_ACTOR, LSTM_TRAIN, BILSTM_TRAIN, RSSM_TRAIN, GRU_TRAIN)}


def _uniform(g, shape, bound):
    return (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0) * bound


def make_rnn_inputs(spec: RnnSpec, seed: int = 0, bias: bool = True) -> dict:
    """Weights, x, lengths, h0, c0 for an RnnSpec (fp32 CPU tensors)."""
    g = torch.Generator().manual_seed(seed)
    bound = 1.0 / math.sqrt(spec.hidden)
    H, nG, Hout, D = spec.hidden, spec.nG, spec.Hout, spec.D
    weights = []
    for layer in range(spec.layers):
        in_w = spec.in_dim if layer == 0 else D * Hout
        for _ in range(D):
            w = {"w_ih": _uniform(g, (nG * H, in_w), bound),
                 "w_hh": _uniform(g, (nG * H, Hout), bound)}
            b_ih = _uniform(g, (nG * H,), bound)
            b_hh = _uniform(g, (nG * H,), bound)
            w["b_ih"] = b_ih if bias else None
            w["b_hh"] = b_hh if bias else None
            w["w_hr"] = _uniform(g, (spec.proj, H), bound) if spec.proj > 0 else None
            weights.append(w)
    x = torch.randn((spec.T, spec.B, spec.in_dim), generator=g, dtype=torch.float32)
    lengths = None
    if spec.varlen is not None:
        lo, hi = spec.varlen
        lengths = torch.randint(lo, hi + 1, (spec.B,), generator=g, dtype=torch.int32)
    h0 = c0 = None
    LD = spec.layers * D
    if spec.h0_std > 0:
        h0 = torch.randn((LD, spec.B, Hout), generator=g, dtype=torch.float32) * spec.h0_std
    if spec.c0_std > 0 and spec.cell == "lstm":
        c0 = torch.randn((LD, spec.B, H), generator=g, dtype=torch.float32) * spec.c0_std
    out = {"weights": weights, "x": x, "lengths": lengths, "h0": h0, "c0": c0}
    if spec.train:  # drawn last: the other draws stay those of the forward workload
        out["dy"] = torch.randn((spec.T, spec.B, D * Hout), generator=g, dtype=torch.float32)
    return out


def make_rssm_inputs(spec: RssmSpec, seed: int = 0) -> dict:
    """RSSM prior weights, actions ~ U(-1, 1), eps ~ N(0, 1), zero or random start.
    With spec.actor_hidden the actions are replaced by the actor's weights
    ("actor", make_rssm_actor); every other draw stays the same."""
    g = torch.Generator().manual_seed(seed)
    S, A, Hd, RH = spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden
    b1 = 1.0 / math.sqrt(S + A)
    bg = 1.0 / math.sqrt(RH)
    w = {
        "W1": _uniform(g, (Hd, S + A), b1), "b1": _uniform(g, (Hd,), b1),
        "W_ih": _uniform(g, (3 * RH, Hd), bg), "W_hh": _uniform(g, (3 * RH, RH), bg),
        "b_ih": _uniform(g, (3 * RH,), bg), "b_hh": _uniform(g, (3 * RH,), bg),
        "W2": _uniform(g, (Hd, RH), 1.0 / math.sqrt(RH)),
        "b2": _uniform(g, (Hd,), 1.0 / math.sqrt(RH)),
        "W3": _uniform(g, (2 * S, Hd), 1.0 / math.sqrt(Hd)),
        "b3": _uniform(g, (2 * S,), 1.0 / math.sqrt(Hd)),
    }
    actions = torch.rand((spec.T, spec.B, A), generator=g, dtype=torch.float32) * 2.0 - 1.0
    eps = torch.randn((spec.T, spec.B, S), generator=g, dtype=torch.float32)
    state0 = belief0 = None
    if spec.state0_std > 0:
        state0 = torch.randn((spec.B, S), generator=g, dtype=torch.float32) * spec.state0_std
    if spec.belief0_std > 0:
        belief0 = torch.randn((spec.B, RH), generator=g, dtype=torch.float32) * spec.belief0_std
    out = {"weights": w, "actions": actions, "eps": eps, "state0": state0, "belief0": belief0}
    if spec.train:  # drawn last: the other draws stay those of the forward workload
        for k, n in (("dmeans", S), ("dstds", S), ("dstates", S), ("dbeliefs", RH)):
            out[k] = torch.randn((spec.T, spec.B, n), generator=g, dtype=torch.float32)
    if spec.actor_hidden:
        out["actions"] = None
        out["actor"] = make_rssm_actor(spec, seed, spec.actor_hidden)
    return out


def make_rssm_actor(spec: RssmSpec, seed: int = 0, actor_hidden: int = 0) -> dict:
    """Weights of the actor of the second unroll variant (actions computed on
    the fly): Wa1 [Ha, S+RH], ba1 [Ha], Wa2 [A, Ha], ba2 [A], U(+-1/sqrt(fan_in)),
    Ha = spec.hidden unless given.  A separate generator (seed + 7919) leaves
    make_rssm_inputs' draws unchanged."""
    g = torch.Generator().manual_seed(seed + 7919)
    S, A, RH = spec.state_dim, spec.action_dim, spec.rnn_hidden
    Ha = actor_hidden or spec.hidden
    b1 = 1.0 / math.sqrt(S + RH)
    b2 = 1.0 / math.sqrt(Ha)
    return {"Wa1": _uniform(g, (Ha, S + RH), b1), "ba1": _uniform(g, (Ha,), b1),
            "Wa2": _uniform(g, (A, Ha), b2), "ba2": _uniform(g, (A,), b2)}
