"""GPU parity of the training use of the unroll: the backward pass through
time of the stacked cells and of the RSSM unroll, through the C ABI, against
the fp64 oracle's backward.

Tolerance: per gradient tensor, max|gpu - ref| / max|ref| <= 1e-4 (fp32
sums over T*B rows and T dependent steps); bf16-weight handles 2e-2.  The
cases that have run on the GPU before come first in this file.
"""
import numpy as np
import pytest
import torch

import oracle
from recurrent_cell_unroll_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

BF16_REL = 2e-2


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _cell(spec):
    return oracle.LSTM if spec.cell == "lstm" else oracle.GRU


# ----------------------------------------------------------------------------- stacked cells

BWD_REL = 1e-4  # per tensor: max|gpu - ref| / max|ref| (fp32 sums over T*B terms, T steps)

BWD_SPECS = [
    wl.LSTM_T80.scaled(T=7, B=5, in_dim=12, hidden=20, layers=2, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(T=6, B=9, in_dim=16, hidden=24, layers=2, dtype="f32"),
    wl.GRU_3L.scaled(T=5, B=3, in_dim=7, hidden=13, layers=1, dtype="f32", h0_std=0.3),
    wl.LSTM_T80.scaled(T=32, B=64, in_dim=256, hidden=512, layers=1),
    wl.GRU_3L.scaled(T=24, B=32, in_dim=128, hidden=256, layers=3, dtype="f32", h0_std=0.1),
    wl.LSTM_T80.scaled(T=1, B=1, in_dim=5, hidden=7, layers=2, c0_std=0.5, h0_std=0.5),
    wl.GRU_3L.scaled(T=9, B=130, in_dim=40, hidden=48, layers=1, dtype="f32", h0_std=0.0),
    # LSTM with projection
    wl.LSTMP_2L.scaled(T=6, B=5, in_dim=12, hidden=20, proj=8, dtype="f32", h0_std=0.5,
                       c0_std=0.5),
    wl.LSTMP_2L.scaled(T=16, B=32, in_dim=64, hidden=128, proj=32, dtype="f32"),
    # bidirectional
    wl.BILSTM_VAR.scaled(T=7, B=5, in_dim=12, hidden=20, layers=2, varlen=None, h0_std=0.5,
                         c0_std=0.5),
    wl.GRU_3L.scaled(T=6, B=9, in_dim=16, hidden=24, layers=2, dtype="f32", bidir=True),
    wl.LSTMP_2L.scaled(T=5, B=4, in_dim=8, hidden=16, proj=6, dtype="f32", bidir=True,
                       h0_std=0.5),
    wl.BILSTM_VAR.scaled(T=32, B=64, in_dim=256, hidden=256, varlen=None),
    # variable lengths (length 1 and T both drawn)
    wl.LSTM_T80.scaled(T=9, B=7, in_dim=12, hidden=20, layers=2, varlen=(1, 9), h0_std=0.5,
                       c0_std=0.5),
    wl.GRU_3L.scaled(T=8, B=9, in_dim=16, hidden=24, layers=2, dtype="f32", varlen=(1, 8),
                     h0_std=0.3),
    wl.BILSTM_VAR.scaled(T=10, B=6, in_dim=12, hidden=20, layers=2, varlen=(1, 10), h0_std=0.5,
                         c0_std=0.5),
    wl.GRU_3L.scaled(T=7, B=5, in_dim=9, hidden=11, layers=1, dtype="f32", bidir=True,
                     varlen=(1, 7)),
    wl.LSTMP_2L.scaled(T=7, B=5, in_dim=8, hidden=16, proj=6, dtype="f32", bidir=True,
                       varlen=(1, 7), h0_std=0.5),
    wl.BILSTM_VAR.scaled(T=40, B=64, in_dim=256, hidden=256, varlen=(5, 40)),
    # batches too large for the reverse-time kernel's K split over a CTA pair
    # (which needs at most 32 rows per batch group): single CTAs, the K slices
    # summed by warp shuffles (38 rows per group) ...
    wl.GRU_3L.scaled(T=4, B=300, in_dim=16, hidden=24, layers=1, dtype="f32", h0_std=0.3),
    # ... and through shared memory (75 rows per group: more than 16 row
    # groups, 26 slices)
    wl.LSTM_T80.scaled(T=3, B=600, in_dim=12, hidden=20, layers=1, h0_std=0.5, c0_std=0.5),
]


def _bwd_id(s):
    return (f"{s.cell}-L{s.layers}-D{s.D}-T{s.T}-B{s.B}-H{s.hidden}-P{s.proj}"
            + ("-varlen" if s.varlen else ""))


@pytest.mark.parametrize("spec", BWD_SPECS, ids=_bwd_id)
def test_backward_parity(spec):
    inp = wl.make_rnn_inputs(spec, seed=12)
    g = torch.Generator().manual_seed(99)
    L, B, H, Ho, D = spec.layers, spec.B, spec.hidden, spec.Hout, spec.D
    dy = torch.randn((spec.T, B, D * Ho), generator=g)
    dhn = torch.randn((L * D, B, Ho), generator=g)
    dcn = torch.randn((L * D, B, H), generator=g) if spec.cell == "lstm" else None
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])

    def d(t):
        return None if t is None else t.to(dev)
    dx, dh0, dc0, grads = net.backward(d(inp["x"]), d(dy), lengths=d(inp["lengths"]),
                                       h0=d(inp["h0"]), c0=d(inp["c0"]), dh_n=d(dhn),
                                       dc_n=d(dcn))
    torch.cuda.synchronize()
    assert net.status() == 0
    ref = oracle.rnn_backward(_cell(spec), inp["x"], inp["weights"], dy, hidden=H,
                              proj=spec.proj, bidirectional=spec.bidir,
                              lengths=inp["lengths"], h0=inp["h0"], c0=inp["c0"], dh_n=dhn,
                              dc_n=dcn)
    if inp["lengths"] is not None:  # no gradient reaches x past a row's end
        dxc = dx.cpu().numpy()
        for b, n in enumerate(inp["lengths"].tolist()):
            assert np.all(dxc[n:, b] == 0.0)
    pairs = [("dx", dx, ref["dx"]), ("dh0", dh0, ref["dh0"])]
    if spec.cell == "lstm":
        pairs.append(("dc0", dc0, ref["dc0"]))
    for i in range(L * D):
        for k in ("w_ih", "w_hh", "b_ih", "b_hh") + (("w_hr",) if spec.proj else ()):
            pairs.append((f"d{k}[{i}]", grads[i][k], ref["d" + k][i]))
    for name, got, want in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    net.close()


BWD_BF16_SPECS = [
    wl.GRU_3L.scaled(T=8, B=130, in_dim=64, hidden=96, layers=2),      # tensor-core forward
    wl.LSTM_T80.scaled(T=9, B=6, in_dim=24, hidden=40, dtype="bf16", h0_std=0.5, c0_std=0.5),
    wl.LSTMP_2L.scaled(T=7, B=5, in_dim=24, hidden=64, proj=16),        # folded forward
    wl.LSTM_T80.scaled(T=9, B=6, in_dim=24, hidden=40, dtype="bf16", varlen=(1, 9)),
    # the 3-layer GRU workload's width: 1024 units, 256 rows (the reverse-time
    # kernel's plan shrinks its K slices to fit), short T, one layer
    wl.GRU_3L.scaled(T=3, B=256, in_dim=64, hidden=1024, layers=1, h0_std=0.1),
    # T*B = 185 rows (not a multiple of 8) and an input width that is not
    # either: the bf16 operand copies are padded row by row
    wl.GRU_3L.scaled(T=5, B=37, in_dim=60, hidden=96, layers=2, h0_std=0.5),
    # input width 13: the weight-gradient GEMMs keep the fp32 path (their
    # output rows need a multiple of 4), the recompute runs on the tensor cores
    wl.LSTM_T80.scaled(T=6, B=20, in_dim=13, hidden=48, dtype="bf16", h0_std=0.5, c0_std=0.5),
    # T*B = 4096 rows: the weight-gradient GEMMs (2 output tiles against
    # 64 K blocks) split K into 4 chunks summed in order
    wl.GRU_3L.scaled(T=64, B=64, in_dim=32, hidden=64, layers=2, h0_std=0.5),
    # the tcgen05 reverse-time path reads h_{t-1} from h0 and the layer's
    # output in place: no h0 (zero rows), both directions, a single step (h0
    # alone), and an input width of 13 (fp32 weight-gradient GEMMs, which
    # take the assembled h_{t-1} sequence)
    wl.GRU_3L.scaled(T=6, B=40, in_dim=32, hidden=64, layers=2, h0_std=0.0),
    wl.GRU_3L.scaled(T=5, B=24, in_dim=16, hidden=32, layers=2, bidir=True, h0_std=0.3),
    wl.GRU_3L.scaled(T=1, B=16, in_dim=16, hidden=32, layers=1, h0_std=0.5),
    wl.GRU_3L.scaled(T=5, B=20, in_dim=13, hidden=32, layers=1, h0_std=0.5),
    # a bidirectional LSTM over variable lengths: both directions' FFMA
    # reverse-time recurrences in one launch, the GEMMs on the tensor cores
    wl.BILSTM_VAR.scaled(T=8, B=12, in_dim=16, hidden=32, varlen=(1, 8), dtype="bf16",
                         h0_std=0.3, c0_std=0.3),
]


@pytest.mark.parametrize("spec", BWD_BF16_SPECS, ids=_bwd_id)
def test_backward_bf16_parity(spec):
    """bf16 handles: the gradient of the model with the bf16-rounded weights
    the forward used, its GEMMs on the tensor cores (operands rounded to bf16
    as the forward's are, fp32 accumulation), against the oracle's fp64
    gradient of the model with the same rounded weights (bf16 tier: relative
    2e-2; the forward's bf16 activation rounding is in the recomputed
    states)."""
    inp = wl.make_rnn_inputs(spec, seed=13)
    g = torch.Generator().manual_seed(98)
    L, D, B, Ho = spec.layers, spec.D, spec.B, spec.Hout
    dy = torch.randn((spec.T, B, D * Ho), generator=g)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_PROFILE, 1)

    def d(t):
        return None if t is None else t.to(dev)
    dx, dh0, dc0, grads = net.backward(d(inp["x"]), d(dy), lengths=d(inp["lengths"]),
                                       h0=d(inp["h0"]), c0=d(inp["c0"]))
    torch.cuda.synchronize()
    assert net.status() == 0
    # the GRU over fixed-length rows (widths of whole 32-unit clusters) takes
    # the tcgen05 reverse-time kernel, every other form the FFMA one
    tc_rec = spec.cell == "gru" and spec.varlen is None and spec.hidden % 32 == 0
    assert ("bwd_recurrent_tc" in net.profile()) == tc_rec, net.profile()
    ref = oracle.rnn_backward(_cell(spec), inp["x"], inp["weights"], dy, hidden=spec.hidden,
                              proj=spec.proj, bidirectional=spec.bidir, lengths=inp["lengths"],
                              h0=inp["h0"], c0=inp["c0"], bf16_weights=True)
    pairs = [("dx", dx, ref["dx"]), ("dh0", dh0, ref["dh0"])]
    for i in range(L * D):
        for k in ("w_ih", "w_hh", "b_ih") + (("w_hr",) if spec.proj else ()):
            pairs.append((f"d{k}[{i}]", grads[i][k], ref["d" + k][i]))
    for name, got, want in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BF16_REL, f"{name}: relative max error {e:.3e}"
    net.close()


# ----------------------------------------------------------------------------- RSSM

RSSM_BWD_SPECS = [
    wl.RSSM_B50,
    wl.RSSM_B50.scaled(T=7, B=3, state_dim=5, action_dim=0, hidden=33, rnn_hidden=17,
                       state0_std=1.0, belief0_std=0.5),
    wl.RSSM_B50.scaled(T=6, B=70, state_dim=13, action_dim=5, hidden=72, rnn_hidden=40,
                       state0_std=1.0, belief0_std=0.5),
]


@pytest.mark.parametrize("spec", RSSM_BWD_SPECS,
                         ids=lambda s: f"T{s.T}-B{s.B}-S{s.state_dim}-A{s.action_dim}-H{s.hidden}")
@pytest.mark.parametrize("which", ["all", "beliefs_only"])
@pytest.mark.parametrize("chain", ["fused", "launches"])
def test_rssm_backward_parity(spec, which, chain):
    """rssm_backward + rssm_get_weight_grads against the oracle's RSSM backward
    (per tensor: max|gpu - ref| / max|ref| <= 1e-4); gradients given for every
    output, or for the beliefs alone (the others NULL); the reverse-time
    chain as one cluster-resident kernel or as separate launches per step."""
    inp = wl.make_rssm_inputs(spec, seed=22)
    g = torch.Generator().manual_seed(97)
    T, B, S, RH = spec.T, spec.B, spec.state_dim, spec.rnn_hidden
    grads = {k: torch.randn((T, B, n), generator=g)
             for k, n in (("dmeans", S), ("dstds", S), ("dstates", S), ("dbeliefs", RH))}
    if which == "beliefs_only":
        grads = {"dbeliefs": grads["dbeliefs"]}
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    if chain == "launches":
        binding.rssm_set_attr(m.h, binding.RCU_ATTR_FORCE_PATH, 1)
    with pytest.raises(RuntimeError, match="no rssm_backward"):
        binding.rssm_get_weight_grads(m.h, {})
    d = lambda t: None if t is None else t.to(dev)
    dstate0, dbelief0, dactions, wg = m.backward(
        d(inp["actions"]), d(inp["eps"]), d(inp["state0"]), d(inp["belief0"]),
        **{k: d(v) for k, v in grads.items()})
    torch.cuda.synchronize()
    assert binding.rssm_get_status(m.h) == 0
    # the fused chain is one launch for all T steps, the other ~9 per step
    n_launch = binding.rssm_last_launch_count(m.h)
    assert (n_launch < 60) if chain == "fused" else (n_launch > 5 * spec.T), n_launch
    ref = oracle.rssm_backward(inp["weights"], inp["actions"], inp["eps"], state0=inp["state0"],
                               belief0=inp["belief0"], **grads)
    pairs = [("dstate0", dstate0), ("dbelief0", dbelief0)]
    if spec.action_dim > 0:
        pairs.append(("dactions", dactions))
    pairs += [("d" + k, wg[k]) for k in binding.RSSM_WEIGHT_NAMES]
    for name, got in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), ref[name])
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    m.close()


# ----------------------------------------------------------------------------- projection clipping rejected, cell clipping

def test_backward_errors():
    spec = BWD_SPECS[0]
    inp = wl.make_rnn_inputs(spec, seed=1)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    with pytest.raises(RuntimeError, match="no rnn_backward"):
        binding.rnn_get_weight_grads(net.h, 0, None, None, None, None)
    net.close()
    # projection clipping sits between W_hr and W_hh and breaks the folded
    # projection recurrence: rejected (cell clipping is covered below)
    spec = wl.LSTMP_2L.scaled(T=4, B=3, in_dim=6, hidden=12, proj=5, dtype="f32")
    inp = wl.make_rnn_inputs(spec, seed=1)
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_clip(binding.RCU_CLIP_PROJ, (-1.0, 1.0))
    x = torch.zeros((spec.T, spec.B, spec.in_dim), device=dev)
    dy = torch.zeros((spec.T, spec.B, spec.Hout), device=dev)
    with pytest.raises(RuntimeError, match="projection clipping"):
        binding.rnn_backward(net.h, spec.T, spec.B, x, None, None, None, dy, None, None, None, None,
                             None)
    net.close()


BWD_CLIP_SPECS = [
    (wl.LSTM_T80.scaled(T=8, B=6, in_dim=12, hidden=20, layers=2, h0_std=0.5, c0_std=0.5),
     (-0.12, 0.15)),
    (wl.LSTMP_2L.scaled(T=7, B=5, in_dim=10, hidden=24, proj=8, dtype="f32", h0_std=0.5,
                        c0_std=0.5), (-0.1, 0.12)),
    (wl.BILSTM_VAR.scaled(T=9, B=7, in_dim=12, hidden=20, varlen=(1, 9), c0_std=0.5),
     (-0.12, 0.15)),
    (wl.LSTM_T80.scaled(T=24, B=16, in_dim=64, hidden=128, layers=1, c0_std=0.3),
     (-0.1, 0.1)),
]


@pytest.mark.parametrize("spec,bounds", BWD_CLIP_SPECS,
                         ids=lambda v: _bwd_id(v) if hasattr(v, "cell") else f"clip{v[1]}")
def test_backward_cell_clip_parity(spec, bounds):
    """Cell-state clipping in the backward pass (the clamp passes dc where the
    unclamped cell value lies within the bounds) against the oracle with the
    same clipping; bounds chosen so that a good share of the cells clamp."""
    inp = wl.make_rnn_inputs(spec, seed=14)
    g = torch.Generator().manual_seed(95)
    L, B, H, Ho, D = spec.layers, spec.B, spec.hidden, spec.Hout, spec.D
    dy = torch.randn((spec.T, B, D * Ho), generator=g)
    dcn = torch.randn((L * D, B, H), generator=g)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_clip(binding.RCU_CLIP_CELL, bounds)

    def d(t):
        return None if t is None else t.to(dev)
    dx, dh0, dc0, grads = net.backward(d(inp["x"]), d(dy), lengths=d(inp["lengths"]),
                                       h0=d(inp["h0"]), c0=d(inp["c0"]), dc_n=d(dcn))
    torch.cuda.synchronize()
    assert net.status() == 0
    ref = oracle.rnn_backward(_cell(spec), inp["x"], inp["weights"], dy, hidden=H,
                              proj=spec.proj, bidirectional=spec.bidir, lengths=inp["lengths"],
                              h0=inp["h0"], c0=inp["c0"], dc_n=dcn, cell_clip=bounds)
    pairs = [("dx", dx, ref["dx"]), ("dh0", dh0, ref["dh0"]), ("dc0", dc0, ref["dc0"])]
    for i in range(L * D):
        for k in ("w_ih", "w_hh", "b_ih", "b_hh") + (("w_hr",) if spec.proj else ()):
            pairs.append((f"d{k}[{i}]", grads[i][k], ref["d" + k][i]))
    for name, got, want in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    net.close()


# ----------------------------------------------------------------------------- RSSM with the actor, phase profile

@pytest.mark.parametrize("spec", [
    wl.RSSM_ACTOR,
    wl.RSSM_B50.scaled(T=6, B=70, state_dim=13, action_dim=5, hidden=72, rnn_hidden=40,
                       state0_std=1.0, belief0_std=0.5, actor_hidden=37),
], ids=lambda s: f"T{s.T}-B{s.B}-S{s.state_dim}-A{s.action_dim}-X{s.actor_hidden}")
def test_rssm_actor_backward_parity(spec):
    """rssm_backward_actor + rssm_get_weight_grads + rssm_get_actor_grads
    against the oracle's backward of the actor variant (per tensor: max|gpu -
    ref| / max|ref| <= 1e-4), including the gradient reaching each action."""
    inp = wl.make_rssm_inputs(spec, seed=24)
    g = torch.Generator().manual_seed(96)
    T, B, S, RH = spec.T, spec.B, spec.state_dim, spec.rnn_hidden
    grads = {k: torch.randn((T, B, n), generator=g)
             for k, n in (("dmeans", S), ("dstds", S), ("dstates", S), ("dbeliefs", RH))}
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    m.set_actor(inp["actor"])
    with pytest.raises(RuntimeError, match="no rssm_backward_actor"):
        binding.rssm_get_actor_grads(m.h, {})
    d = lambda t: None if t is None else t.to(dev)
    dstate0, dbelief0, dactions, wg, ag = m.backward_actor(
        d(inp["eps"]), d(inp["state0"]), d(inp["belief0"]), **{k: d(v) for k, v in grads.items()})
    torch.cuda.synchronize()
    assert binding.rssm_get_status(m.h) == 0
    ref = oracle.rssm_backward(inp["weights"], None, inp["eps"], state0=inp["state0"],
                               belief0=inp["belief0"], actor=inp["actor"], **grads)
    pairs = [("dstate0", dstate0), ("dbelief0", dbelief0), ("dactions", dactions)]
    pairs += [("d" + k, wg[k]) for k in binding.RSSM_WEIGHT_NAMES]
    pairs += [("d" + k, ag[k]) for k in binding.RSSM_ACTOR_NAMES]
    for name, got in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), ref[name])
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    m.close()


def test_rssm_profile_phases():
    """RCU_ATTR_PROFILE on an RSSM handle times the unroll and the three phases
    of rssm_backward, once per call each."""
    spec = wl.RSSM_B50.scaled(T=5, B=4)
    inp = wl.make_rssm_inputs(spec, seed=23)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    m.set_attr(binding.RCU_ATTR_PROFILE, 1)
    binding.rssm_profile_reset(m.h)
    m.backward(inp["actions"].to(dev), inp["eps"].to(dev),
               dbeliefs=torch.ones((spec.T, spec.B, spec.rnn_hidden), device=dev))
    prof = m.profile()
    assert binding.rssm_get_status(m.h) == 0
    for name in ("rssm_unroll", "rssm_bwd_recompute", "rssm_bwd_chain", "rssm_bwd_grads"):
        assert name in prof and prof[name][1] == 1 and prof[name][0] > 0.0, (name, prof)
    # (at least one launch in each of the four ranges)
    assert m.launch_count() >= 4
    m.close()


def test_backward_argument_errors():
    """Degenerate arguments are rejected on the host before any launch: an
    empty sequence or batch, a missing actor, missing actions."""
    spec = wl.LSTM_T80.scaled(T=3, B=2, in_dim=4, hidden=5)
    inp = wl.make_rnn_inputs(spec, seed=3)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    x = torch.zeros((3, 2, 4), device=dev)
    dy = torch.zeros((3, 2, 5), device=dev)
    for T, B in ((0, 2), (3, 0)):
        with pytest.raises(RuntimeError, match="need T, B >= 1"):
            binding.rnn_backward(net.h, T, B, x, None, None, None, dy, None, None, None, None, None)
    net.close()
    rs = wl.RSSM_B50.scaled(T=3, B=2, state_dim=4, action_dim=2, hidden=6, rnn_hidden=5)
    ri = wl.make_rssm_inputs(rs, seed=3)
    m = binding.RSSM(rs.state_dim, rs.action_dim, rs.hidden, rs.rnn_hidden)
    m.set_weights(ri["weights"])
    eps = ri["eps"].to(dev)
    with pytest.raises(RuntimeError, match="actor not set"):
        m.backward_actor(eps)
    with pytest.raises(RuntimeError, match="need T, B >= 1"):
        m.backward(None, eps)  # actions missing with action_dim > 0
    with pytest.raises(RuntimeError, match="need T, B >= 1"):
        binding.rssm_backward(m.h, 0, 2, None, None, ri["actions"].to(dev), eps, None, None, None,
                              None, None, None, None)
    m.close()


# ----------------------------------------------------------------------------- full-size training pass

@pytest.mark.parametrize("spec", [wl.LSTM_TRAIN, wl.BILSTM_TRAIN], ids=lambda s: s.name)
def test_training_pass_full_size(spec):
    """The training workloads at their full size, through rnn_backward as the
    benchmark calls it (seed-0 inputs, the workload's dy, no dh_n / dc_n):
    every gradient tensor against the oracle's backward over all rows."""
    inp = wl.make_rnn_inputs(spec, seed=0)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    d = lambda t: None if t is None else t.to(dev)
    dx, dh0, dc0, grads = net.backward(d(inp["x"]), d(inp["dy"]), lengths=d(inp["lengths"]),
                                       h0=d(inp["h0"]), c0=d(inp["c0"]))
    torch.cuda.synchronize()
    assert net.status() == 0
    ref = oracle.rnn_backward(_cell(spec), inp["x"], inp["weights"], inp["dy"],
                              hidden=spec.hidden, proj=spec.proj, bidirectional=spec.bidir,
                              lengths=inp["lengths"], h0=inp["h0"], c0=inp["c0"])
    pairs = [("dx", dx, ref["dx"]), ("dh0", dh0, ref["dh0"])]
    if spec.cell == "lstm":
        pairs.append(("dc0", dc0, ref["dc0"]))
    for i in range(spec.layers * spec.D):
        for k in ("w_ih", "w_hh", "b_ih", "b_hh"):
            pairs.append((f"d{k}[{i}]", grads[i][k], ref["d" + k][i]))
    for name, got, want in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    net.close()


def test_gru_training_full_width_sampled_rows():
    """The 3-layer GRU training workload's width and batch (1024 units, 256
    rows: two batch groups on the 4-CTA tcgen05 reverse-time kernel) over 16
    steps.  Rows are independent in dx and dh0, so 6 rows spread over both
    batch groups and the TMEM lane quarters are checked against the oracle run
    on those rows alone (the weight gradients, sums over every row, are
    checked at this width over all rows by test_backward_bf16_parity)."""
    spec = wl.GRU_TRAIN.scaled(T=16)
    inp = wl.make_rnn_inputs(spec, seed=0)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_PROFILE, 1)
    d = lambda t: None if t is None else t.to(dev)
    dx, dh0, _, _ = net.backward(d(inp["x"]), d(inp["dy"]), h0=d(inp["h0"]))
    torch.cuda.synchronize()
    assert net.status() == 0
    assert "bwd_recurrent_tc" in net.profile(), net.profile()
    rows = [0, 31, 32, 127, 128, 255]
    ref = oracle.rnn_backward(oracle.GRU, inp["x"][:, rows], inp["weights"], inp["dy"][:, rows],
                              hidden=spec.hidden, h0=inp["h0"][:, rows], bf16_weights=True)
    for name, got, want in (("dx", dx[:, rows], ref["dx"]), ("dh0", dh0[:, rows], ref["dh0"])):
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BF16_REL, f"{name}: relative max error {e:.3e}"
    net.close()


# fp32 handles with RCU_ATTR_FORCE_PATH = 2: every GEMM (input projection,
# recomputed pre-activations, weight and input gradients) runs on the tensor
# cores as a three-term bf16 split at any size; the fp32 bound still holds
F32X6_SPECS = [
    wl.LSTM_T80.scaled(T=9, B=13, in_dim=24, hidden=40, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(dtype="f32", layers=2, T=7, B=21, in_dim=36, hidden=52, h0_std=0.5),
    wl.BILSTM_VAR.scaled(T=12, B=9, in_dim=20, hidden=32, varlen=(1, 12)),
    # 4,480 rows: the weight gradients' reductions run in two chunks
    wl.LSTM_T80.scaled(T=70, B=64, in_dim=16, hidden=24),
]


@pytest.mark.parametrize("spec", F32X6_SPECS, ids=_bwd_id)
def test_fp32_split_tensor_core_gemms(spec):
    inp = wl.make_rnn_inputs(spec, seed=41)
    g = torch.Generator().manual_seed(41)
    dy = torch.randn((spec.T, spec.B, spec.D * spec.Hout), generator=g)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_FORCE_PATH, 2)

    def d(t):
        return None if t is None else t.to(dev)
    y, hn, cn = net.forward(d(inp["x"]), lengths=d(inp["lengths"]), h0=d(inp["h0"]),
                            c0=d(inp["c0"]))
    dx, dh0, dc0, grads = net.backward(d(inp["x"]), d(dy), lengths=d(inp["lengths"]),
                                       h0=d(inp["h0"]), c0=d(inp["c0"]))
    torch.cuda.synchronize()
    assert net.status() == 0
    fwd = oracle.rnn_forward(_cell(spec), inp["x"], inp["weights"], hidden=spec.hidden,
                             bidirectional=spec.bidir, lengths=inp["lengths"], h0=inp["h0"],
                             c0=inp["c0"])
    assert float(np.abs(y.cpu().numpy() - fwd[0]).max()) <= 1e-4
    ref = oracle.rnn_backward(_cell(spec), inp["x"], inp["weights"], dy, hidden=spec.hidden,
                              bidirectional=spec.bidir, lengths=inp["lengths"], h0=inp["h0"],
                              c0=inp["c0"])
    pairs = [("dx", dx, ref["dx"]), ("dh0", dh0, ref["dh0"])]
    for i in range(spec.layers * spec.D):
        for k in ("w_ih", "w_hh", "b_ih", "b_hh"):
            pairs.append((f"d{k}[{i}]", grads[i][k], ref["d" + k][i]))
    for name, got, want in pairs:
        e = _rel(got.cpu().numpy().astype(np.float64), want)
        print(f"{name}: rel {e:.2e}")
        assert e <= BWD_REL, f"{name}: relative max error {e:.3e}"
    net.close()
