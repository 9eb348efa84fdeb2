"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: fp32 path max-abs error <= 1e-4 on every output after all T
steps; bf16-weight path max|gpu - ref| / max|ref| <= 2e-2 per output tensor
(weights rounded to bf16 on both sides); packing indices bit-exact.
Small cases cover several tiles and ragged tails element by element; the
full-size workloads are checked on sampled batch rows, which the oracle
computes exactly (rows are independent).
"""
import numpy as np
import pytest
import torch

import oracle
from recurrent_cell_unroll_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_REL = 2e-2


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _cell(spec):
    return oracle.LSTM if spec.cell == "lstm" else oracle.GRU


def run_gpu(spec, inp, force_path=0, bias=True):
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    if force_path:
        net.set_attr(binding.RCU_ATTR_FORCE_PATH, force_path)
    net.set_weights(inp["weights"])
    lengths = inp["lengths"].to(dev) if inp["lengths"] is not None else None
    h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
    c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
    y, hn, cn = net.forward(inp["x"].to(dev), lengths=lengths, h0=h0, c0=c0)
    st = net.status()
    assert st == 0, f"device status {st}"
    out = (y.cpu().numpy(), hn.cpu().numpy(), None if cn is None else cn.cpu().numpy())
    net.close()
    return out


def run_oracle(spec, inp, rows=None):
    return oracle.rnn_forward(_cell(spec), inp["x"], inp["weights"], hidden=spec.hidden,
                              proj=spec.proj, bidirectional=spec.bidir, lengths=inp["lengths"],
                              h0=inp["h0"], c0=inp["c0"], bf16_weights=spec.dtype == "bf16",
                              rows=rows)


def compare(spec, got, ref, rows=None):
    sel = slice(None) if rows is None else list(rows)
    pairs = [("y", got[0][:, sel], ref[0][:, sel]), ("h_n", got[1][:, sel], ref[1][:, sel])]
    if spec.cell == "lstm":
        pairs.append(("c_n", got[2][:, sel], ref[2][:, sel]))
    for name, g, r in pairs:
        assert np.all(np.isfinite(g)), f"{name} not finite"
        if spec.dtype == "f32":
            e = float(np.abs(g - r).max())
            assert e <= F32_TOL, f"{name}: max-abs error {e:.3e} > {F32_TOL}"
        else:
            e = _rel(g, r)
            assert e <= BF16_REL, f"{name}: relative error {e:.3e} > {BF16_REL}"


SMALL = [
    # fp32 LSTM at the TVM benchmark shape (whole config)
    wl.LSTM_T80,
    wl.LSTM_T80.scaled(T=9, B=7, in_dim=33, hidden=70, c0_std=0.5, h0_std=0.5),
    wl.LSTM_T80.scaled(name="lstm2l", layers=2, T=11, B=37, in_dim=20, hidden=45),
    wl.LSTMP_2L.scaled(T=13, B=5, in_dim=80, hidden=136, proj=40),
    wl.LSTMP_2L.scaled(dtype="f32", T=7, B=9, in_dim=17, hidden=52, proj=12, h0_std=0.3,
                       c0_std=0.3),
    wl.BILSTM_VAR.scaled(T=37, B=13, in_dim=24, hidden=40, varlen=(1, 37)),
    wl.BILSTM_VAR.scaled(layers=2, T=16, B=6, in_dim=8, hidden=20, varlen=(3, 16)),
    wl.GRU_3L.scaled(T=20, B=37, in_dim=72, hidden=200),
    wl.GRU_3L.scaled(dtype="f32", layers=2, bidir=True, T=9, B=5, in_dim=16, hidden=24,
                     varlen=(1, 9)),
    wl.GRU_3L.scaled(layers=1, T=5, B=1, in_dim=8, hidden=1024),
    # fp32 SIMT kernel with 36 gate rows per CTA (9 units): beyond the
    # half-warp tiles' 32, so the 8 x 4 register tiles
    wl.LSTM_T80.scaled(name="lstm_wide", T=4, B=8, in_dim=32, hidden=1280),
    # tensor-core recurrent kernel: two batch groups with a ragged tail, ragged units
    wl.LSTM_T80.scaled(name="lstm_bf16", dtype="bf16", layers=2, T=12, B=150, in_dim=40,
                       hidden=70, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(bidir=True, layers=2, T=15, B=140, in_dim=24, hidden=40, varlen=(1, 15)),
    wl.GRU_3L.scaled(layers=1, T=9, B=256, in_dim=64, hidden=256),
    # LSTMP on the tensor cores (recurrence on m with W_hh W_hr, projection GEMM after)
    wl.LSTMP_2L.scaled(bidir=True, T=9, B=6, in_dim=16, hidden=64, proj=24, h0_std=0.5,
                       c0_std=0.5),
    wl.LSTMP_2L.scaled(layers=3, T=7, B=130, in_dim=32, hidden=128, proj=64),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: f"{s.name}-T{s.T}-B{s.B}-H{s.hidden}")
@pytest.mark.parametrize("path", [0, 1], ids=["auto", "simt"])
def test_small_parity(spec, path):
    inp = wl.make_rnn_inputs(spec, seed=11)
    compare(spec, run_gpu(spec, inp, force_path=path), run_oracle(spec, inp))


def test_no_bias_equals_zero_bias():
    spec = wl.LSTM_T80.scaled(T=6, B=4, in_dim=10, hidden=12)
    inp = wl.make_rnn_inputs(spec, seed=3, bias=False)
    got = run_gpu(spec, inp)
    for w in inp["weights"]:
        w["b_ih"] = torch.zeros(4 * 12)
        w["b_hh"] = torch.zeros(4 * 12)
    ref = run_gpu(spec, inp)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
    compare(spec, got, run_oracle(spec, inp))


def test_pack_indices_bit_exact():
    spec = wl.BILSTM_VAR
    inp = wl.make_rnn_inputs(spec.scaled(in_dim=8, hidden=8), seed=0)
    dev = torch.device("cuda")
    net = binding.RNN("lstm", 1, 8, 8, bidirectional=True)
    net.set_weights(inp["weights"])
    lengths = inp["lengths"].to(dev)
    net.forward(inp["x"].to(dev), lengths=lengths)
    s = torch.empty(spec.B, dtype=torch.int32, device=dev)
    u = torch.empty_like(s)
    bs = torch.empty(spec.T, dtype=torch.int32, device=dev)
    binding.rnn_get_pack(net.h, s, u, bs)
    assert net.status() == 0
    rs, ru, rbs = oracle.pack(inp["lengths"], spec.T)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(u.cpu().numpy(), ru)
    assert np.array_equal(bs.cpu().numpy(), rbs)
    net.close()


def test_padding_is_zero_and_state_at_true_end():
    spec = wl.BILSTM_VAR.scaled(T=20, B=6, in_dim=5, hidden=7, varlen=(1, 20))
    inp = wl.make_rnn_inputs(spec, seed=4)
    got = run_gpu(spec, inp)
    L = inp["lengths"].numpy()
    for b in range(spec.B):
        assert np.all(got[0][L[b]:, b] == 0.0)
    compare(spec, got, run_oracle(spec, inp))


def test_rows_sorted_equal_lengths_and_single_step():
    spec = wl.BILSTM_VAR.scaled(T=1, B=3, in_dim=4, hidden=5, varlen=(1, 1))
    inp = wl.make_rnn_inputs(spec, seed=5)
    compare(spec, run_gpu(spec, inp), run_oracle(spec, inp))
    spec = wl.GRU_3L.scaled(dtype="f32", layers=1, bidir=True, T=6, B=4, in_dim=4, hidden=5,
                            varlen=(6, 6))
    inp = wl.make_rnn_inputs(spec, seed=6)
    compare(spec, run_gpu(spec, inp), run_oracle(spec, inp))


def test_non_canonical_strides_give_same_result():
    spec = wl.LSTM_T80.scaled(T=1, B=4, in_dim=5, hidden=6)
    inp = wl.make_rnn_inputs(spec, seed=7)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    x = inp["x"].to(dev)
    y1, _, _ = net.forward(x)
    x_odd = x.reshape(-1).as_strided((1, 4, 5), (5, 5, 1))  # passes is_contiguous()
    y2, _, _ = net.forward(x_odd)
    assert net.status() == 0
    assert torch.equal(y1, y2)
    net.close()


def test_deterministic_repeat():
    spec = wl.GRU_3L.scaled(T=10, B=9, in_dim=32, hidden=64)
    inp = wl.make_rnn_inputs(spec, seed=8)
    a = run_gpu(spec, inp)
    b = run_gpu(spec, inp)
    for x, y in zip(a, b):
        if x is not None:
            np.testing.assert_array_equal(x, y)


def test_errors_are_reported():
    with pytest.raises(binding.RcuError) as e:
        binding.rnn_create(binding.RCU_GRU, 1, 4, 8, 2, binding.RCU_F32)
    assert e.value.code == binding.RCU_ERR_UNSUPPORTED
    with pytest.raises(binding.RcuError):
        binding.rnn_create(binding.RCU_LSTM, 0, 4, 8, 0, binding.RCU_F32)
    net = binding.RNN("lstm", 1, 4, 8)
    with pytest.raises(binding.RcuError) as e:
        net.forward(torch.zeros(3, 2, 4, device="cuda"))
    assert e.value.code == binding.RCU_ERR_STATE
    net.close()


def test_bad_lengths_flagged_on_device():
    spec = wl.BILSTM_VAR.scaled(T=5, B=3, in_dim=4, hidden=4, varlen=(1, 5))
    inp = wl.make_rnn_inputs(spec, seed=9)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    lengths = torch.tensor([5, 0, 7], dtype=torch.int32, device=dev)
    net.forward(inp["x"].to(dev), lengths=lengths)
    assert net.status() == binding.RCU_ERR_LENGTHS
    y, _, _ = net.forward(inp["x"].to(dev), lengths=inp["lengths"].to(dev))
    assert net.status() == 0
    net.close()


def test_barrier_wait_times_out_and_context_survives():
    """One CTA never arrives at the first step barrier: every wait must end
    with RCU_ERR_TIMEOUT within the bound, and the next call must work."""
    spec = wl.LSTM_T80.scaled(T=4, B=2, in_dim=8, hidden=64)
    inp = wl.make_rnn_inputs(spec, seed=10)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_BARRIER_TIMEOUT_NS, 50_000_000)
    net.set_attr(binding.RCU_ATTR_FORCE_PATH, 1)
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 1)
    net.forward(inp["x"].to(dev))
    assert net.status() == binding.RCU_ERR_TIMEOUT
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 0)
    y, hn, cn = net.forward(inp["x"].to(dev))
    assert net.status() == 0
    ref = run_oracle(spec, inp)
    assert np.abs(y.cpu().numpy() - ref[0]).max() <= F32_TOL
    net.close()


KSPLIT = [
    # two batch groups with a ragged tail; 13 sixteen-unit tiles (odd: the last
    # pair has one tile of zero rows); H not a multiple of 16
    wl.GRU_3L.scaled(layers=2, T=10, B=150, in_dim=40, hidden=200, h0_std=0.5),
    wl.LSTM_T80.scaled(name="lstm_bf16", dtype="bf16", layers=1, T=8, B=129, in_dim=64,
                       hidden=1000, h0_std=0.5, c0_std=0.5),
    # varlen, both directions; odd number of K blocks (3) so the pair splits 2 + 1
    wl.BILSTM_VAR.scaled(dtype="bf16", T=12, B=70, in_dim=24, hidden=150, varlen=(1, 12)),
    wl.GRU_3L.scaled(layers=1, T=6, B=256, in_dim=32, hidden=1024),
]


@pytest.mark.parametrize("spec", KSPLIT, ids=lambda s: f"{s.name}-T{s.T}-B{s.B}-H{s.hidden}")
@pytest.mark.parametrize("ksplit", [1, 2, 4])
def test_tensor_core_k_split(spec, ksplit):
    """h W_hh^T with K kept whole (1) or split over a CTA pair (2) or four
    CTAs (4) whose partial sums are exchanged through distributed shared
    memory."""
    inp = wl.make_rnn_inputs(spec, seed=17)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_attr(binding.RCU_ATTR_FORCE_PATH, 2)
    net.set_attr(binding.RCU_ATTR_TC_KSPLIT, ksplit)
    net.set_attr(binding.RCU_ATTR_PROFILE, 1)
    net.set_weights(inp["weights"])
    lengths = inp["lengths"].to(dev) if inp["lengths"] is not None else None
    h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
    c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
    y, hn, cn = net.forward(inp["x"].to(dev), lengths=lengths, h0=h0, c0=c0)
    assert net.status() == 0
    torch.cuda.synchronize()
    assert "recurrent_tc" in net.profile()
    got = (y.cpu().numpy(), hn.cpu().numpy(), None if cn is None else cn.cpu().numpy())
    compare(spec, got, run_oracle(spec, inp))
    net.close()


# Layer-pipelined LSTMP (unidirectional, bf16, T >= 128): layers run
# concurrently over chunks of steps; ragged last chunk; three layers
PIPE = [
    wl.LSTMP_2L.scaled(T=200, B=32, in_dim=80, hidden=256, proj=64, h0_std=0.5, c0_std=0.5),
    wl.LSTMP_2L.scaled(layers=3, T=131, B=7, in_dim=24, hidden=128, proj=48),
    # no projection: the tensor-core recurrence of each layer writes the next
    # layer's input chunk by chunk (two batch groups, the second ragged)
    wl.GRU_3L.scaled(T=200, B=150, in_dim=40, hidden=96, h0_std=0.5),
    wl.LSTM_T80.scaled(name="lstm_bf16", dtype="bf16", layers=2, T=131, B=37, in_dim=24,
                       hidden=64, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(layers=2, T=129, B=256, in_dim=64, hidden=256),
]


@pytest.mark.parametrize("spec", PIPE,
                         ids=lambda s: f"{s.cell}-L{s.layers}-T{s.T}-B{s.B}-H{s.hidden}-P{s.proj}")
def test_layer_pipelined_forward(spec):
    """The pipelined forward equals the layer-by-layer one bit for bit (every
    GEMM row and recurrent step sees the same operands) and the oracle."""
    inp = wl.make_rnn_inputs(spec, seed=23)
    dev = torch.device("cuda")
    outs = []
    kernel = "recurrent_tc_lstmp" if spec.proj else "recurrent_tc"
    for pipe in (1, 0):
        net = binding.RNN.from_spec(spec)
        net.set_attr(binding.RCU_ATTR_LAYER_PIPELINE, pipe)
        net.set_attr(binding.RCU_ATTR_PROFILE, 1)
        if not spec.proj:
            # the tensor-core recurrence (small shapes would take the cluster kernel)
            net.set_attr(binding.RCU_ATTR_FORCE_PATH, 2)
        net.set_weights(inp["weights"])
        h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
        c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
        y, hn, cn = net.forward(inp["x"].to(dev), h0=h0, c0=c0)
        assert net.status() == 0
        torch.cuda.synchronize()
        prof = net.profile()
        # one recurrent launch per layer and chunk when pipelined, per layer otherwise
        n_rec = prof[kernel][1]
        assert (n_rec > spec.layers) if pipe else (n_rec == spec.layers), prof
        outs.append((y.cpu().numpy(), hn.cpu().numpy(),
                     cn.cpu().numpy() if cn is not None else None))
        net.close()
    for a, b in zip(*outs):
        if a is not None:
            np.testing.assert_array_equal(a, b)
    compare(spec, outs[0], run_oracle(spec, inp))


CLUSTER = [
    wl.LSTM_T80,  # one row: one cluster of 16 CTAs
    wl.LSTM_T80.scaled(T=9, B=7, in_dim=33, hidden=70, c0_std=0.5, h0_std=0.5),
    wl.LSTM_T80.scaled(name="lstm2l", layers=2, T=11, B=37, in_dim=20, hidden=45),
    wl.GRU_3L.scaled(dtype="f32", layers=2, bidir=True, T=9, B=5, in_dim=16, hidden=24,
                     varlen=(1, 9)),
    wl.BILSTM_VAR.scaled(T=21, B=33, in_dim=24, hidden=300, varlen=(1, 21), h0_std=0.3,
                         c0_std=0.3),
    wl.GRU_3L.scaled(dtype="f32", layers=1, T=12, B=37, in_dim=40, hidden=200),
    wl.LSTM_T80.scaled(name="lstm_bf16", dtype="bf16", layers=2, T=12, B=150, in_dim=40,
                       hidden=70, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(bidir=True, layers=2, T=15, B=140, in_dim=24, hidden=40, varlen=(1, 15)),
    # widths whose units split evenly over the cluster (4 and 8 per CTA):
    # several batch slices, variable lengths, both directions
    wl.LSTM_T80.scaled(name="lstm_q4", T=13, B=37, in_dim=30, hidden=64, varlen=(1, 13),
                       h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(name="gru_q8", dtype="f32", layers=2, bidir=True, T=10, B=20, in_dim=12,
                     hidden=128, varlen=(2, 10)),
    wl.LSTM_T80.scaled(name="lstm_bf16_q8", dtype="bf16", layers=2, T=9, B=60, in_dim=16,
                       hidden=128),
]


@pytest.mark.parametrize("spec", CLUSTER, ids=lambda s: f"{s.name}-T{s.T}-B{s.B}-H{s.hidden}")
def test_cluster_resident_kernel(spec):
    """W_hh resident in one thread-block cluster, h exchanged through
    distributed shared memory, clusters on disjoint batch slices."""
    inp = wl.make_rnn_inputs(spec, seed=19)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_attr(binding.RCU_ATTR_FORCE_PATH, 3)
    net.set_attr(binding.RCU_ATTR_PROFILE, 1)
    net.set_weights(inp["weights"])
    lengths = inp["lengths"].to(dev) if inp["lengths"] is not None else None
    h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
    c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
    y, hn, cn = net.forward(inp["x"].to(dev), lengths=lengths, h0=h0, c0=c0)
    assert net.status() == 0
    torch.cuda.synchronize()
    assert "recurrent_cluster" in net.profile()
    got = (y.cpu().numpy(), hn.cpu().numpy(), None if cn is None else cn.cpu().numpy())
    compare(spec, got, run_oracle(spec, inp))
    net.close()


@pytest.mark.parametrize("in_dim", [64, 128, 256, 520])
def test_input_projection_k_split(in_dim):
    """fp32 input GEMM with few output tiles: K split over a 2/4/8-CTA cluster
    (in_dim 64, 128, 256; 520 leaves the last slice short), partial tiles
    summed over distributed shared memory."""
    spec = wl.LSTM_T80.scaled(T=5, B=6, in_dim=in_dim, hidden=40, h0_std=0.3, c0_std=0.3)
    inp = wl.make_rnn_inputs(spec, seed=23)
    for path in (1, 3):
        compare(spec, run_gpu(spec, inp, force_path=path), run_oracle(spec, inp))


@pytest.mark.parametrize("spec", [
    wl.LSTM_T80,
    wl.BILSTM_VAR.scaled(T=40, B=16, in_dim=64, hidden=128, varlen=(5, 40)),
], ids=lambda s: s.name)
def test_opt_in_bf16_conversion_accuracy(spec):
    """An fp32 workload run through the opt-in down-conversion (a bf16 handle:
    weights and MMA operands rounded to bf16, fp32 state and accumulation).
    Parity is asserted against the model the conversion defines (the oracle
    with the same bf16-rounded weights) at the bf16 tolerance; the distance
    from the exact fp32 model (the oracle with unrounded weights) includes
    the weight quantisation, which no tolerance on the pages bounds, so it is
    reported only."""
    inp = wl.make_rnn_inputs(spec, seed=29)
    bspec = spec.scaled(dtype="bf16")
    got = run_gpu(bspec, inp)
    compare(bspec, got, run_oracle(bspec, inp))
    ref = oracle.rnn_forward(_cell(spec), inp["x"], inp["weights"], hidden=spec.hidden,
                             proj=spec.proj, bidirectional=spec.bidir, lengths=inp["lengths"],
                             h0=inp["h0"], c0=inp["c0"], bf16_weights=False)
    errs = {n: _rel(g, r) for n, g, r in zip(("y", "h_n", "c_n"), got, ref) if g is not None}
    print(f"{spec.name}: relative error of the bf16 conversion vs the fp32 model {errs}")
    assert all(np.isfinite(e) for e in errs.values()), errs


CLIP = [
    # (spec, force_path, kernel expected in the profile, cell clip, projection clip)
    (wl.LSTM_T80.scaled(T=12, B=9, in_dim=24, hidden=70, c0_std=0.5, h0_std=0.5), 3,
     "recurrent_cluster", (-0.25, 0.3), None),
    (wl.LSTM_T80.scaled(T=12, B=9, in_dim=24, hidden=70, c0_std=0.5, h0_std=0.5), 1,
     "recurrent_simt", (-0.25, 0.3), None),
    (wl.LSTMP_2L.scaled(dtype="f32", T=9, B=7, in_dim=17, hidden=52, proj=12), 1,
     "recurrent_simt", (-0.2, 0.25), (-0.03, 0.04)),
    (wl.LSTM_T80.scaled(name="lstm_bf16", dtype="bf16", T=12, B=150, in_dim=40, hidden=70,
                        h0_std=0.5, c0_std=0.5), 2, "recurrent_tc", (-0.25, 0.3), None),
    (wl.LSTMP_2L.scaled(T=9, B=130, in_dim=32, hidden=128, proj=64), 0,
     "recurrent_tc_lstmp", (-0.2, 0.25), None),
    (wl.LSTMP_2L.scaled(T=9, B=20, in_dim=32, hidden=128, proj=64), 0,
     "recurrent_simt", (-0.2, 0.25), (-0.05, 0.06)),
]


@pytest.mark.parametrize("spec,path,kernel,cc,pc", CLIP,
                         ids=lambda v: v.name if hasattr(v, "name") else None)
def test_clipping_parity(spec, path, kernel, cc, pc):
    """Cell-state / projection clipping on each recurrent kernel against the
    clipped oracle; the bounds are active (the unclipped result differs)."""
    inp = wl.make_rnn_inputs(spec, seed=31)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    if path:
        net.set_attr(binding.RCU_ATTR_FORCE_PATH, path)
    net.set_attr(binding.RCU_ATTR_PROFILE, 1)
    net.set_weights(inp["weights"])
    net.set_clip(binding.RCU_CLIP_CELL, cc)
    if pc is not None:
        net.set_clip(binding.RCU_CLIP_PROJ, pc)
    h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
    c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
    y, hn, cn = net.forward(inp["x"].to(dev), h0=h0, c0=c0)
    assert net.status() == 0
    torch.cuda.synchronize()
    assert kernel in net.profile()
    ref = oracle.rnn_forward(_cell(spec), inp["x"], inp["weights"], hidden=spec.hidden,
                             proj=spec.proj, h0=inp["h0"], c0=inp["c0"],
                             bf16_weights=spec.dtype == "bf16", cell_clip=cc, proj_clip=pc)
    unclipped = run_oracle(spec, inp)
    # the bounds bite: the clipped output differs by over 5 % of its range
    assert np.abs(ref[0] - unclipped[0]).max() > 0.05 * np.abs(unclipped[0]).max()
    compare(spec, (y.cpu().numpy(), hn.cpu().numpy(), cn.cpu().numpy()), ref)
    net.close()


def test_clip_argument_errors():
    gru = binding.RNN.from_spec(wl.GRU_3L.scaled(layers=1, T=2, B=2, in_dim=4, hidden=8))
    with pytest.raises(binding.RcuError) as e:
        gru.set_clip(binding.RCU_CLIP_CELL, (-1.0, 1.0))
    assert e.value.code == binding.RCU_ERR_UNSUPPORTED
    gru.close()
    lstm = binding.RNN.from_spec(wl.LSTM_T80.scaled(T=2, B=2, in_dim=4, hidden=8))
    with pytest.raises(binding.RcuError) as e:
        lstm.set_clip(binding.RCU_CLIP_PROJ, (-1.0, 1.0))
    assert e.value.code == binding.RCU_ERR_UNSUPPORTED
    with pytest.raises(binding.RcuError) as e:
        lstm.set_clip(binding.RCU_CLIP_CELL, (1.0, -1.0))
    assert e.value.code == binding.RCU_ERR_INVALID
    lstm.set_clip(binding.RCU_CLIP_CELL, None)  # off is always accepted
    lstm.close()


@pytest.mark.parametrize("ksplit", [1, 2, 4])
def test_barrier_timeout_on_tensor_core_path(ksplit):
    spec = wl.GRU_3L.scaled(layers=1, T=4, B=20, in_dim=16, hidden=128)
    inp = wl.make_rnn_inputs(spec, seed=14)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_attr(binding.RCU_ATTR_FORCE_PATH, 2)  # the grid-barrier kernel
    net.set_attr(binding.RCU_ATTR_TC_KSPLIT, ksplit)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_BARRIER_TIMEOUT_NS, 50_000_000)
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 1)
    net.forward(inp["x"].to(dev), h0=inp["h0"].to(dev))
    assert net.status() == binding.RCU_ERR_TIMEOUT
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 0)
    y, _, _ = net.forward(inp["x"].to(dev), h0=inp["h0"].to(dev))
    assert net.status() == 0
    ref = run_oracle(spec, inp)
    assert _rel(y.cpu().numpy(), ref[0]) <= BF16_REL
    net.close()


@pytest.mark.parametrize("dtype,B", [("f32", 9), ("f32", 300), ("bf16", 9)])
def test_backward_recurrence_timeout(dtype, B):
    """A CTA of the reverse-time kernel (FFMA for fp32: its CTA-pair K split
    at 9 rows, single CTAs at 300; tcgen05 for the bf16 GRU) skips its first
    step arrival: the bounded counter wait runs out, the status reads
    RCU_ERR_TIMEOUT, and the next backward on the same handle is correct."""
    spec = wl.GRU_3L.scaled(T=6, B=B, in_dim=16, hidden=24 if dtype == "f32" else 64, layers=2,
                            dtype=dtype)
    inp = wl.make_rnn_inputs(spec, seed=15)
    dy = torch.randn((spec.T, spec.B, spec.hidden), generator=torch.Generator().manual_seed(15))
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    net.set_attr(binding.RCU_ATTR_BARRIER_TIMEOUT_NS, 50_000_000)
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 2)
    net.backward(inp["x"].to(dev), dy.to(dev), h0=inp["h0"].to(dev))
    assert net.status() == binding.RCU_ERR_TIMEOUT
    net.set_attr(binding.RCU_ATTR_TEST_DROP_ARRIVAL, 0)
    dx, _, _, _ = net.backward(inp["x"].to(dev), dy.to(dev), h0=inp["h0"].to(dev))
    assert net.status() == 0
    ref = oracle.rnn_backward(oracle.GRU, inp["x"], inp["weights"], dy, hidden=spec.hidden,
                              h0=inp["h0"], bf16_weights=dtype == "bf16")
    # the backward parity bound of the tier
    assert _rel(dx.cpu().numpy(), ref["dx"]) <= (1e-4 if dtype == "f32" else BF16_REL)
    net.close()


def test_rssm_broadcast_timeout():
    """One CTA skips its first state broadcast: its cluster's bounded mbarrier
    waits run out, rssm_get_status reads RCU_ERR_TIMEOUT, and the next unroll
    on the same handle is correct."""
    spec = wl.RSSM_B50.scaled(T=4, B=9)
    inp = wl.make_rssm_inputs(spec, seed=16)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    binding.rssm_set_attr(m.h, binding.RCU_ATTR_BARRIER_TIMEOUT_NS, 50_000_000)
    binding.rssm_set_attr(m.h, binding.RCU_ATTR_TEST_DROP_ARRIVAL, 1)
    m.unroll(inp["actions"].to(dev), inp["eps"].to(dev))
    assert binding.rssm_get_status(m.h) == binding.RCU_ERR_TIMEOUT
    binding.rssm_set_attr(m.h, binding.RCU_ATTR_TEST_DROP_ARRIVAL, 0)
    outs = m.unroll(inp["actions"].to(dev), inp["eps"].to(dev))
    assert binding.rssm_get_status(m.h) == 0
    ref = oracle.rssm_unroll(inp["weights"], inp["actions"], inp["eps"])
    for o, r in zip(outs, ref):
        assert np.abs(o.cpu().numpy() - r).max() <= F32_TOL
    m.close()


def test_two_handles_two_threads():
    import threading
    spec_a = wl.LSTM_T80.scaled(T=7, B=3, in_dim=9, hidden=33)
    spec_b = wl.GRU_3L.scaled(dtype="f32", layers=1, T=5, B=4, in_dim=6, hidden=17)
    ia, ib = wl.make_rnn_inputs(spec_a, seed=12), wl.make_rnn_inputs(spec_b, seed=13)
    results = {}

    def work(name, spec, inp):
        with torch.cuda.stream(torch.cuda.Stream()):
            results[name] = run_gpu(spec, inp)

    ts = [threading.Thread(target=work, args=("a", spec_a, ia)),
          threading.Thread(target=work, args=("b", spec_b, ib))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    compare(spec_a, results["a"], run_oracle(spec_a, ia))
    compare(spec_b, results["b"], run_oracle(spec_b, ib))


# ----------------------------------------------------------------------------- RSSM

@pytest.mark.parametrize("spec", [
    wl.RSSM_B50,
    wl.RSSM_B50.scaled(T=7, B=3, state_dim=5, action_dim=0, hidden=33, rnn_hidden=17,
                       state0_std=1.0, belief0_std=0.5),
    wl.RSSM_B50.scaled(T=4, B=70, state_dim=30, action_dim=3, hidden=64, rnn_hidden=96),
    # 8 batch rows per cluster (the most): each lane of the shuffle-reduced
    # mat-vecs ends with several sums
    wl.RSSM_B50.scaled(T=5, B=130, state_dim=20, action_dim=6, hidden=100, rnn_hidden=60),
], ids=lambda s: f"T{s.T}-B{s.B}-S{s.state_dim}-H{s.hidden}-RH{s.rnn_hidden}")
def test_rssm_parity(spec):
    inp = wl.make_rssm_inputs(spec, seed=21)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    s0 = inp["state0"].to(dev) if inp["state0"] is not None else None
    b0 = inp["belief0"].to(dev) if inp["belief0"] is not None else None
    outs = m.unroll(inp["actions"].to(dev), inp["eps"].to(dev), s0, b0)
    assert binding.rssm_get_status(m.h) == 0
    ref = oracle.rssm_unroll(inp["weights"], inp["actions"], inp["eps"], state0=inp["state0"],
                             belief0=inp["belief0"])
    for name, o, r in zip(("means", "stds", "states", "beliefs"), outs, ref):
        e = float(np.abs(o.cpu().numpy() - r).max())
        assert e <= F32_TOL, f"{name}: max-abs error {e:.3e}"
    m.close()


@pytest.mark.parametrize("spec,hx", [
    (wl.RSSM_B50, 0),   # actor hidden width = the prior's hidden width
    (wl.RSSM_B50.scaled(T=9, B=70, state_dim=13, action_dim=5, hidden=72, rnn_hidden=40,
                        state0_std=1.0, belief0_std=0.5), 37),
    (wl.RSSM_B50.scaled(T=3, B=1, state_dim=4, action_dim=11, hidden=16, rnn_hidden=9), 3),
    # eight batch rows per cluster through the actor phases too
    (wl.RSSM_B50.scaled(T=4, B=130, state_dim=12, action_dim=4, hidden=48, rnn_hidden=40), 24),
], ids=lambda v: getattr(v, "name", f"hx{v}"))
def test_rssm_actor_parity(spec, hx):
    """Unroll variant 2: the actions come from the actor on the device and
    are fed back; every output and the actions match the oracle."""
    inp = wl.make_rssm_inputs(spec, seed=23)
    actor = wl.make_rssm_actor(spec, seed=23, actor_hidden=hx)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    m.set_actor(actor)
    s0 = inp["state0"].to(dev) if inp["state0"] is not None else None
    b0 = inp["belief0"].to(dev) if inp["belief0"] is not None else None
    outs = m.unroll_actor(inp["eps"].to(dev), s0, b0)
    assert binding.rssm_get_status(m.h) == 0
    assert m.launch_count() == 1
    ref = oracle.rssm_unroll_actor(inp["weights"], actor, inp["eps"], state0=inp["state0"],
                                   belief0=inp["belief0"])
    for name, o, r in zip(("means", "stds", "states", "beliefs", "actions"), outs, ref):
        e = float(np.abs(o.cpu().numpy() - r).max())
        assert e <= F32_TOL, f"{name}: max-abs error {e:.3e}"
    # the given-actions unroll of the same handle is unaffected by the actor
    got = m.unroll(outs[4], inp["eps"].to(dev), s0, b0)
    for o, r in zip(got, outs[:4]):
        assert float((o - r).abs().max()) <= F32_TOL
    m.close()


def test_rssm_actor_errors():
    spec = wl.RSSM_B50.scaled(T=2, B=2, state_dim=4, action_dim=3, hidden=8, rnn_hidden=8)
    inp = wl.make_rssm_inputs(spec, seed=1)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    with pytest.raises(RuntimeError, match="actor not set"):
        m.unroll_actor(inp["eps"].to(dev))
    # an actor wider than one cluster's shared memory holds
    big = wl.make_rssm_actor(spec, actor_hidden=40000)
    with pytest.raises(RuntimeError, match="shared memory"):
        m.set_actor(big)
    m.close()
    m0 = binding.RSSM(spec.state_dim, 0, spec.hidden, spec.rnn_hidden)
    m0.set_weights(wl.make_rssm_inputs(spec.scaled(action_dim=0), seed=1)["weights"])
    with pytest.raises(RuntimeError, match="action_dim"):
        m0.set_actor(wl.make_rssm_actor(spec.scaled(action_dim=1), actor_hidden=4))
    m0.close()


def test_metadata_reuse_across_calls():
    """One handle: fixed-length, variable-length, fixed-length again and another
    T: the fixed-length metadata kept between calls is rebuilt whenever it no
    longer describes the call, so every result matches the oracle."""
    spec = wl.BILSTM_VAR.scaled(T=9, B=6, in_dim=8, hidden=12, bidir=False, varlen=(2, 9))
    inp = wl.make_rnn_inputs(spec, seed=31)
    dev = torch.device("cuda")
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    x = inp["x"].to(dev)
    ref_fixed = oracle.rnn_forward(oracle.LSTM, inp["x"], inp["weights"], hidden=spec.hidden)
    ref_var = run_oracle(spec, inp)
    ref_short = oracle.rnn_forward(oracle.LSTM, inp["x"][:5], inp["weights"], hidden=spec.hidden)
    for kind in ("fixed", "var", "fixed", "fixed", "short", "fixed"):
        if kind == "var":
            y, hn, cn = net.forward(x, lengths=inp["lengths"].to(dev))
            ref = ref_var
        elif kind == "short":
            y, hn, cn = net.forward(x[:5].contiguous())
            ref = ref_short
        else:
            y, hn, cn = net.forward(x)
            ref = ref_fixed
        assert net.status() == 0
        e = np.abs(y.cpu().numpy() - ref[0]).max()
        assert e <= F32_TOL, f"{kind}: {e:.3e}"
        assert np.abs(hn.cpu().numpy() - ref[1]).max() <= F32_TOL
    net.close()


# ----------------------------------------------------------------------------- host-buffer entry points

HOST_SPECS = [
    wl.LSTM_T80.scaled(T=9, B=3, in_dim=20, hidden=24, h0_std=0.5, c0_std=0.5),
    wl.GRU_3L.scaled(T=6, B=130, in_dim=72, hidden=64, layers=2),
    wl.BILSTM_VAR.scaled(T=11, B=7, in_dim=16, hidden=40, varlen=(1, 11)),
    wl.LSTMP_2L.scaled(T=7, B=5, in_dim=24, hidden=64, proj=16),
]


def _host_inputs(spec, inp, pinned):
    def h(t, dtype=torch.float32):
        if t is None:
            return None
        t = t.to(dtype).contiguous()
        return t.pin_memory() if pinned else t.clone()
    return h(inp["x"]), h(inp["lengths"], torch.int32), h(inp["h0"]), h(inp["c0"])


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("spec", HOST_SPECS, ids=lambda s: s.name)
def test_forward_host_equals_device(spec, pinned):
    """rnn_forward_host runs the same kernels as rnn_forward: with pinned
    buffers x is read and y written in place over the CPU-GPU link, with
    pageable ones both are staged.  Outputs are bit-identical."""
    inp = wl.make_rnn_inputs(spec, seed=5)
    ref = run_gpu(spec, inp)
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    x, L, h0, c0 = _host_inputs(spec, inp, pinned)
    LD = spec.layers * spec.D

    def out(*shape):
        t = torch.full(shape, float("nan"))
        return t.pin_memory() if pinned else t
    y = out(spec.T, spec.B, spec.D * spec.Hout)
    hn = out(LD, spec.B, spec.Hout)
    cn = out(LD, spec.B, spec.hidden) if spec.cell == "lstm" else None
    binding.rnn_forward_host(net.h, spec.T, spec.B, x, L, h0, c0, y, hn, cn)
    torch.cuda.synchronize()
    assert net.status() == 0
    assert np.array_equal(y.numpy(), ref[0])
    assert np.array_equal(hn.numpy(), ref[1])
    if cn is not None:
        assert np.array_equal(cn.numpy(), ref[2])
    net.close()


def test_forward_host_single_step_and_tiny_batch():
    """T = 1 (one chunk whatever the attribute) and B = 1 through the host call."""
    for spec in (HOST_SPECS[1].scaled(T=1, B=1), HOST_SPECS[0].scaled(T=1, B=2)):
        inp = wl.make_rnn_inputs(spec, seed=8)
        ref = run_gpu(spec, inp)
        net = binding.RNN.from_spec(spec)
        net.set_attr(binding.RCU_ATTR_HOST_CHUNKS, 4)
        net.set_weights(inp["weights"])
        x, L, h0, c0 = _host_inputs(spec, inp, True)
        LD = spec.layers * spec.D
        y = torch.empty((spec.T, spec.B, spec.D * spec.Hout)).pin_memory()
        hn = torch.empty((LD, spec.B, spec.Hout)).pin_memory()
        cn = torch.empty((LD, spec.B, spec.hidden)).pin_memory() if spec.cell == "lstm" else None
        binding.rnn_forward_host(net.h, spec.T, spec.B, x, L, h0, c0, y, hn, cn)
        torch.cuda.synchronize()
        assert net.status() == 0
        assert np.array_equal(y.numpy(), ref[0]) and np.array_equal(hn.numpy(), ref[1])
        net.close()


@pytest.mark.parametrize("chunks", [2, 3, 16])
@pytest.mark.parametrize("spec", [HOST_SPECS[1], HOST_SPECS[0], HOST_SPECS[3],
                                  HOST_SPECS[2]], ids=lambda s: s.name)
def test_forward_host_chunked_equals_device(spec, chunks):
    """The chunked host pipeline (each chunk a forward of all layers from the
    fp32 state the previous chunk left) gives the unchunked results: exactly
    on the bf16 path, whose GEMM rows do not depend on the chunk size, and to
    fp32 rounding on the fp32 path.  Bidirectional, varlen and projected
    networks take the unchunked path whatever the attribute says."""
    spec = spec.scaled(T=11) if spec.varlen is None else spec
    inp = wl.make_rnn_inputs(spec, seed=6)
    ref = run_gpu(spec, inp)
    net = binding.RNN.from_spec(spec)
    net.set_attr(binding.RCU_ATTR_HOST_CHUNKS, chunks)
    net.set_weights(inp["weights"])
    x, L, h0, c0 = _host_inputs(spec, inp, True)
    LD = spec.layers * spec.D
    y = torch.full((spec.T, spec.B, spec.D * spec.Hout), float("nan")).pin_memory()
    hn = torch.full((LD, spec.B, spec.Hout), float("nan")).pin_memory()
    cn = torch.full((LD, spec.B, spec.hidden), float("nan")).pin_memory() \
        if spec.cell == "lstm" else None
    binding.rnn_forward_host(net.h, spec.T, spec.B, x, L, h0, c0, y, hn, cn)
    torch.cuda.synchronize()
    assert net.status() == 0
    got = [y.numpy(), hn.numpy()] + ([cn.numpy()] if cn is not None else [])
    for g, r in zip(got, ref):
        if spec.dtype == "bf16":
            assert np.array_equal(g, r)
        else:
            assert np.abs(g - r).max() <= 1e-5
    net.close()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_rssm_host_equals_device(pinned):
    spec = wl.RSSM_B50.scaled(T=5, B=11, state0_std=1.0, belief0_std=0.5)
    inp = wl.make_rssm_inputs(spec, seed=9)
    actor = wl.make_rssm_actor(spec, seed=9, actor_hidden=24)
    dev = torch.device("cuda")
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"])
    m.set_actor(actor)
    s0, b0 = inp["state0"], inp["belief0"]
    ref = m.unroll(inp["actions"].to(dev), inp["eps"].to(dev), s0.to(dev), b0.to(dev))
    ref_a = m.unroll_actor(inp["eps"].to(dev), s0.to(dev), b0.to(dev))

    def out(w):
        t = torch.full((spec.T, spec.B, w), float("nan"))
        return t.pin_memory() if pinned else t
    S, RH, A = spec.state_dim, spec.rnn_hidden, spec.action_dim
    got = [out(S), out(S), out(S), out(RH)]
    binding.rssm_unroll_host(m.h, spec.T, spec.B, s0, b0, inp["actions"], inp["eps"], *got)
    got_a = [out(S), out(S), out(S), out(RH), out(A)]
    binding.rssm_unroll_actor_host(m.h, spec.T, spec.B, s0, b0, inp["eps"], *got_a)
    torch.cuda.synchronize()
    assert binding.rssm_get_status(m.h) == 0
    for g, r in zip(got, ref):
        assert torch.equal(g, r.cpu())
    for g, r in zip(got_a, ref_a):
        assert torch.equal(g, r.cpu())
    m.close()


def test_forward_host_rejects_device_tensors():
    spec = HOST_SPECS[0]
    inp = wl.make_rnn_inputs(spec, seed=5)
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    y = torch.empty((spec.T, spec.B, spec.Hout))
    with pytest.raises(ValueError, match="host tensors"):
        binding.rnn_forward_host(net.h, spec.T, spec.B, inp["x"].cuda(), None, None, None, y,
                                 None, None)
    net.close()


# ----------------------------------------------------------------------------- full-size workloads

# Rows checked at full size (sorted order = original order without lengths).
# GRU, B = 256: TMEM lanes 0, 31, 32, 63, 64, 95, 96, 127 of the first
# 128-row batch group, the 127/128 group boundary and lanes of the second
# group.  LSTMP, B = 32 (one group, 32 live lanes): 16 rows spread over it.
# BiLSTM: every row whose length ties another's (the stable sort decides
# their order), the longest and the shortest, and evenly spaced rows.
FULL = [
    (wl.LSTMP_2L, [0, 1, 2, 5, 8, 11, 13, 15, 16, 19, 22, 24, 27, 29, 30, 31]),
    (wl.BILSTM_VAR, None),
    (wl.GRU_3L, [0, 1, 31, 32, 63, 64, 95, 96, 126, 127, 128, 129, 159, 191, 224, 255]),
]


def full_size_rows(inp, B, n=16):
    L = inp["lengths"].numpy()
    vals, counts = np.unique(L, return_counts=True)
    ties = [int(b) for b in range(B) if counts[np.searchsorted(vals, L[b])] > 1]
    rows = set(ties) | {int(np.argmax(L)), int(np.argmin(L))}
    for b in np.linspace(0, B - 1, n).astype(int):
        if len(rows) >= max(n, len(ties) + 2):
            break
        rows.add(int(b))
    return sorted(rows)


def per_element_report(spec, got, ref, rows):
    """Per-element error statistics of the sampled rows: the largest
    |gpu - ref| / |ref| over elements with |ref| >= 10 % of their row's
    max|ref|, and that row-normalised error's maximum (bf16)."""
    out = {}
    for name, g, r in (("y", got[0][:, rows], ref[0][:, rows]),):
        big = np.abs(r) >= 0.1 * np.abs(r).max(axis=(0, 2), keepdims=True)
        rel = np.abs(g - r)[big] / np.abs(r)[big]
        rowmax = np.abs(r).max(axis=(0, 2), keepdims=True)
        out[name] = {"max_rel_large_elems": float(rel.max()),
                     "p999_rel_large_elems": float(np.quantile(rel, 0.999)),
                     "max_row_normalised": float((np.abs(g - r) / np.maximum(rowmax, 1e-30)).max())}
    return out


@pytest.mark.parametrize("spec,rows", FULL, ids=lambda v: getattr(v, "name", "rows"))
def test_full_size_sampled_rows(spec, rows):
    inp = wl.make_rnn_inputs(spec, seed=0)
    if rows is None:
        rows = full_size_rows(inp, spec.B)
        assert len(rows) >= 16
    got = run_gpu(spec, inp)
    ref = run_oracle(spec, inp, rows=rows)
    compare(spec, got, ref, rows=rows)
    if spec.dtype == "bf16":
        # each sampled row against its own max|ref| (a bad row cannot hide
        # behind a larger one); per-element statistics are printed
        rep = per_element_report(spec, got, ref, rows)
        print(f"\n{spec.name} per-element error over {len(rows)} rows: {rep}")
        assert rep["y"]["max_row_normalised"] <= BF16_REL, rep
    if spec.varlen is not None:
        L = inp["lengths"].numpy()
        for b in range(spec.B):
            assert np.all(got[0][L[b]:, b] == 0.0)
