"""Pins for the CPU oracle: it is checked against things other than itself.

- closed forms (zero weights, saturated gates) derived from the cell equations;
- an independent library evaluation (torch float64 on CPU: nn.LSTM with
  proj_size, nn.GRU, nn.GRUCell, pack_padded_sequence) of the modules the
  pages name (pytorch/rl issue 366 Solution; pytorch/pytorch issue 46213);
- invariants (layer composition, reversal for the backward direction,
  packed == per-sequence, batch permutation, identity projection);
- a separately written scalar evaluation on tiny inputs;
- hand-worked golden fixtures under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from recurrent_cell_unroll_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _zero_weights(cell, layers, in_dim, H, D=1, proj=0):
    nG = 4 if cell == oracle.LSTM else 3
    Hout = proj or H
    ws = []
    for layer in range(layers):
        in_w = in_dim if layer == 0 else D * Hout
        for _ in range(D):
            ws.append({"w_ih": np.zeros((nG * H, in_w), np.float32),
                       "w_hh": np.zeros((nG * H, Hout), np.float32),
                       "b_ih": None, "b_hh": None,
                       "w_hr": np.zeros((proj, H), np.float32) if proj else None})
    return ws


def _rand_weights(rng, cell, layers, in_dim, H, D=1, proj=0, scale=0.5):
    nG = 4 if cell == oracle.LSTM else 3
    Hout = proj or H
    ws = []
    for layer in range(layers):
        in_w = in_dim if layer == 0 else D * Hout
        for _ in range(D):
            ws.append({"w_ih": rng.uniform(-scale, scale, (nG * H, in_w)).astype(np.float32),
                       "w_hh": rng.uniform(-scale, scale, (nG * H, Hout)).astype(np.float32),
                       "b_ih": rng.uniform(-scale, scale, nG * H).astype(np.float32),
                       "b_hh": rng.uniform(-scale, scale, nG * H).astype(np.float32),
                       "w_hr": rng.uniform(-scale, scale, (proj, H)).astype(np.float32)
                       if proj else None})
    return ws


# --------------------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_library():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                        # exact ties: low 16 bits 0x8000, both parities of bit 16
                        np.array([0x3f808000, 0x3f818000, 0xbf808000, 0x40490fdb, 0x00018000],
                                 dtype=np.uint32).view(np.float32)])
    ours = oracle.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_weights_flag_equals_prerounded_weights():
    rng = np.random.default_rng(2)
    ws = _rand_weights(rng, oracle.LSTM, 1, 5, 4, proj=3)
    x = rng.standard_normal((6, 2, 5)).astype(np.float32)
    y1, h1, c1 = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=4, proj=3, bf16_weights=True)
    pre = [{k: (None if v is None or k.startswith("b_") else
                torch.from_numpy(v).to(torch.bfloat16).float().numpy()) if k != "b_ih" and k != "b_hh"
            else v for k, v in w.items()} for w in ws]
    y2, h2, c2 = oracle.rnn_forward(oracle.LSTM, x, pre, hidden=4, proj=3)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2) and np.array_equal(c1, c2)
    # and rounding really changes something
    y3, _, _ = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=4, proj=3)
    assert not np.array_equal(y1, y3)


# --------------------------------------------------------------------------- closed forms

def test_lstm_zero_weights_closed_form():
    """Zero weights: i=f=o=1/2, g=0, so c_t = 2^-t c0 and h_t = tanh(c_t)/2."""
    T, B, H = 6, 3, 4
    rng = np.random.default_rng(3)
    x = rng.standard_normal((T, B, 2)).astype(np.float32)
    h0 = rng.standard_normal((1, B, H)).astype(np.float32)
    c0 = rng.standard_normal((1, B, H)).astype(np.float32)
    y, hn, cn = oracle.rnn_forward(oracle.LSTM, x, _zero_weights(oracle.LSTM, 1, 2, H),
                                   hidden=H, h0=h0, c0=c0)
    for t in range(T):
        c_t = c0[0].astype(np.float64) * 2.0 ** -(t + 1)
        np.testing.assert_allclose(y[t], 0.5 * np.tanh(c_t), rtol=0, atol=1e-15)
    np.testing.assert_allclose(cn[0], c0[0] * 2.0 ** -T, rtol=0, atol=1e-15)


def test_lstm_saturated_forget_keeps_cell():
    """b_f = +40, b_i = -40: f = 1, i = 0 to double precision, so c_t = c0."""
    T, B, H, I = 7, 2, 3, 4
    rng = np.random.default_rng(4)
    ws = _rand_weights(rng, oracle.LSTM, 1, I, H, scale=0.3)
    ws[0]["b_ih"][0:H] = -40.0
    ws[0]["b_ih"][H:2 * H] = 40.0
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    c0 = rng.standard_normal((1, B, H)).astype(np.float32)
    _, _, cn = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, c0=c0)
    np.testing.assert_allclose(cn[0], c0[0], rtol=0, atol=1e-15)


def test_lstm_input_path_only():
    """W_hh = 0, i = o = 1, f = 0: h_t = tanh(tanh(W_ig x_t + b_ig + b_hg))."""
    T, B, H, I = 5, 2, 3, 4
    rng = np.random.default_rng(5)
    ws = _rand_weights(rng, oracle.LSTM, 1, I, H)
    ws[0]["w_hh"][:] = 0
    ws[0]["b_ih"][0:H] = 40.0
    ws[0]["b_ih"][H:2 * H] = -40.0
    ws[0]["b_ih"][3 * H:4 * H] = 40.0
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    y, _, _ = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H)
    Wg = ws[0]["w_ih"][2 * H:3 * H].astype(np.float64)
    bg = ws[0]["b_ih"][2 * H:3 * H].astype(np.float64) + ws[0]["b_hh"][2 * H:3 * H]
    expect = np.tanh(np.tanh(np.einsum("hk,tbk->tbh", Wg, x.astype(np.float64)) + bg))
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-14)


def test_gru_zero_weights_closed_form():
    """Zero weights: r = z = 1/2, n = 0, so h_t = 2^-t h0."""
    T, B, H = 6, 3, 5
    rng = np.random.default_rng(6)
    x = rng.standard_normal((T, B, 2)).astype(np.float32)
    h0 = rng.standard_normal((1, B, H)).astype(np.float32)
    y, hn, _ = oracle.rnn_forward(oracle.GRU, x, _zero_weights(oracle.GRU, 1, 2, H),
                                  hidden=H, h0=h0)
    for t in range(T):
        np.testing.assert_allclose(y[t], h0[0] * 2.0 ** -(t + 1), rtol=0, atol=1e-15)


def test_gru_update_gate_limits():
    """z -> 1 keeps h0 exactly; z -> 0 gives h_t = n_t."""
    T, B, H, I = 4, 2, 3, 2
    rng = np.random.default_rng(7)
    ws = _rand_weights(rng, oracle.GRU, 1, I, H, scale=0.3)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    h0 = rng.standard_normal((1, B, H)).astype(np.float32)
    ws[0]["b_ih"][H:2 * H] = 40.0
    y, _, _ = oracle.rnn_forward(oracle.GRU, x, ws, hidden=H, h0=h0)
    for t in range(T):
        np.testing.assert_allclose(y[t], h0[0], rtol=0, atol=1e-15)
    # z -> 0 and W_hh = 0: h_t = tanh(W_in x_t + b_in + r * b_hn), r = sigma(W_ir x + b_ir + b_hr)
    ws[0]["b_ih"][H:2 * H] = -40.0
    ws[0]["w_hh"][:] = 0
    y, _, _ = oracle.rnn_forward(oracle.GRU, x, ws, hidden=H, h0=h0)
    xd = x.astype(np.float64)
    Wi, bi, bh = ws[0]["w_ih"].astype(np.float64), ws[0]["b_ih"], ws[0]["b_hh"]
    r = 1 / (1 + np.exp(-(xd @ Wi[0:H].T + bi[0:H] + bh[0:H])))
    n = np.tanh(xd @ Wi[2 * H:].T + bi[2 * H:] + r * bh[2 * H:])
    np.testing.assert_allclose(y, n, rtol=0, atol=1e-14)


def test_lstm_one_step_by_hand():
    """H = 1, in = 1, T = 1 with simple numbers, evaluated step by step."""
    w = {"w_ih": np.array([[0.5], [-0.25], [1.0], [0.75]], np.float32),
         "w_hh": np.array([[0.125], [0.25], [-0.5], [1.0]], np.float32),
         "b_ih": np.array([0.0, 1.0, 0.0, -0.5], np.float32),
         "b_hh": np.array([0.25, 0.0, 0.5, 0.0], np.float32), "w_hr": None}
    x = np.array([[[2.0]]], np.float32)
    h0 = np.array([[[0.5]]], np.float32)
    c0 = np.array([[[-1.0]]], np.float32)
    y, hn, cn = oracle.rnn_forward(oracle.LSTM, x, [w], hidden=1, h0=h0, c0=c0)
    s = lambda v: 1.0 / (1.0 + math.exp(-v))
    i = s(0.5 * 2 + 0.125 * 0.5 + 0.25)        # 1.3125
    f = s(-0.25 * 2 + 0.25 * 0.5 + 1.0)        # 0.625
    g = math.tanh(1.0 * 2 - 0.5 * 0.5 + 0.5)   # 2.25
    o = s(0.75 * 2 + 1.0 * 0.5 - 0.5)          # 1.5
    c = f * -1.0 + i * g
    assert abs(cn[0, 0, 0] - c) < 1e-15
    assert abs(y[0, 0, 0] - o * math.tanh(c)) < 1e-15


# --------------------------------------------------------------------------- library cross-check

def _torch_rnn(cell, ws, x, H, proj, D, layers, lengths, h0, c0):
    in_dim = x.shape[2]
    kw = dict(input_size=in_dim, hidden_size=H, num_layers=layers, bidirectional=D == 2,
              dtype=torch.float64)
    mod = torch.nn.LSTM(proj_size=proj, **kw) if cell == oracle.LSTM else torch.nn.GRU(**kw)
    with torch.no_grad():
        for layer in range(layers):
            for d in range(D):
                sfx = f"_l{layer}" + ("_reverse" if d else "")
                w = ws[layer * D + d]
                getattr(mod, "weight_ih" + sfx).copy_(torch.from_numpy(w["w_ih"]).double())
                getattr(mod, "weight_hh" + sfx).copy_(torch.from_numpy(w["w_hh"]).double())
                getattr(mod, "bias_ih" + sfx).copy_(torch.from_numpy(w["b_ih"]).double())
                getattr(mod, "bias_hh" + sfx).copy_(torch.from_numpy(w["b_hh"]).double())
                if proj:
                    getattr(mod, "weight_hr" + sfx).copy_(torch.from_numpy(w["w_hr"]).double())
        xt = torch.from_numpy(x).double()
        Hout = proj or H
        B = x.shape[1]
        hz = torch.zeros(layers * D, B, Hout, dtype=torch.float64) if h0 is None else \
            torch.from_numpy(h0).double()
        cz = torch.zeros(layers * D, B, H, dtype=torch.float64) if c0 is None else \
            torch.from_numpy(c0).double()
        state = (hz, cz) if cell == oracle.LSTM else hz
        if lengths is not None:
            packed = torch.nn.utils.rnn.pack_padded_sequence(
                xt, torch.from_numpy(lengths).long(), enforce_sorted=False)
            out, st = mod(packed, state)
            y, _ = torch.nn.utils.rnn.pad_packed_sequence(out, total_length=x.shape[0])
        else:
            y, st = mod(xt, state)
    if cell == oracle.LSTM:
        return y.numpy(), st[0].numpy(), st[1].numpy()
    return y.numpy(), st.numpy(), None


@pytest.mark.parametrize("cell,proj,D,layers,varlen", [
    (oracle.LSTM, 0, 1, 1, False),
    (oracle.LSTM, 0, 2, 2, True),
    (oracle.LSTM, 3, 1, 2, False),
    (oracle.LSTM, 3, 2, 1, True),
    (oracle.GRU, 0, 1, 3, False),
    (oracle.GRU, 0, 2, 2, True),
])
def test_against_torch_float64(cell, proj, D, layers, varlen):
    rng = np.random.default_rng(10 + layers + 3 * D + proj)
    T, B, I, H = 7, 5, 4, 6
    ws = _rand_weights(rng, cell, layers, I, H, D=D, proj=proj)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    Hout = proj or H
    h0 = rng.standard_normal((layers * D, B, Hout)).astype(np.float32)
    c0 = rng.standard_normal((layers * D, B, H)).astype(np.float32)
    lengths = rng.integers(1, T + 1, B).astype(np.int32) if varlen else None
    if varlen:
        lengths[0] = T
    y, hn, cn = oracle.rnn_forward(cell, x, ws, hidden=H, proj=proj, bidirectional=D == 2,
                                   lengths=lengths, h0=h0, c0=c0 if cell == oracle.LSTM else None)
    ty, thn, tcn = _torch_rnn(cell, ws, x, H, proj, D, layers, lengths, h0,
                              c0 if cell == oracle.LSTM else None)
    np.testing.assert_allclose(y, ty, rtol=0, atol=1e-12)
    np.testing.assert_allclose(hn, thn, rtol=0, atol=1e-12)
    if cell == oracle.LSTM:
        np.testing.assert_allclose(cn, tcn, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- invariants

def test_identity_projection_equals_plain_lstm():
    rng = np.random.default_rng(20)
    T, B, I, H = 6, 3, 4, 5
    ws = _rand_weights(rng, oracle.LSTM, 2, I, H, proj=H)
    for w in ws:
        w["w_hr"] = np.eye(H, dtype=np.float32)
    plain = [{k: (None if k == "w_hr" else v) for k, v in w.items()} for w in ws]
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    y1, h1, c1 = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, proj=H)
    y2, h2, c2 = oracle.rnn_forward(oracle.LSTM, x, plain, hidden=H)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2) and np.array_equal(c1, c2)


@pytest.mark.parametrize("cell", [oracle.LSTM, oracle.GRU])
def test_layers_compose(cell):
    rng = np.random.default_rng(21)
    T, B, I, H = 5, 3, 4, 6
    ws = _rand_weights(rng, cell, 2, I, H, D=2)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    y, hn, cn = oracle.rnn_forward(cell, x, ws, hidden=H, bidirectional=True)
    y1, hn1, cn1 = oracle.rnn_forward(cell, x, ws[:2], hidden=H, bidirectional=True)
    # layer 2 sees layer 1's output; round-trip via float32 is exact only in fp64, so
    # compare layer 2 run on the float64 output cast to fp32 with a loose bound
    y2, hn2, _ = oracle.rnn_forward(cell, y1.astype(np.float32), ws[2:], hidden=H,
                                    bidirectional=True)
    np.testing.assert_allclose(hn[:2], hn1, rtol=0, atol=0)
    np.testing.assert_allclose(y, y2, rtol=0, atol=1e-6)
    np.testing.assert_allclose(hn[2:], hn2, rtol=0, atol=1e-6)


@pytest.mark.parametrize("cell", [oracle.LSTM, oracle.GRU])
def test_backward_direction_is_reversed_forward(cell):
    rng = np.random.default_rng(22)
    T, B, I, H = 6, 4, 3, 5
    ws = _rand_weights(rng, cell, 1, I, H, D=2)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    lengths = np.array([6, 3, 5, 1], np.int32)
    y, hn, _ = oracle.rnn_forward(cell, x, ws, hidden=H, bidirectional=True, lengths=lengths)
    for b in range(B):
        L = lengths[b]
        xr = x[:L, b:b + 1][::-1].copy()
        yr, hr, _ = oracle.rnn_forward(cell, xr, [ws[1]], hidden=H)
        np.testing.assert_array_equal(y[:L, b, H:], yr[::-1, 0])
        np.testing.assert_array_equal(hn[1, b], hr[0, 0])
        yf, hf, _ = oracle.rnn_forward(cell, x[:L, b:b + 1], [ws[0]], hidden=H)
        np.testing.assert_array_equal(y[:L, b, :H], yf[:, 0])
        np.testing.assert_array_equal(hn[0, b], hf[0, 0])
        assert np.all(y[L:, b] == 0)


@pytest.mark.parametrize("cell,proj", [(oracle.LSTM, 0), (oracle.LSTM, 2), (oracle.GRU, 0)])
def test_varlen_equals_per_sequence(cell, proj):
    rng = np.random.default_rng(23)
    T, B, I, H = 8, 5, 3, 4
    ws = _rand_weights(rng, cell, 2, I, H, proj=proj)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    lengths = np.array([8, 2, 5, 5, 1], np.int32)
    y, hn, cn = oracle.rnn_forward(cell, x, ws, hidden=H, proj=proj, lengths=lengths)
    for b in range(B):
        L = lengths[b]
        yb, hb, cb = oracle.rnn_forward(cell, x[:L, b:b + 1], ws, hidden=H, proj=proj)
        np.testing.assert_array_equal(y[:L, b], yb[:, 0])
        np.testing.assert_array_equal(hn[:, b], hb[:, 0])
        if cn is not None:
            np.testing.assert_array_equal(cn[:, b], cb[:, 0])
        assert np.all(y[L:, b] == 0)


def test_batch_permutation_and_row_subset():
    rng = np.random.default_rng(24)
    T, B, I, H = 5, 6, 3, 4
    ws = _rand_weights(rng, oracle.GRU, 2, I, H, D=2)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    h0 = rng.standard_normal((4, B, H)).astype(np.float32)
    lengths = np.array([5, 1, 3, 3, 4, 2], np.int32)
    y, hn, _ = oracle.rnn_forward(oracle.GRU, x, ws, hidden=H, bidirectional=True,
                                  lengths=lengths, h0=h0)
    perm = rng.permutation(B)
    yp, hnp, _ = oracle.rnn_forward(oracle.GRU, x[:, perm], ws, hidden=H, bidirectional=True,
                                    lengths=lengths[perm], h0=h0[:, perm])
    np.testing.assert_array_equal(yp, y[:, perm])
    np.testing.assert_array_equal(hnp, hn[:, perm])
    ys, hs, _ = oracle.rnn_forward(oracle.GRU, x, ws, hidden=H, bidirectional=True,
                                   lengths=lengths, h0=h0, rows=[4, 1])
    np.testing.assert_array_equal(ys[:, [4, 1]], y[:, [4, 1]])
    np.testing.assert_array_equal(hs[:, [4, 1]], hn[:, [4, 1]])


# --------------------------------------------------------------------------- separately written scalar loops

def _scalar_lstm(w, xs, h, c, proj, cell_clip=None, proj_clip=None):
    """Independent scalar evaluation of one LSTM(P) direction over a list of steps.
    cell_clip / proj_clip: (lo, hi) bounds applied to c_t and to h_t = W_hr m_t."""
    H = len(c)
    out = []
    for xv in xs:
        def row(r):
            v = float(w["b_ih"][r]) + float(w["b_hh"][r])
            v += sum(float(w["w_ih"][r][k]) * xv[k] for k in range(len(xv)))
            v += sum(float(w["w_hh"][r][k]) * h[k] for k in range(len(h)))
            return v
        sg = lambda v: 1.0 / (1.0 + math.exp(-v))
        m = []
        newc = []
        for j in range(H):
            ig, fg, gg, og = sg(row(j)), sg(row(H + j)), math.tanh(row(2 * H + j)), sg(row(3 * H + j))
            cj = fg * c[j] + ig * gg
            if cell_clip is not None:
                cj = min(max(cj, cell_clip[0]), cell_clip[1])
            newc.append(cj)
            m.append(og * math.tanh(cj))
        c = newc
        if proj:
            h = [sum(float(w["w_hr"][p][j]) * m[j] for j in range(H)) for p in range(proj)]
            if proj_clip is not None:
                h = [min(max(v, proj_clip[0]), proj_clip[1]) for v in h]
        else:
            h = m
        out.append(list(h))
    return out, h, c


def _scalar_gru(w, xs, h):
    H = len(h)
    out = []
    for xv in xs:
        def dot(mat, r, vec):
            return sum(float(mat[r][k]) * vec[k] for k in range(len(vec)))
        sg = lambda v: 1.0 / (1.0 + math.exp(-v))
        new = []
        for j in range(H):
            r = sg(dot(w["w_ih"], j, xv) + float(w["b_ih"][j]) + dot(w["w_hh"], j, h) + float(w["b_hh"][j]))
            z = sg(dot(w["w_ih"], H + j, xv) + float(w["b_ih"][H + j]) + dot(w["w_hh"], H + j, h)
                   + float(w["b_hh"][H + j]))
            n = math.tanh(dot(w["w_ih"], 2 * H + j, xv) + float(w["b_ih"][2 * H + j])
                          + r * (dot(w["w_hh"], 2 * H + j, h) + float(w["b_hh"][2 * H + j])))
            new.append((1 - z) * n + z * h[j])
        h = new
        out.append(list(h))
    return out, h


@pytest.mark.parametrize("cell,proj", [(oracle.LSTM, 0), (oracle.LSTM, 2), (oracle.GRU, 0)])
def test_tiny_scalar_bruteforce(cell, proj):
    rng = np.random.default_rng(30 + proj)
    T, B, I, H = 4, 2, 2, 3
    ws = _rand_weights(rng, cell, 1, I, H, proj=proj)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    Hout = proj or H
    h0 = rng.standard_normal((1, B, Hout)).astype(np.float32)
    c0 = rng.standard_normal((1, B, H)).astype(np.float32)
    y, hn, cn = oracle.rnn_forward(cell, x, ws, hidden=H, proj=proj, h0=h0,
                                   c0=c0 if cell == oracle.LSTM else None)
    for b in range(B):
        xs = [[float(v) for v in x[t, b]] for t in range(T)]
        if cell == oracle.LSTM:
            out, h, c = _scalar_lstm(ws[0], xs, [float(v) for v in h0[0, b]],
                                     [float(v) for v in c0[0, b]], proj)
            np.testing.assert_allclose(cn[0, b], c, rtol=0, atol=1e-13)
        else:
            out, h = _scalar_gru(ws[0], xs, [float(v) for v in h0[0, b]])
        np.testing.assert_allclose(y[:, b], np.array(out), rtol=0, atol=1e-13)
        np.testing.assert_allclose(hn[0, b], h, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- clipping
# Cell-state and projection clipping (cuDNN 7.2 options discussed in "RNN Op
# Changes", apache/mxnet issue 9543): c_t is clamped as soon as it is updated,
# the projected h_t as soon as it is formed.

@pytest.mark.parametrize("proj", [0, 2])
def test_clipped_tiny_scalar_bruteforce(proj):
    rng = np.random.default_rng(41 + proj)
    T, B, I, H = 5, 3, 2, 3
    ws = _rand_weights(rng, oracle.LSTM, 1, I, H, proj=proj, scale=1.5)
    x = rng.standard_normal((T, B, I)).astype(np.float32)
    Hout = proj or H
    h0 = rng.standard_normal((1, B, Hout)).astype(np.float32)
    c0 = rng.standard_normal((1, B, H)).astype(np.float32)
    cc, pc = (-0.3, 0.4), ((-0.2, 0.25) if proj else None)
    y, hn, cn = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, proj=proj, h0=h0, c0=c0,
                                   cell_clip=cc, proj_clip=pc)
    y0, _, _ = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, proj=proj, h0=h0, c0=c0)
    assert np.abs(y - y0).max() > 1e-3  # the bounds are active
    for b in range(B):
        xs = [[float(v) for v in x[t, b]] for t in range(T)]
        out, h, c = _scalar_lstm(ws[0], xs, [float(v) for v in h0[0, b]],
                                 [float(v) for v in c0[0, b]], proj, cc, pc)
        np.testing.assert_allclose(y[:, b], np.array(out), rtol=0, atol=1e-13)
        np.testing.assert_allclose(hn[0, b], h, rtol=0, atol=1e-13)
        np.testing.assert_allclose(cn[0, b], c, rtol=0, atol=1e-13)


def test_cell_clip_saturated_closed_form():
    """i = f = o = 1 (bias +40), W = 0: c_t = c_{t-1} + tanh(b_g) grows linearly,
    so the clipped cell is clamp(t * tanh(b_g), lo, hi) and h_t = tanh(c_t)."""
    H, T = 3, 8
    ws = _zero_weights(oracle.LSTM, 1, 2, H)
    bg = np.array([0.5, -0.5, 0.2], np.float32)
    b = np.concatenate([np.full(H, 40, np.float32), np.full(H, 40, np.float32), bg,
                        np.full(H, 40, np.float32)])
    ws[0]["b_ih"] = b
    x = np.zeros((T, 1, 2), np.float32)
    lo, hi = -0.6, 0.9
    y, hn, cn = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, cell_clip=(lo, hi))
    g = np.tanh(bg.astype(np.float64))
    for t in range(T):
        c = np.clip((t + 1) * g, lo, hi)
        np.testing.assert_allclose(y[t, 0], np.tanh(c), rtol=0, atol=1e-14)
    np.testing.assert_allclose(cn[0, 0], np.clip(T * g, lo, hi), rtol=0, atol=1e-14)


def test_proj_clip_closed_form():
    """Same saturated cell with P = H and W_hr = 10 I: h_t = clamp(10 tanh(c_t), lo, hi)
    and nothing feeds back (W_hh = 0)."""
    H, T = 3, 6
    ws = _zero_weights(oracle.LSTM, 1, 2, H, proj=H)
    bg = np.array([0.05, -0.08, 0.02], np.float32)
    ws[0]["b_ih"] = np.concatenate([np.full(H, 40, np.float32), np.full(H, 40, np.float32), bg,
                                    np.full(H, 40, np.float32)])
    ws[0]["w_hr"] = (10 * np.eye(H)).astype(np.float32)
    x = np.zeros((T, 1, 2), np.float32)
    lo, hi = -0.5, 0.7
    y, hn, _ = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, proj=H, proj_clip=(lo, hi))
    g = np.tanh(bg.astype(np.float64))
    for t in range(T):
        np.testing.assert_allclose(y[t, 0], np.clip(10 * np.tanh((t + 1) * g), lo, hi),
                                   rtol=0, atol=1e-13)


def test_infinite_clip_equals_unclipped():
    rng = np.random.default_rng(47)
    ws = _rand_weights(rng, oracle.LSTM, 2, 3, 4, D=2, proj=2)
    x = rng.standard_normal((6, 3, 3)).astype(np.float32)
    inf = float("inf")
    a = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=4, proj=2, bidirectional=True)
    b = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=4, proj=2, bidirectional=True,
                           cell_clip=(-inf, inf), proj_clip=(-inf, inf))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# --------------------------------------------------------------------------- packing

def test_pack_golden_example():
    g = json.load(open(os.path.join(GOLDEN, "pack_example.json")))
    s, u, bs = oracle.pack(np.array(g["lengths"], np.int32), g["T"])
    assert s.tolist() == g["sorted_idx"]
    assert u.tolist() == g["unsorted_idx"]
    assert bs.tolist() == g["batch_sizes"]
    assert int(bs.sum()) == g["total"]


def test_pack_bruteforce_random():
    rng = np.random.default_rng(40)
    for trial in range(50):
        B = int(rng.integers(1, 70))
        T = int(rng.integers(1, 40))
        lengths = rng.integers(1, T + 1, B).astype(np.int32)
        s, u, bs = oracle.pack(lengths, T)
        expect = sorted(range(B), key=lambda b: (-int(lengths[b]), b))
        assert s.tolist() == expect
        assert all(u[s[i]] == i for i in range(B))
        assert int(bs.sum()) == int(lengths.sum())
        assert all(bs[t] >= bs[t + 1] for t in range(T - 1))
        assert bs[0] == B
        for t in range(T):
            assert bs[t] == int((lengths > t).sum())


def test_pack_rejects_bad_lengths():
    with pytest.raises(ValueError):
        oracle.pack(np.array([3, 0, 2], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.pack(np.array([3, 5, 2], np.int32), 4)


# --------------------------------------------------------------------------- RSSM

def _rssm_torch(w, actions, eps, state0, belief0):
    """The RSSM prior step assembled from torch float64 modules, as the page lays it out."""
    T, B, A = actions.shape
    S = eps.shape[2]
    Hd = w["W1"].shape[0]
    RH = w["W_hh"].shape[1]
    d = lambda a: torch.from_numpy(np.asarray(a)).double()
    lin1 = torch.nn.Linear(S + A, Hd, dtype=torch.float64)
    gru = torch.nn.GRUCell(Hd, RH, dtype=torch.float64)
    lin2 = torch.nn.Linear(RH, Hd, dtype=torch.float64)
    lin3 = torch.nn.Linear(Hd, 2 * S, dtype=torch.float64)
    with torch.no_grad():
        lin1.weight.copy_(d(w["W1"])); lin1.bias.copy_(d(w["b1"]))
        gru.weight_ih.copy_(d(w["W_ih"])); gru.weight_hh.copy_(d(w["W_hh"]))
        gru.bias_ih.copy_(d(w["b_ih"])); gru.bias_hh.copy_(d(w["b_hh"]))
        lin2.weight.copy_(d(w["W2"])); lin2.bias.copy_(d(w["b2"]))
        lin3.weight.copy_(d(w["W3"])); lin3.bias.copy_(d(w["b3"]))
        state = torch.zeros(B, S, dtype=torch.float64) if state0 is None else d(state0)
        belief = torch.zeros(B, RH, dtype=torch.float64) if belief0 is None else d(belief0)
        outs = []
        for t in range(T):
            a = torch.nn.functional.elu(lin1(torch.cat([state, d(actions[t])], dim=-1)))
            belief = gru(a, belief)
            p = lin3(torch.nn.functional.elu(lin2(belief)))
            mean, raw = p[:, :S], p[:, S:]
            std = torch.nn.functional.softplus(raw) + 0.1
            state = mean + d(eps[t]) * std
            outs.append((mean, std, state, belief))
    return [torch.stack([o[i] for o in outs]).numpy() for i in range(4)]


def _rssm_actor_torch(w, actor, eps, state0, belief0):
    """Unroll variant 2 from torch float64 modules: the actor (Linear, ELU,
    Linear, Tanh on [state, belief]) picks each step's action."""
    T, B, S = eps.shape
    Hd = w["W1"].shape[0]
    RH = w["W_hh"].shape[1]
    A, Ha = actor["Wa2"].shape
    d = lambda a: torch.from_numpy(np.asarray(a)).double()
    lin1 = torch.nn.Linear(S + A, Hd, dtype=torch.float64)
    gru = torch.nn.GRUCell(Hd, RH, dtype=torch.float64)
    lin2 = torch.nn.Linear(RH, Hd, dtype=torch.float64)
    lin3 = torch.nn.Linear(Hd, 2 * S, dtype=torch.float64)
    act = torch.nn.Sequential(torch.nn.Linear(S + RH, Ha, dtype=torch.float64), torch.nn.ELU(),
                              torch.nn.Linear(Ha, A, dtype=torch.float64), torch.nn.Tanh())
    with torch.no_grad():
        lin1.weight.copy_(d(w["W1"])); lin1.bias.copy_(d(w["b1"]))
        gru.weight_ih.copy_(d(w["W_ih"])); gru.weight_hh.copy_(d(w["W_hh"]))
        gru.bias_ih.copy_(d(w["b_ih"])); gru.bias_hh.copy_(d(w["b_hh"]))
        lin2.weight.copy_(d(w["W2"])); lin2.bias.copy_(d(w["b2"]))
        lin3.weight.copy_(d(w["W3"])); lin3.bias.copy_(d(w["b3"]))
        act[0].weight.copy_(d(actor["Wa1"])); act[0].bias.copy_(d(actor["ba1"]))
        act[2].weight.copy_(d(actor["Wa2"])); act[2].bias.copy_(d(actor["ba2"]))
        state = torch.zeros(B, S, dtype=torch.float64) if state0 is None else d(state0)
        belief = torch.zeros(B, RH, dtype=torch.float64) if belief0 is None else d(belief0)
        outs = []
        for t in range(T):
            action = act(torch.cat([state, belief], dim=-1))
            a = torch.nn.functional.elu(lin1(torch.cat([state, action], dim=-1)))
            belief = gru(a, belief)
            p = lin3(torch.nn.functional.elu(lin2(belief)))
            mean, raw = p[:, :S], p[:, S:]
            std = torch.nn.functional.softplus(raw) + 0.1
            state = mean + d(eps[t]) * std
            outs.append((mean, std, state, belief, action))
    return [torch.stack([o[i] for o in outs]).numpy() for i in range(5)]


def test_rssm_actor_against_torch_modules():
    spec = wl.RSSM_B50.scaled(T=7, B=5, state_dim=5, action_dim=3, hidden=7, rnn_hidden=6,
                              state0_std=0.5, belief0_std=0.5)
    inp = wl.make_rssm_inputs(spec, seed=43)
    actor = {k: v.numpy() for k, v in wl.make_rssm_actor(spec, seed=43, actor_hidden=4).items()}
    got = oracle.rssm_unroll_actor(inp["weights"], actor, inp["eps"], state0=inp["state0"],
                                   belief0=inp["belief0"])
    ref = _rssm_actor_torch({k: v.numpy() for k, v in inp["weights"].items()}, actor,
                            inp["eps"].numpy(), inp["state0"].numpy(), inp["belief0"].numpy())
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-12)


def test_rssm_constant_actor_equals_given_actions():
    """Zero actor weights with ba2 = atanh(v) act v at every step: the unroll
    equals variant 1 with actions = v."""
    spec = wl.RSSM_B50.scaled(T=6, B=3, state_dim=4, action_dim=2, hidden=5, rnn_hidden=6,
                              belief0_std=0.5)
    inp = wl.make_rssm_inputs(spec, seed=44)
    v = np.array([0.3, -0.6], np.float32)
    actor = {"Wa1": np.zeros((8, 10), np.float32), "ba1": np.ones(8, np.float32),
             "Wa2": np.zeros((2, 8), np.float32), "ba2": np.arctanh(v.astype(np.float64)).astype(np.float32)}
    got = oracle.rssm_unroll_actor(inp["weights"], actor, inp["eps"], belief0=inp["belief0"])
    acts = np.broadcast_to(np.tanh(actor["ba2"].astype(np.float64)), (6, 3, 2)).astype(np.float32)
    ref = oracle.rssm_unroll(inp["weights"], acts.copy(), inp["eps"], belief0=inp["belief0"])
    for g, r in zip(got[:4], ref):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-7)
    np.testing.assert_allclose(got[4], acts, rtol=0, atol=1e-7)


def test_rssm_against_torch_modules():
    spec = wl.RSSM_B50.scaled(T=6, B=4, state_dim=5, action_dim=3, hidden=7, rnn_hidden=6,
                              state0_std=1.0, belief0_std=0.5)
    inp = wl.make_rssm_inputs(spec, seed=3)
    w = {k: v.numpy() for k, v in inp["weights"].items()}
    got = oracle.rssm_unroll(w, inp["actions"], inp["eps"], state0=inp["state0"],
                             belief0=inp["belief0"])
    ref = _rssm_torch(w, inp["actions"].numpy(), inp["eps"].numpy(), inp["state0"].numpy(),
                      inp["belief0"].numpy())
    for g_, r_ in zip(got, ref):
        np.testing.assert_allclose(g_, r_, rtol=0, atol=1e-12)


def test_rssm_zero_weights_golden():
    g = json.load(open(os.path.join(GOLDEN, "rssm_zero_weights.json")))
    assert abs(g["std"] - (math.log(2.0) + 0.1)) < 1e-16
    spec = wl.RSSM_B50.scaled(T=5, B=3)
    inp = wl.make_rssm_inputs(spec, seed=1)
    w = {k: np.zeros_like(v.numpy()) for k, v in inp["weights"].items()}
    means, stds, states, beliefs = oracle.rssm_unroll(w, inp["actions"], inp["eps"])
    assert np.all(means == g["mean"])
    np.testing.assert_allclose(stds, g["std"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(states, g["std"] * inp["eps"].numpy().astype(np.float64),
                               rtol=0, atol=1e-15)
    assert np.all(beliefs == g["belief"])


def test_rssm_rows_and_permutation():
    spec = wl.RSSM_B50.scaled(T=4, B=6, hidden=9, rnn_hidden=8, state0_std=1.0,
                              belief0_std=1.0)
    inp = wl.make_rssm_inputs(spec, seed=5)
    w = {k: v.numpy() for k, v in inp["weights"].items()}
    full = oracle.rssm_unroll(w, inp["actions"], inp["eps"], state0=inp["state0"],
                              belief0=inp["belief0"])
    perm = np.array([3, 0, 5, 1, 4, 2])
    permd = oracle.rssm_unroll(w, inp["actions"].numpy()[:, perm], inp["eps"].numpy()[:, perm],
                               state0=inp["state0"].numpy()[perm],
                               belief0=inp["belief0"].numpy()[perm])
    for f, p in zip(full, permd):
        np.testing.assert_array_equal(p, f[:, perm])
    sub = oracle.rssm_unroll(w, inp["actions"], inp["eps"], state0=inp["state0"],
                             belief0=inp["belief0"], rows=[2, 5])
    for f, s in zip(full, sub):
        np.testing.assert_array_equal(s[:, [2, 5]], f[:, [2, 5]])


def test_workload_generators_are_seeded():
    a = wl.make_rnn_inputs(wl.BILSTM_VAR.scaled(T=20, B=5, in_dim=4, hidden=3, varlen=(2, 20)), 0)
    b = wl.make_rnn_inputs(wl.BILSTM_VAR.scaled(T=20, B=5, in_dim=4, hidden=3, varlen=(2, 20)), 0)
    assert torch.equal(a["x"], b["x"]) and torch.equal(a["lengths"], b["lengths"])
    assert int(a["lengths"].min()) >= 2 and int(a["lengths"].max()) <= 20


# --------------------------------------------------------------------------- backward (BPTT)

def _bptt_case(cell, layers, seed, T=5, B=3, in_dim=4, H=3):
    rng = np.random.default_rng(seed)
    ws = _rand_weights(rng, cell, layers, in_dim, H)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers, B, H))).astype(np.float32)
    c0 = (0.5 * rng.standard_normal((layers, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, H)).astype(np.float32)
    dhn = rng.standard_normal((layers, B, H)).astype(np.float32)
    dcn = rng.standard_normal((layers, B, H)).astype(np.float32)
    if cell == oracle.GRU:
        c0 = dcn = None
    return ws, x, h0, c0, dy, dhn, dcn


@pytest.mark.parametrize("cell,layers", [(oracle.LSTM, 1), (oracle.LSTM, 3), (oracle.GRU, 1),
                                         (oracle.GRU, 2)])
def test_bptt_against_torch_autograd(cell, layers):
    """The oracle's gradients equal torch float64 autograd through nn.LSTM /
    nn.GRU (a library routine) for loss = <y, dy> + <h_n, dh_n> (+ <c_n, dc_n>)."""
    ws, x, h0, c0, dy, dhn, dcn = _bptt_case(cell, layers, seed=10 + layers + 5 * cell)
    T, B, in_dim = x.shape
    H = 3
    g = oracle.rnn_backward(cell, x, ws, dy, hidden=H, h0=h0, c0=c0, dh_n=dhn, dc_n=dcn)
    kw = dict(input_size=in_dim, hidden_size=H, num_layers=layers, dtype=torch.float64)
    mod = torch.nn.LSTM(**kw) if cell == oracle.LSTM else torch.nn.GRU(**kw)
    with torch.no_grad():
        for layer in range(layers):
            for k, name in (("w_ih", "weight_ih"), ("w_hh", "weight_hh"), ("b_ih", "bias_ih"),
                            ("b_hh", "bias_hh")):
                getattr(mod, f"{name}_l{layer}").copy_(torch.from_numpy(ws[layer][k]).double())
    xt = torch.from_numpy(x).double().requires_grad_()
    ht = torch.from_numpy(h0).double().requires_grad_()
    if cell == oracle.LSTM:
        ct = torch.from_numpy(c0).double().requires_grad_()
        y, (hn, cn) = mod(xt, (ht, ct))
        loss = (y * torch.from_numpy(dy).double()).sum() + \
            (hn * torch.from_numpy(dhn).double()).sum() + (cn * torch.from_numpy(dcn).double()).sum()
    else:
        y, hn = mod(xt, ht)
        loss = (y * torch.from_numpy(dy).double()).sum() + (hn * torch.from_numpy(dhn).double()).sum()
    loss.backward()
    tol = dict(rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dh0"], ht.grad.numpy(), **tol)
    if cell == oracle.LSTM:
        np.testing.assert_allclose(g["dc0"], ct.grad.numpy(), **tol)
    for layer in range(layers):
        for k, name in (("dw_ih", "weight_ih"), ("dw_hh", "weight_hh"), ("db_ih", "bias_ih"),
                        ("db_hh", "bias_hh")):
            np.testing.assert_allclose(g[k][layer], getattr(mod, f"{name}_l{layer}").grad.numpy(),
                                       **tol, err_msg=f"{k} layer {layer}")


@pytest.mark.parametrize("cell", [oracle.LSTM, oracle.GRU])
def test_bptt_finite_differences(cell):
    """Central differences of the (separately pinned) oracle forward agree with
    the oracle's backward, for entries of x, h0, c0 and every weight tensor."""
    layers = 2
    ws, x, h0, c0, dy, dhn, dcn = _bptt_case(cell, layers, seed=77 + cell, T=4, B=2)
    H = 3

    def loss(x_, ws_, h0_, c0_):
        y, hn, cn = oracle.rnn_forward(cell, x_, ws_, hidden=H, h0=h0_, c0=c0_)
        v = float((y * dy).sum() + (hn * dhn).sum())
        if cell == oracle.LSTM:
            v += float((cn * dcn).sum())
        return v

    g = oracle.rnn_backward(cell, x, ws, dy, hidden=H, h0=h0, c0=c0, dh_n=dhn, dc_n=dcn)
    eps = np.float32(2.0 ** -10)   # exact in fp32 at these magnitudes
    rng = np.random.default_rng(5)

    def check(arr, grad, rebuild):
        for _ in range(4):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            fd = (loss(*rebuild(hi)) - loss(*rebuild(lo))) / (2 * float(eps))
            assert abs(fd - grad[idx]) <= 1e-5 * max(1.0, abs(grad[idx])), (idx, fd, grad[idx])

    check(x, g["dx"], lambda a: (a, ws, h0, c0))
    check(h0, g["dh0"], lambda a: (x, ws, a, c0))
    if cell == oracle.LSTM:
        check(c0, g["dc0"], lambda a: (x, ws, h0, a))
    for layer in range(layers):
        for k, gk in (("w_ih", "dw_ih"), ("w_hh", "dw_hh"), ("b_ih", "db_ih"), ("b_hh", "db_hh")):
            def rebuild(a, layer=layer, k=k):
                w2 = [dict(w) for w in ws]
                w2[layer][k] = a
                return x, w2, h0, c0
            check(ws[layer][k], g[gk][layer], rebuild)


@pytest.mark.parametrize("layers", [1, 2])
def test_bptt_projection_against_torch_autograd(layers):
    """LSTM with projection: the oracle's gradients (dw_hr included) equal
    torch float64 autograd through nn.LSTM(proj_size=P)."""
    rng = np.random.default_rng(40 + layers)
    T, B, in_dim, H, P = 5, 3, 4, 6, 3
    ws = _rand_weights(rng, oracle.LSTM, layers, in_dim, H, proj=P)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers, B, P))).astype(np.float32)
    c0 = (0.5 * rng.standard_normal((layers, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, P)).astype(np.float32)
    dhn = rng.standard_normal((layers, B, P)).astype(np.float32)
    dcn = rng.standard_normal((layers, B, H)).astype(np.float32)
    g = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=P, h0=h0, c0=c0, dh_n=dhn,
                            dc_n=dcn)
    mod = torch.nn.LSTM(input_size=in_dim, hidden_size=H, num_layers=layers, proj_size=P,
                        dtype=torch.float64)
    names = (("w_ih", "weight_ih"), ("w_hh", "weight_hh"), ("b_ih", "bias_ih"),
             ("b_hh", "bias_hh"), ("w_hr", "weight_hr"))
    with torch.no_grad():
        for layer in range(layers):
            for k, name in names:
                getattr(mod, f"{name}_l{layer}").copy_(torch.from_numpy(ws[layer][k]).double())
    xt = torch.from_numpy(x).double().requires_grad_()
    ht = torch.from_numpy(h0).double().requires_grad_()
    ct = torch.from_numpy(c0).double().requires_grad_()
    y, (hn, cn) = mod(xt, (ht, ct))
    loss = (y * torch.from_numpy(dy).double()).sum() + (hn * torch.from_numpy(dhn).double()).sum() \
        + (cn * torch.from_numpy(dcn).double()).sum()
    loss.backward()
    tol = dict(rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dh0"], ht.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dc0"], ct.grad.numpy(), **tol)
    for layer in range(layers):
        for k, name in names:
            np.testing.assert_allclose(g["d" + k][layer],
                                       getattr(mod, f"{name}_l{layer}").grad.numpy(), **tol,
                                       err_msg=f"d{k} layer {layer}")


def test_bptt_projection_finite_differences():
    rng = np.random.default_rng(55)
    T, B, in_dim, H, P, layers = 4, 2, 3, 5, 2, 2
    ws = _rand_weights(rng, oracle.LSTM, layers, in_dim, H, proj=P)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers, B, P))).astype(np.float32)
    c0 = (0.5 * rng.standard_normal((layers, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, P)).astype(np.float32)
    dhn = rng.standard_normal((layers, B, P)).astype(np.float32)

    def loss(ws_):
        y, hn, _ = oracle.rnn_forward(oracle.LSTM, x, ws_, hidden=H, proj=P, h0=h0, c0=c0)
        return float((y * dy).sum() + (hn * dhn).sum())

    g = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=P, h0=h0, c0=c0, dh_n=dhn)
    eps = np.float32(2.0 ** -10)
    for layer in range(layers):
        for k, gk in (("w_hr", "dw_hr"), ("w_hh", "dw_hh"), ("w_ih", "dw_ih")):
            arr = ws[layer][k]
            for idx in ((0, 0), (arr.shape[0] - 1, arr.shape[1] - 1)):
                hi, lo = arr.copy(), arr.copy()
                hi[idx] += eps
                lo[idx] -= eps
                w_hi = [dict(w) for w in ws]
                w_lo = [dict(w) for w in ws]
                w_hi[layer][k] = hi
                w_lo[layer][k] = lo
                fd = (loss(w_hi) - loss(w_lo)) / (2 * float(eps))
                want = g[gk][layer][idx]
                assert abs(fd - want) <= 1e-5 * max(1.0, abs(want)), (layer, k, idx, fd, want)



@pytest.mark.parametrize("cell,layers,proj", [(oracle.LSTM, 2, 0), (oracle.GRU, 2, 0),
                                              (oracle.LSTM, 2, 3), (oracle.LSTM, 1, 0)])
def test_bptt_bidirectional_against_torch_autograd(cell, layers, proj):
    """Bidirectional stacks: the oracle's gradients equal torch float64
    autograd through nn.LSTM / nn.GRU(bidirectional=True)."""
    rng = np.random.default_rng(60 + layers + 3 * cell + proj)
    T, B, in_dim, H = 5, 3, 4, 5
    Ho = proj or H
    D = 2
    ws = _rand_weights(rng, cell, layers, in_dim, H, D=D, proj=proj)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers * D, B, Ho))).astype(np.float32)
    c0 = (0.5 * rng.standard_normal((layers * D, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, D * Ho)).astype(np.float32)
    dhn = rng.standard_normal((layers * D, B, Ho)).astype(np.float32)
    dcn = rng.standard_normal((layers * D, B, H)).astype(np.float32)
    lstm = cell == oracle.LSTM
    g = oracle.rnn_backward(cell, x, ws, dy, hidden=H, proj=proj, bidirectional=True, h0=h0,
                            c0=c0 if lstm else None, dh_n=dhn, dc_n=dcn if lstm else None)
    kw = dict(input_size=in_dim, hidden_size=H, num_layers=layers, bidirectional=True,
              dtype=torch.float64)
    mod = torch.nn.LSTM(proj_size=proj, **kw) if lstm else torch.nn.GRU(**kw)
    names = (("w_ih", "weight_ih"), ("w_hh", "weight_hh"), ("b_ih", "bias_ih"),
             ("b_hh", "bias_hh")) + ((("w_hr", "weight_hr"),) if proj else ())
    with torch.no_grad():
        for layer in range(layers):
            for d in range(D):
                sfx = f"_l{layer}" + ("_reverse" if d else "")
                for k, name in names:
                    getattr(mod, name + sfx).copy_(torch.from_numpy(ws[layer * D + d][k]).double())
    xt = torch.from_numpy(x).double().requires_grad_()
    ht = torch.from_numpy(h0).double().requires_grad_()
    if lstm:
        ct = torch.from_numpy(c0).double().requires_grad_()
        y, (hn, cn) = mod(xt, (ht, ct))
        loss = (y * torch.from_numpy(dy).double()).sum() + \
            (hn * torch.from_numpy(dhn).double()).sum() + (cn * torch.from_numpy(dcn).double()).sum()
    else:
        y, hn = mod(xt, ht)
        loss = (y * torch.from_numpy(dy).double()).sum() + (hn * torch.from_numpy(dhn).double()).sum()
    loss.backward()
    tol = dict(rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dh0"], ht.grad.numpy(), **tol)
    if lstm:
        np.testing.assert_allclose(g["dc0"], ct.grad.numpy(), **tol)
    for layer in range(layers):
        for d in range(D):
            sfx = f"_l{layer}" + ("_reverse" if d else "")
            for k, name in names:
                np.testing.assert_allclose(g["d" + k][layer * D + d],
                                           getattr(mod, name + sfx).grad.numpy(), **tol,
                                           err_msg=f"d{k}{sfx}")


def test_bptt_bidirectional_finite_differences():
    rng = np.random.default_rng(77)
    T, B, in_dim, H, layers, D = 4, 2, 3, 4, 2, 2
    ws = _rand_weights(rng, oracle.GRU, layers, in_dim, H, D=D)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers * D, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, D * H)).astype(np.float32)

    def loss(x_, ws_):
        y, _, _ = oracle.rnn_forward(oracle.GRU, x_, ws_, hidden=H, bidirectional=True, h0=h0)
        return float((y * dy).sum())

    g = oracle.rnn_backward(oracle.GRU, x, ws, dy, hidden=H, bidirectional=True, h0=h0)
    eps = np.float32(2.0 ** -10)
    for idx in ((0, 0, 0), (T - 1, B - 1, in_dim - 1), (2, 1, 1)):
        hi, lo = x.copy(), x.copy()
        hi[idx] += eps
        lo[idx] -= eps
        fd = (loss(hi, ws) - loss(lo, ws)) / (2 * float(eps))
        assert abs(fd - g["dx"][idx]) <= 1e-5 * max(1.0, abs(g["dx"][idx])), (idx, fd)
    for i in range(layers * D):
        arr = ws[i]["w_hh"]
        for idx in ((0, 0), (arr.shape[0] - 1, arr.shape[1] - 1)):
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            w_hi = [dict(w) for w in ws]
            w_lo = [dict(w) for w in ws]
            w_hi[i]["w_hh"] = hi
            w_lo[i]["w_hh"] = lo
            fd = (loss(x, w_hi) - loss(x, w_lo)) / (2 * float(eps))
            want = g["dw_hh"][i][idx]
            assert abs(fd - want) <= 1e-5 * max(1.0, abs(want)), (i, idx, fd, want)


def test_bptt_bf16_weights_is_fp32_bptt_of_rounded_weights():
    """bf16_weights rounds the weight matrices (not the biases) and nothing
    else: equal, bit for bit, to the fp64 BPTT of pre-rounded weights."""
    rng = np.random.default_rng(90)
    T, B, in_dim, H, P = 4, 3, 5, 6, 3
    ws = _rand_weights(rng, oracle.LSTM, 2, in_dim, H, proj=P)
    rnd = [{k: (v if k in ("b_ih", "b_hh") or v is None else
                torch.from_numpy(v).to(torch.bfloat16).float().numpy())
            for k, v in w.items()} for w in ws]
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    dy = rng.standard_normal((T, B, P)).astype(np.float32)
    a = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=P, bf16_weights=True)
    b = oracle.rnn_backward(oracle.LSTM, x, rnd, dy, hidden=H, proj=P)
    for k in ("dx", "dh0", "dc0"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("dw_ih", "dw_hh", "db_ih", "db_hh", "dw_hr"):
        for u, v in zip(a[k], b[k]):
            assert np.array_equal(u, v), k



@pytest.mark.parametrize("cell,bidir", [(oracle.LSTM, True), (oracle.GRU, False),
                                        (oracle.LSTM, False)])
def test_bptt_varlen_against_torch_autograd(cell, bidir):
    """Variable lengths: the oracle's gradients equal torch float64 autograd
    through pack_padded_sequence -> nn.LSTM / nn.GRU -> pad_packed_sequence
    (h_n of each row at its own last step, zero gradient beyond it)."""
    rng = np.random.default_rng(70 + cell + 2 * bidir)
    T, B, in_dim, H, layers = 6, 4, 3, 5, 2
    D = 2 if bidir else 1
    ws = _rand_weights(rng, cell, layers, in_dim, H, D=D)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    lengths = np.array([6, 2, 4, 4], np.int32)
    h0 = (0.5 * rng.standard_normal((layers * D, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, D * H)).astype(np.float32)
    dhn = rng.standard_normal((layers * D, B, H)).astype(np.float32)
    lstm = cell == oracle.LSTM
    g = oracle.rnn_backward(cell, x, ws, dy, hidden=H, bidirectional=bidir, lengths=lengths,
                            h0=h0, dh_n=dhn)
    kw = dict(input_size=in_dim, hidden_size=H, num_layers=layers, bidirectional=bidir,
              dtype=torch.float64)
    mod = torch.nn.LSTM(**kw) if lstm else torch.nn.GRU(**kw)
    names = (("w_ih", "weight_ih"), ("w_hh", "weight_hh"), ("b_ih", "bias_ih"),
             ("b_hh", "bias_hh"))
    with torch.no_grad():
        for layer in range(layers):
            for d in range(D):
                sfx = f"_l{layer}" + ("_reverse" if d else "")
                for k, name in names:
                    getattr(mod, name + sfx).copy_(torch.from_numpy(ws[layer * D + d][k]).double())
    xt = torch.from_numpy(x).double().requires_grad_()
    ht = torch.from_numpy(h0).double().requires_grad_()
    packed = torch.nn.utils.rnn.pack_padded_sequence(xt, torch.from_numpy(lengths).long(),
                                                     enforce_sorted=False)
    state = (ht, torch.zeros_like(ht)) if lstm else ht
    out, st = mod(packed, state)
    y, _ = torch.nn.utils.rnn.pad_packed_sequence(out, total_length=T)
    hn = st[0] if lstm else st
    loss = (y * torch.from_numpy(dy).double()).sum() + (hn * torch.from_numpy(dhn).double()).sum()
    loss.backward()
    tol = dict(rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dh0"], ht.grad.numpy(), **tol)
    for layer in range(layers):
        for d in range(D):
            sfx = f"_l{layer}" + ("_reverse" if d else "")
            for k, name in names:
                np.testing.assert_allclose(g["d" + k][layer * D + d],
                                           getattr(mod, name + sfx).grad.numpy(), **tol,
                                           err_msg=f"d{k}{sfx}")
    for b in range(B):
        assert np.all(g["dx"][lengths[b]:, b] == 0.0)


# --------------------------------------------------------------------------- RSSM backward

def _rssm_case(seed, T=5, B=3, S=4, A=3, Hd=6, RH=5):
    spec = wl.RSSM_B50.scaled(T=T, B=B, state_dim=S, action_dim=A, hidden=Hd, rnn_hidden=RH,
                              state0_std=1.0, belief0_std=0.5)
    inp = wl.make_rssm_inputs(spec, seed=seed)
    w = {k: v.numpy() for k, v in inp["weights"].items()}
    rng = np.random.default_rng(seed)
    grads = {k: rng.standard_normal((T, B, n)).astype(np.float32)
             for k, n in (("dmeans", S), ("dstds", S), ("dstates", S), ("dbeliefs", RH))}
    return w, inp["actions"].numpy(), inp["eps"].numpy(), inp["state0"].numpy(), \
        inp["belief0"].numpy(), grads


def test_rssm_backward_against_torch_autograd():
    """The oracle's RSSM gradients equal torch float64 autograd through the
    prior step assembled from nn.Linear / nn.GRUCell / ELU / softplus modules,
    for every input and parameter."""
    w, actions, eps, s0, b0, gr = _rssm_case(41)
    T, B, A = actions.shape
    S = eps.shape[2]
    Hd, RH = w["W1"].shape[0], w["W_hh"].shape[1]
    g = oracle.rssm_backward(w, actions, eps, state0=s0, belief0=b0, **gr)
    d = lambda a: torch.from_numpy(np.asarray(a)).double()
    lin1 = torch.nn.Linear(S + A, Hd, dtype=torch.float64)
    gru = torch.nn.GRUCell(Hd, RH, dtype=torch.float64)
    lin2 = torch.nn.Linear(RH, Hd, dtype=torch.float64)
    lin3 = torch.nn.Linear(Hd, 2 * S, dtype=torch.float64)
    params = {"W1": lin1.weight, "b1": lin1.bias, "W_ih": gru.weight_ih, "W_hh": gru.weight_hh,
              "b_ih": gru.bias_ih, "b_hh": gru.bias_hh, "W2": lin2.weight, "b2": lin2.bias,
              "W3": lin3.weight, "b3": lin3.bias}
    with torch.no_grad():
        for k, prm in params.items():
            prm.copy_(d(w[k]))
    st0, bl0, act = d(s0).requires_grad_(), d(b0).requires_grad_(), d(actions).requires_grad_()
    state, belief = st0, bl0
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(T):
        x = torch.nn.functional.elu(lin1(torch.cat([state, act[t]], dim=-1)))
        belief = gru(x, belief)
        p = lin3(torch.nn.functional.elu(lin2(belief)))
        mean = p[:, :S]
        std = torch.nn.functional.softplus(p[:, S:]) + 0.1
        state = mean + d(eps[t]) * std
        loss = loss + (mean * d(gr["dmeans"][t])).sum() + (std * d(gr["dstds"][t])).sum() \
            + (state * d(gr["dstates"][t])).sum() + (belief * d(gr["dbeliefs"][t])).sum()
    loss.backward()
    tol = dict(rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dstate0"], st0.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dbelief0"], bl0.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dactions"], act.grad.numpy(), **tol)
    for k, prm in params.items():
        np.testing.assert_allclose(g["d" + k], prm.grad.numpy(), **tol, err_msg=k)


def test_rssm_backward_finite_differences():
    """Central differences of the (separately pinned) oracle RSSM forward agree
    with the oracle's RSSM backward, for entries of state0, belief0, the
    actions and every weight and bias."""
    w, actions, eps, s0, b0, gr = _rssm_case(43, T=4, B=2)
    g = oracle.rssm_backward(w, actions, eps, state0=s0, belief0=b0, **gr)

    def loss(w_, a_, s_, b_):
        m, sd, st, bl = oracle.rssm_unroll(w_, a_, eps, state0=s_, belief0=b_)
        return float((m * gr["dmeans"]).sum() + (sd * gr["dstds"]).sum()
                     + (st * gr["dstates"]).sum() + (bl * gr["dbeliefs"]).sum())

    # fp64 loss and exact fp32 offsets: the step only trades the O(h^2)
    # truncation term against fp64 round-off
    h = np.float32(2.0 ** -14)
    rng = np.random.default_rng(9)

    def check(arr, grad, rebuild):
        for _ in range(3):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += h
            lo[idx] -= h
            fd = (loss(*rebuild(hi)) - loss(*rebuild(lo))) / (2 * float(h))
            assert abs(fd - grad[idx]) <= 1e-5 * max(1.0, abs(grad[idx])), (idx, fd, grad[idx])

    check(s0, g["dstate0"], lambda a: (w, actions, a, b0))
    check(b0, g["dbelief0"], lambda a: (w, actions, s0, a))
    check(actions, g["dactions"], lambda a: (w, a, s0, b0))
    for k in oracle.RSSM_WEIGHTS:
        def rebuild(a, k=k):
            w2 = dict(w)
            w2[k] = a
            return w2, actions, s0, b0
        check(w[k], g["d" + k], rebuild)


def test_rssm_backward_head_only_closed_form():
    """With only dmeans given and T = 1, the gradient reaching b3 is dmeans
    summed over rows, and the std half of db3 is zero (a closed form)."""
    w, actions, eps, s0, b0, gr = _rssm_case(47, T=1, B=3)
    S = eps.shape[2]
    g = oracle.rssm_backward(w, actions, eps, state0=s0, belief0=b0, dmeans=gr["dmeans"])
    np.testing.assert_allclose(g["db3"][:S], gr["dmeans"][0].astype(np.float64).sum(0),
                               rtol=1e-12, atol=1e-12)
    assert np.all(g["db3"][S:] == 0.0)


def _rssm_actor_case(seed, T=5, B=3, S=4, A=3, Hd=6, RH=5, Ha=7):
    w, _, eps, s0, b0, gr = _rssm_case(seed, T=T, B=B, S=S, A=A, Hd=Hd, RH=RH)
    rng = np.random.default_rng(seed + 1)
    u = lambda shape, fan: (rng.uniform(-1, 1, shape) / np.sqrt(fan)).astype(np.float32)
    actor = {"Wa1": u((Ha, S + RH), S + RH), "ba1": u((Ha,), S + RH),
             "Wa2": u((A, Ha), Ha), "ba2": u((A,), Ha)}
    return w, actor, eps, s0, b0, gr


def test_rssm_actor_backward_against_torch_autograd():
    """Unroll variant 2 (the actor in the loop): the oracle's gradients equal
    torch float64 autograd through the actor (Linear, ELU, Linear, Tanh on
    [state, belief]) and the prior modules, for state0, belief0, every prior
    weight, every actor weight and each produced action."""
    w, actor, eps, s0, b0, gr = _rssm_actor_case(51)
    T, B, S = eps.shape
    Hd, RH = w["W1"].shape[0], w["W_hh"].shape[1]
    A, Ha = actor["Wa2"].shape
    g = oracle.rssm_backward(w, None, eps, state0=s0, belief0=b0, actor=actor, **gr)
    d = lambda a: torch.from_numpy(np.asarray(a)).double()
    lin1 = torch.nn.Linear(S + A, Hd, dtype=torch.float64)
    gru = torch.nn.GRUCell(Hd, RH, dtype=torch.float64)
    lin2 = torch.nn.Linear(RH, Hd, dtype=torch.float64)
    lin3 = torch.nn.Linear(Hd, 2 * S, dtype=torch.float64)
    act1 = torch.nn.Linear(S + RH, Ha, dtype=torch.float64)
    act2 = torch.nn.Linear(Ha, A, dtype=torch.float64)
    params = {"W1": lin1.weight, "b1": lin1.bias, "W_ih": gru.weight_ih, "W_hh": gru.weight_hh,
              "b_ih": gru.bias_ih, "b_hh": gru.bias_hh, "W2": lin2.weight, "b2": lin2.bias,
              "W3": lin3.weight, "b3": lin3.bias, "Wa1": act1.weight, "ba1": act1.bias,
              "Wa2": act2.weight, "ba2": act2.bias}
    with torch.no_grad():
        for k, prm in params.items():
            prm.copy_(d(w[k] if k in w else actor[k]))
    st0, bl0 = d(s0).requires_grad_(), d(b0).requires_grad_()
    state, belief = st0, bl0
    loss = torch.zeros((), dtype=torch.float64)
    acts = []
    for t in range(T):
        action = torch.tanh(act2(torch.nn.functional.elu(act1(torch.cat([state, belief], -1)))))
        action.retain_grad()
        acts.append(action)
        x = torch.nn.functional.elu(lin1(torch.cat([state, action], dim=-1)))
        belief = gru(x, belief)
        p = lin3(torch.nn.functional.elu(lin2(belief)))
        mean = p[:, :S]
        std = torch.nn.functional.softplus(p[:, S:]) + 0.1
        state = mean + d(eps[t]) * std
        loss = loss + (mean * d(gr["dmeans"][t])).sum() + (std * d(gr["dstds"][t])).sum() \
            + (state * d(gr["dstates"][t])).sum() + (belief * d(gr["dbeliefs"][t])).sum()
    loss.backward()
    tol = dict(rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dstate0"], st0.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dbelief0"], bl0.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dactions"], torch.stack([a.grad for a in acts]).numpy(), **tol)
    for k, prm in params.items():
        np.testing.assert_allclose(g["d" + k], prm.grad.numpy(), **tol, err_msg=k)


def test_rssm_actor_backward_finite_differences():
    """Central differences of the (separately pinned) oracle actor unroll agree
    with the oracle's actor-variant backward for state0, belief0 and every
    actor weight and bias."""
    w, actor, eps, s0, b0, gr = _rssm_actor_case(53, T=4, B=2)
    g = oracle.rssm_backward(w, None, eps, state0=s0, belief0=b0, actor=actor, **gr)

    def loss(ac, s_, b_):
        m, sd, st, bl, _ = oracle.rssm_unroll_actor(w, ac, eps, state0=s_, belief0=b_)
        return float((m * gr["dmeans"]).sum() + (sd * gr["dstds"]).sum()
                     + (st * gr["dstates"]).sum() + (bl * gr["dbeliefs"]).sum())

    h = np.float32(2.0 ** -14)
    rng = np.random.default_rng(10)

    def check(arr, grad, rebuild):
        for _ in range(3):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += h
            lo[idx] -= h
            fd = (loss(*rebuild(hi)) - loss(*rebuild(lo))) / (2 * float(h))
            assert abs(fd - grad[idx]) <= 1e-5 * max(1.0, abs(grad[idx])), (idx, fd, grad[idx])

    check(s0, g["dstate0"], lambda a: (actor, a, b0))
    check(b0, g["dbelief0"], lambda a: (actor, s0, a))
    for k in ("Wa1", "ba1", "Wa2", "ba2"):
        def rebuild(a, k=k):
            ac = dict(actor)
            ac[k] = a
            return ac, s0, b0
        check(actor[k], g["d" + k], rebuild)


def test_rssm_constant_actor_backward_reduces_to_given_actions():
    """Zero actor weights with ba2 = atanh(v) act v whatever the state: the
    prior's gradients equal the given-actions backward with actions = v, no
    gradient reaches Wa1 or ba1 (Wa2 = 0 stops it), and dba2 = (1 - v^2) times
    the summed action gradients."""
    w, _, eps, s0, b0, gr = _rssm_case(57, T=5, B=3, A=2)
    v = np.array([0.3, -0.6], np.float32)
    Ha, S, RH = 4, eps.shape[2], w["W_hh"].shape[1]
    actor = {"Wa1": np.zeros((Ha, S + RH), np.float32), "ba1": np.ones(Ha, np.float32),
             "Wa2": np.zeros((2, Ha), np.float32),
             "ba2": np.arctanh(v.astype(np.float64)).astype(np.float32)}
    got = oracle.rssm_backward(w, None, eps, state0=s0, belief0=b0, actor=actor, **gr)
    acts = np.tanh(actor["ba2"].astype(np.float64))
    ref = oracle.rssm_backward(w, np.broadcast_to(acts, (5, 3, 2)).astype(np.float32), eps,
                               state0=s0, belief0=b0, **gr)
    for k in ["dstate0", "dbelief0", "dactions"] + ["d" + n for n in oracle.RSSM_WEIGHTS]:
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-6, atol=1e-6, err_msg=k)
    assert np.all(got["dWa1"] == 0.0) and np.all(got["dba1"] == 0.0)
    np.testing.assert_allclose(got["dba2"], (1 - acts ** 2) * got["dactions"].sum((0, 1)),
                               rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- backward with clipping

def _clipped_lstm_loss(x, ws, H, P, h0, c0, dy, dhn, dcn, cclip, pclip):
    """A stacked unidirectional LSTM (optionally with projection) written out
    with torch.clamp on the cell state and the projection, float64; returns the
    loss <y, dy> + <h_n, dhn> + <c_n, dcn>."""
    L = len(ws)
    Ho = P if P else H
    layer_in = x
    loss = torch.zeros((), dtype=torch.float64)
    for l in range(L):
        w = ws[l]
        h, c = h0[l], c0[l]
        ys = []
        for t in range(layer_in.shape[0]):
            z = layer_in[t] @ w["w_ih"].T + w["b_ih"] + h @ w["w_hh"].T + w["b_hh"]
            i, f, g, o = z.split(H, dim=-1)
            c = torch.sigmoid(f) * c + torch.sigmoid(i) * torch.tanh(g)
            if cclip is not None:
                c = torch.clamp(c, cclip[0], cclip[1])
            m = torch.sigmoid(o) * torch.tanh(c)
            h = m @ w["w_hr"].T if P else m
            if P and pclip is not None:
                h = torch.clamp(h, pclip[0], pclip[1])
            ys.append(h)
        layer_in = torch.stack(ys)
        loss = loss + (h * dhn[l]).sum() + (c * dcn[l]).sum()
    return loss + (layer_in * dy).sum()


@pytest.mark.parametrize("proj", [0, 4])
def test_bptt_clipping_against_torch_autograd(proj):
    """Cell-state (and projection) clipping: the oracle's gradients equal
    torch float64 autograd through the clamps, with bounds that clamp a good
    share of the values."""
    rng = np.random.default_rng(81 + proj)
    T, B, in_dim, H, layers = 6, 3, 4, 5, 2
    ws = _rand_weights(rng, oracle.LSTM, layers, in_dim, H, proj=proj, scale=1.5)
    Ho = proj if proj else H
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    h0 = (0.5 * rng.standard_normal((layers, B, Ho))).astype(np.float32)
    c0 = (0.5 * rng.standard_normal((layers, B, H))).astype(np.float32)
    dy = rng.standard_normal((T, B, Ho)).astype(np.float32)
    dhn = rng.standard_normal((layers, B, Ho)).astype(np.float32)
    dcn = rng.standard_normal((layers, B, H)).astype(np.float32)
    cclip, pclip = (-0.3, 0.4), ((-0.2, 0.25) if proj else None)
    g = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=proj, h0=h0, c0=c0,
                            dh_n=dhn, dc_n=dcn, cell_clip=cclip, proj_clip=pclip)
    d = lambda a: torch.from_numpy(np.asarray(a)).double()
    tw = [{k: (d(v).requires_grad_() if v is not None else None) for k, v in w.items()}
          for w in ws]
    xt, h0t, c0t = d(x).requires_grad_(), d(h0).requires_grad_(), d(c0).requires_grad_()
    loss = _clipped_lstm_loss(xt, tw, H, proj, h0t, c0t, d(dy), d(dhn), d(dcn), cclip, pclip)
    loss.backward()
    # the bounds do clamp (else this would test nothing)
    y, _, cn = oracle.rnn_forward(oracle.LSTM, x, ws, hidden=H, proj=proj, h0=h0, c0=c0)
    assert (np.abs(cn) > 0.4).any() and (y.max() > 0.25 if proj else True)
    tol = dict(rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dh0"], h0t.grad.numpy(), **tol)
    np.testing.assert_allclose(g["dc0"], c0t.grad.numpy(), **tol)
    for l in range(layers):
        for k in ("w_ih", "w_hh", "b_ih", "b_hh") + (("w_hr",) if proj else ()):
            np.testing.assert_allclose(g["d" + k][l], tw[l][k].grad.numpy(), **tol,
                                       err_msg=f"d{k}[{l}]")


def test_bptt_cell_clip_to_zero_stops_every_gradient():
    """Clamping the cell state to [0, 0] makes every c_t and h_t zero whatever
    the inputs (a closed form): no output depends on any input, weight or
    initial state, so dx, dh0, dc0 and all weight gradients are exactly 0."""
    rng = np.random.default_rng(85)
    T, B, in_dim, H = 5, 2, 3, 4
    ws = _rand_weights(rng, oracle.LSTM, 1, in_dim, H)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    dy = rng.standard_normal((T, B, H)).astype(np.float32)
    dcn = rng.standard_normal((1, B, H)).astype(np.float32)
    g = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, dc_n=dcn, cell_clip=(0.0, 0.0))
    for k in ("dx", "dh0", "dc0"):
        assert np.all(g[k] == 0.0), k
    for k in ("dw_ih", "dw_hh", "db_ih", "db_hh"):
        assert np.all(g[k][0] == 0.0), k


def test_bptt_infinite_clip_bounds_change_nothing():
    rng = np.random.default_rng(86)
    T, B, in_dim, H, P = 5, 2, 3, 6, 4
    ws = _rand_weights(rng, oracle.LSTM, 2, in_dim, H, proj=P)
    x = rng.standard_normal((T, B, in_dim)).astype(np.float32)
    dy = rng.standard_normal((T, B, P)).astype(np.float32)
    inf = float("inf")
    a = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=P)
    b = oracle.rnn_backward(oracle.LSTM, x, ws, dy, hidden=H, proj=P, cell_clip=(-inf, inf),
                            proj_clip=(-inf, inf))
    for k in ("dx", "dh0", "dc0"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("dw_ih", "dw_hh", "db_ih", "db_hh", "dw_hr"):
        for l in range(2):
            assert np.array_equal(a[k][l], b[k][l]), k
