"""The RCU_DEBUG build of the library on the GPU: its device bounds checks
(the stand-in for a memory checker, which is not available on the GPUs this
library is tested on) stay silent on valid calls, and its results match the
oracle.  It runs in a child process, since a process loads one librcu."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import oracle
from recurrent_cell_unroll_gb300 import _build, binding, workloads as wl
binding.load(_build.build(debug=True))
dev = torch.device("cuda")
cases = [
    (wl.GRU_3L.scaled(layers=2, T=9, B=150, in_dim=40, hidden=200, h0_std=0.5), 2),
    (wl.BILSTM_VAR.scaled(T=12, B=13, in_dim=24, hidden=40, varlen=(1, 12)), 1),
    (wl.LSTMP_2L.scaled(T=9, B=6, in_dim=16, hidden=64, proj=24), 0),
]
for spec, path in cases:
    inp = wl.make_rnn_inputs(spec, seed=31)
    net = binding.RNN.from_spec(spec)
    if path:
        net.set_attr(binding.RCU_ATTR_FORCE_PATH, path)
    net.set_weights(inp["weights"])
    L = inp["lengths"].to(dev) if inp["lengths"] is not None else None
    h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
    y, hn, cn = net.forward(inp["x"].to(dev), lengths=L, h0=h0)
    st = net.status()
    assert st == 0, (spec.name, st, binding.load().rcu_last_error())
    ref = oracle.rnn_forward(oracle.LSTM if spec.cell == "lstm" else oracle.GRU, inp["x"],
                             inp["weights"], hidden=spec.hidden, proj=spec.proj,
                             bidirectional=spec.bidir, lengths=inp["lengths"], h0=inp["h0"],
                             bf16_weights=spec.dtype == "bf16")
    e = float(np.abs(y.cpu().numpy() - ref[0]).max() / np.abs(ref[0]).max())
    assert e <= (2e-2 if spec.dtype == "bf16" else 1e-4), (spec.name, e)
    net.close()
# the tcgen05 reverse-time kernel of the GRU (two batch groups, the second ragged)
spec = wl.GRU_3L.scaled(T=6, B=150, in_dim=24, hidden=64, layers=2, h0_std=0.5)
inp = wl.make_rnn_inputs(spec, seed=33)
dy = torch.randn((spec.T, spec.B, spec.hidden), generator=torch.Generator().manual_seed(33))
net = binding.RNN.from_spec(spec)
net.set_weights(inp["weights"])
net.set_attr(binding.RCU_ATTR_PROFILE, 1)
dx, dh0, _, _ = net.backward(inp["x"].to(dev), dy.to(dev), h0=inp["h0"].to(dev))
st = net.status()
assert st == 0, (spec.name, st, binding.load().rcu_last_error())
assert "bwd_recurrent_tc" in net.profile(), net.profile()
ref = oracle.rnn_backward(oracle.GRU, inp["x"], inp["weights"], dy, hidden=spec.hidden,
                          h0=inp["h0"], bf16_weights=True)
for got, want in ((dx, ref["dx"]), (dh0, ref["dh0"])):
    e = float(np.abs(got.cpu().numpy() - want).max() / np.abs(want).max())
    assert e <= 2e-2, ("backward", e)
net.close()
# the FFMA reverse-time kernel with its K split over a CTA pair (fp32 LSTM)
spec = wl.LSTM_T80.scaled(T=7, B=9, in_dim=12, hidden=40, layers=2, h0_std=0.5, c0_std=0.5)
inp = wl.make_rnn_inputs(spec, seed=35)
dy = torch.randn((spec.T, spec.B, spec.hidden), generator=torch.Generator().manual_seed(35))
net = binding.RNN.from_spec(spec)
net.set_weights(inp["weights"])
dx, dh0, dc0, _ = net.backward(inp["x"].to(dev), dy.to(dev), h0=inp["h0"].to(dev),
                               c0=inp["c0"].to(dev))
st = net.status()
assert st == 0, (spec.name, st, binding.load().rcu_last_error())
ref = oracle.rnn_backward(oracle.LSTM, inp["x"], inp["weights"], dy, hidden=spec.hidden,
                          h0=inp["h0"], c0=inp["c0"])
for got, want in ((dx, ref["dx"]), (dh0, ref["dh0"]), (dc0, ref["dc0"])):
    e = float(np.abs(got.cpu().numpy() - want).max() / np.abs(want).max())
    assert e <= 1e-4, ("fp32 backward", e)
net.close()
print("debug build ok")
"""


def test_debug_build_checks_stay_silent_and_results_match():
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "debug build ok" in r.stdout
