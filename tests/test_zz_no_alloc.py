"""The allocation-free LSTM entry point against the regular one and the oracle.

rnn_lstm_forward_noalloc exists for callers that must not allocate device
memory (a host framework that owns the device heap, a fixed memory budget, a
loop that cannot pay for an allocation).  Its scratch lives in a fixed device
array inside the library, so this file checks that two calls in a row (the
second one reusing the scratch the first one left behind) both match the
handle-based rnn_forward and the fp64 CPU oracle within the fp32 tolerance of
the other tests.  One case has hidden = 1024 with a batch that fills the
kernel's shared-memory plan to its limit.  The file is named to be collected
last, and it passes run alone as well.
"""
import numpy as np
import pytest
import torch

import oracle
from recurrent_cell_unroll_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4

CASES = [
    wl.LSTM_T80.scaled(T=21, B=6, in_dim=40, hidden=97, h0_std=0.5, c0_std=0.5),
    # hidden 1024 and 32 rows: the largest batch chunk whose shared-memory
    # plan still fits beside the kernel's static shared memory; 10.5 MB of
    # scratch, inside the 16 MiB array
    wl.LSTM_T80.scaled(T=16, B=32, in_dim=64, hidden=1024, h0_std=0.5, c0_std=0.5),
]


def _regular(spec, inp, dev):
    net = binding.RNN.from_spec(spec)
    net.set_weights(inp["weights"])
    h0 = inp["h0"].to(dev)
    c0 = inp["c0"].to(dev)
    y, hn, cn = net.forward(inp["x"].to(dev), h0=h0, c0=c0)
    assert net.status() == 0
    net.close()
    return y, hn, cn


@pytest.mark.parametrize("spec", CASES, ids=lambda s: f"T{s.T}-B{s.B}-H{s.hidden}")
def test_noalloc_matches_regular_entry_point_and_oracle_twice(spec):
    dev = torch.device("cuda")
    inp = wl.make_rnn_inputs(spec, seed=41)
    y_reg, hn_reg, cn_reg = _regular(spec, inp, dev)
    y_or, hn_or, cn_or = oracle.rnn_forward(oracle.LSTM, inp["x"], inp["weights"],
                                            hidden=spec.hidden, h0=inp["h0"], c0=inp["c0"])
    w = {k: (None if v is None else v.to(dev)) for k, v in inp["weights"][0].items()}
    x = inp["x"].to(dev)
    h0, c0 = inp["h0"][0].to(dev), inp["c0"][0].to(dev)
    for call in range(2):
        y = torch.full_like(y_reg, float("nan"))
        hn = torch.full((spec.B, spec.hidden), float("nan"), device=dev)
        cn = torch.full_like(hn, float("nan"))
        binding.rnn_lstm_forward_noalloc(spec.T, spec.B, spec.in_dim, spec.hidden, x, w["w_ih"],
                                         w["w_hh"], w["b_ih"], w["b_hh"], h0, c0, y, hn, cn)
        # the existing entry point
        assert float((y - y_reg).abs().max()) <= F32_TOL, f"call {call}: y differs"
        assert float((hn - hn_reg[0]).abs().max()) <= F32_TOL, f"call {call}: h_n differs"
        assert float((cn - cn_reg[0]).abs().max()) <= F32_TOL, f"call {call}: c_n differs"
        # the oracle
        assert np.abs(y.cpu().numpy() - y_or).max() <= F32_TOL, f"call {call}: y vs oracle"
        assert np.abs(hn.cpu().numpy() - hn_or[0]).max() <= F32_TOL, f"call {call}: h_n vs oracle"
        assert np.abs(cn.cpu().numpy() - cn_or[0]).max() <= F32_TOL, f"call {call}: c_n vs oracle"


def test_noalloc_rejects_problems_beyond_its_scratch():
    dev = torch.device("cuda")
    T, B, I, H = 64, 64, 8, 1024  # needs ~268 MB of scratch
    x = torch.zeros((T, B, I), device=dev)
    W_ih = torch.zeros((4 * H, I), device=dev)
    W_hh = torch.zeros((4 * H, H), device=dev)
    y = torch.zeros((T, B, H), device=dev)
    with pytest.raises(binding.RcuError) as e:
        binding.rnn_lstm_forward_noalloc(T, B, I, H, x, W_ih, W_hh, y=y)
    assert e.value.code == binding.RCU_ERR_UNSUPPORTED
