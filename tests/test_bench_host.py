"""Host-side logic of bench.py on CPU: workload arithmetic, and the
max-over-ranks / sum-over-ranks reductions of the multi-process (torchrun)
path run as two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from recurrent_cell_unroll_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, local, ws = bench.dist_init("gloo")
    mx = bench.dist_max(float(10 + rank))
    sm = bench.dist_sum(float(1 + rank))
    bench.dist_barrier()
    q.put((r, ws, mx, sm))
    torch.distributed.destroy_process_group()


def test_two_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == 11.0 and r[3] == 3.0 for r in res)


def test_single_process_reductions_are_identity():
    assert bench.dist_max(3.5) == 3.5 and bench.dist_sum(2.0) == 2.0


def _flops(spec, inp=None):
    inp = inp or {"lengths": None}
    return bench.total_flops(spec, inp)


def test_flop_counts_match_the_workload_definitions():
    # GRU bf16 3 layers T512 B256 1024: 6 dense ops of 2*131072*3072*1024
    assert _flops(wl.GRU_3L) == 6 * 2 * 131072 * 3072 * 1024
    # LSTMP: layer 1 in-GEMM 2*32000*4096*80, recurrent 2*32000*(4096*256+256*1024)
    lstmp = 2 * 32000 * 4096 * 80 + 2 * 32000 * 4096 * 256 + \
        2 * 2 * 32000 * (4096 * 256 + 256 * 1024)
    assert _flops(wl.LSTMP_2L) == lstmp
    assert abs(_flops(wl.LSTMP_2L) / 1e9 - 255.9) < 0.1
    # RSSM: 586.4 kFLOP per row-step
    assert _flops(wl.RSSM_B50) == 586400 * 2500
    # LSTM T80: 83.9 M + 41.9 M
    assert _flops(wl.LSTM_T80) == 2 * 80 * 1024 * 512 + 2 * 80 * 1024 * 256


def test_varlen_counts_use_the_true_lengths():
    spec = wl.BILSTM_VAR.scaled(T=10, B=3, varlen=(1, 10))
    inp = {"lengths": torch.tensor([10, 4, 1], dtype=torch.int32)}
    f = bench.kernel_flops(spec, inp)
    assert f["input_gemm"] == [2 * 15 * 2 * 4 * 512 * 256]
    assert f["recurrent"] == [2 * 15 * 2 * 4 * 512 * 512]
    assert bench.units(spec, inp) == 30


def test_fp32_alu_peak():
    assert abs(bench.fp32_alu_peak_tflops(152, 2070.0) - 80.55) < 0.01


def test_reference_arm_prints_oracle_line(capsys, monkeypatch):
    monkeypatch.setitem(bench.WORKLOADS, "tiny", wl.LSTM_T80.scaled(T=5, B=2, in_dim=8,
                                                                     hidden=8))
    monkeypatch.setattr(bench, "WORKLOADS", dict(bench.WORKLOADS))
    import argparse
    args = argparse.Namespace(steps=2, warmup=3, seed=0)
    line = bench.run_reference(args, bench.WORKLOADS["tiny"])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_step_trace_medians():
    """Phase medians of the step-trace helper (host arithmetic only)."""
    import numpy as np
    from recurrent_cell_unroll_gb300 import step_trace
    tr = np.zeros((5, 16))
    tr[:, 0] = [0, 100, 200, 300, 400]
    tr[:, 3] = tr[:, 0] + 10
    tr[:, 4] = tr[:, 0] + 30
    tr[:, 1] = tr[:, 0] + 60
    got = dict(step_trace._medians(tr, step_trace.PHASES["recurrent_cluster"]))
    assert got == {"mat-vec": 10.0, "gates": 20.0, "h_t sent": 30.0}
    # phases whose stamps are absent are skipped
    assert step_trace._medians(tr, [(5, 6, "absent")]) == []
