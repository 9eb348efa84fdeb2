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


def test_training_flops_are_forward_plus_bptt():
    """forward 2MG(K+H); backward: recompute 2MG(K+H), dh recurrence 2MGH,
    dW_ih + dW_hh 2MG(K+H), dx 2MGK (G = 4H for the LSTM)."""
    spec = wl.LSTM_TRAIN
    inp = wl.make_rnn_inputs(spec.scaled(T=2, B=2), seed=0)
    inp["lengths"] = None
    fl = bench.kernel_flops(spec, inp)
    M, H, K = spec.B * spec.T, spec.hidden, spec.in_dim
    G = 4 * H
    assert fl["input_gemm"] == [2 * M * G * K] and fl["recurrent"] == [2 * M * G * H]
    assert fl["bwd_recompute_gemm"] == [2 * M * G * (K + H)]
    assert fl["bwd_recurrent"] == [2 * M * G * H]
    assert fl["bwd_weight_gemm"] == [2 * M * G * (K + H)]
    assert fl["bwd_dx_gemm"] == [2 * M * G * K]
    assert "dy" in inp and inp["dy"].shape == (2, 2, H)


def test_bidirectional_varlen_training_flops():
    """Bidirectional, variable length: one entry per (layer, direction), M =
    the processed row-steps (the sum of the lengths), the upper layer's K =
    2 * hidden; the training draws leave the forward workload's inputs
    unchanged."""
    spec = wl.BILSTM_TRAIN.scaled(layers=2, T=6, B=3, varlen=(2, 6))
    inp = wl.make_rnn_inputs(spec, seed=4)
    fwd = wl.make_rnn_inputs(spec.scaled(train=False), seed=4)
    assert torch.equal(inp["x"], fwd["x"]) and torch.equal(inp["lengths"], fwd["lengths"])
    fl = bench.kernel_flops(spec, inp)
    M, H, K = int(inp["lengths"].sum()), spec.hidden, spec.in_dim
    G = 4 * H
    ks = [K, K, 2 * H, 2 * H]
    assert fl["bwd_recompute_gemm"] == [2 * M * G * (k + H) for k in ks]
    assert fl["bwd_recurrent"] == [2 * M * G * H] * 4
    assert fl["bwd_weight_gemm"] == [2 * M * G * (k + H) for k in ks]
    assert fl["bwd_dx_gemm"] == [2 * M * G * k for k in ks]
    assert inp["dy"].shape == (6, 3, 2 * H)


def test_rssm_training_flops_and_draws():
    """RSSM training pass: one FLOP entry per timed phase of rssm_backward (the
    unroll, the recompute, the reverse-time chain, the gradients), and the
    output-gradient draws leave the forward workload's inputs unchanged."""
    spec = wl.RSSM_TRAIN.scaled(T=3, B=2)
    inp = wl.make_rssm_inputs(spec, seed=2)
    fwd = wl.make_rssm_inputs(spec.scaled(train=False), seed=2)
    for k in ("actions", "eps"):
        assert torch.equal(inp[k], fwd[k])
    S, A, Hd, RH = spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden
    for k, n in (("dmeans", S), ("dstds", S), ("dstates", S), ("dbeliefs", RH)):
        assert inp[k].shape == (3, 2, n)
    fl = bench.kernel_flops(spec, inp)
    rs = 6
    prior = 2 * (Hd * (S + A) + 3 * RH * Hd + 3 * RH * RH + Hd * RH + 2 * S * Hd)
    assert fl == {"rssm_unroll": [prior * rs], "rssm_bwd_recompute": [prior * rs],
                  "rssm_bwd_chain": [2 * (3 * S * Hd + Hd * RH + 3 * RH * RH + 3 * RH * Hd)
                                     * rs],
                  "rssm_bwd_grads": [(prior + 2 * A * Hd) * rs]}
    assert bench.oracle_serial(spec) and not bench.oracle_serial(wl.RSSM_B50)


def test_traffic_table_names_real_workloads_and_kernels():
    """Every captured traffic entry belongs to a bench workload and to a kernel
    name the roofline can report for it."""
    names = {s.name for s in bench.WORKLOADS.values()}
    kinds = {"recurrent_tc", "recurrent_tc_lstmp", "recurrent_simt", "recurrent_cluster",
             "rssm_unroll", "bwd_recurrent", "bwd_recurrent_tc", "rssm_bwd_chain"}
    for (workload, kernel), traffic in bench.TRAFFIC.items():
        assert workload in names, workload
        assert kernel in kinds, kernel
        assert traffic > 0


def _chunk_starts(T, n):
    # the chunked host pipeline's split: q steps, n-2 equal chunks, q steps
    q = max(1, T // (4 * (n - 2) + 2)) if n >= 3 else 0
    mid = n - 2 if n >= 3 else n
    span = T - 2 * q
    t = [0] + ([q] if q else []) + [q + span * i // mid for i in range(1, mid + 1)]
    return t + ([T] if q else [])


def test_host_chunk_boundaries_cover_every_step_once():
    for T in range(1, 300):
        for n in range(2, 17):
            if n > T:
                continue
            t = _chunk_starts(T, n)
            steps = [b - a for a, b in zip(t, t[1:])]
            assert t[0] == 0 and t[-1] == T and min(steps) >= 1 and len(steps) <= 16
    assert _chunk_starts(512, 8) == [0, 19, 98, 177, 256, 335, 414, 493, 512]
    # the automatic split of the 512-step GRU (one chunk per 64 steps, at most 6)
    assert _chunk_starts(512, 6) == [0, 28, 142, 256, 370, 484, 512]


def test_topology_cpu_affinity_parsing():
    """The GPU's local CPUs come from the "CPU Affinity" column of nvidia-smi's
    topology matrix (tab-separated, ranges and lists)."""
    import bench
    text = ("\tGPU0\tGPU1\tCPU Affinity\tNUMA Affinity\tGPU NUMA ID\n"
            "GPU0\t X \tNV18\t0-3,8\t0\t2\n"
            "GPU1\tNV18\t X \t4-7\t1\t3\n\n"
            "Legend:\n\n  X    = Self\n")
    assert bench.parse_topo_affinity(text, 0) == {0, 1, 2, 3, 8}
    assert bench.parse_topo_affinity(text, 1) == {4, 5, 6, 7}
    assert bench.parse_topo_affinity(text, 2) is None
    assert bench.parse_topo_affinity("no table here", 0) is None


def test_bf16_peak_choice_follows_the_timed_region():
    import bench
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "measured"}
    assert bench.bf16_peak(peaks, 0.3)[0] == 1900.0
    assert bench.bf16_peak(peaks, None)[0] == 1900.0
    assert bench.bf16_peak(peaks, 5.0)[0] == 1700.0


def test_oracle_sample_prefix_and_plan():
    """A bounded CPU sample cuts the workload to a prefix of its steps (the
    varlen lengths clamped, the training gradients cut too) and sizes rows x
    steps to the budget: a row that does not fit becomes one row over fewer
    steps."""
    spec = wl.BILSTM_TRAIN.scaled(T=30, B=4, in_dim=8, hidden=8, varlen=(5, 30))
    inp = wl.make_rnn_inputs(spec, seed=1)
    sp, ip = bench.prefix(spec, inp, 7)
    assert sp.T == 7 and ip["x"].shape[0] == 7 and ip["dy"].shape[0] == 7
    assert int(ip["lengths"].max()) <= 7 and inp["lengths"].max() > 7
    assert bench.prefix(spec, inp, 30)[0] is spec
    rows, Tp = bench.sample_plan(spec, inp, cores=2, budget_s=60.0)
    assert Tp == spec.T and rows == [0, 1]
    rows, Tp = bench.sample_plan(spec, inp, cores=2, budget_s=1e-9)
    assert rows == [0, 1] and Tp == 1
    cb = bench.cpu_baseline(spec, inp, budget_s=0.5)
    assert cb["value"] > 0 and cb["kind"] == "oracle"
    rs = wl.RSSM_TRAIN.scaled(T=9, B=3)
    sp, ip = bench.prefix(rs, wl.make_rssm_inputs(rs, seed=2), 4)
    assert sp.T == 4 and ip["eps"].shape[0] == 4 and ip["dbeliefs"].shape[0] == 4


def test_roofline_bound_follows_the_kernel():
    """A tcgen05 kernel is held to the tensor peak, an FFMA kernel to the FP32
    ALU peak, whatever the handle's dtype; the tcgen05 reverse-time kernel
    counts the reverse-time recurrence's FLOPs."""
    spec = wl.GRU_TRAIN.scaled(T=4, B=8, in_dim=16, hidden=32)
    inp = wl.make_rnn_inputs(spec, seed=0)
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2000.0,
             "source": "test"}
    fl = bench.kernel_flops(spec, inp)
    tc = bench._roofline(spec, inp, {"bwd_recurrent_tc": (2.0, 2), "bwd_prep": (1.0, 2)},
                         peaks, 148, region_s=0.1, steps=2)
    assert tc["bound"] == "tensor" and tc["peak"] == 1900.0
    assert tc["algorithmic_flop_per_launch"] == sum(fl["bwd_recurrent"])
    ffma = bench._roofline(spec, inp, {"bwd_recurrent": (2.0, 2)}, peaks, 148, region_s=0.1,
                           steps=2)
    assert ffma["bound"] == "alu" and ffma["peak"] == round(bench.fp32_alu_peak_tflops(148, 2000.0), 1)
