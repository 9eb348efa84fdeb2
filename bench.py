"""Benchmark of the time-unrolled recurrent forward pass on GB300.

One "step" = one full forward of the workload through the C ABI (length sort
and packing, every layer's input-projection GEMM and persistent recurrent
kernel, output streaming).  Default workload: the 3-layer bf16 GRU
(T=512, B=256, 1024 -> 1024), the largest of the five shapes; --workload picks
another.  Metric: (batch x timesteps)/s, i.e. B*T per second of device time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (batch rows are independent: weak scaling, no collective on the data
path); the reported time is the max over ranks.  --impl reference times the
fp64 CPU oracle on the host cores instead (the only baseline this method has).
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from recurrent_cell_unroll_gb300 import workloads as wl  # noqa: E402

WORKLOADS = {
    "lstm": wl.LSTM_T80, "rssm": wl.RSSM_B50, "lstmp": wl.LSTMP_2L,
    "bilstm": wl.BILSTM_VAR, "gru": wl.GRU_3L, "rssm_actor": wl.RSSM_ACTOR,
    "lstm_train": wl.LSTM_TRAIN, "bilstm_train": wl.BILSTM_TRAIN, "rssm_train": wl.RSSM_TRAIN,
    "gru_train": wl.GRU_TRAIN,
}
METRIC = "(batch×timesteps)/s"
UNIT = "(B·T)/s"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- distributed helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, ws


def dist_init(backend: str):
    rank, local, ws = dist_info()
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return rank, local, ws


def dist_barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def dist_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_sum(value: float, device=None) -> float:
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- workload arithmetic

def units(spec, inp) -> int:
    """B*T of one step (the metric's unit count; padded T for varlen)."""
    return spec.B * spec.T


def active_rows(spec, inp) -> int:
    """Sum over rows of processed steps (= B*T without lengths)."""
    if isinstance(spec, wl.RssmSpec) or inp.get("lengths") is None:
        return spec.B * spec.T
    return int(inp["lengths"].sum())


def kernel_flops(spec, inp) -> dict:
    """Algorithmic FLOPs per launch of each kernel kind (2 per multiply-add)."""
    if isinstance(spec, wl.RssmSpec):
        S, A, Hd, RH = spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden
        prior = 2 * (Hd * (S + A) + 3 * RH * Hd + 3 * RH * RH + Hd * RH + 2 * S * Hd)
        Hx = spec.actor_hidden
        per = prior + 2 * (Hx * (S + RH) + A * Hx)
        rs = spec.B * spec.T
        if not spec.train:
            return {"rssm": [per * rs]}
        # training pass, per phase of rssm_backward (names of its timed spans):
        # the unroll again; the same products over all rows; the reverse-time
        # chain (W3^T, W2^T, W_hh^T, W_ih^T and the state columns of W1^T per
        # row-step); the weight gradients and the action gradient
        chain = 2 * (2 * S * Hd + Hd * RH + 3 * RH * RH + 3 * RH * Hd + S * Hd)
        return {"rssm_unroll": [per * rs], "rssm_bwd_recompute": [prior * rs],
                "rssm_bwd_chain": [chain * rs], "rssm_bwd_grads": [(prior + 2 * A * Hd) * rs]}
    M = active_rows(spec, inp)
    D, nG, H, Ho, P = spec.D, spec.nG, spec.hidden, spec.Hout, spec.proj
    gemm, rec = [], []
    for layer in range(spec.layers):
        K = spec.in_dim if layer == 0 else D * Ho
        gemm.append(2 * M * D * nG * H * K)
        rec.append(2 * M * D * (nG * H * Ho + (P * H if P else 0)))
    out = {"input_gemm": gemm, "recurrent": rec}
    if getattr(spec, "train", False):
        # backward through time, per (layer, direction): the dh recurrence
        # (W_hh^T dz, or (W_hh W_hr)^T dz with a projection: width H either
        # way), dW_ih, dW_hh, dX; the recompute GEMMs repeat the forward's
        # (counted, they run).  M counts processed row-steps only.
        G = nG * H
        ks = [spec.in_dim if layer == 0 else D * Ho for layer in range(spec.layers)
              for _ in range(D)]
        out["bwd_recompute_gemm"] = [2 * M * G * (k + Ho) for k in ks]
        out["bwd_recurrent"] = [2 * M * G * H for _ in ks]
        out["bwd_weight_gemm"] = [2 * M * G * (k + Ho) for k in ks]
        out["bwd_dx_gemm"] = [2 * M * G * k for k in ks]
    return out


def total_flops(spec, inp) -> int:
    return sum(sum(v) for v in kernel_flops(spec, inp).values())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def fp32_alu_peak_tflops(nsm: int, mhz: float) -> float:
    """FFMA peak: SMs x 128 fp32 lanes x 2 FLOP x clock."""
    return nsm * 128 * 2 * mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms in the background;
    start() returns once the first sample has arrived, so samples fall inside
    a timed region that begins after it."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        deadline = time.time() + 3.0
        while not self.lines and time.time() < deadline and self.proc.poll() is None:
            time.sleep(0.01)
        self.lines.clear()  # keep only samples taken from here on

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm

def make_rssm_train_runner(spec, inp, dev):
    """A training pass of the RSSM unroll: rssm_backward (which runs the unroll
    again) and the weight gradients."""
    from recurrent_cell_unroll_gb300 import binding
    m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
    m.set_weights(inp["weights"], device=dev)
    names = ("actions", "eps", "state0", "belief0", "dmeans", "dstds", "dstates", "dbeliefs")
    d = {k: (None if inp[k] is None else inp[k].to(dev)) for k in names}
    T, B, S, A, RH = spec.T, spec.B, spec.state_dim, spec.action_dim, spec.rnn_hidden
    dstate0 = torch.empty((B, S), device=dev)
    dbelief0 = torch.empty((B, RH), device=dev)
    dactions = torch.empty((T, B, A), device=dev) if A > 0 else None
    shapes = binding.rssm_weight_shapes(S, A, spec.hidden, RH)
    grads = {k: torch.empty(shapes[k], device=dev) for k in binding.RSSM_WEIGHT_NAMES}

    def step():
        binding.rssm_backward(m.h, T, B, d["state0"], d["belief0"], d["actions"], d["eps"],
                              d["dmeans"], d["dstds"], d["dstates"], d["dbeliefs"], dstate0,
                              dbelief0, dactions)
        binding.rssm_get_weight_grads(m.h, grads)

    def launches():
        return binding.rssm_last_launch_count(m.h)

    def profile_on():
        m.set_attr(binding.RCU_ATTR_PROFILE, 1)
        binding.rssm_profile_reset(m.h)

    def profile_read():
        prof = m.profile()
        m.set_attr(binding.RCU_ATTR_PROFILE, 0)
        return prof

    def e2e_io():
        # no host-buffer form of the backward: pinned host tensors copied in and
        # out around the device call, all on the launching stream
        hin = {k: inp[k].contiguous().pin_memory() for k in names if inp[k] is not None}
        outs = [dstate0, dbelief0] + ([dactions] if dactions is not None else []) + \
            list(grads.values())
        hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]

        def call():
            for k, v in hin.items():
                d[k].copy_(v, non_blocking=True)
            step()
            for o, hbuf in zip(outs, hout):
                hbuf.copy_(o, non_blocking=True)
        return list(hin.values()), hout, call

    def status():
        return binding.rssm_get_status(m.h)
    return step, launches, profile_on, profile_read, e2e_io, status, m


def make_runner(spec, inp, dev, tc_ksplit=0):
    from recurrent_cell_unroll_gb300 import binding
    if isinstance(spec, wl.RssmSpec) and spec.train:
        return make_rssm_train_runner(spec, inp, dev)
    if isinstance(spec, wl.RssmSpec):
        m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
        m.set_weights(inp["weights"], device=dev)
        d = {k: (None if inp[k] is None else inp[k].to(dev)) for k in
             ("actions", "eps", "state0", "belief0")}
        T, B, S, RH = spec.T, spec.B, spec.state_dim, spec.rnn_hidden
        outs = [torch.empty((T, B, S), device=dev) for _ in range(3)] + \
            [torch.empty((T, B, RH), device=dev)]
        if spec.actor_hidden:
            m.set_actor(inp["actor"], device=dev)
            outs.append(torch.empty((T, B, spec.action_dim), device=dev))

        def step():
            if spec.actor_hidden:
                binding.rssm_unroll_actor(m.h, T, B, d["state0"], d["belief0"], d["eps"], *outs)
            else:
                binding.rssm_unroll(m.h, T, B, d["state0"], d["belief0"], d["actions"],
                                    d["eps"], *outs)

        def launches():
            return binding.rssm_last_launch_count(m.h)

        def profile_on():
            pass

        def profile_read():
            return None

        def e2e_io():
            # pinned host buffers through the host-buffer entry point
            hin = {k: (None if inp[k] is None else inp[k].contiguous().pin_memory())
                   for k in ("state0", "belief0", "actions", "eps")}
            hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]

            def call():
                if spec.actor_hidden:
                    binding.rssm_unroll_actor_host(m.h, T, B, hin["state0"], hin["belief0"],
                                                   hin["eps"], *hout)
                else:
                    binding.rssm_unroll_host(m.h, T, B, hin["state0"], hin["belief0"],
                                             hin["actions"], hin["eps"], *hout)
            return [v for v in hin.values() if v is not None], hout, call

        def status():
            return binding.rssm_get_status(m.h)
        return step, launches, profile_on, profile_read, e2e_io, status, m

    net = binding.RNN.from_spec(spec)
    if tc_ksplit:
        net.set_attr(binding.RCU_ATTR_TC_KSPLIT, tc_ksplit)
    net.set_weights(inp["weights"], device=dev)
    d = {k: (None if inp[k] is None else inp[k].to(dev)) for k in ("x", "lengths", "h0", "c0")}
    T, B = spec.T, spec.B
    if spec.train:
        return make_train_runner(spec, inp, dev, net, d)
    y = torch.empty((T, B, spec.D * spec.Hout), device=dev)
    hn = torch.empty((spec.layers * spec.D, B, spec.Hout), device=dev)
    cn = torch.empty((spec.layers * spec.D, B, spec.hidden), device=dev) \
        if spec.cell == "lstm" else None

    def step():
        binding.rnn_forward(net.h, T, B, d["x"], d["lengths"], d["h0"], d["c0"], None, y, hn, cn)

    def launches():
        return net.launch_count()

    def profile_on():
        net.set_attr(binding.RCU_ATTR_PROFILE, 1)
        binding.rnn_profile_reset(net.h)

    def profile_read():
        prof = net.profile()
        net.set_attr(binding.RCU_ATTR_PROFILE, 0)
        return prof

    def e2e_io():
        # pinned host buffers through the host-buffer entry point
        hin = {k: (None if inp[k] is None else inp[k].contiguous().pin_memory())
               for k in ("x", "lengths", "h0", "c0")}
        hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in (y, hn)] + \
            ([torch.empty(cn.shape, dtype=cn.dtype, pin_memory=True)] if cn is not None else [None])

        def call():
            binding.rnn_forward_host(net.h, T, B, hin["x"], hin["lengths"], hin["h0"], hin["c0"],
                                     *hout)
        return [v for v in hin.values() if v is not None], [o for o in hout if o is not None], call

    def status():
        return net.status()
    return step, launches, profile_on, profile_read, e2e_io, status, net


def make_train_runner(spec, inp, dev, net, d):
    """A training pass: rnn_backward (which runs the forward again keeping every
    layer's output) and the weight gradients of every layer and direction."""
    from recurrent_cell_unroll_gb300 import binding
    T, B, H, L, D, Ho, P = spec.T, spec.B, spec.hidden, spec.layers, spec.D, spec.Hout, spec.proj
    G = spec.nG * H
    dy = inp["dy"].to(dev)
    dx = torch.empty_like(d["x"])
    dh0 = torch.empty((L * D, B, Ho), device=dev)
    dc0 = torch.empty((L * D, B, H), device=dev) if spec.cell == "lstm" else None
    grads = []  # over layer * D + direction: dW_ih, dW_hh, db_ih, db_hh, dW_hr
    for i in range(L * D):
        k = spec.in_dim if i // D == 0 else D * Ho
        grads.append([torch.empty((G, k), device=dev), torch.empty((G, Ho), device=dev),
                      torch.empty((G,), device=dev), torch.empty((G,), device=dev),
                      torch.empty((P, H), device=dev) if P else None])

    def step():
        binding.rnn_backward(net.h, T, B, d["x"], d["lengths"], d["h0"], d["c0"], dy, None, None,
                             dx, dh0, dc0)
        for i in range(L * D):
            layer, direction = divmod(i, D)
            binding.rnn_get_weight_grads(net.h, layer, *grads[i][:4], dW_hr=grads[i][4],
                                         direction=direction)

    def launches():
        return net.launch_count()

    def profile_on():
        net.set_attr(binding.RCU_ATTR_PROFILE, 1)
        binding.rnn_profile_reset(net.h)

    def profile_read():
        prof = net.profile()
        net.set_attr(binding.RCU_ATTR_PROFILE, 0)
        return prof

    def e2e_io():
        # no host-buffer form of the backward: pinned host tensors copied in and
        # out around the device call, all on the launching stream
        hin = {"x": inp["x"].contiguous().pin_memory(), "dy": inp["dy"].contiguous().pin_memory()}
        if d["lengths"] is not None:
            hin["lengths"] = inp["lengths"].contiguous().pin_memory()
        outs = [dx] + [g for gl in grads for g in gl if g is not None]
        hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]

        def call():
            d["x"].copy_(hin["x"], non_blocking=True)
            dy.copy_(hin["dy"], non_blocking=True)
            if "lengths" in hin:
                d["lengths"].copy_(hin["lengths"], non_blocking=True)
            step()
            for o, hbuf in zip(outs, hout):
                hbuf.copy_(o, non_blocking=True)
        return list(hin.values()), hout, call

    def status():
        return net.status()
    return step, launches, profile_on, profile_read, e2e_io, status, net


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# workload's dominant kernel, from single-pass ncu captures of the full-size
# workloads (the mean over the captured launches); a kernel changed after its
# capture must be taken out of this table (its traffic is then null).
TRAFFIC = {
    ("gru_bf16_3L_T512_B256_1024", "recurrent_tc"): 1961.3e6,
    ("lstmp_bf16_2L_T1000_B32_80x1024p256", "recurrent_tc_lstmp"): 43.7e6,
    ("bilstm_f32_varlen_B64_T500_256x512", "recurrent_simt"): 358.1e6,
    ("lstm_f32_T80_B1_512x256", "recurrent_cluster"): 1.41e6,
    ("rssm_f32_B50_T50_S20_A6_H200", "rssm_unroll"): 1.55e6,
    ("rssm_actor_f32_B50_T50_S20_A6_H200_X200", "rssm_unroll"): 1.69e6,
    ("lstm_train_f32_T500_B64_256x512", "bwd_recurrent"): 633.6e6,
    ("bilstm_train_f32_varlen_B64_T500_256x512", "bwd_recurrent"): 941.7e6,
    ("rssm_train_f32_B50_T50_S20_A6_H200", "rssm_bwd_chain"): 18.7e6,
    ("gru_train_bf16_3L_T512_B256_1024", "bwd_recurrent_tc"): 6688.3e6,
}


# A timed region shorter than this runs at the burst tensor rate (the
# measured bf16 peak of a short GEMM); a longer one settles under the power
# cap, where the sustained measurement applies.
SUSTAINED_AFTER_S = 2.0


def bf16_peak(peaks, region_s):
    """(TFLOP/s, note) of the bf16 tensor peak that applies to a timed region."""
    if region_s is not None and region_s >= SUSTAINED_AFTER_S:
        return peaks["bf16_tflops_sustained"], \
            f"bf16 dense, sustained ({peaks['source']}): timed region {region_s:.2f} s"
    return peaks["bf16_tflops"], f"bf16 dense, burst ({peaks['source']}): timed region " + \
        ("unknown" if region_s is None else f"{region_s:.2f} s") + \
        f" < {SUSTAINED_AFTER_S:.0f} s"


def roofline(spec, inp, prof, peaks, nsm, step_ms=None, region_s=None, steps=1):
    """Roofline of the dominant kernel from the live event timings."""
    r = _roofline(spec, inp, prof, peaks, nsm, step_ms, region_s, steps)
    if r is not None:
        tr = TRAFFIC.get((spec.name, r["kernel"]))
        r["traffic"] = tr
        if tr is not None:
            r["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    return r


def on_tensor_cores(kernel):
    """The kernels named *_tc* (the bf16 input GEMM and the tcgen05
    recurrences) run their contraction on the tensor cores; every other kernel
    (the SIMT and cluster-resident recurrences, the whole backward pass) is
    FP32 FFMA work, even on a bf16 handle."""
    return "_tc" in kernel


def _roofline(spec, inp, prof, peaks, nsm, step_ms=None, region_s=None, steps=1):
    if isinstance(spec, wl.RssmSpec) and not spec.train:
        # one kernel per step: its launch time is the event-timed step
        per_launch = kernel_flops(spec, inp)["rssm"][0]
        achieved = per_launch / (step_ms / 1e3) / 1e12
        peak = fp32_alu_peak_tflops(nsm, peaks["sm_max_mhz"])
        return {"kernel": "rssm_unroll", "bound": "alu", "achieved": round(achieved, 4),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 6),
                "traffic": None, "peak_note": "fp32 FFMA: SMs x 128 lanes x 2 x max SM clock",
                "avg_launch_ms": round(step_ms, 4), "launches": 1,
                "algorithmic_flop_per_launch": per_launch}
    if not prof:
        return None
    name, (ms, n) = max(prof.items(), key=lambda kv: kv[1][0])
    fl = kernel_flops(spec, inp)
    kind = name if name in fl else "recurrent" if name.startswith("recurrent") else (
        "input_gemm" if name.startswith("input_gemm") else
        "bwd_recurrent" if name.startswith("bwd_recurrent") else None)
    if kind is None:
        return None
    # the kind's FLOPs of all timed steps over its launches (one launch per
    # layer, or one per chunk of steps when the layers are pipelined)
    per_launch = sum(fl[kind]) * steps / n
    avg_s = ms / 1e3 / n
    achieved = per_launch / avg_s / 1e12
    if on_tensor_cores(name):
        peak, note = bf16_peak(peaks, region_s)
        bound = "tensor"
    else:
        peak, bound, note = fp32_alu_peak_tflops(nsm, peaks["sm_max_mhz"]), "alu", \
            "fp32 FFMA: SMs x 128 lanes x 2 x max SM clock"
    return {"kernel": name, "bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 5), "traffic": None,
            "peak_note": note, "avg_launch_ms": round(avg_s * 1e3, 4), "launches": n,
            "algorithmic_flop_per_launch": per_launch}


def flush_l2(buf):
    buf.add_(1.0)


def run_ours(args, spec, rank, local, ws):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from recurrent_cell_unroll_gb300 import binding
    binding.load()
    inp = (wl.make_rssm_inputs(spec, seed=args.seed + rank) if isinstance(spec, wl.RssmSpec)
           else wl.make_rnn_inputs(spec, seed=args.seed + rank))
    step, launches, profile_on, profile_read, e2e_io, status, keep = make_runner(
        spec, inp, dev, args.tc_ksplit)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(int(2 * L2_BYTES // 4), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        step()
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps, L2 flushed between steps (outside the events)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    profile_on()
    dist_barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    # no garbage-collector pass while the host enqueues the timed work
    gc.collect()
    gc.disable()
    t_wall = time.perf_counter()
    n_launch = 0
    try:
        for i in range(args.steps):
            flush_l2(flush)
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
            n_launch += launches()
        torch.cuda.synchronize(dev)
    finally:
        gc.enable()
    wall = time.perf_counter() - t_wall
    dist_barrier()
    clk = clocks.stop()
    dev_ms = sum(a.elapsed_time(b) for a, b in evs)
    prof = profile_read()
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    max_ms = dist_max(dev_ms, dev)
    all_units = dist_sum(units(spec, inp) * args.steps, dev)
    value = all_units / (max_ms / 1e3)

    # ---- end to end: the library's host-buffer entry point on pinned host
    #      inputs and outputs (every byte crosses the CPU-GPU link each step)
    #      (--e2e-steps 0 skips it, e.g. for a profiler's launch list of the
    #      timed region alone)
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, spec, e2e_io, status, keep, dev, stream, local,
                      max_ms / args.steps)

    peaks = load_peaks()
    extra = {}
    if not isinstance(spec, wl.RssmSpec) and inp.get("lengths") is not None:
        # varlen: also the rate of real (unpadded) row-steps
        sum_len = int(inp["lengths"].sum())
        extra["tokens_per_s"] = round(dist_sum(sum_len * args.steps, dev) / (max_ms / 1e3), 1)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4),
        "us_per_timestep": round(max_ms / args.steps * 1e3 / spec.T, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if getattr(spec, "dtype", "f32") == "bf16" else "f32",
        "data": "synthetic",
        "config": workload_config(spec, inp, ws),
        "roofline": roofline(spec, inp, prof, peaks, nsm, dev_ms / args.steps, wall, args.steps),
        "path_roofline": path_roofline(spec, inp, peaks, nsm, max_ms / args.steps, wall),
        "kernels": {k: {"ms_total": round(v[0], 3), "launches": v[1]} for k, v in prof.items()}
        if prof else None,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
        **extra,
    }
    return line, inp


def gpu_cpu_affinity(index: int):
    """CPUs nvidia-smi names as local to GPU `index` ("CPU Affinity" of
    `nvidia-smi topo -m`), as a set, or None when it cannot be read."""
    try:
        out = subprocess.run(["nvidia-smi", "topo", "-m"], capture_output=True, text=True,
                             timeout=20).stdout
    except (OSError, subprocess.SubprocessError):
        return None
    cpus = parse_topo_affinity(out, index)
    if cpus is None:
        return None
    return (cpus & os.sched_getaffinity(0)) or None


def parse_topo_affinity(out: str, index: int):
    """The "CPU Affinity" cell of GPU `index` in `nvidia-smi topo -m` output
    (tab-separated; ranges like 0-71,144-215) as a set of CPUs, or None."""
    lines = [ln for ln in out.splitlines() if ln.strip()]
    if not lines:
        return None
    head = lines[0].split("\t")
    col = next((i for i, h in enumerate(head) if "CPU Affinity" in h), None)
    if col is None:
        return None
    for ln in lines[1:]:
        f = ln.split("\t")
        if f and f[0].strip() == f"GPU{index}" and len(f) > col:
            cpus = set()
            for part in f[col].strip().split(","):
                if "-" in part:
                    lo, hi = part.split("-")
                    cpus.update(range(int(lo), int(hi) + 1))
                elif part.strip().isdigit():
                    cpus.add(int(part))
            return cpus or None
    return None


def link_rates(host_in, host_out, dev, stream):
    """GB/s of one host->device copy of the largest input and one device->host
    copy of the largest output, each alone on the stream (after one untimed
    copy of each), so the end-to-end figure can be read against the link."""
    def timed(dst, src):
        dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return src.numel() * src.element_size() / (a.elapsed_time(b) / 1e3) / 1e9
    big_in = max(host_in, key=lambda t: t.numel() * t.element_size())
    big_out = max(host_out, key=lambda t: t.numel() * t.element_size())
    d_in = torch.empty(big_in.shape, dtype=big_in.dtype, device=dev)
    d_out = torch.empty(big_out.shape, dtype=big_out.dtype, device=dev)
    r = {"h2d_gbs": round(timed(d_in, big_in), 1), "d2h_gbs": round(timed(big_out, d_out), 1),
         "h2d_probe_bytes": big_in.numel() * big_in.element_size(),
         "d2h_probe_bytes": big_out.numel() * big_out.element_size()}
    del d_in, d_out
    return r


def run_e2e(args, spec, e2e_io, status, keep, dev, stream, local, device_ms):
    """The end-to-end leg: the public host-buffer call on pinned host buffers,
    every step's inputs in and outputs out inside the timed region.  The
    process runs on the GPU's local CPUs meanwhile (so the pinned buffers are
    allocated on the GPU's NUMA node); the line records how the call moved
    the data and the link's own rate for one copy each way."""
    from recurrent_cell_unroll_gb300 import binding
    old_aff = os.sched_getaffinity(0)
    local_cpus = gpu_cpu_affinity(local)
    if local_cpus:
        os.sched_setaffinity(0, local_cpus)
    try:
        host_in, host_out, host_call = e2e_io()
        h2d = sum(v.numel() * v.element_size() for v in host_in)
        d2h = sum(o.numel() * o.element_size() for o in host_out)
        e2e_steps = max(1, args.e2e_steps)
        # untimed warm-up calls until the call time is steady: the first calls
        # after the staging buffers, copy streams and pinned buffers are set
        # up ran up to 3x slower than the steady step (two in a row within
        # 10 %, at least W calls, at most 20)
        prev, warm = None, 0
        while warm < 20:
            wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            wa.record(stream)
            host_call()
            wb.record(stream)
            torch.cuda.synchronize(dev)
            cur = wa.elapsed_time(wb)
            warm += 1
            if warm >= max(3, args.warmup) and prev is not None and abs(cur - prev) <= 0.1 * prev:
                break
            prev = cur
        dist_barrier()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
        gc.collect()
        gc.disable()
        try:
            t_host = time.perf_counter()
            for i in range(e2e_steps):
                evs[i][0].record(stream)
                host_call()
                evs[i][1].record(stream)
            t_host = time.perf_counter() - t_host
            torch.cuda.synchronize(dev)
        finally:
            gc.enable()
        per = [a.elapsed_time(b) for a, b in evs]
        e2e_ms = dist_max(sum(per) / e2e_steps, dev)
        e2e_value = dist_sum(units(spec, None), dev) / (e2e_ms / 1e3)
        st = status()
        if st != 0:
            raise RuntimeError(f"device status {st} in the end-to-end loop")
        link = link_rates(host_in, host_out, dev, stream)
        plan = None
        if isinstance(keep, binding.RNN) and not getattr(spec, "train", False):
            plan = binding.rnn_host_plan(keep.h)
    finally:
        os.sched_setaffinity(0, old_aff)
    return {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "ms_per_step_each": [round(x, 3) for x in per], "steps": e2e_steps,
            # (the value is the mean; an occasional host-side stall of one call
            # shows here and in the list)
            "ms_per_step_median": round(sorted(per)[len(per) // 2], 4),
            "warmup_calls": warm,
            # host time to issue the calls: well under the device time means
            # the host ran ahead of the GPU
            "host_issue_ms_per_step": round(t_host * 1e3 / e2e_steps, 3),
            "device_ms_per_step": round(device_ms, 4),
            "link": link,
            "h2d_ms_alone": round(h2d / (link["h2d_gbs"] * 1e9) * 1e3, 3),
            "d2h_ms_alone": round(d2h / (link["d2h_gbs"] * 1e9) * 1e3, 3),
            "host_plan": plan,
            "cpu_affinity": (f"{min(local_cpus)}-{max(local_cpus)} ({len(local_cpus)} CPUs, "
                             "local to the GPU)") if local_cpus else "unchanged",
            "call": ("rssm_backward + rssm_get_weight_grads, pinned host copies on the stream"
                     if getattr(spec, "train", False) else
                     "rssm_unroll_actor_host" if getattr(spec, "actor_hidden", 0) else
                     "rssm_unroll_host") if isinstance(spec, wl.RssmSpec) else
            ("rnn_backward + rnn_get_weight_grads, pinned host copies on the stream"
             if getattr(spec, "train", False) else "rnn_forward_host"),
            "host_buffers": "pinned"}


def path_roofline(spec, inp, peaks, nsm, ms_step, region_s=None):
    """Whole-step roofline: max(FLOPs / peak(dtype), compulsory bytes / HBM)."""
    fl = total_flops(spec, inp)
    if getattr(spec, "dtype", "f32") == "bf16":
        peak = bf16_peak(peaks, region_s)[0] * 1e12
    else:
        peak = fp32_alu_peak_tflops(nsm, peaks["sm_max_mhz"]) * 1e12
    t_flop = fl / peak
    byt = compulsory_bytes(spec, inp)
    t_byte = byt / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_flop, t_byte)
    return {"flop": fl, "compulsory_bytes": byt, "roofline_ms": round(t_roof * 1e3, 4),
            "frac": round(t_roof * 1e3 / ms_step, 5)}


def compulsory_bytes(spec, inp) -> int:
    if isinstance(spec, wl.RssmSpec):
        S, A, Hd, RH = spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden
        w = Hd * (S + A + 1) + 3 * RH * (Hd + RH + 2) + Hd * (RH + 1) + 2 * S * (Hd + 1)
        Hx = spec.actor_hidden
        w += Hx * (S + RH + 1) + A * (Hx + 1)
        # actions are read when given, written when the actor makes them
        io = spec.T * spec.B * (A + S + 3 * S + RH)
        if spec.train:
            # weights in, their gradients out; actions, eps and the four output
            # gradients in, the action gradient out
            return 4 * (2 * w + io + spec.T * spec.B * A)
        return 4 * (w + io)
    es = 2 if spec.dtype == "bf16" else 4
    D, nG, H, Ho = spec.D, spec.nG, spec.hidden, spec.Hout
    w = 0
    for layer in range(spec.layers):
        K = spec.in_dim if layer == 0 else D * Ho
        w += D * (nG * H * (K + Ho) * es + 2 * nG * H * 4 + (spec.proj * H * es if spec.proj else 0))
    M = active_rows(spec, inp)
    x = M * spec.in_dim * 4
    y = spec.T * spec.B * D * Ho * 4
    if getattr(spec, "train", False):
        # x and dy in, dx and the weight gradients out
        return 2 * w + 2 * x + y
    st = spec.layers * D * spec.B * (Ho + (H if spec.cell == "lstm" else 0)) * 4
    h0 = st if (inp.get("h0") is not None) else 0
    return w + x + y + st + h0


def workload_config(spec, inp, ws):
    c = {"workload": spec.name, "T": spec.T, "B": spec.B, "replicas": ws,
         "l2": "inputs larger than L2" if input_bytes(spec, inp) > L2_BYTES
         else "L2 flushed between timed steps (256 MB write)"}
    if isinstance(spec, wl.RssmSpec):
        c.update(state_dim=spec.state_dim, action_dim=spec.action_dim, hidden=spec.hidden,
                 rnn_hidden=spec.rnn_hidden, actor_hidden=spec.actor_hidden or None,
                 train=spec.train or None)
    else:
        c.update(cell=spec.cell, layers=spec.layers, in_dim=spec.in_dim, hidden=spec.hidden,
                 proj=spec.proj, bidirectional=spec.bidir, train=spec.train or None,
                 varlen=None if inp.get("lengths") is None else
                 {"sum_len": int(inp["lengths"].sum()), "range": list(spec.varlen)})
    c["l2_flush_each_step"] = True
    return c


def input_bytes(spec, inp):
    if isinstance(spec, wl.RssmSpec):
        a = inp["actions"].numel() * 4 if inp["actions"] is not None else 0
        return a + inp["eps"].numel() * 4
    return inp["x"].numel() * 4


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_sample(spec, inp, rows, threads):
    import oracle
    t0 = time.perf_counter()
    if isinstance(spec, wl.RssmSpec) and spec.train:
        sel = list(rows)
        sub = (lambda t, dim: None if t is None else t[:, sel] if dim == 1 else t[sel])
        oracle.rssm_backward(inp["weights"], sub(inp["actions"], 1), sub(inp["eps"], 1),
                             state0=sub(inp["state0"], 0), belief0=sub(inp["belief0"], 0),
                             **{k: sub(inp[k], 1) for k in ("dmeans", "dstds", "dstates",
                                                            "dbeliefs")})
    elif isinstance(spec, wl.RssmSpec) and spec.actor_hidden:
        oracle.rssm_unroll_actor(inp["weights"], inp["actor"], inp["eps"], state0=inp["state0"],
                                 belief0=inp["belief0"], rows=rows, threads=threads)
    elif isinstance(spec, wl.RssmSpec):
        oracle.rssm_unroll(inp["weights"], inp["actions"], inp["eps"], state0=inp["state0"],
                           belief0=inp["belief0"], rows=rows, threads=threads)
    elif spec.train:
        sel = list(rows)
        sub = (lambda t, dim: None if t is None else t[:, sel] if dim == 1 else t[sel])
        oracle.rnn_backward(oracle.LSTM if spec.cell == "lstm" else oracle.GRU,
                            sub(inp["x"], 1), inp["weights"], sub(inp["dy"], 1),
                            hidden=spec.hidden, proj=spec.proj, bidirectional=spec.bidir,
                            lengths=sub(inp["lengths"], 0), h0=sub(inp["h0"], 1),
                            c0=sub(inp["c0"], 1), bf16_weights=spec.dtype == "bf16",
                            threads=threads)
    else:
        oracle.rnn_forward(oracle.LSTM if spec.cell == "lstm" else oracle.GRU, inp["x"],
                           inp["weights"], hidden=spec.hidden, proj=spec.proj,
                           bidirectional=spec.bidir, lengths=inp["lengths"], h0=inp["h0"],
                           c0=inp["c0"], bf16_weights=spec.dtype == "bf16", rows=rows,
                           threads=threads)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_serial(spec) -> bool:
    """The RSSM backward oracle takes its rows one after another on one thread
    (its weight gradients sum over them)."""
    return isinstance(spec, wl.RssmSpec) and spec.train


def prefix(spec, inp, Tp):
    """The workload cut to its first Tp steps (every step of a recurrence
    costs the same, so (B*T)/s of the prefix is that of the whole)."""
    if Tp >= spec.T:
        return spec, inp
    out = dict(inp)
    if isinstance(spec, wl.RssmSpec):
        for k in ("actions", "eps", "dmeans", "dstds", "dstates", "dbeliefs"):
            if out.get(k) is not None:
                out[k] = out[k][:Tp]
    else:
        out["x"] = inp["x"][:Tp]
        if inp.get("dy") is not None:
            out["dy"] = inp["dy"][:Tp]
        if inp.get("lengths") is not None:
            out["lengths"] = inp["lengths"].clamp(max=Tp)
    return spec.scaled(T=Tp), out


def sample_plan(spec, inp, cores, budget_s):
    """(rows, steps) of a bounded oracle sample: one row timed over a short
    prefix gives the cost of a row-step; then as many rows as the budget
    allows over all steps (at most one per core unless the oracle is
    serial), or, when a whole row exceeds the budget, one row over the
    longest prefix that fits."""
    T0 = min(spec.T, 16)
    sp, ip = prefix(spec, inp, T0)
    per_step = oracle_sample(sp, ip, [0], 1) / T0
    per_row = per_step * spec.T
    if oracle_serial(spec):
        # rows one after another on one thread: as many whole rows as fit
        if per_row <= budget_s:
            return list(range(max(1, min(spec.B, int(budget_s / max(per_row, 1e-9)))))), spec.T
        return [0], max(1, min(spec.T, int(budget_s / max(per_step, 1e-9))))
    # one row per core, in parallel: all steps when a whole row fits the
    # budget, else the longest prefix that does
    rows = list(range(max(1, min(spec.B, cores))))
    if per_row <= budget_s:
        return rows, spec.T
    return rows, max(1, min(spec.T, int(budget_s / max(per_step, 1e-9))))


def cpu_baseline(spec, inp, budget_s=20.0):
    import oracle
    oracle.build()
    cores = cpu_cores()
    rows, Tp = sample_plan(spec, inp, cores, budget_s)
    sp, ip = prefix(spec, inp, Tp)
    threads = 1 if oracle_serial(spec) else min(cores, len(rows))
    t = oracle_sample(sp, ip, rows, threads)
    value = len(rows) * Tp / t
    steps = f"all {spec.T} steps" if Tp == spec.T else f"the first {Tp} of {spec.T} steps"
    return {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {spec.B} batch rows, {steps}, all layers "
                      f"(rows are independent, every step costs the same), fp64, "
                      f"{threads} threads",
            "seconds": round(t, 3)}


def run_reference(args, spec):
    import oracle
    oracle.build()
    inp = (wl.make_rssm_inputs(spec, seed=args.seed) if isinstance(spec, wl.RssmSpec)
           else wl.make_rnn_inputs(spec, seed=args.seed))
    cores = cpu_cores()
    # size each step so that warm-up + timed steps stay within ~3 minutes
    budget = max(1.0, min(20.0, 180.0 / max(1, args.steps + args.warmup)))
    rows, Tp = sample_plan(spec, inp, cores, budget)
    sp, ip = prefix(spec, inp, Tp)
    threads = 1 if oracle_serial(spec) else min(cores, len(rows))
    for _ in range(args.warmup):
        oracle_sample(sp, ip, rows, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_sample(sp, ip, rows, threads)
    value = len(rows) * Tp * args.steps / t
    steps = f"all {spec.T} steps" if Tp == spec.T else f"the first {Tp} of {spec.T} steps"
    sample = (f"{len(rows)} of {spec.B} batch rows per step, {steps}, all layers, "
              f"fp64, {threads} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(spec, inp, 1),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- the other configs

# The shapes the metric is also quoted on, measured after the headline
# workload in the same run (1 GPU only): the TVM page's LSTM, the RSSM prior,
# the 2-layer LSTMP, the variable-length bidirectional LSTM, the RSSM with
# the actor in the loop, and the training passes (forward + backward through
# time) of the LSTM, the variable-length bidirectional LSTM, the RSSM and the
# 3-layer GRU.
CONFIG_WORKLOADS = ("lstm", "rssm", "lstmp", "bilstm", "rssm_actor", "lstm_train",
                    "bilstm_train", "rssm_train", "gru_train")


def run_configs(args, rank, local, ws):
    """One compact entry per config: throughput, per-step latency, the
    dominant kernel's and the whole path's roofline fractions, the
    end-to-end rate and a bounded CPU-oracle sample."""
    out = {}
    for name in CONFIG_WORKLOADS:
        spec = WORKLOADS[name]
        sub = argparse.Namespace(**vars(args))
        sub.steps = max(3, min(args.steps, 10))
        sub.e2e_steps = min(args.e2e_steps, 3)
        line, inp = run_ours(sub, spec, rank, local, ws)
        rf, pr, e2e = line["roofline"] or {}, line["path_roofline"] or {}, line["e2e"] or {}
        entry = {
            "value": line["value"], "unit": UNIT, "dtype": line["dtype"], "steps": sub.steps,
            "ms_per_step": line["ms_per_step"], "us_per_timestep": line["us_per_timestep"],
            "roofline": {k: rf.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit",
                                                "frac", "avg_launch_ms", "traffic")},
            "path_roofline": {k: pr.get(k) for k in ("roofline_ms", "frac")},
            "e2e": {k: e2e.get(k) for k in ("value", "ms_per_step", "host_plan")} if e2e
            else None,
            "clocks": line["clocks"],
        }
        if "tokens_per_s" in line:
            entry["tokens_per_s"] = line["tokens_per_s"]
        if not args.no_cpu_baseline:
            entry["cpu_baseline"] = cpu_baseline(spec, inp, args.config_cpu_budget)
        out[spec.name] = entry
        del line, inp
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gru", choices=sorted(WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="steps of the host-buffer end-to-end leg (0 = skip it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configs measured after the default workload")
    ap.add_argument("--config-cpu-budget", type=float, default=6.0,
                    help="seconds of CPU-oracle work per extra config")
    ap.add_argument("--T", type=int, default=0,
                    help="override the sequence length (small cases for profiler captures)")
    ap.add_argument("--dtype", default="", choices=["", "f32", "bf16"],
                    help="override the workload's weight type (bf16 on an fp32 workload is the "
                         "opt-in down-conversion to the tensor cores)")
    ap.add_argument("--tc-ksplit", type=int, default=0, choices=[0, 1, 2, 4],
                    help="tensor-core recurrence: CTAs splitting K (0 = the library's choice)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    spec = WORKLOADS[args.workload]
    if args.dtype and not isinstance(spec, wl.RssmSpec) and args.dtype != spec.dtype:
        spec = spec.scaled(dtype=args.dtype, name=f"{spec.name}@{args.dtype}")
    if args.T > 0:
        kw = {"T": args.T, "name": f"{spec.name}@T{args.T}"}
        if getattr(spec, "varlen", None) is not None:
            kw["varlen"] = (min(spec.varlen[0], args.T), args.T)
        spec = spec.scaled(**kw)
    rank, local, ws = dist_info()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, spec)), flush=True)
        return 0

    rank, local, ws = dist_init("nccl")
    line, inp = run_ours(args, spec, rank, local, ws)
    if rank == 0:
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(spec, inp, args.cpu_budget)
        else:
            line["cpu_baseline"] = None
        if (ws == 1 and not args.no_configs and args.workload == "gru" and args.T == 0 and
                not args.dtype and not args.tc_ksplit):
            line["configs"] = run_configs(args, rank, local, ws)
        print(json.dumps(line), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
