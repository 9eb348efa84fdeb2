"""Per-step phase timings of the first layer's recurrent kernel.

Runs one workload a few times, then once with the library's step trace on
(RCU_ATTR_TRACE / rnn_get_trace, rssm_get_trace: CUDA global-timer stamps of
CTA 0, resolution about 256 ns) and prints the median time between stamps.

    python -m recurrent_cell_unroll_gb300.step_trace --workload gru --T 64 [--ksplit 1]
        [--all-ctas] [--backward]

--all-ctas (tensor-core recurrence): every CTA's stamps for steps 16..23, to
see how far apart the CTAs publish h_t and how long the last publication
takes to reach the other CTAs.

--backward: a training pass instead, and the stamps of layer 0's
reverse-time recurrence (the tensor-core kernel of a bf16 GRU, else the
FFMA kernel).

Which stamps exist depends on the kernel that ran (named by the profile):
tensor-core recurrence, portable SIMT recurrence, cluster-resident
recurrence, or the RSSM unroll.  See include/rcu.h for the slot meanings.
"""
import argparse
import sys

import numpy as np
import torch

from . import binding
from . import workloads as wl

WORKLOADS = {"lstm": wl.LSTM_T80, "rssm": wl.RSSM_B50, "lstmp": wl.LSTMP_2L,
             "bilstm": wl.BILSTM_VAR, "gru": wl.GRU_3L, "rssm_actor": wl.RSSM_ACTOR,
             "lstm_train": wl.LSTM_TRAIN, "bilstm_train": wl.BILSTM_TRAIN}

# (from slot, to slot, label) per kernel
PHASES = {
    "recurrent_tc": [(0, 1, "step barrier seen -> first h stage landed"),
                     (1, 8, "h stages streamed, MMAs issued"),
                     (8, 3, "last stage -> epilogue has the accumulator"),
                     (3, 5, "TMEM read (and partial sums sent)"),
                     (5, 11, "partner's partial sums received"),
                     (11, 13, "gates"),
                     (13, 6, "next step's G loads issued, h_t stored"),
                     (5, 6, "-> gates done, h_t stored"),
                     (6, 4, "h_t published")],
    "recurrent_simt": [(0, 3, "h_{t-1} rows loaded"), (3, 4, "mat-vec"),
                       (4, 1, "gates, h_t stored"), (1, 2, "step barrier")],
    "recurrent_cluster": [(0, 3, "mat-vec"), (3, 4, "gates"), (4, 1, "h_t sent")],
    "bwd_recurrent_tc": [(0, 1, "every dR_{t+1} published -> first stage landed"),
                         (1, 2, "dR stages streamed, MMAs issued"),
                         (2, 3, "last MMA issued -> epilogue has the accumulator"),
                         (3, 4, "accumulator read, partial sums sent"),
                         (4, 5, "peers' partial sums received"),
                         (5, 6, "gate gradients, dR_t stored and published"),
                         (6, 7, "gradient stores for the GEMMs"),
                         (7, 8, "next step's activations")],
    "bwd_recurrent": [(0, 1, "gate gradients of the CTA's units"),
                      (1, 2, "step barrier"),
                      (2, 3, "W_hh^T dR_t (dR_t staged from L2)"),
                      (3, 4, "K-slice partial sums")],
    "rssm": [(0, 5, "actor: ELU layer, tanh layer"), (5, 1, "Linear+ELU on [state, action]"),
             (0, 1, "[actor and] Linear+ELU on [state, action]"), (1, 2, "GRUCell"),
             (2, 3, "Linear+ELU"), (3, 4, "Linear, softplus, sample")],
}


def _medians(tr, phases):
    out = []
    for a, b, label in phases:
        if not (np.any(tr[:, a]) and np.any(tr[:, b])):
            continue
        out.append((label, float(np.median(tr[:, b] - tr[:, a]))))
    return out


ALL_S0, ALL_N, ALL_CTAS = 16, 8, 1024  # the library's all-CTA trace window


def all_cta_summary(rows: np.ndarray):
    """rows [ALL_N, ALL_CTAS, 16] of stamps.  Per step t (of the window):
    spread of the CTAs' publication times (slot 4), and the time from the
    last publication of step t to the first / median / last CTA seeing
    step t+1's barrier (slot 0)."""
    live = np.any(rows[0] != 0, axis=1)
    R = rows[:, live, :].astype(np.float64)
    out = {"ctas": int(live.sum())}
    spread, first, med, last, land, mma = [], [], [], [], [], []
    for i in range(ALL_N - 1):
        pub, nxt = R[i, :, 4], R[i + 1, :, 0]
        if not (np.all(pub) and np.all(nxt)):
            continue
        spread.append(pub.max() - pub.min())
        first.append(nxt.min() - pub.max())
        med.append(np.median(nxt) - pub.max())
        last.append(nxt.max() - pub.max())
        land.append(np.median(R[i + 1, :, 1] - R[i + 1, :, 0]))
        mma.append(np.median(R[i + 1, :, 2] - R[i + 1, :, 1]))
    if spread:
        out.update({
            "publish_spread_ns": float(np.median(spread)),
            "last_publish_to_first_barrier_seen_ns": float(np.median(first)),
            "last_publish_to_median_barrier_seen_ns": float(np.median(med)),
            "last_publish_to_last_barrier_seen_ns": float(np.median(last)),
            "median_barrier_seen_to_first_stage_ns": float(np.median(land)),
            "median_first_stage_to_last_mma_ns": float(np.median(mma))})
        # which CTAs publish last, most often
        lastc = [int(np.argmax(R[i, :, 4])) for i in range(ALL_N) if np.all(R[i, :, 4])]
        out["last_publisher_ctas"] = lastc
    return out


def run(workload: str, T: int = 0, ksplit: int = 0, seed: int = 0, all_ctas: bool = False,
        backward: bool = False):
    spec = WORKLOADS[workload]
    if T > 0:
        kw = {"T": T}
        if getattr(spec, "varlen", None) is not None:
            kw["varlen"] = (min(spec.varlen[0], T), T)
        spec = spec.scaled(**kw)
    dev = torch.device("cuda")
    if isinstance(spec, wl.RssmSpec):
        inp = wl.make_rssm_inputs(spec, seed=seed)
        m = binding.RSSM(spec.state_dim, spec.action_dim, spec.hidden, spec.rnn_hidden)
        m.set_weights(inp["weights"])
        e = inp["eps"].to(dev)
        if spec.actor_hidden:
            m.set_actor(inp["actor"])
            run1 = lambda: m.unroll_actor(e)  # noqa: E731
        else:
            a = inp["actions"].to(dev)
            run1 = lambda: m.unroll(a, e)  # noqa: E731
        for _ in range(3):
            run1()
        binding.rssm_set_attr(m.h, binding.RCU_ATTR_TRACE, 1)
        run1()
        tr = binding.rssm_get_trace(m.h, spec.T).numpy().astype(np.float64)
        kernel = "rssm"
    else:
        if backward:
            spec = spec.scaled(train=True)
        inp = wl.make_rnn_inputs(spec, seed=seed)
        net = binding.RNN.from_spec(spec)
        if ksplit:
            net.set_attr(binding.RCU_ATTR_TC_KSPLIT, ksplit)
        net.set_weights(inp["weights"])
        x = inp["x"].to(dev)
        h0 = inp["h0"].to(dev) if inp["h0"] is not None else None
        c0 = inp["c0"].to(dev) if inp["c0"] is not None else None
        L = inp["lengths"].to(dev) if inp["lengths"] is not None else None
        if backward:
            dy = inp["dy"].to(dev)
            run1 = lambda: net.backward(x, dy, lengths=L, h0=h0, c0=c0)  # noqa: E731
            for _ in range(3):
                run1()
            net.set_attr(binding.RCU_ATTR_TRACE, 1)
            net.set_attr(binding.RCU_ATTR_PROFILE, 1)
            run1()
            torch.cuda.synchronize()
            if net.status() != 0:
                raise RuntimeError("device status after the traced backward")
            kernel = ("bwd_recurrent_tc" if any(n.startswith("bwd_recurrent_tc")
                                                for n in net.profile()) else "bwd_recurrent")
            tr = binding.rnn_get_trace(net.h, spec.T + 1).numpy().astype(np.float64)
            net.close()
            body = tr[2:max(3, spec.T - 1)]
            pub = 6 if kernel == "bwd_recurrent_tc" else 0
            period = float(np.median(np.diff(body[:, pub]))) if len(body) > 1 else float("nan")
            res = {"workload": spec.name, "T": spec.T, "kernel": kernel,
                   "step_period_ns": period, "phases_ns": _medians(body, PHASES[kernel])}
            if kernel == "bwd_recurrent_tc":
                res["barrier_ns"] = float(np.median(body[1:, 0] - body[:-1, 6]))
            return res
        for _ in range(3):
            net.forward(x, lengths=L, h0=h0, c0=c0)
        net.set_attr(binding.RCU_ATTR_TRACE, 2 if all_ctas else 1)
        net.set_attr(binding.RCU_ATTR_PROFILE, 1)
        net.forward(x, lengths=L, h0=h0, c0=c0)
        torch.cuda.synchronize()
        if net.status() != 0:
            raise RuntimeError("device status after the traced forward")
        names = net.profile()
        kernel = next((k for k in ("recurrent_tc", "recurrent_cluster", "recurrent_simt")
                       if any(n.startswith(k) for n in names)), "recurrent_simt")
        rows = spec.T + (ALL_N * ALL_CTAS if all_ctas else 0)
        full = binding.rnn_get_trace(net.h, rows).numpy()
        tr = full[:spec.T].astype(np.float64)
        allc = full[spec.T:].reshape(ALL_N, ALL_CTAS, 16) if all_ctas else None
        net.close()
    body = tr[2:max(3, spec.T - 1)]  # skip the first steps (cold) and the last
    period = float(np.median(np.diff(body[:, 0]))) if len(body) > 1 else float("nan")
    res = {"workload": spec.name, "T": spec.T, "kernel": kernel, "step_period_ns": period,
           "phases_ns": _medians(body, PHASES[kernel])}
    if not isinstance(spec, wl.RssmSpec) and all_ctas:
        res["all_ctas"] = all_cta_summary(allc)
    if kernel == "recurrent_tc" and np.any(body[:, 10]):
        res["mma_thread_cycles"] = {"issuing": float(np.median(body[:, 10])),
                                    "waiting": float(np.median(body[:, 9]))}
        res["barrier_ns"] = float(np.median(body[1:, 0] - body[:-1, 4]))
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="gru", choices=sorted(WORKLOADS))
    ap.add_argument("--T", type=int, default=64, help="sequence length (0 = the workload's)")
    ap.add_argument("--ksplit", type=int, default=0, choices=[0, 1, 2, 4])
    ap.add_argument("--all-ctas", action="store_true",
                    help="also every CTA's stamps for steps 16..23 (tensor-core kernel)")
    ap.add_argument("--backward", action="store_true",
                    help="trace the tensor-core reverse-time recurrence of a training pass")
    args = ap.parse_args(argv)
    r = run(args.workload, args.T, args.ksplit, all_ctas=args.all_ctas, backward=args.backward)
    print(f"{r['workload']} T={r['T']} kernel={r['kernel']} "
          f"step period (median) {r['step_period_ns']:.0f} ns")
    for label, v in r["phases_ns"]:
        print(f"  {label:45s} {v:8.0f} ns")
    if "mma_thread_cycles" in r:
        c = r["mma_thread_cycles"]
        print(f"  MMA thread clock cycles: issuing {c['issuing']:.0f}, waiting {c['waiting']:.0f}")
        print(f"  {'h_t published -> next step barrier seen':45s} {r['barrier_ns']:8.0f} ns")
    elif "barrier_ns" in r:
        print(f"  {'dR_t published -> next step barrier seen':45s} {r['barrier_ns']:8.0f} ns")
    if "all_ctas" in r:
        for k, v in r["all_ctas"].items():
            print(f"  all CTAs: {k:45s} {v}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
