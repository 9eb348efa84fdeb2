// Host side of the C ABI's RSSM prior (include/rcu.h): the handle, weights
// and actor, the unroll (device and host buffers) and its backward pass
// through time.  Every step runs in this library's kernels.
#include <algorithm>
#include <cstdint>

#include "rcu.h"
#include "common.cuh"
#include "internal.h"
#include "api_host.h"

using namespace rcu;
using namespace rcu_api;

// ---------------------------------------------------------------------------
// RSSM handle

struct rcu_rssm_s : EventProfiler {
  int S, A, Hd, RH;
  int device, nsm;
  DevBuf W1, b1, Wih, Whh, bih, bhh, W2, b2, W3, b3;
  bool set = false;
  // actor of unroll variant 2 (rssm_set_actor)
  int Hx = 0;
  DevBuf Wa1, ba1, Wa2, ba2;
  int launches = 0;
  DevBuf ctl;  // device error word
  int64_t timeout_ns = 2000000000LL;  // bound on each wait for a broadcast vector
  int drop_send = 0;                  // testing: RCU_ATTR_TEST_DROP_ARRIVAL
  int force_path = 0;                 // RCU_ATTR_FORCE_PATH: 1 = backward chain as separate launches
  bool trace = false;
  DevBuf trace_buf;
  int trace_T = 0;
  // rssm_unroll_host / rssm_unroll_actor_host staging buffers
  DevBuf io_s0, io_b0, io_act, io_eps, io_out[5];
  // rssm_backward: workspace and the weight gradients of the last call (gwa:
  // the actor's, after rssm_backward_actor)
  DevBuf bw, gw, gwa;
  bool grads_ready = false, actor_grads_ready = false;
  // timed spans (RCU_ATTR_PROFILE); launches are counted by the callers
  void begin(const char *name, cudaStream_t s) { prof_begin(name, s); }
  void end(cudaStream_t s) { prof_end(s); }
};

extern "C" int rssm_set_attr(rcu_rssm_t h, int attr, int64_t value) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_set_attr: NULL handle");
  if (attr == RCU_ATTR_BARRIER_TIMEOUT_NS) {
    if (value <= 0) return fail(RCU_ERR_INVALID, "timeout must be > 0");
    h->timeout_ns = value;
    return RCU_OK;
  }
  if (attr == RCU_ATTR_TEST_DROP_ARRIVAL) {
    h->drop_send = value != 0;
    return RCU_OK;
  }
  if (attr == RCU_ATTR_PROFILE) {
    h->profile = value != 0;
    return RCU_OK;
  }
  if (attr == RCU_ATTR_FORCE_PATH) {
    if (value != 0 && value != 1) return fail(RCU_ERR_INVALID, "RSSM force_path must be 0 or 1");
    h->force_path = (int)value;
    return RCU_OK;
  }
  if (attr != RCU_ATTR_TRACE) return fail(RCU_ERR_INVALID, "rssm_set_attr: unknown attribute %d", attr);
  h->trace = value != 0;
  return RCU_OK;
}

extern "C" int rssm_get_trace(rcu_rssm_t h, int64_t *host_out, int n_steps, void *stream) {
  if (!h || !host_out || n_steps < 0) return fail(RCU_ERR_INVALID, "rssm_get_trace: bad arguments");
  if (!h->trace_buf.p) return fail(RCU_ERR_STATE, "rssm_get_trace: no traced unroll");
  const int n = std::min(n_steps, h->trace_T);
  CU(cudaStreamSynchronize((cudaStream_t)stream));
  CU(cudaMemcpy(host_out, h->trace_buf.p, (size_t)n * 16 * 8, cudaMemcpyDeviceToHost));
  return RCU_OK;
}

extern "C" int rssm_create(rcu_rssm_t *out, int state_dim, int action_dim, int hidden,
                           int rnn_hidden) {
  if (!out) return fail(RCU_ERR_INVALID, "rssm_create: out is NULL");
  *out = nullptr;
  if (state_dim < 1 || action_dim < 0 || hidden < 1 || rnn_hidden < 1)
    return fail(RCU_ERR_INVALID, "rssm_create: dims must be >= 1 (action_dim >= 0)");
  if (!rssm_supported(state_dim, action_dim, hidden, rnn_hidden))
    return fail(RCU_ERR_UNSUPPORTED, "rssm_create: weights do not fit one cluster's shared memory");
  auto *h = new rcu_rssm_s();
  h->S = state_dim; h->A = action_dim; h->Hd = hidden; h->RH = rnn_hidden;
  h->nsm = device_sm_count(&h->device);
  if (h->ctl.ensure(256) != cudaSuccess) { delete h; return fail(RCU_ERR_CUDA, "rssm_create: alloc"); }
  cudaMemset(h->ctl.p, 0, 256);
  *out = h;
  return RCU_OK;
}

extern "C" int rssm_set_weights(rcu_rssm_t h, const float *W1, const float *b1, const float *W_ih,
                                const float *W_hh, const float *b_ih, const float *b_hh,
                                const float *W2, const float *b2, const float *W3, const float *b3,
                                void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_set_weights: NULL handle");
  if (!W1 || !W_ih || !W_hh || !W2 || !W3)
    return fail(RCU_ERR_INVALID, "rssm_set_weights: weight matrices are required");
  cudaStream_t s = (cudaStream_t)stream;
  const int S = h->S, A = h->A, Hd = h->Hd, RH = h->RH;
  struct Item { DevBuf *dst; const float *src; size_t n; };
  Item items[] = {{&h->W1, W1, (size_t)Hd * (S + A)}, {&h->b1, b1, (size_t)Hd},
                  {&h->Wih, W_ih, (size_t)3 * RH * Hd}, {&h->Whh, W_hh, (size_t)3 * RH * RH},
                  {&h->bih, b_ih, (size_t)3 * RH}, {&h->bhh, b_hh, (size_t)3 * RH},
                  {&h->W2, W2, (size_t)Hd * RH}, {&h->b2, b2, (size_t)Hd},
                  {&h->W3, W3, (size_t)2 * S * Hd}, {&h->b3, b3, (size_t)2 * S}};
  for (auto &it : items) {
    CU(it.dst->ensure(std::max<size_t>(it.n, 1) * 4));
    if (it.src)
      CU(cudaMemcpyAsync(it.dst->p, it.src, it.n * 4, cudaMemcpyDeviceToDevice, s));
    else
      CU(cudaMemsetAsync(it.dst->p, 0, it.n * 4, s));
  }
  CU(cudaStreamSynchronize(s));
  h->set = true;
  return RCU_OK;
}

extern "C" int rssm_set_actor(rcu_rssm_t h, int actor_hidden, const float *Wa1, const float *ba1,
                              const float *Wa2, const float *ba2, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_set_actor: NULL handle");
  if (actor_hidden < 1 || !Wa1 || !Wa2 || h->A < 1)
    return fail(RCU_ERR_INVALID, "rssm_set_actor: need actor_hidden >= 1, Wa1, Wa2, action_dim >= 1");
  if (!rssm_supported(h->S, h->A, h->Hd, h->RH, actor_hidden))
    return fail(RCU_ERR_UNSUPPORTED, "rssm_set_actor: weights do not fit one cluster's shared memory");
  cudaStream_t s = (cudaStream_t)stream;
  const int S = h->S, A = h->A, RH = h->RH, Hx = actor_hidden;
  struct Item { DevBuf *dst; const float *src; size_t n; };
  Item items[] = {{&h->Wa1, Wa1, (size_t)Hx * (S + RH)}, {&h->ba1, ba1, (size_t)Hx},
                  {&h->Wa2, Wa2, (size_t)A * Hx}, {&h->ba2, ba2, (size_t)A}};
  for (auto &it : items) {
    CU(it.dst->ensure(std::max<size_t>(it.n, 1) * 4));
    if (it.src)
      CU(cudaMemcpyAsync(it.dst->p, it.src, it.n * 4, cudaMemcpyDeviceToDevice, s));
    else
      CU(cudaMemsetAsync(it.dst->p, 0, it.n * 4, s));
  }
  CU(cudaStreamSynchronize(s));
  h->Hx = Hx;
  return RCU_OK;
}

static int rssm_run(rcu_rssm_t h, bool with_actor, int T, int B, const float *state0,
                    const float *belief0, const float *actions, const float *eps, float *means,
                    float *stds, float *states, float *beliefs, float *actions_out, void *stream) {
  const char *fn = with_actor ? "rssm_unroll_actor" : "rssm_unroll";
  if (!h) return fail(RCU_ERR_INVALID, "%s: NULL handle", fn);
  h->launches = 0;
  if (!h->set) return fail(RCU_ERR_STATE, "%s: weights not set", fn);
  if (with_actor && h->Hx < 1) return fail(RCU_ERR_STATE, "%s: actor not set", fn);
  if (T < 0 || B < 0) return fail(RCU_ERR_INVALID, "%s: T and B must be >= 0", fn);
  if (T == 0 || B == 0) return RCU_OK;
  if ((!with_actor && h->A > 0 && !actions) || !eps || !means || !stds || !states || !beliefs)
    return fail(RCU_ERR_INVALID, "%s: actions (without an actor), eps and all outputs are required",
                fn);
  RssmParams p{};
  p.S = h->S; p.A = h->A; p.Hd = h->Hd; p.RH = h->RH; p.T = T; p.B = B;
  p.W1 = (const float *)h->W1.p; p.b1 = (const float *)h->b1.p;
  p.Wih = (const float *)h->Wih.p; p.Whh = (const float *)h->Whh.p;
  p.bih = (const float *)h->bih.p; p.bhh = (const float *)h->bhh.p;
  p.W2 = (const float *)h->W2.p; p.b2 = (const float *)h->b2.p;
  p.W3 = (const float *)h->W3.p; p.b3 = (const float *)h->b3.p;
  p.state0 = state0; p.belief0 = belief0; p.actions = actions; p.eps = eps;
  p.means = means; p.stds = stds; p.states = states; p.beliefs = beliefs;
  if (with_actor) {
    p.actions = nullptr;
    p.Hx = h->Hx;
    p.Wa1 = (const float *)h->Wa1.p; p.ba1 = (const float *)h->ba1.p;
    p.Wa2 = (const float *)h->Wa2.p; p.ba2 = (const float *)h->ba2.p;
    p.actions_out = actions_out;
  }
  p.err = (int *)h->ctl.p;
  p.timeout_ns = (uint64_t)h->timeout_ns;
  p.drop_send = h->drop_send;
  p.trace = nullptr;
  if (h->trace) {
    CU(h->trace_buf.ensure((size_t)T * 16 * 8));
    CU(cudaMemsetAsync(h->trace_buf.p, 0, (size_t)T * 16 * 8, (cudaStream_t)stream));
    h->trace_T = T;
    p.trace = (unsigned long long *)h->trace_buf.p;
  }
  int clusters = 0;
  h->begin(with_actor ? "rssm_unroll_actor" : "rssm_unroll", (cudaStream_t)stream);
  cudaError_t e = launch_rssm(p, h->nsm, (cudaStream_t)stream, &clusters);
  h->end((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rssm kernel launch: %s", cudaGetErrorString(e));
  h->launches = 1;
  return RCU_OK;
}

extern "C" int rssm_unroll(rcu_rssm_t h, int T, int B, const float *state0, const float *belief0,
                           const float *actions, const float *eps, float *means, float *stds,
                           float *states, float *beliefs, void *stream) {
  return rssm_run(h, false, T, B, state0, belief0, actions, eps, means, stds, states, beliefs,
                  nullptr, stream);
}

extern "C" int rssm_unroll_actor(rcu_rssm_t h, int T, int B, const float *state0,
                                 const float *belief0, const float *eps, float *means, float *stds,
                                 float *states, float *beliefs, float *actions_out, void *stream) {
  return rssm_run(h, true, T, B, state0, belief0, nullptr, eps, means, stds, states, beliefs,
                  actions_out, stream);
}

// Host-buffer form of both unrolls: inputs staged, outputs in place when
// page-locked (written by the kernel over the CPU-GPU link), else staged.
static int rssm_run_host(rcu_rssm_t h, bool with_actor, int T, int B, const float *state0,
                         const float *belief0, const float *actions, const float *eps,
                         float *means, float *stds, float *states, float *beliefs,
                         float *actions_out, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm host unroll: NULL handle");
  if (T <= 0 || B <= 0)
    return rssm_run(h, with_actor, T, B, state0, belief0, actions, eps, means, stds, states,
                    beliefs, actions_out, stream);
  const size_t TB = (size_t)T * B;
  HostIO io{(cudaStream_t)stream, {}};
  const void *ds0, *db0, *dact, *deps;
  CU(io.in(state0, (size_t)B * h->S * 4, h->io_s0, false, &ds0));
  CU(io.in(belief0, (size_t)B * h->RH * 4, h->io_b0, false, &db0));
  CU(io.in(with_actor ? nullptr : actions, TB * h->A * 4, h->io_act, false, &dact));
  CU(io.in(eps, TB * h->S * 4, h->io_eps, false, &deps));
  void *d[5];
  float *outs[5] = {means, stds, states, beliefs, actions_out};
  const size_t w[5] = {(size_t)h->S, (size_t)h->S, (size_t)h->S, (size_t)h->RH, (size_t)h->A};
  for (int i = 0; i < 5; ++i) CU(io.out(outs[i], TB * w[i] * 4, h->io_out[i], true, &d[i]));
  const int rc = rssm_run(h, with_actor, T, B, (const float *)ds0, (const float *)db0,
                          (const float *)dact, (const float *)deps, (float *)d[0], (float *)d[1],
                          (float *)d[2], (float *)d[3], (float *)d[4], stream);
  if (rc != RCU_OK) return rc;
  CU(io.finish());
  return RCU_OK;
}

extern "C" int rssm_unroll_host(rcu_rssm_t h, int T, int B, const float *state0,
                                const float *belief0, const float *actions, const float *eps,
                                float *means, float *stds, float *states, float *beliefs,
                                void *stream) {
  return rssm_run_host(h, false, T, B, state0, belief0, actions, eps, means, stds, states, beliefs,
                       nullptr, stream);
}

extern "C" int rssm_unroll_actor_host(rcu_rssm_t h, int T, int B, const float *state0,
                                      const float *belief0, const float *eps, float *means,
                                      float *stds, float *states, float *beliefs,
                                      float *actions_out, void *stream) {
  return rssm_run_host(h, true, T, B, state0, belief0, nullptr, eps, means, stds, states, beliefs,
                       actions_out, stream);
}

// Backward pass through time of the unroll with given actions.  The forward
// is run again (states and beliefs kept); every quantity off the reverse-time
// chain is then recomputed over all T*B rows (GEMMs, ELU, the GRU gates by
// the same activation scan as the stacked-RNN backward); the chain runs one
// step at a time as five batched mat-vecs between elementwise kernels; the
// weight and action gradients are GEMMs over all rows afterwards.
// With the actor (unroll variant 2) the actions are the forward's own: the
// actor's layers are recomputed over all rows like the prior's, and each step
// of the chain also takes the gradient reaching a_t back through tanh, Wa2,
// ELU and Wa1 into s_{t-1} and h_{t-1}.
static int rssm_backward_run(rcu_rssm_t h, bool with_actor, int T, int B, const float *state0,
                             const float *belief0, const float *actions, const float *eps,
                             const float *dmeans, const float *dstds, const float *dstates,
                             const float *dbeliefs, float *dstate0, float *dbelief0,
                             float *dactions, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_backward: NULL handle");
  h->launches = 0;
  if (!h->set) return fail(RCU_ERR_STATE, "rssm_backward: weights not set");
  if (with_actor && h->Hx < 1) return fail(RCU_ERR_STATE, "rssm_backward_actor: actor not set");
  if (T < 1 || B < 1 || !eps || (!with_actor && h->A > 0 && !actions))
    return fail(RCU_ERR_INVALID, "rssm_backward: need T, B >= 1, eps and actions (action_dim > 0)");
  if ((size_t)T * B > (size_t)INT32_MAX / 8)
    return fail(RCU_ERR_UNSUPPORTED, "rssm_backward: T*B too large");
  cudaStream_t s = (cudaStream_t)stream;
  const int S = h->S, A = h->A, Hd = h->Hd, RH = h->RH, G = 3 * RH, SA = S + A, S2 = 2 * S;
  const int Hx = with_actor ? h->Hx : 0, SR = S + RH;
  const int M = T * B;
  // the weight-gradient groups' shapes (dZ width, Y width), for the scratch
  // of their chunk partials: W1, W_ih, W_hh, W2, W3 (and the actor's Wa2, Wa1)
  const WgradGroup wshape[7] = {{nullptr, Hd, nullptr, SA}, {nullptr, G, nullptr, Hd},
                                {nullptr, G, nullptr, RH}, {nullptr, Hd, nullptr, RH},
                                {nullptr, S2, nullptr, Hd}, {nullptr, A, nullptr, Hx},
                                {nullptr, Hx, nullptr, SR}};
  size_t off = 0;
  auto take = [&](size_t n) { size_t r = off; off += (n + 63) & ~size_t(63); return r; };
  const size_t o_mean = take((size_t)M * S), o_std = take((size_t)M * S),
               o_st = take((size_t)M * S), o_bel = take((size_t)M * RH),
               o_in = take((size_t)M * SA), o_u = take((size_t)M * Hd), o_x = take((size_t)M * Hd),
               o_hp = take((size_t)M * RH), o_zi = take((size_t)M * G), o_zh = take((size_t)M * G),
               o_v = take((size_t)M * Hd), o_q = take((size_t)M * Hd), o_p = take((size_t)M * S2),
               o_dp = take((size_t)M * S2), o_dv = take((size_t)M * Hd),
               o_da = take((size_t)M * G), o_dr = take((size_t)M * G), o_du = take((size_t)M * Hd),
               o_tq = take((size_t)B * Hd), o_thq = take((size_t)B * RH),
               o_gh = take((size_t)B * RH), o_dhz = take((size_t)B * RH),
               o_tx = take((size_t)B * Hd), o_cs = take((size_t)B * S),
               o_w3t = take((size_t)Hd * S2), o_w2t = take((size_t)RH * Hd),
               o_whht = take((size_t)RH * G), o_wiht = take((size_t)Hd * G),
               o_w1st = take((size_t)S * Hd), o_w1at = take((size_t)std::max(A, 1) * Hd),
               o_wg = take(wgrad_scratch_floats(wshape, with_actor ? 7 : 5, M));
  // actor only: its actions, inputs [s_{t-1}, h_{t-1}], layers and gradients
  const size_t na = with_actor ? 1 : 0;
  const size_t o_acts = take(na * M * A), o_xa = take(na * M * SR), o_ua = take(na * M * Hx),
               o_ha = take(na * M * Hx), o_dact = take(na * M * A), o_dva = take(na * M * A),
               o_dha = take(na * M * Hx), o_tdha = take(na * B * Hx), o_csa = take(na * B * S),
               o_ga = take(na * B * RH), o_wa2t = take(na * Hx * A), o_wa1st = take(na * S * Hx),
               o_wa1ht = take(na * RH * Hx);
  CU(h->bw.ensure(off * 4));
  float *ws = (float *)h->bw.p;
  float *means = ws + o_mean, *stds = ws + o_std, *states = ws + o_st, *bel = ws + o_bel;
  float *IN = ws + o_in, *U = ws + o_u, *X = ws + o_x, *HP = ws + o_hp, *ZI = ws + o_zi,
        *ZH = ws + o_zh, *V = ws + o_v, *Q = ws + o_q, *Pm = ws + o_p, *DP = ws + o_dp,
        *DV = ws + o_dv, *DA = ws + o_da, *DR = ws + o_dr, *DU = ws + o_du;
  float *TQ = ws + o_tq, *THQ = ws + o_thq, *GH = ws + o_gh, *DHZ = ws + o_dhz, *TX = ws + o_tx,
        *CS = ws + o_cs;
  float *W3T = ws + o_w3t, *W2T = ws + o_w2t, *WhhT = ws + o_whht, *WihT = ws + o_wiht,
        *W1sT = ws + o_w1st, *W1aT = ws + o_w1at, *WG = ws + o_wg;
  float *ACTS = ws + o_acts, *XA = ws + o_xa, *UA = ws + o_ua, *HA = ws + o_ha,
        *DACT = ws + o_dact, *DVA = ws + o_dva, *DHA = ws + o_dha, *TDHA = ws + o_tdha,
        *CSA = ws + o_csa, *GA = ws + o_ga, *Wa2T = ws + o_wa2t, *Wa1sT = ws + o_wa1st,
        *Wa1hT = ws + o_wa1ht;
  const float *Wa1 = (const float *)h->Wa1.p, *ba1 = (const float *)h->ba1.p;
  const float *Wa2 = (const float *)h->Wa2.p;
  const float *W1 = (const float *)h->W1.p, *b1 = (const float *)h->b1.p;
  const float *Wih = (const float *)h->Wih.p, *Whh = (const float *)h->Whh.p;
  const float *bih = (const float *)h->bih.p, *bhh = (const float *)h->bhh.p;
  const float *W2 = (const float *)h->W2.p, *b2 = (const float *)h->b2.p;
  const float *W3 = (const float *)h->W3.p, *b3 = (const float *)h->b3.p;
  h->grads_ready = false;
  h->actor_grads_ready = false;
  // ---- forward again (clears and may set the handle's error word); with the
  // actor it also returns the actions it produced
  int rc = rssm_run(h, with_actor, T, B, state0, belief0, with_actor ? nullptr : actions, eps,
                    means, stds, states, bel, with_actor ? ACTS : nullptr, stream);
  if (rc != RCU_OK) return rc;
  const float *acts = with_actor ? ACTS : actions;
  int launches = h->launches;
  int *err = (int *)h->ctl.p;
  cudaError_t e = cudaSuccess;
  auto gemm = [&](const float *Xp, int ldx, const float *Wp, int ldw, const float *bias, float *Gp,
                  int ldg, int m, int n, int k) {
    if (e == cudaSuccess)
      e = launch_gemm_simt<float, float>(Xp, ldx, Wp, ldw, bias, Gp, ldg, m, nullptr, n, k, s, err);
    ++launches;
  };
  auto tr = [&](const float *in, int R, int C, int ldi, float *out, int ldo) {
    if (e == cudaSuccess) e = launch_transpose(in, R, C, ldi, out, ldo, s);
    ++launches;
  };
  // ---- everything off the reverse-time chain, over all T*B rows
  h->begin("rssm_bwd_recompute", s);
  if (belief0) CU(cudaMemcpyAsync(HP, belief0, (size_t)B * RH * 4, cudaMemcpyDeviceToDevice, s));
  else CU(cudaMemsetAsync(HP, 0, (size_t)B * RH * 4, s));      // h_{t-1}
  if (T > 1)
    CU(cudaMemcpyAsync(HP + (size_t)B * RH, bel, (size_t)(T - 1) * B * RH * 4,
                       cudaMemcpyDeviceToDevice, s));
  if (e == cudaSuccess) e = launch_rssm_inputs(T, B, S, A, state0, states, acts, IN, s);
  ++launches;
  gemm(IN, SA, W1, SA, b1, U, Hd, M, Hd, SA);                    // u = W1 [s, a] + b1
  if (e == cudaSuccess) e = launch_elu(U, X, (size_t)M * Hd, s);  // x = ELU(u)
  ++launches;
  if (with_actor) {
    // actor input [s_{t-1}, h_{t-1}] (the inputs kernel with h_{t-1} in the
    // action slot), ua = Wa1 [s, h] + ba1, ha = ELU(ua)
    if (e == cudaSuccess) e = launch_rssm_inputs(T, B, S, RH, state0, states, HP, XA, s);
    ++launches;
    gemm(XA, SR, Wa1, SR, ba1, UA, Hx, M, Hx, SR);
    if (e == cudaSuccess) e = launch_elu(UA, HA, (size_t)M * Hx, s);
    ++launches;
    tr(Wa2, A, Hx, Hx, Wa2T, A);            // [Hx][A]
    tr(Wa1, Hx, S, SR, Wa1sT, Hx);          // state columns, [S][Hx]
    tr(Wa1 + S, Hx, RH, SR, Wa1hT, Hx);     // belief columns, [RH][Hx]
  }
  gemm(X, Hd, Wih, Hd, bih, ZI, G, M, G, Hd);                    // input-side gate pre-activations
  gemm(HP, RH, Whh, RH, bhh, ZH, G, M, G, RH);                   // hidden-side
  if (e == cudaSuccess) e = launch_bwd_prep(T, B, RH, RCU_GRU, ZI, ZH, nullptr, nullptr, nullptr, s);
  ++launches;                                                    // ZI <- r, z, n
  gemm(bel, RH, W2, RH, b2, V, Hd, M, Hd, RH);                   // v = W2 h + b2
  if (e == cudaSuccess) e = launch_elu(V, Q, (size_t)M * Hd, s);  // q = ELU(v)
  ++launches;
  gemm(Q, Hd, W3, Hd, b3, Pm, S2, M, S2, Hd);                    // p = W3 q + b3
  // the given-actions chain runs as one cluster kernel with the weights
  // resident (it reads them untransposed) when they fit; otherwise, and with
  // the actor, as batched mat-vecs between elementwise kernels
  const bool fused = !with_actor && h->force_path != 1 && rssm_bwd_chain_supported(S, A, Hd, RH);
  // transposed weights for the chain's mat-vecs (X W^T form of the GEMM)
  if (!fused) {
    tr(W3, S2, Hd, Hd, W3T, S2);
    tr(W2, Hd, RH, RH, W2T, Hd);
    tr(Whh, G, RH, RH, WhhT, G);
    tr(Wih, G, Hd, Hd, WihT, G);
    tr(W1, Hd, S, SA, W1sT, Hd);
  }
  if (A > 0) tr(W1 + S, Hd, A, SA, W1aT, Hd);
  h->end(s);
  if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rssm_backward: recompute: %s", cudaGetErrorString(e));
  // ---- the reverse-time chain (one timed span over all its launches)
  h->begin("rssm_bwd_chain", s);
  if (fused) {
    RssmBwdChainParams cp{};
    cp.S = S; cp.A = A; cp.Hd = Hd; cp.RH = RH; cp.T = T; cp.B = B;
    cp.W1 = W1; cp.Wih = Wih; cp.Whh = Whh; cp.W2 = W2; cp.W3 = W3;
    cp.dmeans = dmeans; cp.dstds = dstds; cp.dstates = dstates; cp.dbeliefs = dbeliefs;
    cp.eps = eps; cp.p = Pm; cp.v = V; cp.u = U; cp.gates = ZI; cp.zh = ZH; cp.hp = HP;
    cp.DP = DP; cp.DV = DV; cp.DA = DA; cp.DR = DR; cp.DU = DU;
    cp.cs_out = CS;  // ds_{-1}
    cp.gh_out = GH;  // dh_{-1}, the W_hh^T dR_0 and z_0 dh_0 parts together
    cp.err = err;
    cp.timeout_ns = (uint64_t)h->timeout_ns;
    e = launch_rssm_bwd_chain(cp, h->nsm, s);
    ++launches;
    CU(cudaMemsetAsync(DHZ, 0, (size_t)B * RH * 4, s));  // already in GH
  } else {
    CU(cudaMemsetAsync(GH, 0, (size_t)B * RH * 4, s));
    CU(cudaMemsetAsync(DHZ, 0, (size_t)B * RH * 4, s));
    CU(cudaMemsetAsync(CS, 0, (size_t)B * S * 4, s));
  }
  for (int t = T - 1; !fused && t >= 0 && e == cudaSuccess; --t) {
    const size_t r0 = (size_t)t * B;
    e = launch_rssm_sample_grad(t, B, S, dmeans, dstds, dstates, eps, Pm, CS, DP, s);
    ++launches;
    gemm(DP + r0 * S2, S2, W3T, S2, nullptr, TQ, Hd, B, Hd, S2);      // dq = W3^T dp
    if (e == cudaSuccess) e = launch_elu_grad(TQ, V + r0 * Hd, DV + r0 * Hd, (size_t)B * Hd, s);
    ++launches;
    gemm(DV + r0 * Hd, Hd, W2T, Hd, nullptr, THQ, RH, B, RH, Hd);     // W2^T dv
    if (e == cudaSuccess)
      e = launch_rssm_gru_grad(t, B, RH, dbeliefs, THQ, GH, DHZ, ZI, ZH, HP, DA, DR, s);
    ++launches;
    gemm(DR + r0 * G, G, WhhT, G, nullptr, GH, RH, B, RH, G);          // W_hh^T dR_t
    gemm(DA + r0 * G, G, WihT, G, nullptr, TX, Hd, B, Hd, G);          // dx = W_ih^T dA_t
    if (e == cudaSuccess) e = launch_elu_grad(TX, U + r0 * Hd, DU + r0 * Hd, (size_t)B * Hd, s);
    ++launches;
    gemm(DU + r0 * Hd, Hd, W1sT, Hd, nullptr, CS, S, B, S, Hd);       // ds_{t-1} part
    if (with_actor) {
      // the gradient reaching a_t, back through tanh, Wa2, ELU and Wa1
      gemm(DU + r0 * Hd, Hd, W1aT, Hd, nullptr, DACT + r0 * A, A, B, A, Hd);
      if (e == cudaSuccess)
        e = launch_tanh_grad(DACT + r0 * A, ACTS + r0 * A, DVA + r0 * A, (size_t)B * A, s);
      ++launches;
      gemm(DVA + r0 * A, A, Wa2T, A, nullptr, TDHA, Hx, B, Hx, A);
      if (e == cudaSuccess) e = launch_elu_grad(TDHA, UA + r0 * Hx, DHA + r0 * Hx, (size_t)B * Hx, s);
      ++launches;
      gemm(DHA + r0 * Hx, Hx, Wa1sT, Hx, nullptr, CSA, S, B, S, Hx);  // into ds_{t-1}
      if (e == cudaSuccess) e = launch_add(CS, CSA, (size_t)B * S, s);
      ++launches;
      gemm(DHA + r0 * Hx, Hx, Wa1hT, Hx, nullptr, GA, RH, B, RH, Hx); // into dh_{t-1}
      if (e == cudaSuccess) e = launch_add(GH, GA, (size_t)B * RH, s);
      ++launches;
    }
  }
  h->end(s);
  if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rssm_backward: recurrence: %s", cudaGetErrorString(e));
  h->begin("rssm_bwd_grads", s);
  if (dstate0) CU(cudaMemcpyAsync(dstate0, CS, (size_t)B * S * 4, cudaMemcpyDeviceToDevice, s));
  if (dbelief0) {
    CU(cudaMemcpyAsync(dbelief0, GH, (size_t)B * RH * 4, cudaMemcpyDeviceToDevice, s));
    e = launch_add(dbelief0, DHZ, (size_t)B * RH, s);
    ++launches;
  }
  if (with_actor && dactions)
    CU(cudaMemcpyAsync(dactions, DACT, (size_t)M * A * 4, cudaMemcpyDeviceToDevice, s));
  else if (A > 0 && dactions)
    gemm(DU, Hd, W1aT, Hd, nullptr, dactions, A, M, A, Hd);
  // ---- weight gradients: dW = dZ^T Y and db = column sums of dZ, every
  // layer's in one grouped pair of launches over the row-major activations
  const size_t nW[10] = {(size_t)Hd * SA, (size_t)Hd, (size_t)G * Hd, (size_t)G * RH, (size_t)G,
                         (size_t)G, (size_t)Hd * RH, (size_t)Hd, (size_t)S2 * Hd, (size_t)S2};
  size_t tot = 0;
  for (size_t v : nW) tot += v;
  CU(h->gw.ensure(tot * 4));
  float *gp[10];
  gp[0] = (float *)h->gw.p;
  for (int i = 1; i < 10; ++i) gp[i] = gp[i - 1] + nW[i - 1];
  WgradGroup wg[7] = {{DU, Hd, IN, SA, gp[0], gp[1]}, {DA, G, X, Hd, gp[2], gp[4]},
                      {DR, G, HP, RH, gp[3], gp[5]}, {DV, Hd, bel, RH, gp[6], gp[7]},
                      {DP, S2, Q, Hd, gp[8], gp[9]}};
  int ng = 5;
  if (with_actor) {
    // dWa2 = dVa^T ha, dba2; dWa1 = dHa^T [s, h], dba1
    CU(h->gwa.ensure(((size_t)Hx * SR + Hx + (size_t)A * Hx + A) * 4));
    float *gWa1 = (float *)h->gwa.p, *gba1 = gWa1 + (size_t)Hx * SR, *gWa2 = gba1 + Hx,
          *gba2 = gWa2 + (size_t)A * Hx;
    wg[ng++] = {DVA, A, HA, Hx, gWa2, gba2};
    wg[ng++] = {DHA, Hx, XA, SR, gWa1, gba1};
  }
  if (e == cudaSuccess) e = launch_wgrad(wg, ng, M, WG, s);
  launches += 2;
  h->end(s);
  if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rssm_backward: gradients: %s", cudaGetErrorString(e));
  h->grads_ready = true;
  h->actor_grads_ready = with_actor;
  h->launches = launches;
  return RCU_OK;
}

extern "C" int rssm_backward(rcu_rssm_t h, int T, int B, const float *state0,
                             const float *belief0, const float *actions, const float *eps,
                             const float *dmeans, const float *dstds, const float *dstates,
                             const float *dbeliefs, float *dstate0, float *dbelief0,
                             float *dactions, void *stream) {
  return rssm_backward_run(h, false, T, B, state0, belief0, actions, eps, dmeans, dstds, dstates,
                           dbeliefs, dstate0, dbelief0, dactions, stream);
}

extern "C" int rssm_backward_actor(rcu_rssm_t h, int T, int B, const float *state0,
                                   const float *belief0, const float *eps, const float *dmeans,
                                   const float *dstds, const float *dstates,
                                   const float *dbeliefs, float *dstate0, float *dbelief0,
                                   float *dactions, void *stream) {
  return rssm_backward_run(h, true, T, B, state0, belief0, nullptr, eps, dmeans, dstds, dstates,
                           dbeliefs, dstate0, dbelief0, dactions, stream);
}

extern "C" int rssm_get_actor_grads(rcu_rssm_t h, float *dWa1, float *dba1, float *dWa2,
                                    float *dba2, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_get_actor_grads: NULL handle");
  if (!h->actor_grads_ready)
    return fail(RCU_ERR_STATE, "rssm_get_actor_grads: no rssm_backward_actor has run");
  const int SR = h->S + h->RH, Hx = h->Hx, A = h->A;
  const size_t n[4] = {(size_t)Hx * SR, (size_t)Hx, (size_t)A * Hx, (size_t)A};
  float *dst[4] = {dWa1, dba1, dWa2, dba2};
  const float *src = (const float *)h->gwa.p;
  for (int i = 0; i < 4; ++i) {
    if (dst[i])
      CU(cudaMemcpyAsync(dst[i], src, n[i] * 4, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    src += n[i];
  }
  return RCU_OK;
}

extern "C" int rssm_get_weight_grads(rcu_rssm_t h, float *dW1, float *db1, float *dW_ih,
                                     float *dW_hh, float *db_ih, float *db_hh, float *dW2,
                                     float *db2, float *dW3, float *db3, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_get_weight_grads: NULL handle");
  if (!h->grads_ready) return fail(RCU_ERR_STATE, "rssm_get_weight_grads: no rssm_backward has run");
  const int S = h->S, A = h->A, Hd = h->Hd, RH = h->RH, G = 3 * RH;
  const size_t nW[10] = {(size_t)Hd * (S + A), (size_t)Hd, (size_t)G * Hd, (size_t)G * RH,
                         (size_t)G, (size_t)G, (size_t)Hd * RH, (size_t)Hd, (size_t)2 * S * Hd,
                         (size_t)2 * S};
  float *dst[10] = {dW1, db1, dW_ih, dW_hh, db_ih, db_hh, dW2, db2, dW3, db3};
  const float *src = (const float *)h->gw.p;
  for (int i = 0; i < 10; ++i) {
    if (dst[i])
      CU(cudaMemcpyAsync(dst[i], src, nW[i] * 4, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    src += nW[i];
  }
  return RCU_OK;
}

extern "C" int rssm_profile_entry(rcu_rssm_t h, int i, const char **name, double *total_ms,
                                  int64_t *count) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_profile_entry: NULL handle");
  return h->entry(i, name, total_ms, count);
}

extern "C" int rssm_profile_reset(rcu_rssm_t h) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_profile_reset: NULL handle");
  h->reset();
  return RCU_OK;
}

extern "C" int rssm_get_status(rcu_rssm_t h, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rssm_get_status: NULL handle");
  CU(cudaStreamSynchronize((cudaStream_t)stream));
  CU(cudaGetLastError());
  int v = 0;
  CU(cudaMemcpy(&v, h->ctl.p, sizeof v, cudaMemcpyDeviceToHost));
  CU(cudaMemset(h->ctl.p, 0, sizeof v));
  return status_from_dev(v);
}

extern "C" int rssm_last_launch_count(rcu_rssm_t h) { return h ? h->launches : -1; }

extern "C" int rssm_destroy(rcu_rssm_t h) {
  if (!h) return RCU_OK;
  cudaDeviceSynchronize();
  delete h;
  return RCU_OK;
}
