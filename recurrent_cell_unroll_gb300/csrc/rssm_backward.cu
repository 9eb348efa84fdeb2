// Backward pass through time of the RSSM prior unroll with given actions:
// the training use of the unroll behind "[Feature Request] CUDNN version of
// RSSM" (pytorch/rl issue 366, Motivation: the Python loop over the prior
// dominates the training step; the step itself is the issue's Solution,
// RSSMPrior.forward with the first unroll_rssm).
//
// One step of the prior, per row:
//   u = W1 [s_{t-1}, a_t] + b1,  x = ELU(u),  h_t = GRUCell(x, h_{t-1}),
//   v = W2 h_t + b2,  q = ELU(v),  p = W3 q + b3,
//   mean = p[:S],  std = softplus(p[S:]) + 0.1,  s_t = mean + eps_t * std.
// Everything that does not depend on the reverse-time chain is recomputed
// over all T*B rows at once (GEMMs and elementwise kernels from the forward's
// saved states and beliefs).  The chain itself, ds_t -> dp -> dv -> dh_t ->
// gate gradients -> du -> ds_{t-1} and dh_{t-1}, runs one step at a time as
// small batched mat-vecs (B rows) between the elementwise kernels here; the
// weight and action gradients are GEMMs over all rows after the sweep.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace rcu {

namespace {

constexpr int EW = 256;

inline unsigned ew_blocks(size_t n) {
  return (unsigned)std::min<size_t>((n + EW - 1) / EW, 65535u * 8);
}

// IN[t][b] = [s_{t-1}, a_t]: s_{-1} = state0 (NULL: 0), then the states
__global__ void rssm_inputs_kernel(int T, int B, int S, int A, const float *__restrict__ state0,
                                   const float *__restrict__ states,
                                   const float *__restrict__ actions, float *__restrict__ in) {
  const int SA = S + A;
  const size_t n = (size_t)T * B * SA;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e % SA);
    const size_t r = e / SA;  // t * B + b
    const int t = (int)(r / B), b = (int)(r % B);
    float v;
    if (j < S)
      v = t == 0 ? (state0 ? state0[(size_t)b * S + j] : 0.f) : states[(r - B) * S + j];
    else
      v = actions[r * A + (j - S)];
    in[e] = v;
  }
}

__global__ void elu_kernel(const float *__restrict__ pre, float *__restrict__ post, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const float u = pre[e];
    post[e] = u > 0.f ? u : expm1f(u);
  }
}

// out = g * ELU'(pre), ELU'(u) = 1 for u > 0, exp(u) otherwise
__global__ void elu_grad_kernel(const float *__restrict__ g, const float *__restrict__ pre,
                                float *__restrict__ out, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const float u = pre[e];
    out[e] = g[e] * (u > 0.f ? 1.f : expf(u));
  }
}

// out = g * (1 - y^2), the gradient through y = tanh(v)
__global__ void tanh_grad_kernel(const float *__restrict__ g, const float *__restrict__ y,
                                 float *__restrict__ out, size_t n) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const float v = y[e];
    out[e] = g[e] * (1.f - v * v);
  }
}

// Sample and head at step t: ds = dstates_t + cs (the part from step t+1),
// dmean = dmeans_t + ds, dstd = dstds_t + ds * eps_t;  dp = [dmean,
// dstd * softplus'(p_std)] with softplus' = sigmoid.  p: [T*B][2S] head
// outputs; dp written at row t*B + b of DP [T*B][2S].
__global__ void rssm_sample_grad_kernel(int t, int B, int S, const float *__restrict__ dmeans,
                                        const float *__restrict__ dstds,
                                        const float *__restrict__ dstates,
                                        const float *__restrict__ eps, const float *__restrict__ p,
                                        const float *__restrict__ cs, float *__restrict__ dp) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= B * S) return;
  const int b = e / S, j = e % S;
  const size_t r = (size_t)t * B + b, o = r * S + j;
  const float ds = (dstates ? dstates[o] : 0.f) + cs[e];
  const float dmean = (dmeans ? dmeans[o] : 0.f) + ds;
  const float dsd = (dstds ? dstds[o] : 0.f) + ds * eps[o];
  dp[r * 2 * S + j] = dmean;
  dp[r * 2 * S + S + j] = dsd * sigmoid_f(p[r * 2 * S + S + j]);
}

// GRU cell at step t: dh = dbeliefs_t + dhq (through the head) + gh (W_hh^T
// dR_{t+1}) + dhz (z_{t+1} dh_{t+1}); gate gradients into DA (input side) and
// DR (hidden side) at rows t*B + b; dhz <- z_t dh (read, then overwritten).
// gates: activated r, z, n [T*B][3RH]; zh: hidden-side pre-activations
// (n part: W_hn h_{t-1} + b_hn); hp: h_{t-1} [T*B][RH].
__global__ void rssm_gru_grad_kernel(int t, int B, int RH, const float *__restrict__ dbeliefs,
                                     const float *__restrict__ dhq, const float *__restrict__ gh,
                                     float *__restrict__ dhz, const float *__restrict__ gates,
                                     const float *__restrict__ zh, const float *__restrict__ hp,
                                     float *__restrict__ DA, float *__restrict__ DR) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= B * RH) return;
  const int b = e / RH, j = e % RH, G = 3 * RH;
  const size_t r = (size_t)t * B + b;
  const float dh = (dbeliefs ? dbeliefs[r * RH + j] : 0.f) + dhq[e] + gh[e] + dhz[e];
  const float *g = gates + r * G;
  const float rg = g[j], z = g[RH + j], n = g[2 * RH + j];
  const float hn = zh[r * G + 2 * RH + j];
  const float dn = dh * (1.f - z), dz = dh * (hp[r * RH + j] - n);
  const float dan = dn * (1.f - n * n);
  const float ar = dan * hn * rg * (1.f - rg), az = dz * z * (1.f - z);
  float *da = DA + r * G, *dr = DR + r * G;
  da[j] = ar; da[RH + j] = az; da[2 * RH + j] = dan;
  dr[j] = ar; dr[RH + j] = az; dr[2 * RH + j] = dan * rg;
  dhz[e] = dh * z;
}

}  // namespace

cudaError_t launch_rssm_inputs(int T, int B, int S, int A, const float *state0,
                               const float *states, const float *actions, float *in,
                               cudaStream_t s) {
  const size_t n = (size_t)T * B * (S + A);
  if (n == 0) return cudaSuccess;
  rssm_inputs_kernel<<<ew_blocks(n), EW, 0, s>>>(T, B, S, A, state0, states, actions, in);
  return cudaGetLastError();
}

cudaError_t launch_elu(const float *pre, float *post, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  elu_kernel<<<ew_blocks(n), EW, 0, s>>>(pre, post, n);
  return cudaGetLastError();
}

cudaError_t launch_elu_grad(const float *g, const float *pre, float *out, size_t n,
                            cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  elu_grad_kernel<<<ew_blocks(n), EW, 0, s>>>(g, pre, out, n);
  return cudaGetLastError();
}

cudaError_t launch_tanh_grad(const float *g, const float *y, float *out, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  tanh_grad_kernel<<<ew_blocks(n), EW, 0, s>>>(g, y, out, n);
  return cudaGetLastError();
}

cudaError_t launch_rssm_sample_grad(int t, int B, int S, const float *dmeans, const float *dstds,
                                    const float *dstates, const float *eps, const float *p,
                                    const float *cs, float *dp, cudaStream_t s) {
  rssm_sample_grad_kernel<<<ceil_div(B * S, EW), EW, 0, s>>>(t, B, S, dmeans, dstds, dstates, eps,
                                                              p, cs, dp);
  return cudaGetLastError();
}

cudaError_t launch_rssm_gru_grad(int t, int B, int RH, const float *dbeliefs, const float *dhq,
                                 const float *gh, float *dhz, const float *gates, const float *zh,
                                 const float *hp, float *DA, float *DR, cudaStream_t s) {
  rssm_gru_grad_kernel<<<ceil_div(B * RH, EW), EW, 0, s>>>(t, B, RH, dbeliefs, dhq, gh, dhz,
                                                            gates, zh, hp, DA, DR);
  return cudaGetLastError();
}

}  // namespace rcu
