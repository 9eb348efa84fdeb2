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

// ---- weight gradients of several layers in two launches: for each group,
// dW[o][k] = sum_m dZ[m][o] Y[m][k] and db[o] = sum_m dZ[m][o], read from the
// row-major activations directly (Y is extended by a column of ones, whose
// output column is db).  The rows are split into S chunks: the first kernel
// writes each chunk's partial 64 x 64 tiles, the second sums the chunks in
// order, so the result does not depend on timing.
constexpr int WGT = 64, WGM = 32, WG_NT = 256;

__global__ void __launch_bounds__(WG_NT) wgrad_partial_kernel(const WgradParams p) {
  __shared__ __align__(16) float sdz[WGM][WGT];
  __shared__ __align__(16) float sy[WGM][WGT];
  int gi = 0;
  while (gi + 1 < p.ngroups && (int)blockIdx.x >= p.g[gi + 1].tile0) ++gi;
  const WgradGroup &g = p.g[gi];
  const int tkn = ceil_div(g.ny + 1, WGT);
  const int t = (int)blockIdx.x - g.tile0, o0 = (t / tkn) * WGT, k0 = (t % tkn) * WGT;
  const int m0 = (int)blockIdx.y * p.mchunk, m1 = min(p.M, m0 + p.mchunk);
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int lc = tid % WGT, lr = tid / WGT;  // loader: column, first row
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int o = o0 + lc, k = k0 + lc;
  for (int mb = m0; mb < m1; mb += WGM) {
#pragma unroll
    for (int q = 0; q < WGM / 4; ++q) {
      const int r = lr + 4 * q, m = mb + r;
      const bool in = m < m1;
      sdz[r][lc] = (in && o < g.nz) ? __ldg(g.dz + (size_t)m * g.nz + o) : 0.f;
      sy[r][lc] = !in ? 0.f : k < g.ny ? __ldg(g.y + (size_t)m * g.ny + k) : (k == g.ny ? 1.f : 0.f);
    }
    __syncthreads();
#pragma unroll 8
    for (int mm = 0; mm < WGM; ++mm) {
      const float4 a = *reinterpret_cast<const float4 *>(&sdz[mm][ty * 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&sy[mm][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  // this chunk's partial tile: [o][ny + 1] rows of the group's slot
  float *part = p.part + (size_t)blockIdx.y * p.total + g.off;
  const int w = g.ny + 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int oo = o0 + ty * 4 + i;
    if (oo >= g.nz) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kk = k0 + tx * 4 + j;
      if (kk < w) part[(size_t)oo * w + kk] = acc[i][j];
    }
  }
}

__global__ void wgrad_sum_kernel(const WgradParams p) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.total;
       e += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int c = 0; c < p.S; ++c) v += p.part[(size_t)c * p.total + e];
    int gi = 0;
    while (gi + 1 < p.ngroups && e >= p.g[gi + 1].off) ++gi;
    const WgradGroup &g = p.g[gi];
    const size_t l = e - g.off, w = (size_t)g.ny + 1;
    const size_t o = l / w, k = l % w;
    if (k < (size_t)g.ny) g.dW[o * g.ny + k] = v;
    else g.db[o] = v;
  }
}

}  // namespace

size_t wgrad_scratch_floats(const WgradGroup *g, int n, int M) {
  size_t tot = 0;
  for (int i = 0; i < n; ++i) tot += (size_t)g[i].nz * (g[i].ny + 1);
  return tot * (size_t)ceil_div(std::max(M, 1), WG_ROWS_PER_CHUNK);
}

cudaError_t launch_wgrad(const WgradGroup *groups, int n, int M, float *scratch, cudaStream_t s) {
  if (n < 1 || n > WG_MAX_GROUPS || M < 1) return cudaErrorInvalidValue;
  WgradParams p{};
  p.ngroups = n;
  p.M = M;
  p.S = ceil_div(M, WG_ROWS_PER_CHUNK);
  p.mchunk = WG_ROWS_PER_CHUNK;
  p.part = scratch;
  int tiles = 0;
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    p.g[i] = groups[i];
    if (p.g[i].nz < 1 || p.g[i].ny < 0) return cudaErrorInvalidValue;
    p.g[i].tile0 = tiles;
    p.g[i].off = off;
    tiles += ceil_div(p.g[i].nz, WGT) * ceil_div(p.g[i].ny + 1, WGT);
    off += (size_t)p.g[i].nz * (p.g[i].ny + 1);
  }
  p.total = off;
  if (p.S > 65535) return cudaErrorInvalidValue;
  wgrad_partial_kernel<<<dim3(tiles, p.S), WG_NT, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  wgrad_sum_kernel<<<(unsigned)std::min<size_t>((off + 255) / 256, 4096), 256, 0, s>>>(p);
  return cudaGetLastError();
}

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
