// Fused RSSM prior unroll ("[Feature Request] CUDNN version of RSSM",
// pytorch/rl issue 366: RSSMPrior.forward and the first unroll_rssm).
//
// The per-step chain is four dependent dense ops
//   a = ELU(W1 [state, action_t] + b1)            (Hd outputs)
//   belief = GRUCell(a, belief)                   (RH units, 3 gates each)
//   q = ELU(W2 belief + b2)                       (Hd outputs)
//   p = W3 q + b3 -> mean, std = softplus + 0.1, state = mean + eps_t * std
// which the Python loop on the page runs as ~10 launches per step.  Here one
// launch runs all T steps.  A thread-block cluster of RC CTAs holds one copy
// of every weight, each CTA the rows of the outputs it owns, resident in
// shared memory (transposed, so threads read consecutive words).  Each phase
// computes the CTA's output slice for the cluster's batch rows and
// broadcasts it into every CTA's shared memory through distributed shared
// memory, followed by a cluster barrier (a hardware barrier: it cannot hang
// and needs no timeout).  Clusters take disjoint batch slices and never
// wait on each other.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace rcu {

namespace {

constexpr int RC = 8;    // CTAs per cluster
constexpr int NT = 256;
constexpr int MAXBC = 8; // batch rows per cluster (register accumulators)

struct Dims {
  int S, A, Hd, RH, Ha, Ua, Sa, Bc;
};

__host__ __device__ inline Dims make_dims(int S, int A, int Hd, int RH, int Bc) {
  Dims d;
  d.S = S; d.A = A; d.Hd = Hd; d.RH = RH;
  d.Ha = ceil_div(Hd, RC);
  d.Ua = ceil_div(RH, RC);
  d.Sa = ceil_div(S, RC);
  d.Bc = Bc;
  return d;
}

// shared-memory carve-up (floats)
struct Layout {
  size_t w1, b1, wih, whh, bih, bhh, w2, b2, w3, b3;   // weights (transposed [k][o])
  size_t st, av, bel, qv, total;                        // vectors
};
__host__ __device__ inline Layout make_layout(const Dims &d) {
  Layout L;
  size_t o = 0;
  auto take = [&](size_t n) { size_t r = o; o += (n + 3) & ~size_t(3); return r; };
  L.w1 = take((size_t)(d.S + d.A) * d.Ha);
  L.b1 = take(d.Ha);
  L.wih = take((size_t)d.Hd * 3 * d.Ua);
  L.whh = take((size_t)d.RH * 3 * d.Ua);
  L.bih = take(3 * d.Ua);
  L.bhh = take(3 * d.Ua);
  L.w2 = take((size_t)d.RH * d.Ha);
  L.b2 = take(d.Ha);
  L.w3 = take((size_t)d.Hd * 2 * d.Sa);
  L.b3 = take(2 * d.Sa);
  L.st = take((size_t)d.Bc * d.S);
  L.av = take((size_t)d.Bc * d.Hd);
  L.bel = take((size_t)2 * d.Bc * d.RH);
  L.qv = take((size_t)d.Bc * d.Hd);
  L.total = o;
  return L;
}

__device__ __forceinline__ float elu_f(float v) { return v > 0.f ? v : expm1f(v); }
__device__ __forceinline__ float softplus_f(float v) {
  return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
}

// out[r][o] = sum_k Wt[k*O + o] * v[r*ldv + k] for o < O, r < nr; every
// thread takes one output column and all rows (nr <= MAXBC accumulators);
// columns beyond the block size loop.
template <int NR>
__device__ __forceinline__ void matvec_rows(const float *Wt, int O, int K, const float *v, int ldv,
                                            int o, float (&acc)[MAXBC]) {
#pragma unroll
  for (int r = 0; r < MAXBC; ++r) acc[r] = 0.f;
  for (int k = 0; k < K; ++k) {
    const float w = Wt[(size_t)k * O + o];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = fmaf(w, v[r * ldv + k], acc[r]);
  }
}

template <int NR>
__global__ void __cluster_dims__(RC, 1, 1) __launch_bounds__(NT, 1)
    rssm_kernel(const RssmParams p, int Bc) {
  extern __shared__ __align__(16) float sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int q = blockIdx.x / RC;
  const int b0 = q * Bc;
  const int nr = min(Bc, p.B - b0);  // rows of this cluster (uniform across the cluster)
  const Dims d = make_dims(p.S, p.A, p.Hd, p.RH, Bc);
  const Layout L = make_layout(d);
  const int S = d.S, A = d.A, Hd = d.Hd, RH = d.RH, SA = S + A;
  const int i0 = c * d.Ha, ni = max(0, min(d.Ha, Hd - i0));   // owned a / q outputs
  const int j0 = c * d.Ua, nj = max(0, min(d.Ua, RH - j0));   // owned GRU units
  const int s0 = c * d.Sa, ns = max(0, min(d.Sa, S - s0));    // owned state entries
  const int tid = threadIdx.x;

  // ---- resident weights, transposed to [k][o]
  for (int e = tid; e < SA * d.Ha; e += NT) {
    const int k = e / d.Ha, o = e % d.Ha;
    sm[L.w1 + e] = o < ni ? p.W1[(size_t)(i0 + o) * SA + k] : 0.f;
  }
  for (int o = tid; o < d.Ha; o += NT) {
    sm[L.b1 + o] = (o < ni && p.b1) ? p.b1[i0 + o] : 0.f;
    sm[L.b2 + o] = (o < ni && p.b2) ? p.b2[i0 + o] : 0.f;
  }
  for (int e = tid; e < Hd * 3 * d.Ua; e += NT) {
    const int k = e / (3 * d.Ua), o = e % (3 * d.Ua), g = o / d.Ua, j = o % d.Ua;
    sm[L.wih + e] = j < nj ? p.Wih[(size_t)(g * RH + j0 + j) * Hd + k] : 0.f;
  }
  for (int e = tid; e < RH * 3 * d.Ua; e += NT) {
    const int k = e / (3 * d.Ua), o = e % (3 * d.Ua), g = o / d.Ua, j = o % d.Ua;
    sm[L.whh + e] = j < nj ? p.Whh[(size_t)(g * RH + j0 + j) * RH + k] : 0.f;
  }
  for (int o = tid; o < 3 * d.Ua; o += NT) {
    const int g = o / d.Ua, j = o % d.Ua;
    sm[L.bih + o] = (j < nj && p.bih) ? p.bih[g * RH + j0 + j] : 0.f;
    sm[L.bhh + o] = (j < nj && p.bhh) ? p.bhh[g * RH + j0 + j] : 0.f;
  }
  for (int e = tid; e < RH * d.Ha; e += NT) {
    const int k = e / d.Ha, o = e % d.Ha;
    sm[L.w2 + e] = o < ni ? p.W2[(size_t)(i0 + o) * RH + k] : 0.f;
  }
  for (int e = tid; e < Hd * 2 * d.Sa; e += NT) {
    const int k = e / (2 * d.Sa), o = e % (2 * d.Sa), h = o / d.Sa, j = o % d.Sa;
    sm[L.w3 + e] = j < ns ? p.W3[(size_t)(h * S + s0 + j) * Hd + k] : 0.f;
  }
  for (int o = tid; o < 2 * d.Sa; o += NT) {
    const int h = o / d.Sa, j = o % d.Sa;
    sm[L.b3 + o] = (j < ns && p.b3) ? p.b3[h * S + s0 + j] : 0.f;
  }
  // ---- initial state / belief of the cluster's rows (full vectors, every CTA)
  for (int e = tid; e < Bc * S; e += NT) {
    const int r = e / S, k = e % S;
    sm[L.st + e] = (r < nr && p.state0) ? p.state0[(size_t)(b0 + r) * S + k] : 0.f;
  }
  for (int e = tid; e < Bc * RH; e += NT) {
    const int r = e / RH, k = e % RH;
    sm[L.bel + e] = (r < nr && p.belief0) ? p.belief0[(size_t)(b0 + r) * RH + k] : 0.f;
  }
  for (int e = tid; e < Bc * Hd; e += NT) { sm[L.av + e] = 0.f; sm[L.qv + e] = 0.f; }
  cluster.sync();

  float *rem[RC];
#pragma unroll
  for (int r = 0; r < RC; ++r) rem[r] = cluster.map_shared_rank(sm, r);

  float acc[MAXBC], acc2[MAXBC];
  for (int t = 0; t < p.T; ++t) {
    const int cur = t & 1;
    float *bel_cur = sm + L.bel + (size_t)cur * Bc * RH;
    const size_t bel_nxt = L.bel + (size_t)(cur ^ 1) * Bc * RH;
    // ---- phase 1: a = ELU(W1 [state, action] + b1), owned outputs
    if (tid < ni) {
      const int o = tid;
      matvec_rows<NR>(sm + L.w1, d.Ha, S, sm + L.st, S, o, acc);
      for (int k = 0; k < A; ++k) {
        const float w = sm[L.w1 + (size_t)(S + k) * d.Ha + o];
#pragma unroll
        for (int r = 0; r < NR; ++r)
          if (r < nr) acc[r] = fmaf(w, __ldg(p.actions + ((size_t)t * p.B + b0 + r) * A + k), acc[r]);
      }
      const float bb = sm[L.b1 + o];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float a = elu_f(acc[r] + bb);
#pragma unroll
        for (int x = 0; x < RC; ++x) rem[x][L.av + (size_t)r * Hd + i0 + o] = a;
      }
    }
    cluster.sync();
    // ---- phase 2: GRUCell(a, belief) for owned units
    if (tid < nj) {
      const int j = tid;
      float gi[3][MAXBC], gh[3][MAXBC];
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        matvec_rows<NR>(sm + L.wih, 3 * d.Ua, Hd, sm + L.av, Hd, g * d.Ua + j, acc);
        matvec_rows<NR>(sm + L.whh, 3 * d.Ua, RH, bel_cur, RH, g * d.Ua + j, acc2);
#pragma unroll
        for (int r = 0; r < MAXBC; ++r) {
          gi[g][r] = acc[r] + sm[L.bih + g * d.Ua + j];
          gh[g][r] = acc2[r] + sm[L.bhh + g * d.Ua + j];
        }
      }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float rg = sigmoid_f(gi[0][r] + gh[0][r]);
        const float zg = sigmoid_f(gi[1][r] + gh[1][r]);
        const float ng = tanh_f(gi[2][r] + rg * gh[2][r]);
        const float hb = (1.f - zg) * ng + zg * bel_cur[r * RH + j0 + j];
#pragma unroll
        for (int x = 0; x < RC; ++x) rem[x][bel_nxt + (size_t)r * RH + j0 + j] = hb;
        if (r < nr) p.beliefs[((size_t)t * p.B + b0 + r) * RH + j0 + j] = hb;
      }
    }
    cluster.sync();
    // ---- phase 3: q = ELU(W2 belief + b2), owned outputs
    if (tid < ni) {
      const int o = tid;
      matvec_rows<NR>(sm + L.w2, d.Ha, RH, sm + bel_nxt, RH, o, acc);
      const float bb = sm[L.b2 + o];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float qv = elu_f(acc[r] + bb);
#pragma unroll
        for (int x = 0; x < RC; ++x) rem[x][L.qv + (size_t)r * Hd + i0 + o] = qv;
      }
    }
    cluster.sync();
    // ---- phase 4: p = W3 q + b3 -> mean, std, sampled state (owned entries)
    if (tid < ns) {
      const int j = tid;
      matvec_rows<NR>(sm + L.w3, 2 * d.Sa, Hd, sm + L.qv, Hd, j, acc);
      matvec_rows<NR>(sm + L.w3, 2 * d.Sa, Hd, sm + L.qv, Hd, d.Sa + j, acc2);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float mean = acc[r] + sm[L.b3 + j];
        const float sd = softplus_f(acc2[r] + sm[L.b3 + d.Sa + j]) + 0.1f;
        float st = mean;
        if (r < nr) {
          const size_t o = ((size_t)t * p.B + b0 + r) * S + s0 + j;
          st = fmaf(__ldg(p.eps + o), sd, mean);
          p.means[o] = mean;
          p.stds[o] = sd;
          p.states[o] = st;
        }
#pragma unroll
        for (int x = 0; x < RC; ++x) rem[x][L.st + (size_t)r * S + s0 + j] = st;
      }
    }
    cluster.sync();
  }
}

int pick_bc(int B, int nsm) {
  int clusters = nsm / RC;
  if (clusters < 1) clusters = 1;
  int bc = ceil_div(B, clusters);
  if (bc < 1) bc = 1;
  if (bc > MAXBC) bc = MAXBC;
  return bc;
}

size_t smem_bytes(int S, int A, int Hd, int RH, int Bc) {
  return make_layout(make_dims(S, A, Hd, RH, Bc)).total * sizeof(float);
}

template <int NR>
cudaError_t launch_nr(const RssmParams &p, int Bc, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute((const void *)rssm_kernel<NR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rssm_kernel<NR><<<grid, NT, smem, s>>>(p, Bc);
  return cudaGetLastError();
}

}  // namespace

bool rssm_supported(int S, int A, int Hd, int RH) {
  if (S < 1 || A < 0 || Hd < 1 || RH < 1) return false;
  if (ceil_div(Hd, RC) > NT || ceil_div(RH, RC) > NT || ceil_div(S, RC) > NT) return false;
  return smem_bytes(S, A, Hd, RH, 1) <= 227 * 1024;
}

cudaError_t launch_rssm(const RssmParams &p, int nsm, cudaStream_t s, int *clusters_used) {
  int Bc = pick_bc(p.B, nsm);
  while (Bc > 1 && smem_bytes(p.S, p.A, p.Hd, p.RH, Bc) > 227 * 1024) --Bc;
  const size_t smem = smem_bytes(p.S, p.A, p.Hd, p.RH, Bc);
  const int clusters = ceil_div(p.B, Bc);
  if (clusters_used) *clusters_used = clusters;
  const int grid = clusters * RC;
  switch (Bc) {
    case 1: return launch_nr<1>(p, Bc, grid, smem, s);
    case 2: return launch_nr<2>(p, Bc, grid, smem, s);
    case 3: return launch_nr<3>(p, Bc, grid, smem, s);
    case 4: return launch_nr<4>(p, Bc, grid, smem, s);
    case 5: return launch_nr<5>(p, Bc, grid, smem, s);
    case 6: return launch_nr<6>(p, Bc, grid, smem, s);
    case 7: return launch_nr<7>(p, Bc, grid, smem, s);
    default: return launch_nr<8>(p, Bc, grid, smem, s);
  }
}

}  // namespace rcu
