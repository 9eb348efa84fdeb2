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
// shared memory ([o][k]).  Each phase is a batched mat-vec over the
// cluster's batch rows: a group of 8 or 16 lanes per 4 outputs splits K and
// sums its partials by shuffles, and the CTA's output slice is broadcast into
// every CTA's shared memory with
// asynchronous distributed-shared-memory stores (st.async), each counting its
// bytes on the receiving CTA's mbarrier for that vector.  A CTA starts the
// next phase as soon as all bytes of the vector it needs have landed: no
// cluster-wide barrier and no release fence per phase.  A CTA can finish
// phase k+1 only after every CTA has sent its phase-k output (after reading
// its phase-k inputs), so no vector is overwritten while a peer still reads
// it.  Clusters take disjoint batch slices and never wait on each other.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace rcu {

namespace {

constexpr int RC = 8;    // CTAs per cluster
constexpr int NT = 512;
constexpr int MAXBC = 8; // batch rows per cluster
constexpr size_t PRELOAD_MAX = 32 * 1024;  // bytes of actions+eps kept in shared memory
constexpr size_t SMEM_CAP = 227 * 1024 - 64;  // dynamic shared memory per CTA (64 B static)

__host__ __device__ inline int r4(int v) { return (v + 3) & ~3; }

struct Dims {
  int S, A, Hd, RH, Ha, Ua, Sa, Bc;
  // padded widths (multiples of 4 floats, so rows start 16-byte aligned)
  int Hap, U3p, S2p, Hdp, RHp, SAp;
  // actor in the loop (Hx = actor hidden width, 0 = none): outputs per CTA
  // and padded widths
  int Hx, Hxa, Axa, Hxap, Axap, Hxp, SRp;
};

__host__ __device__ inline Dims make_dims(int S, int A, int Hd, int RH, int Bc, int Hx = 0) {
  Dims d;
  d.S = S; d.A = A; d.Hd = Hd; d.RH = RH;
  d.Ha = ceil_div(Hd, RC);
  d.Ua = ceil_div(RH, RC);
  d.Sa = ceil_div(S, RC);
  d.Bc = Bc;
  d.Hap = r4(d.Ha);
  d.U3p = r4(3 * d.Ua);
  d.S2p = r4(2 * d.Sa);
  d.Hdp = r4(Hd);
  d.RHp = r4(RH);
  d.SAp = r4(S + A);
  d.Hx = Hx;
  d.Hxa = Hx > 0 ? ceil_div(Hx, RC) : 0;
  d.Axa = Hx > 0 ? ceil_div(A, RC) : 0;
  d.Hxap = r4(d.Hxa);
  d.Axap = r4(d.Axa);
  d.Hxp = r4(Hx);
  d.SRp = Hx > 0 ? r4(S + RH) : 0;
  return d;
}

// shared-memory carve-up (floats)
struct Layout {
  size_t w1, b1, wih, whh, bih, bhh, w2, b2, w3, b3;  // weights ([o][k], both padded)
  size_t wa1, ba1, wa2, ba2;                           // actor weights (same form)
  size_t st, in1, av, bel, qv;                         // vectors, [Bc][padded width]
  size_t ain, hx;                                      // actor input [state, belief], hidden
  size_t part1, part2;                                 // a phase's sums
  size_t act, eps;                                     // preloaded actions / noise
  size_t total;
  bool preload;
};
__host__ __device__ inline Layout make_layout(const Dims &d, int T) {
  Layout L;
  size_t o = 0;
  auto take = [&](size_t n) { size_t r = o; o += (n + 3) & ~size_t(3); return r; };
  // weights [o][k] (the outputs this CTA owns, rows padded to a multiple of
  // 4; k padded likewise)
  L.w1 = take((size_t)d.Hap * d.SAp);
  L.b1 = take(d.Hap);
  L.wih = take((size_t)d.U3p * d.Hdp);
  L.whh = take((size_t)d.U3p * d.RHp);
  L.bih = take(d.U3p);
  L.bhh = take(d.U3p);
  L.w2 = take((size_t)d.Hap * d.RHp);
  L.b2 = take(d.Hap);
  L.w3 = take((size_t)d.S2p * d.Hdp);
  L.b3 = take(d.S2p);
  L.wa1 = take(d.Hx > 0 ? (size_t)d.Hxap * d.SRp : 0);
  L.ba1 = take(d.Hx > 0 ? d.Hxap : 0);
  L.wa2 = take(d.Hx > 0 ? (size_t)d.Axap * d.Hxp : 0);
  L.ba2 = take(d.Hx > 0 ? d.Axap : 0);
  L.st = take((size_t)d.Bc * d.S);
  L.in1 = take((size_t)d.Bc * d.SAp);
  // a (phase 1 -> 2) and q (phase 3 -> 4) share storage: peers write q only
  // after the cluster barrier that ends phase 2, when every CTA has read a,
  // and write a only after the step's last barrier, when q has been read
  L.av = take((size_t)d.Bc * d.Hdp);
  L.qv = L.av;
  L.bel = take((size_t)2 * d.Bc * d.RHp);
  int wmax = d.Hap > d.U3p ? d.Hap : d.U3p;
  if (d.S2p > wmax) wmax = d.S2p;
  if (d.Hxap > wmax) wmax = d.Hxap;
  if (d.Axap > wmax) wmax = d.Axap;
  L.part1 = take((size_t)d.Bc * wmax);  // a phase's sums, [Bc][outputs]
  // the actor's input row and hidden layer live in the phase-2 sums:
  // both are used between the step's last barrier and phase 2, and peers
  // write the hidden layer only after that barrier
  const size_t ain_n = (size_t)d.Bc * d.SRp, hx_n = d.Hx > 0 ? (size_t)d.Bc * d.Hxp : 0;
  size_t p2 = (size_t)d.Bc * d.U3p;
  if (ain_n + hx_n > p2) p2 = ain_n + hx_n;
  L.part2 = take(p2);
  L.ain = L.part2;
  L.hx = L.part2 + ain_n;
  // actions are preloaded only when given (with an actor they are computed),
  // and only while the preload fits beside everything else
  const size_t na = d.Hx > 0 ? 0 : (size_t)T * d.Bc * d.A, ne = (size_t)T * d.Bc * d.S;
  L.preload = (na + ne) * 4 <= PRELOAD_MAX &&
              (o + ((na + 3) & ~size_t(3)) + ((ne + 3) & ~size_t(3))) * 4 <= SMEM_CAP;
  L.act = take(L.preload ? na : 0);
  L.eps = take(L.preload ? ne : 0);
  L.total = o;
  return L;
}

__device__ __forceinline__ float elu_f(float v) { return v > 0.f ? v : expm1f(v); }
__device__ __forceinline__ float softplus_f(float v) {
  return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
}

// out[r*Op + o] = sum over k < K of Wo[o*ldw + k] * V[r*ldv + k], for o < Op
// (a multiple of 4), r < NR.  Threads [t0, t0 + nthr) (nthr a multiple of
// 32) take part: SL consecutive lanes share a group of 4 outputs and split K
// between them (lane l: columns 4l, 4l + 4*SL, ...; every load 16 bytes at
// consecutive addresses across the lanes, and the weights [o][k] rows, so no
// bank conflicts), then sum their 4 x NR partials by a shuffle
// reduce-scatter that leaves each lane whole sums to store.  No shared-memory
// partials and no CTA barrier inside; ldw and ldv are multiples of 4, the
// weights' columns from K up to ldw are zero, and V's are not read.
template <int NR, int SL>
__device__ __forceinline__ void matvec_sl(const float *Wo, int ldw, int Op, int K,
                                          const float *V, int ldv, float *out, int t0, int nthr) {
  static_assert(SL == 8 || SL == 16, "8 or 16 lanes per output group");
  constexpr int NV = 4 * NR;
  constexpr int PER0 = (NV + SL - 1) / SL;
  constexpr int PER = PER0 <= 1 ? 1 : (PER0 <= 2 ? 2 : (PER0 <= 4 ? 4 : 8));  // sums per lane
  constexpr int NVP = SL * PER;
  const int t = threadIdx.x - t0;
  if (t < 0 || t >= nthr) return;  // (whole warps: t0 and nthr are multiples of 32)
  const int ng = Op / 4, slots = nthr / SL;
  const int slot = t / SL, l = t % SL, lane = threadIdx.x & 31;
  const int wslot0 = (t / 32) * (32 / SL);  // this warp's first slot
  const int K4 = (K + 3) & ~3;
  for (int base = 0; base < ng; base += slots) {
    if (base + wslot0 >= ng) break;  // no group of this warp left (warp-uniform)
    const int og = base + slot;
    const bool valid = og < ng;
    float a[NR][4];
#pragma unroll
    for (int r = 0; r < NR; ++r) a[r][0] = a[r][1] = a[r][2] = a[r][3] = 0.f;
    if (valid) {
      const float *w0 = Wo + (size_t)og * 4 * ldw;
      for (int k = 4 * l; k < K4; k += 4 * SL) {
        float4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const float4 *>(w0 + (size_t)i * ldw + k);
        const int rem = K - k;  // (>= 1; below 4 in the last chunk only)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float4 v = *reinterpret_cast<const float4 *>(V + (size_t)r * ldv + k);
          if (rem < 4) {  // the row's padding may hold another phase's values
            v.w = 0.f;
            if (rem < 3) v.z = 0.f;
            if (rem < 2) v.y = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            a[r][i] = fmaf(v.x, w[i].x, fmaf(v.y, w[i].y, fmaf(v.z, w[i].z, fmaf(v.w, w[i].w, a[r][i]))));
        }
      }
    }
    float v[NVP];
#pragma unroll
    for (int i = 0; i < NVP; ++i) v[i] = i < NV ? a[i / 4][i % 4] : 0.f;
    // each step keeps half of the values (the upper half on lanes with bit
    // m set) plus the partner lane's same half: lane l ends with entries
    // PER*l .. PER*l + PER - 1 summed over its SL lanes
#pragma unroll
    for (int h = NVP / 2, m = SL / 2; m >= 1; h >>= 1, m >>= 1) {
      const bool up = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = up ? v[i] : v[i + h];
        const float keep = up ? v[i + h] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
    if (valid) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = PER * l + i, r = idx / 4, j = idx % 4;
        if (r < NR) out[(size_t)r * Op + og * 4 + j] = v[i];
      }
    }
  }
}

// Load rows [row0, row0 + n) of a row-major [rows][K] matrix into shared
// memory dst[o * ldw + k] (k < K); other entries are left as they are (zero).
__device__ __forceinline__ void load_rows(const float *src, int K, int row0, int n, int ldw,
                                          float *dst) {
  for (int e = threadIdx.x; e < n * K; e += NT) {
    const int o = e / K, k = e % K;
    dst[(size_t)o * ldw + k] = src[(size_t)(row0 + o) * K + k];
  }
}

// 4-byte asynchronous store into cluster CTA shared memory (address from
// mapa), completing as 4 bytes of complete_tx on that CTA's mbarrier
__device__ __forceinline__ void st_async_b32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   addr),
               "r"(__float_as_uint(v)), "r"(bar)
               : "memory");
}
// the broadcast vectors, one mbarrier each
enum Vec { V_ST = 0, V_HX, V_ACT, V_AV, V_BEL, V_QV, NVEC };

__device__ __forceinline__ float part_sum(const float *part, int Op, int r, int o) {
  return part[(size_t)r * Op + o];
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
  const bool actor = p.Wa1 != nullptr;  // unroll variant 2: actions from the actor
  const Dims d = make_dims(p.S, p.A, p.Hd, p.RH, Bc, actor ? p.Hx : 0);
  const Layout L = make_layout(d, p.T);
  const int S = d.S, A = d.A, Hd = d.Hd, RH = d.RH, SA = S + A;
  const int Hdp = d.Hdp, RHp = d.RHp, SAp = d.SAp;
  const int i0 = c * d.Ha, ni = max(0, min(d.Ha, Hd - i0));   // owned a / q outputs
  const int j0 = c * d.Ua, nj = max(0, min(d.Ua, RH - j0));   // owned GRU units
  const int s0 = c * d.Sa, ns = max(0, min(d.Sa, S - s0));    // owned state entries
  const int x0 = c * d.Hxa, nx = actor ? max(0, min(d.Hxa, d.Hx - x0)) : 0;  // actor hidden
  const int a0 = c * d.Axa, na = actor ? max(0, min(d.Axa, A - a0)) : 0;      // actions
  const int tid = threadIdx.x;
  const bool tr = p.trace && blockIdx.x == 0 && tid == 0;
  if (tr) p.trace[11] = globaltimer_ns();

  // ---- every padding column and vector starts at zero
  for (size_t e = tid; e < L.total; e += NT) sm[e] = 0.f;
  __syncthreads();
  // ---- resident weights, [o][k] rows of the owned outputs (others zero)
  load_rows(p.W1, SA, i0, ni, SAp, sm + L.w1);
  for (int o = tid; o < d.Ha; o += NT) {
    sm[L.b1 + o] = (o < ni && p.b1) ? p.b1[i0 + o] : 0.f;
    sm[L.b2 + o] = (o < ni && p.b2) ? p.b2[i0 + o] : 0.f;
  }
  for (int g = 0; g < 3; ++g) {
    load_rows(p.Wih, Hd, g * RH + j0, nj, Hdp, sm + L.wih + (size_t)g * d.Ua * Hdp);
    load_rows(p.Whh, RH, g * RH + j0, nj, RHp, sm + L.whh + (size_t)g * d.Ua * RHp);
  }
  for (int o = tid; o < 3 * d.Ua; o += NT) {
    const int g = o / d.Ua, j = o % d.Ua;
    sm[L.bih + o] = (j < nj && p.bih) ? p.bih[g * RH + j0 + j] : 0.f;
    sm[L.bhh + o] = (j < nj && p.bhh) ? p.bhh[g * RH + j0 + j] : 0.f;
  }
  load_rows(p.W2, RH, i0, ni, RHp, sm + L.w2);
  for (int h = 0; h < 2; ++h)
    load_rows(p.W3, Hd, h * S + s0, ns, Hdp, sm + L.w3 + (size_t)h * d.Sa * Hdp);
  for (int o = tid; o < 2 * d.Sa; o += NT) {
    const int h = o / d.Sa, j = o % d.Sa;
    sm[L.b3 + o] = (j < ns && p.b3) ? p.b3[h * S + s0 + j] : 0.f;
  }
  if (actor) {
    load_rows(p.Wa1, S + RH, x0, nx, d.SRp, sm + L.wa1);
    load_rows(p.Wa2, d.Hx, a0, na, d.Hxp, sm + L.wa2);
    for (int o = tid; o < d.Hxa; o += NT) sm[L.ba1 + o] = (o < nx && p.ba1) ? p.ba1[x0 + o] : 0.f;
    for (int o = tid; o < d.Axa; o += NT) sm[L.ba2 + o] = (o < na && p.ba2) ? p.ba2[a0 + o] : 0.f;
  }
  // ---- initial state / belief of the cluster's rows (full vectors, every CTA)
  for (int e = tid; e < Bc * S; e += NT) {
    const int r = e / S, k = e % S;
    sm[L.st + e] = (r < nr && p.state0) ? p.state0[(size_t)(b0 + r) * S + k] : 0.f;
  }
  for (int e = tid; e < Bc * RH; e += NT) {
    const int r = e / RH, k = e % RH;
    sm[L.bel + (size_t)r * RHp + k] =
        (r < nr && p.belief0) ? p.belief0[(size_t)(b0 + r) * RH + k] : 0.f;
  }
  if (L.preload) {
    for (int e = tid; e < (actor ? 0 : p.T * Bc * A); e += NT) {
      const int t = e / (Bc * A), r = (e / A) % Bc, k = e % A;
      sm[L.act + e] = r < nr ? p.actions[((size_t)t * p.B + b0 + r) * A + k] : 0.f;
    }
    for (int e = tid; e < p.T * Bc * S; e += NT) {
      const int t = e / (Bc * S), r = (e / S) % Bc, k = e % S;
      sm[L.eps + e] = r < nr ? p.eps[((size_t)t * p.B + b0 + r) * S + k] : 0.f;
    }
  }
  __shared__ uint64_t vbar[NVEC];
  __shared__ int s_ok;
  if (tid == 0) {
    for (int v = 0; v < NVEC; ++v) tc::mbar_init(&vbar[v], 1);
    tc::fence_mbar_init();
  }
  // every CTA's vectors are initialised and its mbarriers exist before any
  // peer sends
  cluster.sync();
  if (tr) p.trace[12] = globaltimer_ns();

  // shared-memory window of each cluster CTA, and its mbarriers
  const uint32_t sm0 = (uint32_t)__cvta_generic_to_shared(sm);
  uint32_t rsm[RC], rbar[RC];
#pragma unroll
  for (int r = 0; r < RC; ++r) {
    rsm[r] = tc::mapa_shared(sm0, (uint32_t)r);
    rbar[r] = tc::mapa_shared((uint32_t)__cvta_generic_to_shared(&vbar[0]), (uint32_t)r);
  }
  // send value v to float offset `off` of every CTA, counted on vector `vec`
  auto bcast = [&](size_t off, float v, int vec) {
#pragma unroll
    for (int r = 0; r < RC; ++r)
      st_async_b32(rsm[r] + (uint32_t)(off * 4), v, rbar[r] + (uint32_t)(vec * 8));
  };
  // bytes each CTA receives per use of each vector
  uint32_t vbytes[NVEC];
  vbytes[V_ST] = (uint32_t)(Bc * S * 4);
  vbytes[V_HX] = (uint32_t)(Bc * (actor ? d.Hx : 0) * 4);
  vbytes[V_ACT] = (uint32_t)(Bc * A * 4);
  vbytes[V_AV] = (uint32_t)(Bc * Hd * 4);
  vbytes[V_BEL] = (uint32_t)(Bc * RH * 4);
  vbytes[V_QV] = (uint32_t)(Bc * Hd * 4);
  uint32_t uses = 0;  // thread 0: completed uses per vector, 4 bits each
  volatile int abort_ = 0;
  const uint64_t tmo = p.timeout_ns;
  // wait until vector `vec` of this use has fully landed (bounded)
  auto wait_vec = [&](int vec) -> bool {
    if (tid == 0) {
      const uint32_t n = (uses >> (4 * vec)) & 15u;
      tc::mbar_arrive_expect_tx(&vbar[vec], vbytes[vec]);
      s_ok = tc::mbar_wait(&vbar[vec], n & 1u, p.err, &abort_, tmo);
      uses = (uses & ~(15u << (4 * vec))) | (((n + 1) & 15u) << (4 * vec));
    }
    __syncthreads();
    return s_ok != 0;
  };
  bool ok = true;

  float *part1 = sm + L.part1, *part2 = sm + L.part2;

  for (int t = 0; t < p.T; ++t) {
    const int cur = t & 1;
    // the state of step t-1 (broadcast at the end of its phase 4)
    if (t > 0 && !(ok = wait_vec(V_ST))) break;
    if (tr) p.trace[t * 16 + 0] = globaltimer_ns();
    float *bel_cur = sm + L.bel + (size_t)cur * Bc * RHp;
    const size_t bel_nxt = L.bel + (size_t)(cur ^ 1) * Bc * RHp;
    if (actor) {
      // ---- actor, hidden layer: x = ELU(Wa1 [state, belief] + ba1), owned outputs
      const int SR = S + RH;
      for (int e = tid; e < Bc * SR; e += NT) {
        const int r = e / SR, k = e % SR;
        sm[L.ain + (size_t)r * d.SRp + k] =
            k < S ? sm[L.st + (size_t)r * S + k] : bel_cur[(size_t)r * RHp + (k - S)];
      }
      __syncthreads();
      matvec_sl<NR, 16>(sm + L.wa1, d.SRp, d.Hxap, SR, sm + L.ain, d.SRp, part1, 0, NT);
      __syncthreads();
      for (int e = tid; e < nx * Bc; e += NT) {
        const int o = e % nx, r = e / nx;
        const float xv = elu_f(part_sum(part1, d.Hxap, r, o) + sm[L.ba1 + o]);
        bcast(L.hx + (size_t)r * d.Hxp + x0 + o, xv, V_HX);
      }
      if (!(ok = wait_vec(V_HX))) break;
      // ---- actor, output: action = tanh(Wa2 x + ba2), owned entries, placed
      //      straight into every CTA's phase-1 input row
      matvec_sl<NR, 16>(sm + L.wa2, d.Hxp, d.Axap, d.Hx, sm + L.hx, d.Hxp, part1, 0, NT);
      __syncthreads();
      for (int e = tid; e < na * Bc; e += NT) {
        const int j = e % na, r = e / na;
        const float av = tanh_f(part_sum(part1, d.Axap, r, j) + sm[L.ba2 + j]);
        bcast(L.in1 + (size_t)r * SAp + S + a0 + j, av, V_ACT);
        if (r < nr && p.actions_out) p.actions_out[((size_t)t * p.B + b0 + r) * A + a0 + j] = av;
      }
      if (!(ok = wait_vec(V_ACT))) break;
      if (tr) p.trace[t * 16 + 5] = globaltimer_ns();
    }
    // ---- phase 1: a = ELU(W1 [state, action] + b1), owned outputs (with the
    //      actor only the state part of the input row is filled here)
    for (int e = tid; e < Bc * (actor ? S : SA); e += NT) {
      const int SW = actor ? S : SA;
      const int r = e / SW, k = e % SW;
      float v;
      if (k < S) v = sm[L.st + (size_t)r * S + k];
      else if (L.preload) v = sm[L.act + ((size_t)t * Bc + r) * A + (k - S)];
      else v = r < nr ? __ldg(p.actions + ((size_t)t * p.B + b0 + r) * A + (k - S)) : 0.f;
      sm[L.in1 + (size_t)r * SAp + k] = v;
    }
    __syncthreads();
    matvec_sl<NR, 16>(sm + L.w1, SAp, d.Hap, SA, sm + L.in1, SAp, part1, 0, NT);
    __syncthreads();
    if (tr) p.trace[t * 16 + 10] = clock64();
    for (int e = tid; e < ni * Bc; e += NT) {
      const int o = e % ni, r = e / ni;
      const float a = elu_f(part_sum(part1, d.Hap, r, o) + sm[L.b1 + o]);
      bcast(L.av + (size_t)r * Hdp + i0 + o, a, V_AV);
    }
    if (!(ok = wait_vec(V_AV))) break;
    if (tr) p.trace[t * 16 + 1] = globaltimer_ns();
    // ---- phase 2: GRUCell(a, belief) for owned units
    const long long c2 = clock64();
    // (the two products side by side, each on half of the threads)
    matvec_sl<NR, 8>(sm + L.wih, Hdp, d.U3p, Hd, sm + L.av, Hdp, part1, 0, NT / 2);
    matvec_sl<NR, 8>(sm + L.whh, RHp, d.U3p, RH, bel_cur, RHp, part2, NT / 2, NT / 2);
    __syncthreads();
    if (tr) p.trace[t * 16 + 8] = clock64() - c2;
    for (int e = tid; e < nj * Bc; e += NT) {
      const int j = e % nj, r = e / nj;
      const int O = d.U3p;
      float gi[3], gh[3];
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        gi[g] = part_sum(part1, O, r, g * d.Ua + j) + sm[L.bih + g * d.Ua + j];
        gh[g] = part_sum(part2, O, r, g * d.Ua + j) + sm[L.bhh + g * d.Ua + j];
      }
      const float rg = sigmoid_f(gi[0] + gh[0]);
      const float zg = sigmoid_f(gi[1] + gh[1]);
      const float ng = tanh_f(gi[2] + rg * gh[2]);
      const float hb = (1.f - zg) * ng + zg * bel_cur[(size_t)r * RHp + j0 + j];
      bcast(bel_nxt + (size_t)r * RHp + j0 + j, hb, V_BEL);
      if (r < nr) p.beliefs[((size_t)t * p.B + b0 + r) * RH + j0 + j] = hb;
    }
    if (tr) p.trace[t * 16 + 9] = clock64() - c2;
    if (!(ok = wait_vec(V_BEL))) break;
    if (tr) p.trace[t * 16 + 2] = globaltimer_ns();
    // ---- phase 3: q = ELU(W2 belief + b2), owned outputs
    matvec_sl<NR, 16>(sm + L.w2, RHp, d.Hap, RH, sm + bel_nxt, RHp, part1, 0, NT);
    __syncthreads();
    for (int e = tid; e < ni * Bc; e += NT) {
      const int o = e % ni, r = e / ni;
      const float qv = elu_f(part_sum(part1, d.Hap, r, o) + sm[L.b2 + o]);
      bcast(L.qv + (size_t)r * Hdp + i0 + o, qv, V_QV);
    }
    if (!(ok = wait_vec(V_QV))) break;
    if (tr) p.trace[t * 16 + 3] = globaltimer_ns();
    // ---- phase 4: p = W3 q + b3 -> mean, std, sampled state (owned entries)
    matvec_sl<NR, 16>(sm + L.w3, Hdp, d.S2p, Hd, sm + L.qv, Hdp, part1, 0, NT);
    __syncthreads();
    for (int e = tid; e < ns * Bc; e += NT) {
      const int j = e % ns, r = e / ns;
      const float mean = part_sum(part1, d.S2p, r, j) + sm[L.b3 + j];
      const float sd =
          softplus_f(part_sum(part1, d.S2p, r, d.Sa + j) + sm[L.b3 + d.Sa + j]) + 0.1f;
      float st = mean;
      if (r < nr) {
        const size_t o = ((size_t)t * p.B + b0 + r) * S + s0 + j;
        const float ev = L.preload ? sm[L.eps + ((size_t)t * Bc + r) * S + s0 + j] : __ldg(p.eps + o);
        st = fmaf(ev, sd, mean);
        p.means[o] = mean;
        p.stds[o] = sd;
        p.states[o] = st;
      }
      // the last step's state feeds no further step: not sent
      if (t + 1 < p.T && !(p.drop_send && t == 0 && blockIdx.x == 0))
        bcast(L.st + (size_t)r * S + s0 + j, st, V_ST);
    }
    if (p.trace) __syncthreads();  // (trace only: this CTA's phase 4 is done)
    if (tr) p.trace[t * 16 + 4] = globaltimer_ns();
  }
  // On a normal exit every byte sent to this CTA has been waited for.  After
  // a failed wait, peers may still be sending: every CTA leaves its loop (a
  // bounded wait or the error word ends each one), then the whole cluster
  // meets, and each CTA gives stores already issued time to land before its
  // shared memory goes away.
  if (!ok && tid == 0) atomicCAS(p.err, DEV_OK, DEV_TIMEOUT);
  cluster.sync();
  if (!ok || ld_volatile_int(p.err) != DEV_OK) {
    const uint64_t until = globaltimer_ns() + 20000;  // 20 us
    while (globaltimer_ns() < until) {
    }
  }
}

// ---------------------------------------------------------------------------
// Reverse-time chain of the backward pass through the unroll (given
// actions), the training use of the prior behind the same page.  Per step t,
// from T-1 down to 0, for each row:
//   ds = dstates_t + ds_t(from t+1),  dmean = dmeans_t + ds,
//   dstd = dstds_t + ds * eps_t,  dp = [dmean, dstd * sigmoid(p_std)];
//   dv = (W3^T dp) * ELU'(v);
//   dh = dbeliefs_t + W2^T dv + W_hh^T dR_{t+1} + z_{t+1} * dh_{t+1};
//   GRU gate gradients dA (input side) and dR (hidden side) from r, z, n,
//   the hidden-side n pre-activation and h_{t-1};
//   du = (W_ih^T dA) * ELU'(u);  ds_{t-1} = W1[:, :S]^T du.
// Everything off this chain (the forward's activations, the weight and
// action gradients) is GEMMs over all rows outside the kernel.  As in the
// forward kernel, a cluster of RC CTAs holds the weights (here transposed for
// W^T x, each CTA the columns of the outputs it owns, and every CTA all of
// W1's state columns), the rows of one batch slice run through four phases
// per step, and the three vectors every CTA needs in full (dv, dR with dA,
// du) are broadcast with st.async into every CTA's shared memory, each
// counted on that vector's mbarrier.  A CTA sends a vector of step t-1 only
// after every CTA has sent du of step t, which each does after reading all
// three vectors of step t, so one buffer per vector suffices.
constexpr int MAXBC_BWD = 4;

struct BwdDims {
  int S, Hd, RH, Bc, Ha, Ua, Hap, Uap, Sp, S2p, Hdp, G3p;
};
__host__ __device__ inline BwdDims make_bdims(int S, int Hd, int RH, int Bc) {
  BwdDims d;
  d.S = S; d.Hd = Hd; d.RH = RH; d.Bc = Bc;
  d.Ha = ceil_div(Hd, RC);
  d.Ua = ceil_div(RH, RC);
  d.Hap = r4(d.Ha);
  d.Uap = r4(d.Ua);
  d.Sp = r4(S);
  d.S2p = r4(2 * S);
  d.Hdp = r4(Hd);
  d.G3p = r4(3 * RH);
  return d;
}
struct BwdLayout {
  size_t w3, w2, whh, wih, w1s;       // weights, [o][k] (columns of W as rows)
  size_t dp, dv, dra, du, cs, gh, dhz;  // vectors, [Bc][padded width]
  size_t part1, part2, total;
};
__host__ __device__ inline BwdLayout make_blayout(const BwdDims &d) {
  BwdLayout L;
  size_t o = 0;
  auto take = [&](size_t n) { size_t r = o; o += (n + 3) & ~size_t(3); return r; };
  L.w3 = take((size_t)d.Hap * d.S2p);   // W3^T dp -> owned outputs of Hd
  L.w2 = take((size_t)d.Uap * d.Hdp);   // W2^T dv -> owned units
  L.whh = take((size_t)d.Uap * d.G3p);  // W_hh^T dR -> owned units
  L.wih = take((size_t)d.Hap * d.G3p);  // W_ih^T dA -> owned outputs of Hd
  L.w1s = take((size_t)d.Sp * d.Hdp);   // W1[:, :S]^T du -> every state entry
  L.dp = take((size_t)d.Bc * d.S2p);
  L.dv = take((size_t)d.Bc * d.Hdp);
  L.dra = take((size_t)d.Bc * 2 * d.G3p);  // per row: dR [3RH], then dA [3RH]
  L.du = take((size_t)d.Bc * d.Hdp);
  L.cs = take((size_t)d.Bc * d.Sp);
  L.gh = take((size_t)d.Bc * d.Uap);
  L.dhz = take((size_t)d.Bc * d.Uap);
  int wmax = d.Hap > d.Uap ? d.Hap : d.Uap;
  if (d.Sp > wmax) wmax = d.Sp;
  L.part1 = take((size_t)d.Bc * wmax);  // a phase's sums, [Bc][outputs]
  L.part2 = take((size_t)d.Bc * wmax);
  L.total = o;
  return L;
}

// dst[o * ldw + k] = src[k * ld + col0 + o] for k < K, o < n (a column
// slice of a row-major matrix, kept as rows [o][k]; other entries are left
// as they are, zero)
__device__ __forceinline__ void load_cols(const float *src, int ld, int K, int col0, int n,
                                          int ldw, float *dst) {
  for (int e = threadIdx.x; e < n * K; e += NT) {
    const int k = e / n, o = e % n;
    dst[(size_t)o * ldw + k] = src[(size_t)k * ld + col0 + o];
  }
}

enum BVec { BV_DV = 0, BV_DRA, BV_DU, NBVEC };

template <int NR>
__global__ void __cluster_dims__(RC, 1, 1) __launch_bounds__(NT, 1)
    rssm_bwd_chain_kernel(const RssmBwdChainParams p, int Bc) {
  extern __shared__ __align__(16) float sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int b0 = (int)(blockIdx.x / RC) * Bc;
  const int nr = min(Bc, p.B - b0);  // rows of this cluster (uniform across the cluster)
  const BwdDims d = make_bdims(p.S, p.Hd, p.RH, Bc);
  const BwdLayout L = make_blayout(d);
  const int S = d.S, Hd = d.Hd, RH = d.RH, G = 3 * RH, S2 = 2 * S;
  const int i0 = c * d.Ha, ni = max(0, min(d.Ha, Hd - i0));  // owned outputs of Hd
  const int j0 = c * d.Ua, nj = max(0, min(d.Ua, RH - j0));  // owned GRU units
  const int tid = threadIdx.x;
  const int ldra = 2 * d.G3p;

  for (size_t e = tid; e < L.total; e += NT) sm[e] = 0.f;
  __syncthreads();
  load_cols(p.W3, Hd, S2, i0, ni, d.S2p, sm + L.w3);
  load_cols(p.W2, RH, Hd, j0, nj, d.Hdp, sm + L.w2);
  load_cols(p.Whh, RH, G, j0, nj, d.G3p, sm + L.whh);
  load_cols(p.Wih, Hd, G, i0, ni, d.G3p, sm + L.wih);
  load_cols(p.W1, S + p.A, Hd, 0, S, d.Hdp, sm + L.w1s);
  __shared__ uint64_t vbar[NBVEC];
  __shared__ int s_ok;
  if (tid == 0) {
    for (int v = 0; v < NBVEC; ++v) tc::mbar_init(&vbar[v], 1);
    tc::fence_mbar_init();
  }
  // every CTA's buffers are zero and its mbarriers exist before any peer sends
  cluster.sync();

  const uint32_t sm0 = (uint32_t)__cvta_generic_to_shared(sm);
  uint32_t rsm[RC], rbar[RC];
#pragma unroll
  for (int r = 0; r < RC; ++r) {
    rsm[r] = tc::mapa_shared(sm0, (uint32_t)r);
    rbar[r] = tc::mapa_shared((uint32_t)__cvta_generic_to_shared(&vbar[0]), (uint32_t)r);
  }
  auto bcast = [&](size_t off, float v, int vec) {
#pragma unroll
    for (int r = 0; r < RC; ++r)
      st_async_b32(rsm[r] + (uint32_t)(off * 4), v, rbar[r] + (uint32_t)(vec * 8));
  };
  uint32_t vbytes[NBVEC];
  vbytes[BV_DV] = (uint32_t)(Bc * Hd * 4);
  vbytes[BV_DRA] = (uint32_t)(Bc * 2 * G * 4);
  vbytes[BV_DU] = (uint32_t)(Bc * Hd * 4);
  uint32_t uses = 0;  // thread 0: completed uses per vector, 4 bits each
  volatile int abort_ = 0;
  const uint64_t tmo = p.timeout_ns;
  auto wait_vec = [&](int vec) -> bool {
    if (tid == 0) {
      const uint32_t n = (uses >> (4 * vec)) & 15u;
      tc::mbar_arrive_expect_tx(&vbar[vec], vbytes[vec]);
      s_ok = tc::mbar_wait(&vbar[vec], n & 1u, p.err, &abort_, tmo);
      uses = (uses & ~(15u << (4 * vec))) | (((n + 1) & 15u) << (4 * vec));
    }
    __syncthreads();
    return s_ok != 0;
  };
  float *part1 = sm + L.part1, *part2 = sm + L.part2;
  bool ok = true;

  for (int t = p.T - 1; t >= 0; --t) {
    const size_t rt = (size_t)t * p.B + b0;  // packed row of (t, b0)
    // ---- phase 1: dp of the sample and head (every CTA, all of its rows),
    //      dv = (W3^T dp) * ELU'(v) for the owned outputs, broadcast
    for (int e = tid; e < Bc * S; e += NT) {
      const int r = e / S, j = e % S;
      float dm = 0.f, dsd = 0.f;
      if (r < nr) {
        const size_t o = (rt + r) * S + j;
        const float ds = (p.dstates ? p.dstates[o] : 0.f) + sm[L.cs + (size_t)r * d.Sp + j];
        dm = (p.dmeans ? p.dmeans[o] : 0.f) + ds;
        dsd = ((p.dstds ? p.dstds[o] : 0.f) + ds * p.eps[o]) *
              sigmoid_f(p.p[(rt + r) * S2 + S + j]);
        if (c == 0) {
          p.DP[(rt + r) * S2 + j] = dm;
          p.DP[(rt + r) * S2 + S + j] = dsd;
        }
      }
      sm[L.dp + (size_t)r * d.S2p + j] = dm;
      sm[L.dp + (size_t)r * d.S2p + S + j] = dsd;
    }
    __syncthreads();
    matvec_sl<NR, 16>(sm + L.w3, d.S2p, d.Hap, S2, sm + L.dp, d.S2p, part1, 0, NT);
    __syncthreads();
    for (int e = tid; e < ni * Bc; e += NT) {
      const int o = e % ni, r = e / ni;
      float dv = 0.f;
      if (r < nr) {
        const float vv = p.v[(rt + r) * Hd + i0 + o];
        dv = part_sum(part1, d.Hap, r, o) * (vv > 0.f ? 1.f : expf(vv));
        p.DV[(rt + r) * Hd + i0 + o] = dv;
      }
      bcast(L.dv + (size_t)r * d.Hdp + i0 + o, dv, BV_DV);
    }
    if (!(ok = wait_vec(BV_DV))) break;
    // ---- phase 2: dh of the owned units, their gate gradients; dR and dA broadcast
    matvec_sl<NR, 16>(sm + L.w2, d.Hdp, d.Uap, Hd, sm + L.dv, d.Hdp, part1, 0, NT);
    __syncthreads();
    for (int e = tid; e < nj * Bc; e += NT) {
      const int jj = e % nj, r = e / nj, j = j0 + jj;
      float ar = 0.f, az = 0.f, dan = 0.f, rg = 0.f;
      if (r < nr) {
        const size_t row = rt + r;
        const float dh = (p.dbeliefs ? p.dbeliefs[row * RH + j] : 0.f) +
                         part_sum(part1, d.Uap, r, jj) + sm[L.gh + (size_t)r * d.Uap + jj] +
                         sm[L.dhz + (size_t)r * d.Uap + jj];
        const float *g = p.gates + row * G;
        rg = g[j];
        const float z = g[RH + j], n = g[2 * RH + j];
        const float hn = p.zh[row * G + 2 * RH + j];
        const float dn = dh * (1.f - z), dz = dh * (p.hp[row * RH + j] - n);
        dan = dn * (1.f - n * n);
        ar = dan * hn * rg * (1.f - rg);
        az = dz * z * (1.f - z);
        float *da = p.DA + row * G, *dr = p.DR + row * G;
        da[j] = ar; da[RH + j] = az; da[2 * RH + j] = dan;
        dr[j] = ar; dr[RH + j] = az; dr[2 * RH + j] = dan * rg;
        sm[L.dhz + (size_t)r * d.Uap + jj] = dh * z;
      }
      const size_t rb = L.dra + (size_t)r * ldra;
      bcast(rb + j, ar, BV_DRA);
      bcast(rb + RH + j, az, BV_DRA);
      bcast(rb + 2 * RH + j, dan * rg, BV_DRA);
      bcast(rb + d.G3p + j, ar, BV_DRA);
      bcast(rb + d.G3p + RH + j, az, BV_DRA);
      bcast(rb + d.G3p + 2 * RH + j, dan, BV_DRA);
    }
    if (!(ok = wait_vec(BV_DRA))) break;
    // ---- phase 3: W_hh^T dR for the owned units (carried to step t-1),
    //      du = (W_ih^T dA) * ELU'(u) for the owned outputs, broadcast
    // (the two products side by side, each on half of the threads)
    matvec_sl<NR, 16>(sm + L.whh, d.G3p, d.Uap, G, sm + L.dra, ldra, part1, 0, NT / 2);
    matvec_sl<NR, 16>(sm + L.wih, d.G3p, d.Hap, G, sm + L.dra + d.G3p, ldra, part2, NT / 2,
                      NT / 2);
    __syncthreads();
    for (int e = tid; e < nj * Bc; e += NT) {
      const int jj = e % nj, r = e / nj;
      sm[L.gh + (size_t)r * d.Uap + jj] = part_sum(part1, d.Uap, r, jj);
    }
    for (int e = tid; e < ni * Bc; e += NT) {
      const int o = e % ni, r = e / ni;
      float du = 0.f;
      if (r < nr) {
        const float uu = p.u[(rt + r) * Hd + i0 + o];
        du = part_sum(part2, d.Hap, r, o) * (uu > 0.f ? 1.f : expf(uu));
        p.DU[(rt + r) * Hd + i0 + o] = du;
      }
      bcast(L.du + (size_t)r * d.Hdp + i0 + o, du, BV_DU);
    }
    if (!(ok = wait_vec(BV_DU))) break;
    // ---- phase 4: ds_{t-1} = W1[:, :S]^T du (every CTA, every state entry)
    matvec_sl<NR, 16>(sm + L.w1s, d.Hdp, d.Sp, Hd, sm + L.du, d.Hdp, part1, 0, NT);
    __syncthreads();
    for (int e = tid; e < Bc * S; e += NT) {
      const int r = e / S, k = e % S;
      sm[L.cs + (size_t)r * d.Sp + k] = part_sum(part1, d.Sp, r, k);
    }
    __syncthreads();
  }
  if (ok) {
    // gradients reaching the initial state and belief
    for (int e = tid; e < nr * S; e += NT) {
      const int r = e / S, k = e % S;
      if (c == 0 && p.cs_out) p.cs_out[(size_t)(b0 + r) * S + k] = sm[L.cs + (size_t)r * d.Sp + k];
    }
    for (int e = tid; e < nr * nj; e += NT) {
      const int r = e / nj, jj = e % nj;
      if (p.gh_out)
        p.gh_out[(size_t)(b0 + r) * RH + j0 + jj] =
            sm[L.gh + (size_t)r * d.Uap + jj] + sm[L.dhz + (size_t)r * d.Uap + jj];
    }
  }
  // exit as the forward kernel: on a normal exit every byte sent here has
  // been waited for; after a failed wait the cluster meets and each CTA lets
  // stores already issued land before its shared memory goes away
  if (!ok && tid == 0) atomicCAS(p.err, DEV_OK, DEV_TIMEOUT);
  cluster.sync();
  if (!ok || ld_volatile_int(p.err) != DEV_OK) {
    const uint64_t until = globaltimer_ns() + 20000;  // 20 us
    while (globaltimer_ns() < until) {
    }
  }
}

size_t bwd_smem_bytes(int S, int Hd, int RH, int Bc) {
  return make_blayout(make_bdims(S, Hd, RH, Bc)).total * sizeof(float);
}

template <int NR>
cudaError_t launch_bwd_nr(const RssmBwdChainParams &p, int Bc, int grid, size_t smem,
                          cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute((const void *)rssm_bwd_chain_kernel<NR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rssm_bwd_chain_kernel<NR><<<grid, NT, smem, s>>>(p, Bc);
  return cudaGetLastError();
}

int pick_bc(int B, int nsm) {
  int clusters = nsm / RC;
  if (clusters < 1) clusters = 1;
  int bc = ceil_div(B, clusters);
  if (bc < 1) bc = 1;
  if (bc > MAXBC) bc = MAXBC;
  return bc;
}

template <int NR>
cudaError_t launch_nr(const RssmParams &p, int Bc, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute((const void *)rssm_kernel<NR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rssm_kernel<NR><<<grid, NT, smem, s>>>(p, Bc);
  return cudaGetLastError();
}

size_t smem_bytes(int S, int A, int Hd, int RH, int Bc, int T, int Hx = 0) {
  return make_layout(make_dims(S, A, Hd, RH, Bc, Hx), T).total * sizeof(float);
}

}  // namespace

bool rssm_supported(int S, int A, int Hd, int RH, int Hx) {
  if (S < 1 || A < 0 || Hd < 1 || RH < 1 || Hx < 0 || (Hx > 0 && A < 1)) return false;
  return smem_bytes(S, A, Hd, RH, 1, 0, Hx) <= SMEM_CAP;
}

// Clusters of RC CTAs that can be resident at once with this shared-memory
// size (a cluster needs RC free SMs in one GPC, so this is below nsm / RC).
int resident_clusters(size_t smem, int Bc, int nsm) {
  const void *fn;
  switch (Bc) {
    case 1: fn = (const void *)rssm_kernel<1>; break;
    case 2: fn = (const void *)rssm_kernel<2>; break;
    case 3: fn = (const void *)rssm_kernel<3>; break;
    case 4: fn = (const void *)rssm_kernel<4>; break;
    case 5: fn = (const void *)rssm_kernel<5>; break;
    case 6: fn = (const void *)rssm_kernel<6>; break;
    case 7: fn = (const void *)rssm_kernel<7>; break;
    default: fn = (const void *)rssm_kernel<8>; break;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return std::max(1, nsm / RC);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(RC);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = RC;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return std::max(1, nsm / RC);
  }
  return n;
}

bool rssm_bwd_chain_supported(int S, int A, int Hd, int RH) {
  if (S < 1 || A < 0 || Hd < 1 || RH < 1) return false;
  return bwd_smem_bytes(S, Hd, RH, 1) <= SMEM_CAP;
}

cudaError_t launch_rssm_bwd_chain(const RssmBwdChainParams &p, int nsm, cudaStream_t s) {
  int Bc = std::min(pick_bc(p.B, nsm), MAXBC_BWD);
  while (Bc > 1 && bwd_smem_bytes(p.S, p.Hd, p.RH, Bc) > SMEM_CAP) --Bc;
  const size_t smem = bwd_smem_bytes(p.S, p.Hd, p.RH, Bc);
  if (smem > SMEM_CAP) return cudaErrorInvalidConfiguration;
  const int grid = ceil_div(p.B, Bc) * RC;
  switch (Bc) {
    case 1: return launch_bwd_nr<1>(p, Bc, grid, smem, s);
    case 2: return launch_bwd_nr<2>(p, Bc, grid, smem, s);
    case 3: return launch_bwd_nr<3>(p, Bc, grid, smem, s);
    default: return launch_bwd_nr<4>(p, Bc, grid, smem, s);
  }
}

cudaError_t launch_rssm(const RssmParams &p, int nsm, cudaStream_t s, int *clusters_used) {
  const int hx = p.Wa1 ? p.Hx : 0;
  int Bc = pick_bc(p.B, nsm);
  while (Bc > 1 && smem_bytes(p.S, p.A, p.Hd, p.RH, Bc, p.T, hx) > SMEM_CAP) --Bc;
  // all clusters should be resident together: grow the batch slice until they are
  for (int it = 0; it < MAXBC; ++it) {
    const int room = resident_clusters(smem_bytes(p.S, p.A, p.Hd, p.RH, Bc, p.T, hx), Bc, nsm);
    if (ceil_div(p.B, Bc) <= room || Bc >= MAXBC) break;
    if (smem_bytes(p.S, p.A, p.Hd, p.RH, Bc + 1, p.T, hx) > SMEM_CAP) break;
    ++Bc;
  }
  const size_t smem = smem_bytes(p.S, p.A, p.Hd, p.RH, Bc, p.T, hx);
  if (smem > SMEM_CAP) return cudaErrorInvalidConfiguration;
  const int clusters = ceil_div(p.B, Bc);
  if (clusters_used) *clusters_used = clusters;
  switch (Bc) {
    case 1: return launch_nr<1>(p, Bc, clusters * RC, smem, s);
    case 2: return launch_nr<2>(p, Bc, clusters * RC, smem, s);
    case 3: return launch_nr<3>(p, Bc, clusters * RC, smem, s);
    case 4: return launch_nr<4>(p, Bc, clusters * RC, smem, s);
    case 5: return launch_nr<5>(p, Bc, clusters * RC, smem, s);
    case 6: return launch_nr<6>(p, Bc, clusters * RC, smem, s);
    case 7: return launch_nr<7>(p, Bc, clusters * RC, smem, s);
    default: return launch_nr<8>(p, Bc, clusters * RC, smem, s);
  }
}

}  // namespace rcu
