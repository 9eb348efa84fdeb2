// Backward pass through time (BPTT) of the stacked unidirectional LSTM / GRU,
// fp32: the training use of the unrolled cell behind "[Feature Request] CUDNN
// version of RSSM" (pytorch/rl issue 366, Motivation: the loop dominates
// training) and "Integrating CuDNN API for LSTMs with projections"
// (pytorch/pytorch issue 46213, the training discussion).
//
// The sequential part is only the recurrence of the hidden-state gradient,
//     dh_{t-1} = W_hh^T dR_t (+ z_t * dh_t for the GRU),
// which bwd_rec_kernel runs as one persistent cooperative launch over all
// steps in reverse time: each CTA owns U hidden units of a batch group with
// W_hh columns resident in shared memory (its own units', or with K split
// over a CTA pair, the pair's units over half of K: bwd_rec_pair_kernel),
// computes the gate gradients of its units from the saved activations,
// publishes them, crosses one bounded barrier per batch group, and forms its
// units' dh_{t-1} from everyone's gate gradients.  Everything else is parallel over steps: the pre-activations
// are recomputed as two GEMMs (X W_ih^T, H_prev W_hh^T) once every layer's
// output sequence is known, the LSTM cell sequence is one elementwise scan
// (bwd_prep_kernel), and the weight and input gradients are GEMMs over all
// T*B rows (through transposes) plus a deterministic column sum for the
// biases.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int NT = 512;

// ---- activations and the LSTM cell scan.  zin holds X W_ih^T + b_ih on
// entry and the activated gates on exit (LSTM i, f, g, o; GRU r, z, n);
// zh = H_prev W_hh^T + b_hh is only read.  cs[t][b][u] = c_t (LSTM);
// ms[t][b][u] = m_t = o tanh(c_t) when ms is given (LSTM with projection).
// Cell clipping (cr given): cr[t][b][u] = f c' + i g before the clamp, and
// c_t = clamp(that, clo, chi) as in the forward.
__global__ void bwd_prep_kernel(int T, int B, int H, int cell, float *__restrict__ zin,
                                const float *__restrict__ zh, const float *__restrict__ c0,
                                float *__restrict__ cs, float *__restrict__ ms,
                                float *__restrict__ cr, float clo, float chi) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= B * H) return;
  const int b = e / H, u = e % H;
  const int nG = cell == CELL_LSTM ? 4 : 3, G = nG * H;
  float c = (cell == CELL_LSTM && c0) ? c0[(size_t)b * H + u] : 0.f;
  // Only c carries from step to step: the pre-activations of SD steps are
  // loaded before any of them is used, so their memory latencies overlap
  // (the loop is otherwise one dependent round trip per step).
  constexpr int SD = 8;
  for (int t0 = 0; t0 < T; t0 += SD) {
    float pa[SD][4], ph[SD][4];
#pragma unroll
    for (int j = 0; j < SD; ++j) {
      if (t0 + j >= T) break;
      const size_t r = (size_t)(t0 + j) * B + b;
      const float *a = zin + r * G, *h = zh + r * G;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q >= nG) break;
        pa[j][q] = a[q * H + u];
        ph[j][q] = h[q * H + u];
      }
    }
#pragma unroll
    for (int j = 0; j < SD; ++j) {
      if (t0 + j >= T) break;
      const size_t r = (size_t)(t0 + j) * B + b;
      float *a = zin + r * G;
      if (cell == CELL_LSTM) {
        const float i = sigmoid_f(pa[j][0] + ph[j][0]);
        const float f = sigmoid_f(pa[j][1] + ph[j][1]);
        const float g = tanh_f(pa[j][2] + ph[j][2]);
        const float o = sigmoid_f(pa[j][3] + ph[j][3]);
        c = f * c + i * g;
        if (cr) {
          cr[r * H + u] = c;
          c = fminf(fmaxf(c, clo), chi);
        }
        cs[r * H + u] = c;
        if (ms) ms[r * H + u] = o * tanh_f(c);
        a[u] = i; a[H + u] = f; a[2 * H + u] = g; a[3 * H + u] = o;
      } else {
        const float rg = sigmoid_f(pa[j][0] + ph[j][0]);
        const float z = sigmoid_f(pa[j][1] + ph[j][1]);
        const float n = tanh_f(pa[j][2] + rg * ph[j][2]);
        a[u] = rg; a[H + u] = z; a[2 * H + u] = n;
      }
    }
  }
}

constexpr int UMAX = 16;  // hidden units per CTA (register tile width)
// dynamic shared memory of the reverse-time kernel: the opt-in per-block
// limit (227 KB) less room for its static shared memory (the barrier flag)
constexpr size_t SMEM_CAP = 227 * 1024 - 64;

// a row length clamped to [1, T] (the forward flags out-of-range lengths in
// the status word and runs them clamped the same way)
__device__ __forceinline__ int clamp_len(int len, int T) { return len < 1 ? 1 : (len > T ? T : len); }

// 16-byte asynchronous global -> shared copy (cached in L2 only)
__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct BwdParams {
  int T, B, H, cell, U;
  int Gp, KC, KS;     // gate width padded to 4; staged chunk of dR columns; K slices
  int NB;             // staging buffers (chunks in flight: NB - 1)
  int KP, Gh;         // CTAs splitting K (1 or 2); K columns each holds
  int BS, NUG;        // batch rows per CTA; unit groups (CTA = batch group x unit group)
  int per;            // CTAs of this problem (batch groups x unit groups)
  const float *Whh;   // [nG*H][ldw], PyTorch row order
  int ldw;
  const float *gates; // [T*B][G] activated gates
  const float *zh;    // GRU: [T*B][G] hidden-side pre-activations (n part: W_hn h' + b_hn)
  const float *cs;    // LSTM: [T*B][H] c_t
  const float *c0;    // LSTM: [B][H] or NULL
  const float *hp;    // GRU: [T*B][H] h_{t-1}
  const float *dy;    // [T*B][H]
  const float *dhn, *dcn;  // [B][H] or NULL
  const int32_t *lengths;  // [B] or NULL: row b runs steps 0 .. len_b - 1 only
  const float *cr;    // LSTM cell clipping: [T*B][H] unclamped c_t, or NULL
  float clo, chi;     // its bounds: the clamp passes dc where clo <= cr <= chi
  float *DA, *DR;     // [T*B][G]: input-side and hidden-side gate gradients (LSTM: DR == DA)
  float *dh0, *dc0;   // [B][H] or NULL
  unsigned *ctr;
  int *err;
  uint64_t timeout_ns;
  int drop_arrival;
  unsigned long long *trace;  // NULL, or stamps of CTA 0 (row = reverse step)
};

__device__ __forceinline__ void prefetch_l2(const float *q) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
}

__device__ __forceinline__ void rstamp(const BwdParams &p, int s, int slot) {
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 0)
    p.trace[(size_t)s * 16 + slot] = globaltimer_ns();
}

// KP = 1: the CTA holds W_hh^T columns of its own U units over all K = G.
// KP = 2: a cluster of two CTAs (unit groups 2i, 2i + 1 of one batch group)
// splits K: each holds the pair's 2U units over its half of K, stages only
// that half of dR_t (so all of it is in flight at once), and sends the
// partial sums of the other CTA's units into that CTA's shared memory
// (st.async, counted on its mbarrier).
template <int KP>
__device__ __forceinline__ void bwd_rec_body(const BwdParams &p, const int bid) {
  extern __shared__ __align__(16) float sm[];
  __shared__ uint64_t xbar;       // KP = 2: the peer's partial sums of this CTA's units
  __shared__ unsigned peer_sent;  // KP = 2: steps the peer sent (stored by the peer at exit)
  __shared__ int s_go, s_abort;
  const int H = p.H, B = p.B, U = p.U;
  const bool lstm = p.cell == CELL_LSTM;
  const int G = (lstm ? 4 : 3) * H;
  if (KP > 1 && tc::cluster_nctarank() != (uint32_t)KP) {
    // the K split needs its peer: never address a peer that is not there
    if (threadIdx.x == 0) atomicCAS(p.err, DEV_OK, DEV_CONFIG);
    return;
  }
  // CTA = (batch group bgi: rows [b0, b0 + Bl), unit group ug: units [u0, u0 + nu));
  // batch groups never wait on each other (rows are independent)
  const int BS = p.BS, ug = bid % p.NUG, bgi = bid / p.NUG;
  const int b0 = bgi * BS, Bl = max(0, min(BS, B - b0));
  const int u0 = ug * U, nu = max(0, min(U, H - u0));
  const int kr = KP > 1 ? (ug & 1) : 0;  // this CTA's K share (its rank in the pair)
  const int pu0 = (ug - kr) * U;         // first unit of the W_hh^T columns held
  const int Gp = p.Gp, Gh = p.Gh, KC = p.KC, KS = p.KS, KCP = KC + 4;
  const int kbase = kr * Gh, Kr = max(0, min(Gh, Gp - kbase));  // this CTA's K columns
  float *WT = sm;  // [KP*U][Gh]: WT[j][n] = W_hh[kbase + n][pu0 + j], zero padded
  const int NB = p.NB, PS = BS * U + 1;  // (PS: K-slice stride, padded off a multiple of 32 banks)
  float *xs = WT + (size_t)KP * U * Gh;  // [NB][BS][KCP]: staged columns of dR_t (ring)
  float *part = xs + (size_t)NB * BS * KCP;  // K-slice partial sums (rec_part_floats)
  float *dhrec = part + (KS % 32 == 0 ? (size_t)ceil_div(BS, 4) * KP * (KS / 32) * 64
                                      : (size_t)KS * PS);  // [BS][U]: W_hh^T dR part of dh_t
  float *dcs = dhrec + (size_t)BS * U;   // [BS][U]: LSTM dc carried to the previous step
  float *dhz = dcs + (size_t)BS * U;     // [BS][U]: GRU z * dh (direct path)
  float *recv = dhz + (size_t)BS * U;    // KP = 2, [BS][U]: the peer's partial sums
  unsigned *ctr = p.ctr + bgi;
  const int tid = threadIdx.x;
  for (int e = tid; e < KP * U * Gh; e += NT) {
    const int j = e / Gh, n = e % Gh, unit = pu0 + j, k = kbase + n;
    WT[e] = (unit < H && k < G) ? p.Whh[(size_t)k * p.ldw + unit] : 0.f;
  }
  for (int e = tid; e < BS * U; e += NT) {
    const int b = e / U, j = e % U;
    const bool ok = j < nu && b < Bl;
    dhrec[e] = (ok && p.dhn) ? p.dhn[(size_t)(b0 + b) * H + u0 + j] : 0.f;
    dcs[e] = (ok && lstm && p.dcn) ? p.dcn[(size_t)(b0 + b) * H + u0 + j] : 0.f;
    dhz[e] = 0.f;
  }
  uint32_t peer_recv = 0, peer_bar = 0;
  unsigned x_sent = 0;          // steps whose partial sums this CTA has sent
  int x_posted = 0, x_done = 0;  // thread 0: receive phases armed / completed
  if (KP > 1) {
    if (tid == 0) {
      tc::mbar_init(&xbar, 1);
      peer_sent = 0;
      s_abort = 0;
      tc::fence_mbar_init();
    }
    __syncthreads();
    tc::cluster_sync();  // the peer's barrier exists before any store into it
    peer_recv = tc::mapa_shared(tc::smem_u32(recv), (uint32_t)(kr ^ 1));
    peer_bar = tc::mapa_shared(tc::smem_u32(&xbar), (uint32_t)(kr ^ 1));
  }
  __syncthreads();
  const bool vec = (G & 3) == 0;
  const int RG = ceil_div(Bl, 4);
  bool ok = true;
  for (int t = p.T - 1, it = 1; t >= 0; --t, ++it) {
    rstamp(p, it - 1, 0);
    // ---- gate gradients of this CTA's units at step t
    for (int e = tid; e < Bl * U; e += NT) {
      const int bl = e / U, j = e % U;
      if (j >= nu) continue;
      const int u = u0 + j, b = b0 + bl;
      const size_t r = (size_t)t * B + b;
      if (!RCU_DCHECK(b < B && u < H && r < (size_t)p.T * B, p.err)) continue;
      if (t > 0 && !(p.lengths && t - 1 >= clamp_len(p.lengths[b], p.T))) {
        // the next step's (t - 1) inputs of this (row, unit) into L2 while
        // the barrier and the mat-vec run: its gate phase then waits for L2,
        // not HBM (rows past their end at t - 1 read nothing there)
        const size_t rn = r - B;
        prefetch_l2(p.dy + rn * H + u);
        for (int q = 0; q < (lstm ? 4 : 3); ++q) prefetch_l2(p.gates + rn * G + q * H + u);
        if (lstm) {
          prefetch_l2(p.cs + rn * H + u);
          if (t > 1) prefetch_l2(p.cs + (rn - B) * H + u);
          if (p.cr) prefetch_l2(p.cr + rn * H + u);
        } else {
          prefetch_l2(p.zh + rn * G + 2 * H + u);
          prefetch_l2(p.hp + rn * H + u);
        }
      }
      float *da = p.DA + r * G;
      if (p.lengths && t >= clamp_len(p.lengths[b], p.T)) {
        // a step past the row's end: no gate gradient, and the carried dh
        // (zero: dh_n enters through dy at the row's last step) and dc pass
        // through unchanged
        float *dr = p.DR + r * G;
        for (int q = 0; q < (lstm ? 4 : 3); ++q) da[q * H + u] = 0.f;
        if (!lstm)
          for (int q = 0; q < 3; ++q) dr[q * H + u] = 0.f;
        continue;
      }
      const float dh = p.dy[r * H + u] + dhrec[e];
      const float *g = p.gates + r * G;
      if (lstm) {
        const float i = g[u], f = g[H + u], gg = g[2 * H + u], o = g[3 * H + u];
        const float c = p.cs[r * H + u];
        const float cp = t > 0 ? p.cs[(r - B) * H + u] : (p.c0 ? p.c0[(size_t)b * H + u] : 0.f);
        const float tc = tanh_f(c);
        float dc = dcs[e] + dh * o * (1.f - tc * tc);
        if (p.cr) {  // through the cell-state clamp
          const float v = p.cr[r * H + u];
          if (v < p.clo || v > p.chi) dc = 0.f;
        }
        da[u] = dc * gg * i * (1.f - i);
        da[H + u] = dc * cp * f * (1.f - f);
        da[2 * H + u] = dc * i * (1.f - gg * gg);
        da[3 * H + u] = dh * tc * o * (1.f - o);
        dcs[e] = dc * f;
      } else {
        const float rg = g[u], z = g[H + u], n = g[2 * H + u];
        const float hn = p.zh[r * G + 2 * H + u];
        const float hprev = p.hp[r * H + u];
        const float dn = dh * (1.f - z);
        const float dz = dh * (hprev - n);
        const float dan = dn * (1.f - n * n);
        const float ar = dan * hn * rg * (1.f - rg);
        const float az = dz * z * (1.f - z);
        float *dr = p.DR + r * G;
        da[u] = ar; da[H + u] = az; da[2 * H + u] = dan;
        dr[u] = ar; dr[H + u] = az; dr[2 * H + u] = dan * rg;
        dhz[e] = dh * z;
      }
    }
    rstamp(p, it - 1, 1);
    // every CTA's gate gradients of step t are published
    if (!group_barrier(ctr, (unsigned)it * p.NUG, p.err, p.timeout_ns,
                       p.drop_arrival && blockIdx.x == 0 && it == 1)) {
      ok = false;
      break;
    }
    rstamp(p, it - 1, 2);
    // ---- dh_{t-1} of this CTA's units: W_hh^T dR_t (+ z dh).  dR_t is staged
    // in chunks of KC columns with coalesced loads; thread (row group of 4,
    // K slice) keeps a 4 x U register tile and walks the chunk's float4
    // columns interleaved by K slice (consecutive threads read consecutive
    // 16-byte words: no bank conflicts); the K-slice partials are summed last.
    const float *drt = (lstm ? p.DA : p.DR) + (size_t)t * B * G + kbase;
    // thread = (row group, unit half of the held columns, K slice)
    const int rg = tid / (KP * KS), hh = (tid / KS) % KP, ksl = tid % KS;
    const bool comp = rg < RG;
    float acc[4][UMAX];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < UMAX; ++j) acc[r][j] = 0.f;
    const int nch = ceil_div(Kr, KC);
    // stage chunk c of dR_t into buffer c % NB: cp.async when rows are
    // 16-byte aligned (G a multiple of 4), else plain loads; one commit group
    // per call (empty past the last chunk, so the group count stays uniform)
    auto stage = [&](int c) {
      if (c >= nch) {
        cp_async_commit();
        return;
      }
      const int k0 = c * KC, kc4 = min(KC, Kr - k0) >> 2;
      float *xb = xs + (size_t)(c % NB) * BS * KCP;
      for (int e = tid; e < Bl * kc4; e += NT) {
        const int b = e / kc4, q = e % kc4, k = k0 + 4 * q;
        const float *src = drt + (size_t)(b0 + b) * G + k;
        float *dst = xb + (size_t)b * KCP + 4 * q;
        if (!RCU_DCHECK(b0 + b < B && kbase + k + 4 <= Gp, p.err)) continue;
        if (vec) {
          cp_async16(dst, src);
        } else {
          const int kg = kbase + k;  // the column in dR_t
          float4 v;
          v.x = kg < G ? __ldcg(src) : 0.f;
          v.y = kg + 1 < G ? __ldcg(src + 1) : 0.f;
          v.z = kg + 2 < G ? __ldcg(src + 2) : 0.f;
          v.w = kg + 3 < G ? __ldcg(src + 3) : 0.f;
          *reinterpret_cast<float4 *>(dst) = v;
        }
      }
      cp_async_commit();
    };
    // NB - 1 chunks in flight while one is multiplied
    for (int c = 0; c < NB - 1; ++c) stage(c);
    for (int c = 0; c < nch; ++c) {
      stage(c + NB - 1);  // into the buffer multiplied in the previous round
      if (NB == 4) cp_async_wait<3>();
      else if (NB == 3) cp_async_wait<2>();
      else cp_async_wait<1>();
      __syncthreads();
      const int k0 = c * KC, kc4 = min(KC, Kr - k0) >> 2;
      const float *xb = xs + (size_t)(c % NB) * BS * KCP;
      const float *wh = WT + (size_t)hh * U * Gh + k0;
      if (comp) {
        for (int q = ksl; q < kc4; q += KS) {
          float4 x[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int b = 4 * rg + r;
            x[r] = b < Bl ? *reinterpret_cast<const float4 *>(xb + (size_t)b * KCP + 4 * q)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < UMAX; ++j) {
            if (j >= U) break;
            const float4 w = *reinterpret_cast<const float4 *>(wh + (size_t)j * Gh + 4 * q);
#pragma unroll
            for (int r = 0; r < 4; ++r)
              acc[r][j] = fmaf(x[r].x, w.x, fmaf(x[r].y, w.y, fmaf(x[r].z, w.z,
                                                   fmaf(x[r].w, w.w, acc[r][j]))));
          }
        }
      }
      __syncthreads();  // buffer c % NB is refilled by stage(c + NB) next round
    }
    cp_async_wait<0>();  // (only empty groups remain)
    rstamp(p, it - 1, 3);
    if (KS % 32 == 0) {
      // A warp's 32 lanes are 32 K slices of one row group: reduce-scatter
      // the 4 x 16 tile over the lanes by shuffles (each step keeps half the
      // values, summed with the partner lane's), so lane l ends with tile
      // entries sbase(l) and sbase(l) + 1 summed over its warp; then the
      // row group's KS / 32 warps are summed through shared memory.
      static_assert(UMAX == 16, "the reduce-scatter walks a 4 x 16 tile");
      if (comp) {
        float v[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = acc[i / 16][i % 16];
        const int lane = tid & 31;
#pragma unroll
        for (int h = 32, m = 16; h >= 2; h >>= 1, m >>= 1) {
          const bool up = (lane & m) != 0;
#pragma unroll
          for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        const int sbase = ((lane >> 4) & 1) * 32 + ((lane >> 3) & 1) * 16 +
                          ((lane >> 2) & 1) * 8 + ((lane >> 1) & 1) * 4 + (lane & 1) * 2;
        float *pw = part + (size_t)((rg * KP + hh) * (KS / 32) + ksl / 32) * 64;
        pw[sbase] = v[0];
        pw[sbase + 1] = v[1];
      }
      __syncthreads();
      const int KW = KS / 32;
      // the sum over the warps of (row group, unit half h) for entry e
      auto psum = [&](int e, int h) {
        const int b = e / U, j = e % U;
        const float *pr = part + (size_t)((b / 4) * KP + h) * KW * 64 + (b % 4) * 16 + j;
        float v = 0.f;
        for (int w = 0; w < KW; ++w) v += pr[(size_t)w * 64];
        return v;
      };
      if (KP > 1) {
        // this CTA's sums of the peer's units to the peer (all BS x U
        // entries: a fixed byte count; rows past Bl are never read)
        for (int e = tid; e < BS * U; e += NT)
          tc::st_async_f32(peer_recv + (uint32_t)e * 4u, e < Bl * U ? psum(e, kr ^ 1) : 0.f,
                           peer_bar);
        x_sent = (unsigned)it;
        if (tid == 0) {
          tc::mbar_arrive_expect_tx(&xbar, (uint32_t)(BS * U * 4));
          x_posted = it;
          s_go = tc::mbar_wait_cluster(&xbar, (uint32_t)(it - 1) & 1u, p.err, &s_abort,
                                       p.timeout_ns);
          if (s_go) x_done = it;
        }
        __syncthreads();
        if (!s_go) {
          ok = false;
          break;
        }
        for (int e = tid; e < Bl * U; e += NT)
          dhrec[e] = (lstm ? 0.f : dhz[e]) + psum(e, kr) + recv[e];
      } else {
        for (int e = tid; e < Bl * U; e += NT) dhrec[e] = (lstm ? 0.f : dhz[e]) + psum(e, 0);
      }
    } else {
      if (comp) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int b = 4 * rg + r;
          if (b >= Bl) break;
#pragma unroll
          for (int j = 0; j < UMAX; ++j)
            if (j < U) part[(size_t)ksl * PS + b * U + j] = acc[r][j];
        }
      }
      __syncthreads();
      for (int e = tid; e < Bl * U; e += NT) {
        float v = 0.f;
        for (int q = 0; q < KS; ++q) v += part[(size_t)q * PS + e];
        dhrec[e] = (lstm ? 0.f : dhz[e]) + v;
      }
    }
    __syncthreads();
    rstamp(p, it - 1, 4);
  }
  for (int e = tid; ok && e < Bl * U; e += NT) {
    const int b = e / U, j = e % U;
    if (j >= nu || !RCU_DCHECK(b0 + b < B && u0 + j < H, p.err)) continue;
    if (p.dh0) p.dh0[(size_t)(b0 + b) * H + u0 + j] = dhrec[e];
    if (lstm && p.dc0) p.dc0[(size_t)(b0 + b) * H + u0 + j] = dcs[e];
  }
  if (KP > 1) {
    // Exit: tell the peer how many steps of sums it will have received from
    // this CTA, while it is certainly resident (neither passes the cluster
    // barrier below before both arrive), then wait (bounded) for a step the
    // peer sent but this CTA did not consume.  Nothing after the barrier
    // touches the peer's shared memory.
    __syncthreads();
    if (tid == 0) {
      const uint32_t dst = tc::mapa_shared(tc::smem_u32(&peer_sent), (uint32_t)(kr ^ 1));
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(x_sent) : "memory");
    }
    tc::cluster_sync();
    if (tid == 0) {
      const unsigned ps = *reinterpret_cast<volatile unsigned *>(&peer_sent);
      if ((int)ps > x_done) {
        if (x_posted == x_done) tc::mbar_arrive_expect_tx(&xbar, (uint32_t)(BS * U * 4));
        volatile int never = 0;
        tc::mbar_wait(&xbar, (uint32_t)x_done & 1u, nullptr, &never, 100000000ull);
      }
    }
  }
}

// p's problem on the first p.per CTAs; q's (a second direction of the same
// shape, its own pointers and counters) on the next q.per, if the grid has them
__global__ void __launch_bounds__(NT, 1) bwd_rec_kernel(const BwdParams p, const BwdParams q) {
  if ((int)blockIdx.x < p.per) bwd_rec_body<1>(p, (int)blockIdx.x);
  else bwd_rec_body<1>(q, (int)blockIdx.x - p.per);
}
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
    bwd_rec_pair_kernel(const BwdParams p, const BwdParams q) {
  // (p.per is even: a pair never straddles the two problems)
  if ((int)blockIdx.x < p.per) bwd_rec_body<2>(p, (int)blockIdx.x);
  else bwd_rec_body<2>(q, (int)blockIdx.x - p.per);
}

// out[c][r] = in[r][c] for an R x C row-major matrix (ldi, ldo: row strides),
// written as fp32 or rounded to bf16 (the tensor-core GEMM operand)
template <typename OT>
__global__ void transpose_kernel(const float *__restrict__ in, int R, int C, int ldi,
                                 OT *__restrict__ out, int ldo) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = in[(size_t)r * ldi + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < R && c < C) out[(size_t)c * ldo + r] = Op<OT>::from_f(tile[threadIdx.x][i]);
  }
}

// The same transposes for 16-byte aligned rows, in 64 x 64 tiles: 16-byte
// loads and stores (4 rows of the input are 4 consecutive outputs), 64 bytes
// in flight per thread.  out (fp32, 16-byte aligned) and outb (bf16, 8-byte
// aligned) are each optional; ldi and ldo are multiples of 4.
constexpr int TT = 64;
__global__ void __launch_bounds__(256) transpose64_kernel(const float *__restrict__ in, int R,
                                                          int C, int ldi, float *__restrict__ out,
                                                          __nv_bfloat16 *__restrict__ outb,
                                                          int ldo) {
  __shared__ float tile[TT][TT + 1];
  const int r0 = blockIdx.x * TT, c0 = blockIdx.y * TT;  // (rows on x: no 65535 limit)
  const int lx = threadIdx.x % 16, ly = threadIdx.x / 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = ly + 16 * i, r = r0 + rr, c = c0 + 4 * lx;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < R) {
      const float *src = in + (size_t)r * ldi + c;
      if (c + 3 < C) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(src));
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < C) v[q] = src[q];
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) tile[rr][4 * lx + q] = v[q];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int cc = ly + 16 * i, c = c0 + cc, r = r0 + 4 * lx;
    if (c >= C) continue;
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = tile[4 * lx + q][cc];
    const size_t o = (size_t)c * ldo + r;
    if (r + 3 < R) {
      if (out) *reinterpret_cast<float4 *>(out + o) = make_float4(v[0], v[1], v[2], v[3]);
      if (outb) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(outb + o) = pk;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (r + q < R) {
          if (out) out[o + q] = v[q];
          if (outb) outb[o + q] = __float2bfloat16_rn(v[q]);
        }
    }
  }
}

// out[c][r] = in[r][c] in fp32, and outb[c][r] = bf16(in[r][c]) when outb
// is given (one read of the input for both)
__global__ void transpose_dual_kernel(const float *__restrict__ in, int R, int C, int ldi,
                                      float *__restrict__ out, __nv_bfloat16 *__restrict__ outb,
                                      int ldo) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = in[(size_t)r * ldi + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < R && c < C) {
      const float v = tile[threadIdx.x][i];
      out[(size_t)c * ldo + r] = v;
      if (outb) outb[(size_t)c * ldo + r] = __float2bfloat16_rn(v);
    }
  }
}

// out[r][c] = bf16(in[r][c]) for an R x C row-major matrix (row strides ldi, ldo)
__global__ void convert_rows_kernel(const float *__restrict__ in, int R, int C, int ldi,
                                    __nv_bfloat16 *__restrict__ out, int ldo) {
  for (int r = blockIdx.x; r < R; r += gridDim.x)
    for (int c = threadIdx.x; c < C; c += blockDim.x)
      out[(size_t)r * ldo + c] = __float2bfloat16_rn(in[(size_t)r * ldi + c]);
}

// the same, 8 columns per thread: two 16-byte loads, one 16-byte store
// (C, ldi and ldo multiples of 8, both pointers 16-byte aligned)
__global__ void convert_rows8_kernel(const float *__restrict__ in, int R, int C8, int ldi,
                                     __nv_bfloat16 *__restrict__ out, int ldo) {
  const size_t n = (size_t)R * C8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / (size_t)C8;
    const int c = (int)(i - r * (size_t)C8) * 8;
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(in + r * ldi + c));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(in + r * ldi + c + 4));
    const __nv_bfloat162 v0 = __floats2bfloat162_rn(a.x, a.y), v1 = __floats2bfloat162_rn(a.z, a.w),
                         v2 = __floats2bfloat162_rn(b.x, b.y), v3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t *>(&v0);
    o.y = *reinterpret_cast<const uint32_t *>(&v1);
    o.z = *reinterpret_cast<const uint32_t *>(&v2);
    o.w = *reinterpret_cast<const uint32_t *>(&v3);
    *reinterpret_cast<uint4 *>(out + r * ldo + c) = o;
  }
}

// deterministic column sums of an M x N row-major matrix: chunk partials,
// then the chunks summed in order
constexpr int CS_ROWS = 1024;
__global__ void colsum_partial_kernel(const float *__restrict__ A, int M, int N,
                                      float *__restrict__ part) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int m0 = blockIdx.y * CS_ROWS, m1 = min(M, m0 + CS_ROWS);
  float s = 0.f;
  for (int m = m0; m < m1; ++m) s += A[(size_t)m * N + n];
  part[(size_t)blockIdx.y * N + n] = s;
}
__global__ void colsum_final_kernel(const float *__restrict__ part, int chunks, int N,
                                    float *__restrict__ out) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float s = 0.f;
  for (int c = 0; c < chunks; ++c) s += part[(size_t)c * N + n];
  out[n] = s;
}

struct RecPlan { int U, Gp, KC, KS, BS, NUG, NBG, NB, KP, Gh; size_t smem; };
// partial sums: [KS][BS*U + 1], or with the warp reduce-scatter (KS a
// multiple of 32) one 4 x 16 tile per warp
size_t rec_part_floats(int U, int BS, int KS, int KP) {
  return KS % 32 == 0 ? (size_t)ceil_div(BS, 4) * KP * (KS / 32) * 64
                      : (size_t)KS * ((size_t)BS * U + 1);
}
size_t rec_smem(int U, int Gh, int BS, int KC, int KS, int NB, int KP) {
  return ((size_t)KP * U * Gh + (size_t)NB * BS * (KC + 4) + rec_part_floats(U, BS, KS, KP) +
          (3 + (KP > 1 ? 1 : 0)) * (size_t)BS * U) *
         sizeof(float);
}
// The grid is NBG batch groups x NUG unit groups (at most one CTA per SM: the
// launch is cooperative).  Every CTA streams its rows of dR_t from L2 each
// step, NBG * NUG * BS * G / KP floats in all, so more units per CTA (fewer
// unit groups) and a K split over a CTA pair (KP = 2: half the columns per
// CTA) mean less traffic: the batch is split as far as the register tile
// (UMAX units) and shared memory (W_hh^T columns, staged chunks of at least
// 4 * KS columns) allow.  KC: chunk width, a multiple of 4 * KS, at most 512.
// allow_pair = false: KP = 1 only.
RecPlan plan_rec(int H, int B, int nG, int nsm, bool allow_pair) {
  RecPlan best{};
  long long best_traffic = -1;
  for (int nbg = 1; nbg <= 8 && nbg <= ceil_div(B, 4); nbg *= 2) {
    for (int kp = 1; kp <= (allow_pair ? 2 : 1); ++kp) {
      RecPlan r{};
      r.NBG = nbg;
      r.KP = kp;
      r.BS = ceil_div(B, nbg);
      const int per = std::max(1, std::min(H, nsm / nbg));
      if (kp == 1) {
        r.U = ceil_div(H, per);
        r.NUG = ceil_div(H, r.U);
      } else {
        // pairs of unit groups, 2U units per pair
        const int pairs = std::max(1, std::min(ceil_div(H, 2), per / 2));
        r.U = ceil_div(H, 2 * pairs);
        r.NUG = 2 * ceil_div(H, 2 * r.U);
      }
      r.Gp = round_up(nG * H, 4);
      r.Gh = kp == 1 ? r.Gp : round_up(ceil_div(r.Gp, 2), 4);
      const int RG = ceil_div(r.BS, 4);
      if (r.U > UMAX || RG > NT || r.NUG * nbg > nsm) continue;
      // K split: only with the warp reduce-scatter (a warp = one row group
      // and unit half), and with a K block for each CTA
      if (kp > 1 && (RG * kp > 16 || r.Gh >= r.Gp)) continue;
      // K slices per row group: up to 16 row groups (per unit half), every
      // thread, the slices a multiple of 32 so that a warp holds one row
      // group and sums its slices by shuffles; more row groups: at most 32
      // slices summed through shared memory, halved while their partial
      // tiles (KS * BS * U floats) keep the plan from fitting (the 256-row,
      // 1024-unit GRU fits with 4).
      // Staging: NB buffers of KC columns, NB - 1 chunks in flight while one
      // is multiplied; the most columns in flight wins, up to all of the
      // CTA's K columns (ties: fewer buffers).  Rings deeper than two need
      // chunks of at least 128 columns.
      bool fits = false;
      const int ks0 = RG * kp <= 16 ? (NT / (RG * kp)) / 32 * 32
                                    : std::max(1, std::min(32, NT / RG));
      for (r.KS = ks0; r.KS >= 1 && !fits; r.KS /= 2) {
        int best_score = 0;
        for (int nb = 2; nb <= 4; ++nb) {
          int kc = std::min(512, round_up(r.Gh, 4 * r.KS));
          while (kc > 4 * r.KS && rec_smem(r.U, r.Gh, r.BS, kc, r.KS, nb, kp) > SMEM_CAP)
            kc -= 4 * r.KS;
          if (rec_smem(r.U, r.Gh, r.BS, kc, r.KS, nb, kp) > SMEM_CAP) continue;
          if (nb > 2 && kc < 128) continue;
          const int score = std::min((nb - 1) * kc, round_up(r.Gh, 4 * r.KS));
          if (score > best_score) {
            best_score = score;
            r.NB = nb;
            r.KC = kc;
          }
        }
        if (best_score > 0) {
          r.smem = rec_smem(r.U, r.Gh, r.BS, r.KC, r.KS, r.NB, kp);
          fits = true;
          break;
        }
      }
      if (!fits) continue;
      const long long traffic = (long long)nbg * r.NUG * r.BS * (kp == 1 ? 2 : 1);
      if (best_traffic < 0 || traffic < best_traffic) {
        best = r;
        best_traffic = traffic;
      }
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_bwd_prep(int T, int B, int H, int cell, float *zin, const float *zh,
                            const float *c0, float *cs, float *ms, cudaStream_t s, float *cr,
                            float clo, float chi) {
  const int n = B * H;
  bwd_prep_kernel<<<ceil_div(n, 64), 64, 0, s>>>(T, B, H, cell, zin, zh, c0, cs, ms, cr, clo,
                                                 chi);
  return cudaGetLastError();
}

namespace {
__global__ void add_kernel(float *__restrict__ dst, const float *__restrict__ src, size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] += src[i];
}
}  // namespace

namespace {
// out[s][b][c] = in[t][b][col0 + c] (row stride ldi), t = s, or reversed
// within the row's length: t = len_b-1-s for s < len_b, t = s past it
// V = 4: w, ldi and col0 multiples of 4 and both buffers 16-byte aligned
// (each thread moves 4 consecutive columns)
template <int V>
__global__ void gather_steps_kernel(const float *__restrict__ in, int ldi, int col0, int w, int T,
                                    int B, int reverse, const int32_t *__restrict__ lengths,
                                    float *__restrict__ out) {
  const int wv = w / V;
  const size_t n = (size_t)T * B * wv;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(e % wv) * V;
    const size_t row = e / wv;  // s * B + b
    const int sidx = (int)(row / B), b = (int)(row % B);
    // reversal within each row's own length; steps past it stay in place
    const int len = lengths ? clamp_len(lengths[b], T) : T;
    const int t = (reverse && sidx < len) ? len - 1 - sidx : sidx;
    const float *src = in + ((size_t)t * B + b) * ldi + col0 + c;
    if constexpr (V == 4)
      *reinterpret_cast<float4 *>(out + row * w + c) = *reinterpret_cast<const float4 *>(src);
    else
      out[row * w + c] = *src;
  }
}
// out[t][b][:] = in[t][b][:] (+ dhn[b][:] at t = len_b - 1) for t < len_b, 0
// past the row's end; out may equal in (V = 4 as above)
template <int V>
__global__ void mask_steps_kernel(const float *in, int w, int T, int B,
                                  const int32_t *__restrict__ lengths,
                                  const float *__restrict__ dhn, float *out) {
  const int wv = w / V;
  const size_t n = (size_t)T * B * wv;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(e % wv) * V;
    const size_t row = e / wv;
    const int t = (int)(row / B), b = (int)(row % B);
    const int len = clamp_len(lengths[b], T);
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) v[q] = 0.f;
    if (t < len) {
#pragma unroll
      for (int q = 0; q < V; ++q) v[q] = in[row * w + c + q];
      if (dhn && t == len - 1)
#pragma unroll
        for (int q = 0; q < V; ++q) v[q] += dhn[(size_t)b * w + c + q];
    }
    if constexpr (V == 4)
      *reinterpret_cast<float4 *>(out + row * w + c) = make_float4(v[0], v[1], v[2], v[3]);
    else
      out[row * w + c] = v[0];
  }
}
}  // namespace

static bool al16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

cudaError_t launch_gather_steps(const float *in, int ldi, int col0, int w, int T, int B,
                                bool reverse, const int32_t *lengths, float *out,
                                cudaStream_t s) {
  const size_t n = (size_t)T * B * w;
  if (n == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 65535u * 8);
  if (w % 4 == 0 && ldi % 4 == 0 && col0 % 4 == 0 && al16(in) && al16(out))
    gather_steps_kernel<4><<<blocks, 256, 0, s>>>(in, ldi, col0, w, T, B, reverse ? 1 : 0,
                                                  lengths, out);
  else
    gather_steps_kernel<1><<<blocks, 256, 0, s>>>(in, ldi, col0, w, T, B, reverse ? 1 : 0,
                                                  lengths, out);
  return cudaGetLastError();
}

cudaError_t launch_mask_steps(const float *in, int w, int T, int B, const int32_t *lengths,
                              const float *dhn, float *out, cudaStream_t s) {
  const size_t n = (size_t)T * B * w;
  if (n == 0) return cudaSuccess;
  if (!lengths) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 65535u * 8);
  if (w % 4 == 0 && al16(in) && al16(out) && (!dhn || al16(dhn)))
    mask_steps_kernel<4><<<blocks, 256, 0, s>>>(in, w, T, B, lengths, dhn, out);
  else
    mask_steps_kernel<1><<<blocks, 256, 0, s>>>(in, w, T, B, lengths, dhn, out);
  return cudaGetLastError();
}

cudaError_t launch_add(float *dst, const float *src, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  add_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(dst, src, n);
  return cudaGetLastError();
}

int bwd_units_per_cta(int H, int B, int nG, int nsm) { return plan_rec(H, B, nG, nsm, false).U; }

static BwdParams bwd_params(const BwdRecArgs &a, const RecPlan &rp) {
  BwdParams p{};
  p.T = a.T; p.B = a.B; p.H = a.H; p.cell = a.cell; p.U = rp.U;
  p.Gp = rp.Gp; p.KC = rp.KC; p.KS = rp.KS; p.BS = rp.BS; p.NUG = rp.NUG; p.NB = rp.NB;
  p.KP = rp.KP; p.Gh = rp.Gh; p.per = rp.NBG * rp.NUG;
  p.Whh = a.Whh; p.ldw = a.ldw;
  p.gates = a.gates; p.zh = a.zh; p.cs = a.cs; p.c0 = a.c0; p.hp = a.hp;
  p.dy = a.dy; p.dhn = a.dhn; p.dcn = a.dcn; p.lengths = a.lengths;
  p.cr = a.cr; p.clo = a.clo; p.chi = a.chi;
  p.DA = a.DA; p.DR = a.DR; p.dh0 = a.dh0; p.dc0 = a.dc0;
  p.ctr = a.ctr; p.err = a.err; p.timeout_ns = a.timeout_ns; p.drop_arrival = a.drop_arrival;
  p.trace = a.trace;
  return p;
}

cudaError_t launch_bwd_rec(const BwdRecArgs &a, int nsm, cudaStream_t s, const BwdRecArgs *a2) {
  const int nG = a.cell == CELL_LSTM ? 4 : 3, nd = a2 ? 2 : 1;
  if (a2 && (a2->T != a.T || a2->B != a.B || a2->H != a.H || a2->cell != a.cell))
    return cudaErrorInvalidValue;
  for (int pass = 0; pass < 2; ++pass) {
    // the K split over CTA pairs first; without it if that cluster grid
    // cannot be co-resident.  Two problems share the SMs half and half.
    const RecPlan rp = plan_rec(a.H, a.B, nG, nsm / nd, pass == 0);
    if (rp.U < 1) return cudaErrorInvalidConfiguration;
    if (pass == 1 && rp.KP > 1) return cudaErrorInvalidConfiguration;
    BwdParams p = bwd_params(a, rp), q = bwd_params(a2 ? *a2 : a, rp);
    const int grid = nd * p.per;
    const size_t smem = rp.smem;
    const void *fn = rp.KP > 1 ? (const void *)bwd_rec_pair_kernel : (const void *)bwd_rec_kernel;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {&p, &q};
    if (rp.KP == 1) return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(NT), args, smem, s);
    if (tc_launch_clustered(fn, grid, NT, 2, smem, args, s, &e)) return e;
  }
  return cudaErrorInvalidConfiguration;
}

// the 64 x 64 vectorised kernel when rows and buffers are aligned for it
static bool t64_ok(const float *in, int ldi, const float *out, const __nv_bfloat16 *outb,
                   int ldo) {
  auto al = [](const void *q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; };
  return ldi % 4 == 0 && ldo % 4 == 0 && al(in, 16) && (!out || al(out, 16)) &&
         (!outb || al(outb, 8));
}
static cudaError_t launch_t64(const float *in, int R, int C, int ldi, float *out,
                              __nv_bfloat16 *outb, int ldo, cudaStream_t s) {
  if (ceil_div(C, TT) > 65535) return cudaErrorInvalidValue;
  transpose64_kernel<<<dim3(ceil_div(R, TT), ceil_div(C, TT)), 256, 0, s>>>(in, R, C, ldi, out,
                                                                           outb, ldo);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const float *in, int R, int C, int ldi, float *out, int ldo,
                             cudaStream_t s) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (t64_ok(in, ldi, out, nullptr, ldo)) return launch_t64(in, R, C, ldi, out, nullptr, ldo, s);
  transpose_kernel<float><<<dim3(ceil_div(C, 32), ceil_div(R, 32)), dim3(32, 8), 0, s>>>(
      in, R, C, ldi, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const float *in, int R, int C, int ldi, __nv_bfloat16 *out,
                                  int ldo, cudaStream_t s) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (t64_ok(in, ldi, nullptr, out, ldo)) return launch_t64(in, R, C, ldi, nullptr, out, ldo, s);
  transpose_kernel<__nv_bfloat16><<<dim3(ceil_div(C, 32), ceil_div(R, 32)), dim3(32, 8), 0, s>>>(
      in, R, C, ldi, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_transpose_dual(const float *in, int R, int C, int ldi, float *out,
                                  __nv_bfloat16 *outb, int ldo, cudaStream_t s) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (t64_ok(in, ldi, out, outb, ldo)) return launch_t64(in, R, C, ldi, out, outb, ldo, s);
  transpose_dual_kernel<<<dim3(ceil_div(C, 32), ceil_div(R, 32)), dim3(32, 8), 0, s>>>(
      in, R, C, ldi, out, outb, ldo);
  return cudaGetLastError();
}

cudaError_t launch_convert_rows_bf16(const float *in, int R, int C, int ldi, __nv_bfloat16 *out,
                                     int ldo, cudaStream_t s) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (C % 8 == 0 && ldi % 8 == 0 && ldo % 8 == 0 && (reinterpret_cast<uintptr_t>(in) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const size_t n = (size_t)R * (C / 8);
    const int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)std::max(nsm, 1) * 8);
    convert_rows8_kernel<<<grid, 256, 0, s>>>(in, R, C / 8, ldi, out, ldo);
    return cudaGetLastError();
  }
  convert_rows_kernel<<<std::min(R, 65535), 256, 0, s>>>(in, R, C, ldi, out, ldo);
  return cudaGetLastError();
}

size_t colsum_scratch_floats(int M, int N) { return (size_t)ceil_div(M, CS_ROWS) * N; }

cudaError_t launch_colsum(const float *A, int M, int N, float *scratch, float *out,
                          cudaStream_t s) {
  const int chunks = ceil_div(M, CS_ROWS);
  colsum_partial_kernel<<<dim3(ceil_div(N, 256), chunks), 256, 0, s>>>(A, M, N, scratch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colsum_final_kernel<<<ceil_div(N, 256), 256, 0, s>>>(scratch, chunks, N, out);
  return cudaGetLastError();
}

}  // namespace rcu
