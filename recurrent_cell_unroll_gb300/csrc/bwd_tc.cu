// Reverse-time recurrence of the GRU backward pass on the 5th-generation
// tensor cores (bf16 handles, fixed-length batches): the training use of the
// unrolled cell behind "[Feature Request] CUDNN version of RSSM" (pytorch/rl
// issue 366, Motivation: the loop dominates training).
//
// The only sequential part of the GRU's backward pass is
//     dh_t = dy_t + z_{t+1} (.) dh_{t+1} + W_hh^T dR_{t+1},
// where dR_{t+1} holds the hidden-side gate gradients of step t+1, which in
// turn need dh_{t+1}.  One cooperative launch runs every step in reverse
// time, the forward kernel's structure with the roles of the operands swapped:
//   - B operand: W_hh^T rows of the cluster's units, one K share per CTA,
//     resident in shared memory for the whole sequence;
//   - A operand: dR_{t+1} of the batch group, bf16, streamed from the
//     L2-resident exchange buffer by TMA through a ring of 16 KB stages;
//   - D: 128 TMEM lanes (batch rows) x the cluster's units, fp32.
// A cluster of KS CTAs owns (128-row batch group, 16*KS units); each CTA
// accumulates its 1/KS of K = 3H over all the cluster's units, hands each
// peer the partial sums of the peer's 16 units through distributed shared
// memory (st.async, counted on the peer's mbarrier), and finalises 16 units.
// Its 16 epilogue warps (thread = batch row = TMEM lane, 4 units) then form
// dh_t and the gate gradients of step t,
//     dn = dh (1 - z), dz = dh (h' - n), an = dn (1 - n^2),
//     ar = an hn r (1 - r), az = dz z (1 - z)       (hn = W_hn h' + b_hn),
//     DA = [ar, az, an], DR = [ar, az, an r],        carried z dh,
// with the gates r, z, n activated a step ahead from the recomputed
// pre-activations of both sides, write the gradients for the GEMMs after
// the loop, and publish DR_t in bf16 (the precision of every MMA operand of
// the bf16 forward) with one red.release per CTA on a bounded step counter
// per batch group.
#include <cudaTypedefs.h>

#include <algorithm>

#include "tc.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int UNITS = 16;       // hidden units each CTA finalises
constexpr int BG = 128;         // batch rows per CTA (MMA M)
constexpr int BK = 64;          // K per stage (128 bytes of bf16)
constexpr int A_STAGE = BG * BK * 2;
constexpr int EPI_WARPS = 16;   // 4 per TMEM lane quarter
constexpr int UPT = UNITS / 4;  // units per epilogue thread
constexpr int NT = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int MAX_STAGES = 8;

struct BMaps {
  CUtensorMap dr;  // [2*B rows][3H cols] bf16 (row stride Kx): the dR exchange, box 64 x a_rows
  CUtensorMap wt;  // [H rows][3H cols] bf16 (row stride Kx): W_hh^T, box 64 x N
  int a_rows;      // 128, or round_up(B, 8) when one batch group holds the whole batch
};

struct BCtl {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], wbar, tfull, tfree, mdone, xfull;
  uint32_t tmem_base;
  int abort;
  int go;   // epilogue: result of the per-step accumulator wait
  int go2;  // epilogue: result of the per-step partial-sum wait
  // peer_sent[r] = steps whose partial sums cluster rank r sent to this CTA,
  // stored here by rank r itself before the final cluster barrier
  uint32_t peer_sent[4];
  // per lane quarter: the column sums of DA and DR over its 32 rows
  float bred[4][2][3][UNITS];
};

struct BGeo {
  int N, nkb, nkbm, stages;
  size_t w_bytes, x_bytes, smem;
};

// K = 3H split over KS CTAs; N = the cluster's 16*KS units
__host__ __device__ inline BGeo make_bgeo(int G, int KS) {
  BGeo g;
  g.N = UNITS * KS;
  g.nkb = ceil_div(G, BK);
  g.nkbm = ceil_div(g.nkb, KS);
  g.w_bytes = (size_t)g.nkbm * g.N * 128;
  // partial sums received from the other KS-1 CTAs: [KS-1][4 parts][128 rows] float4
  g.x_bytes = (size_t)(KS - 1) * 4 * BG * 16;
  const size_t fixed = 1024 + g.w_bytes + g.x_bytes + 2048;  // + the control block
  const int st = (int)((SMEM_LIMIT - (long long)fixed) / A_STAGE);
  g.stages = st > MAX_STAGES ? MAX_STAGES : st;
  g.smem = fixed + (size_t)(g.stages > 0 ? g.stages : 0) * A_STAGE;
  return g;
}

// a K split over ks CTAs fits: a ring of at least 3 stages and a K block for
// every CTA
bool bks_fits(int G, int ks) {
  const BGeo g = make_bgeo(G, ks);
  return g.stages >= 3 && (ks - 1) * g.nkbm < g.nkb;
}

int choose_ks(int H) {
  const int G = 3 * H;
  if (H % (UNITS * 4) == 0 && bks_fits(G, 4)) return 4;
  if (H % (UNITS * 2) == 0 && bks_fits(G, 2)) return 2;
  return 0;
}

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}
__device__ __forceinline__ void tmem_ld4_nowait(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ float4 ldg4(const float *p) {
  return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st4(float *p, float a, float b, float c, float d) {
  *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// Step trace: CTA 0's stamps of reverse step s (row s; slots as documented
// with rnn_get_trace)
__device__ __forceinline__ void bstamp(const TcBwdParams &p, int s, int slot) {
  if (p.trace && blockIdx.x == 0) p.trace[(size_t)s * 16 + slot] = globaltimer_ns();
}

template <int KS>
__device__ __forceinline__ void bwd_body(const BMaps &maps, const TcBwdParams &p) {
  static_assert(KS == 2 || KS == 4, "K is split over 2 or 4 CTAs");
  if (tc::cluster_nctarank() != (uint32_t)KS) {
    // the K split needs its peers: never address a peer that is not there
    if (threadIdx.x == 0) atomicCAS(p.err, DEV_OK, DEV_CONFIG);
    return;
  }
  constexpr int N = UNITS * KS;
  constexpr uint32_t TCOLS = N <= 32 ? 32 : (N <= 64 ? 64 : 128);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int H = p.H, G = 3 * H, B = p.B, T = p.T;
  const BGeo geo = make_bgeo(G, KS);
  const int STG = geo.stages;
  uint8_t *sW = smem;                  // resident B operand: nkbm blocks of N x 128 B
  uint8_t *sA = smem + geo.w_bytes;    // ring of STG stages of 128 x 128 B
  float4 *xbuf = reinterpret_cast<float4 *>(sA + (size_t)STG * A_STAGE);
  BCtl *ctl = reinterpret_cast<BCtl *>(reinterpret_cast<uint8_t *>(xbuf) + geo.x_bytes);

  const int NU = H / UNITS;  // CTAs per batch group
  const int bg = blockIdx.x / NU, cu = blockIdx.x % NU;
  const int kr = cu % KS;                      // this CTA's K share (= rank in its cluster)
  const int ugc = cu / KS;                     // the cluster's unit group (N units)
  const int u0 = ugc * N + kr * UNITS, row0 = bg * BG;
  const int kb0 = kr * geo.nkbm;
  const int nk = min(geo.nkb, kb0 + geo.nkbm) - kb0;  // K blocks of this CTA (>= 1)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int *abort = &ctl->abort;
  const uint64_t tmo = p.timeout_ns;
  // one step counter per batch group, on its own 128-byte line; a CTA arrives
  // after it has consumed its peers' partial sums of the step, and a peer
  // sends for the next step only after the counter has moved on: the partial-
  // sum buffer is reused step after step, at most one step in flight
  unsigned *ctr = p.ctr + (size_t)bg * 32 + 16;
  const unsigned n_wait = (unsigned)NU;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    tc::mbar_init(&ctl->wbar, 1);
    tc::mbar_init(&ctl->tfull, 1);
    tc::mbar_init(&ctl->tfree, EPI_WARPS);
    tc::mbar_init(&ctl->mdone, 1);
    tc::mbar_init(&ctl->xfull, 1);
    ctl->abort = 0;
    for (int i = 0; i < 4; ++i) ctl->peer_sent[i] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, TCOLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // the peers' barriers exist before any partial-sum store
  tc::tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  int x_left = 0;       // thread 64: phases consumed (negated - 1 if one more is armed)
  uint32_t x_sent = 0;  // thread 64: steps whose partial sums this CTA has sent

  // Step s = 0 .. T handles reverse step t = T - 1 - s: its MMA (s >= 1)
  // forms W_hh^T dR_{t+1}, its epilogue the gradients of step t (t >= 0) or
  // dh0 (t = -1).
  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&maps.dr);
      tc::prefetch_tmap(&maps.wt);
      // resident W_hh^T: rows [ugc*N, ugc*N + N), K blocks [kb0, kb0 + nk)
      tc::mbar_arrive_expect_tx(&ctl->wbar, (uint32_t)(nk * N * 128));
      for (int i = 0; i < nk; ++i)
        tc::tma_load_2d(sW + (size_t)i * N * 128, &maps.wt, &ctl->wbar, (kb0 + i) * BK, ugc * N);
      int stage = 0;
      uint32_t phase = 0;
      int pend_stage[MAX_STAGES], npend = 0;
      uint32_t pend_phase[MAX_STAGES];
      for (int s = 1; s <= T; ++s) {
        // every CTA of the batch group has published dR_{t+1} (its step s-1)
        const unsigned target = n_wait * (unsigned)s;
        if (ld_acquire_gpu(ctr) < target) {
          const uint64_t deadline = globaltimer_ns() + tmo;
          uint32_t spins = 0;
          bool ok = true;
          while (ld_acquire_gpu(ctr) < target) {
            if ((++spins & 63u) == 0) {
              if (*abort || ld_volatile_int(p.err) != DEV_OK) { ok = false; break; }
              if (globaltimer_ns() > deadline) {
                atomicCAS(p.err, DEV_OK, DEV_TIMEOUT);
                ok = false;
                break;
              }
            }
          }
          if (!ok) { *abort = 1; break; }
        }
        bstamp(p, s, 0);
        fence_proxy_async_global();
        const int t1 = T - s;  // dR_{t+1} lives in buffer t1 & 1
        const int arow = (t1 & 1) * B + row0;
        for (int i = 0; i < nk; ++i) {
          if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, p.err, abort, tmo)) goto producer_out;
          tc::mbar_arrive_expect_tx(&ctl->full[stage], (uint32_t)(maps.a_rows * BK * 2));
          tc::tma_load_2d(sA + (size_t)stage * A_STAGE, &maps.dr, &ctl->full[stage],
                          (kb0 + i) * BK, arow);
          pend_stage[npend % MAX_STAGES] = stage;
          pend_phase[npend % MAX_STAGES] = phase;
          ++npend;
          if (++stage == STG) { stage = 0; phase ^= 1; }
        }
      }
    producer_out:
      if (*abort) {
        // the copies already issued land before the CTA leaves (bounded waits
        // that ignore the abort flag)
        volatile int never = 0;
        tc::mbar_wait(&ctl->wbar, 0, nullptr, &never, 100000000ull);
        const int n = npend < STG ? npend : STG;
        for (int i = 0; i < n; ++i) {
          const int k = (npend - 1 - i) % MAX_STAGES;
          tc::mbar_wait(&ctl->full[pend_stage[k]], pend_phase[k], nullptr, &never, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BG, N);
      const uint64_t adesc0 = tc::smem_desc_sw128(tc::smem_u32(sA));
      const uint64_t bdesc0 = tc::smem_desc_sw128(tc::smem_u32(sW));
      const uint32_t bstep = (uint32_t)(N * 128) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = tc::mbar_wait(&ctl->wbar, 0, p.err, abort, tmo);
      for (int s = 1; ok && s <= T; ++s) {
        // the epilogue has read the previous step's accumulator
        if (!tc::mbar_wait(&ctl->tfree, (uint32_t)((s - 1) & 1) ^ 1u, p.err, abort, tmo)) break;
        tc::tc_fence_after();
        uint64_t bd = bdesc0;
        for (int i = 0; i < nk; ++i, bd += bstep) {
          if (!tc::mbar_wait(&ctl->full[stage], phase, p.err, abort, tmo)) { ok = false; break; }
          if (i == 0) bstamp(p, s, 1);
          const uint64_t ad = adesc0 + (uint64_t)(stage * (A_STAGE >> 4));
          tc::mma4_bf16_commit(tbase, ad, bd, idesc, i != 0, &ctl->empty[stage]);
          if (++stage == STG) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        bstamp(p, s, 2);
        tc::mma_commit(&ctl->tfull);
      }
      // drain: every MMA issued above completes before TMEM is released
      tc::mma_commit(&ctl->mdone);
      volatile int never = 0;
      tc::mbar_wait(&ctl->mdone, 0, nullptr, &never, 100000000ull);
    }
  } else {
    // ---------------- epilogue: 16 warps; warp -> (TMEM lane quarter q, 4 units)
    const int q = warp % 4;
    const int part = (warp - 2) / 4;  // units [part*4, part*4+4) of the CTA's 16
    const int r = q * 32 + lane;      // batch row in the group = TMEM lane
    const int b = row0 + r;
    const bool row_ok = b < B;
    const int ub = u0 + part * UPT;   // first unit of this thread
    const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
    const uint32_t own_col = (uint32_t)(kr * UNITS + part * UPT);
    // Peers i = 0..KS-2 are the other ranks in order.  The partial sums for
    // peer pr's units go into pr's buffer in the slot of this sender (its
    // rank among pr's peers): slot*(4*128) + part*128 + r, one float4.
    constexpr int NP = KS - 1;
    constexpr int SLOT = 4 * BG;
    uint32_t peer_x[NP], peer_bar[NP], peer_col[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int pr = i < kr ? i : i + 1;
      const int slot = kr < pr ? kr : kr - 1;
      peer_x[i] = tc::mapa_shared(tc::smem_u32(xbuf + (size_t)slot * SLOT), (uint32_t)pr);
      peer_bar[i] = tc::mapa_shared(tc::smem_u32(&ctl->xfull), (uint32_t)pr);
      peer_col[i] = (uint32_t)(pr * UNITS + part * UPT);
    }
    int x_posted = 0, x_done = 0;  // thread 64: phases armed / completed
    float dhz[UPT], act[6][UPT];   // carried z dh; the step's saved activations
    float sa[3][UPT], sr[3][UPT];  // this row's sums of DA and DR over the steps
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
      for (int j = 0; j < UPT; ++j) sa[g][j] = sr[g][j] = 0.f;
#pragma unroll
    for (int j = 0; j < UPT; ++j) dhz[j] = (row_ok && p.dhn) ? p.dhn[(size_t)b * H + ub + j] : 0.f;
    // the activations of step t for this row and units: r, z, n, hn, h', dy
    // (a step ahead, off the critical path; the gates are activated here
    // from both sides' pre-activations with the precise fp32 functions)
    auto load_act = [&](int t) {
      if (!row_ok || t < 0) return;
      const size_t row = (size_t)t * B + b;
      if (!RCU_DCHECK(row < (size_t)p.ldz && ub + UPT <= H, p.err)) return;
      // lanes are consecutive batch rows: every load of a warp reads 128
      // contiguous bytes
      const size_t ld = (size_t)p.ldz;
      const float *a = p.zin + (size_t)ub * ld + row, *hz = p.zh + (size_t)ub * ld + row;
      const float *hq = p.hp + (size_t)ub * ld + row, *dq = p.dy + (size_t)ub * ld + row;
      float f[8][UPT];
#pragma unroll
      for (int j = 0; j < UPT; ++j) {
        f[0][j] = __ldg(a + (size_t)j * ld);
        f[1][j] = __ldg(a + ((size_t)H + j) * ld);
        f[2][j] = __ldg(a + ((size_t)2 * H + j) * ld);
        f[3][j] = __ldg(hz + (size_t)j * ld);
        f[4][j] = __ldg(hz + ((size_t)H + j) * ld);
        f[5][j] = __ldg(hz + ((size_t)2 * H + j) * ld);
        f[6][j] = __ldg(hq + (size_t)j * ld);
        f[7][j] = __ldg(dq + (size_t)j * ld);
      }
#pragma unroll
      for (int j = 0; j < UPT; ++j) {
        const float rg = sigmoid_f(f[0][j] + f[3][j]);
        act[0][j] = rg;
        act[1][j] = sigmoid_f(f[1][j] + f[4][j]);
        act[2][j] = tanh_f(f[2][j] + rg * f[5][j]);
        act[3][j] = f[5][j];
        act[4][j] = f[6][j];
        act[5][j] = f[7][j];
      }
    };
    load_act(T - 1);
    for (int s = 0; s <= T; ++s) {
      const int t = T - 1 - s;
      float acc[UPT] = {0.f, 0.f, 0.f, 0.f};
      if (s >= 1) {
        // W_hh^T dR_{t+1}: this CTA's K share from TMEM, the peers' shares
        // of this CTA's units through shared memory
        if (threadIdx.x == 64) {
          ctl->go = tc::mbar_wait(&ctl->tfull, (uint32_t)(s - 1) & 1u, p.err, abort, tmo);
          bstamp(p, s, 3);
        }
        epi_bar();
        if (!ctl->go) break;
        tc::tc_fence_after();
        uint32_t ra[4], rp[NP][4];
        tmem_ld4_nowait(tl + own_col, ra);
#pragma unroll
        for (int i = 0; i < NP; ++i) tmem_ld4_nowait(tl + peer_col[i], rp[i]);
        tmem_wait_ld();
        tc::tc_fence_before();
        if (lane == 0) tc::mbar_arrive(&ctl->tfree);
#pragma unroll
        for (int i = 0; i < NP; ++i)
          tc::st_async_v4(peer_x[i] + (uint32_t)((part * BG + r) * 16), __uint_as_float(rp[i][0]),
                          __uint_as_float(rp[i][1]), __uint_as_float(rp[i][2]),
                          __uint_as_float(rp[i][3]), peer_bar[i]);
        if (threadIdx.x == 64) {
          bstamp(p, s, 4);
          x_sent = (uint32_t)s;
          tc::mbar_arrive_expect_tx(&ctl->xfull, (uint32_t)geo.x_bytes);
          x_posted = s;
          ctl->go2 = tc::mbar_wait_cluster(&ctl->xfull, (uint32_t)(s - 1) & 1u, p.err, abort, tmo);
          if (ctl->go2) x_done = s;
          bstamp(p, s, 5);
        }
        epi_bar();
        if (!ctl->go2) break;
#pragma unroll
        for (int j = 0; j < UPT; ++j) acc[j] = __uint_as_float(ra[j]);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const float4 v = xbuf[(size_t)i * SLOT + part * BG + r];
          acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
        }
      }
      if (t < 0) {
        // dh_{-1}: the gradient reaching h0
        if (row_ok && p.dh0 && RCU_DCHECK(ub + UPT <= H, p.err))
          st4(p.dh0 + (size_t)b * H + ub, dhz[0] + acc[0], dhz[1] + acc[1], dhz[2] + acc[2],
              dhz[3] + acc[3]);
        break;
      }
      // (every epilogue thread reaches the same barriers: the warps of a
      // ragged batch tail hold rows on both sides of B)
      const size_t row = (size_t)t * B + b;
      float da[3][UPT], dr[3][UPT];
      if (row_ok && RCU_DCHECK(t < T && (size_t)(2 * H + ub + UPT) <= (size_t)p.Kx, p.err)) {
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
          const float rg = act[0][j], z = act[1][j], n = act[2][j], hn = act[3][j],
                      hprev = act[4][j];
          const float dh = act[5][j] + dhz[j] + acc[j];
          const float dn = dh * (1.f - z);
          const float dz = dh * (hprev - n);
          const float an = dn * (1.f - n * n);
          const float ar = an * hn * rg * (1.f - rg);
          const float az = dz * z * (1.f - z);
          da[0][j] = ar; da[1][j] = az; da[2][j] = an;
          dr[0][j] = ar; dr[1][j] = az; dr[2][j] = an * rg;
          dhz[j] = dh * z;
        }
#pragma unroll
        for (int g = 0; g < 3; ++g)
#pragma unroll
          for (int j = 0; j < UPT; ++j) {
            sa[g][j] += da[g][j];
            sr[g][j] += dr[g][j];
          }
        // the next step's MMA operand first: it is on the critical path
        __nv_bfloat16 *xo = p.xdr + ((size_t)(t & 1) * B + b) * p.Kx + ub;
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(dr[g][0], dr[g][1]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(dr[g][2], dr[g][3]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t *>(&lo);
          pk.y = *reinterpret_cast<uint32_t *>(&hi);
          *reinterpret_cast<uint2 *>(xo + (size_t)g * H) = pk;
        }
      }
      fence_proxy_async_global();
      epi_bar();
      if (threadIdx.x == 64) {
        red_release_gpu_add(ctr, (p.drop_arrival && blockIdx.x == 0 && s == 0) ? 0u : 1u);
        bstamp(p, s, 6);
      }
      if (row_ok && RCU_DCHECK(row < (size_t)T * B && (!p.dat || row < (size_t)p.ldt), p.err)) {
        // off the critical path: the gate gradients for the GEMMs after the loop
        if (p.DA) {
#pragma unroll
          for (int g = 0; g < 3; ++g) {
            st4(p.DA + row * G + (size_t)g * H + ub, da[g][0], da[g][1], da[g][2], da[g][3]);
            st4(p.DR + row * G + (size_t)g * H + ub, dr[g][0], dr[g][1], dr[g][2], dr[g][3]);
          }
        }
        if (p.dat) {
          // transposed: a warp's 32 rows are 32 consecutive elements
#pragma unroll
          for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int j = 0; j < UPT; ++j) {
              const size_t c = (size_t)(g * H + ub + j) * p.ldt + row;
              p.dat[c] = __float2bfloat16_rn(da[g][j]);
              p.drt[c] = __float2bfloat16_rn(dr[g][j]);
            }
        }
        if (p.dab) {
#pragma unroll
          for (int g = 0; g < 3; ++g) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(da[g][0], da[g][1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(da[g][2], da[g][3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t *>(&lo);
            pk.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(p.dab + row * p.ldab + (size_t)g * H + ub) = pk;
          }
        }
      }
      if (threadIdx.x == 64) bstamp(p, s, 7);
      load_act(t - 1);
      if (threadIdx.x == 64) bstamp(p, s, 8);
    }
    if (threadIdx.x == 64) x_left = x_done < x_posted ? -x_done - 1 : x_done;
    if (p.bsum) {
      // the batch group's column sums of DA and DR over this CTA's units:
      // across the warp's 32 rows by shuffles, then across the 4 lane
      // quarters in a fixed order (deterministic)
#pragma unroll
      for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int j = 0; j < UPT; ++j)
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            sa[g][j] += __shfl_xor_sync(0xffffffffu, sa[g][j], off);
            sr[g][j] += __shfl_xor_sync(0xffffffffu, sr[g][j], off);
          }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < 3; ++g)
#pragma unroll
          for (int j = 0; j < UPT; ++j) {
            ctl->bred[q][0][g][part * UPT + j] = sa[g][j];
            ctl->bred[q][1][g][part * UPT + j] = sr[g][j];
          }
      }
      epi_bar();
      const int e = threadIdx.x - 64;  // 2 x 3 x 16 sums
      if (e < 2 * 3 * UNITS) {
        const int w = e / (3 * UNITS), g = (e / UNITS) % 3, u = e % UNITS;
        const float v = ctl->bred[0][w][g][u] + ctl->bred[1][w][g][u] + ctl->bred[2][w][g][u] +
                        ctl->bred[3][w][g][u];
        if (RCU_DCHECK(bg < ceil_div(B, BG) && u0 + u < H, p.err))
          p.bsum[((size_t)w * ceil_div(B, BG) + bg) * G + (size_t)g * H + u0 + u] = v;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 64) {
    // Tell every peer how many steps of partial sums it will have received
    // from this CTA, while the peer is certain to be resident (it cannot pass
    // the cluster barrier below before this CTA arrives): nothing after that
    // barrier touches another CTA's shared memory.
    for (int pr = 0; pr < KS; ++pr) {
      if (pr == kr) continue;
      const uint32_t dst = tc::mapa_shared(tc::smem_u32(&ctl->peer_sent[kr]), (uint32_t)pr);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(x_sent) : "memory");
    }
  }
  tc::cluster_sync();
  if (threadIdx.x == 64) {
    // after an early exit a peer may have sent one step more than this CTA
    // consumed; those stores land here, so wait for them (bounded)
    const int done = x_left < 0 ? -x_left - 1 : x_left;
    uint32_t peer_sent = 0;
    for (int pr = 0; pr < KS; ++pr) {
      if (pr == kr) continue;
      const uint32_t v = *reinterpret_cast<volatile uint32_t *>(&ctl->peer_sent[pr]);
      peer_sent = v > peer_sent ? v : peer_sent;
    }
    if ((int)peer_sent > done) {
      if (x_left >= 0) tc::mbar_arrive_expect_tx(&ctl->xfull, (uint32_t)geo.x_bytes);
      volatile int never = 0;
      tc::mbar_wait(&ctl->xfull, (uint32_t)done & 1u, nullptr, &never, 100000000ull);
    }
  }
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, TCOLS);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
    bwd_tc_pair_kernel(const __grid_constant__ BMaps maps, const TcBwdParams p) {
  bwd_body<2>(maps, p);
}
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(NT, 1)
    bwd_tc_quad_kernel(const __grid_constant__ BMaps maps, const TcBwdParams p) {
  bwd_body<4>(maps, p);
}

}  // namespace

bool tc_bwd_supported(int H, int B, int nsm) {
  if (H < UNITS || B < 1) return false;
  if (choose_ks(H) == 0) return false;
  return (long long)ceil_div(B, BG) * (H / UNITS) <= nsm;
}

int tc_bwd_counters(int B) { return ceil_div(B, BG) * 32 + 32; }

cudaError_t launch_tc_bwd(const TcBwdParams &pin, int nsm, cudaStream_t s) {
  (void)nsm;
  TcBwdParams p = pin;
  const int H = p.H, G = 3 * H, NBG = ceil_div(p.B, BG);
  int ks = choose_ks(H);
  if (ks == 0) return cudaErrorInvalidValue;
  auto aligned16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  if ((p.Kx % 8) || p.Kx < G || (p.ldz % 4) || p.ldz < p.T * p.B || !aligned16(p.zin) || !aligned16(p.zh) || !aligned16(p.hp) ||
      !aligned16(p.dy) || (p.DA && (!aligned16(p.DA) || !p.DR || !aligned16(p.DR))) ||
      (p.dh0 && !aligned16(p.dh0)) || !aligned16(p.xdr) || !aligned16(p.wt) ||
      (p.dat && (!p.drt || p.ldt < p.T * p.B)) || (p.dab && (!aligned16(p.dab) || (p.ldab % 8) ||
                                                             p.ldab < G)))
    return cudaErrorInvalidValue;
  BMaps maps;
  maps.a_rows = NBG == 1 ? round_up(p.B, 8) : BG;
  if (!tc_map_2d(&maps.dr, p.xdr, 2LL * p.B, G, p.Kx, maps.a_rows)) return cudaErrorInvalidValue;
  const int grid = NBG * (H / UNITS);
  for (;;) {
    const BGeo geo = make_bgeo(G, ks);
    if (!tc_map_2d(&maps.wt, p.wt, H, G, p.Kx, geo.N)) return cudaErrorInvalidValue;
    const void *fn = ks == 4 ? (const void *)bwd_tc_quad_kernel : (const void *)bwd_tc_pair_kernel;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)geo.smem);
    if (e != cudaSuccess) return e;
    void *args[] = {&maps, &p};
    if (tc_launch_clustered(fn, grid, NT, ks, geo.smem, args, s, &e)) return e;
    // that cluster grid cannot be co-resident: a smaller split
    if (ks == 4 && H % (UNITS * 2) == 0 && bks_fits(G, 2)) {
      ks = 2;
      continue;
    }
    return cudaErrorInvalidConfiguration;
  }
}

}  // namespace rcu
