// Persistent recurrent kernel on the 5th-generation tensor cores (bf16 path).
//
// One cooperative launch runs every timestep of one layer.  CTA (d, bg, ug)
// owns direction d, batch rows [bg*128, bg*128+128) (sorted order) and
// hidden units [ug*16, ug*16+16).  Per step it computes
//     R[b, n] = sum_k h_{t-1}[b, k] * W_hh[row(n), k]
// with tcgen05.mma (M = 128 batch rows, N = 16 units x gates, K = Hout),
//   - B operand: the CTA's W_hh rows (all gates of its 16 units), loaded once
//     by TMA and resident in shared memory for the whole sequence;
//   - A operand: h_{t-1} of the batch group, bf16, streamed from the L2-
//     resident exchange buffer by TMA through a ring of 16 KB stages;
//   - D: 128 TMEM lanes x N fp32 columns.
// Four epilogue warps (thread = batch row = TMEM lane) keep h and c of their
// row's 16 units in registers for the whole sequence, add the precomputed
// input projection G, apply the gates (LSTM: sigmoid/tanh, c update; GRU:
// r, z, n with the reset gate on the hidden-side n pre-activation incl. its
// bias), and write h_t (bf16 exchange buffer, output).  A bounded
// release/acquire counter over the CTAs of (d, bg) crosses each step.
// This is the "recurrent hidden-hidden dense" of "[TOPI] TE implementation of
// LSTM using scan" (apache/tvm PR 11531) with the gate and activation math
// inlined, as that page's benchmark did.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int UNITS = 16;       // hidden units each CTA finalises
constexpr int BG = 128;         // batch rows per CTA (MMA M)
constexpr int BK = 64;          // K per stage (128 bytes of bf16)
constexpr int EPI_WARPS = 16;   // 4 per TMEM lane quarter
constexpr int UPT = UNITS / 4;  // units per epilogue thread
constexpr int NT = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int MAX_STAGES = 8;

struct Maps {
  CUtensorMap hx;    // [D*2*B rows][K cols], ld Kp, bf16, box 64 x a_rows
  CUtensorMap w[2];  // per direction [NU16*nG*16 rows][K cols], ld Kp, bf16, box 64 x N
  // Tiled input and output streams (fixed-length batches: a step's rows are
  // contiguous): G as [T][B][ldG] fp32 and the layer outputs as [T][B][ldo]
  // (fp32 y and / or the bf16 packed rows for the next layer), boxes of 16
  // bytes of columns (4 fp32 or 8 bf16) x a_rows rows x 1 step, so that in
  // shared memory each box is a strip of 16-byte rows: a warp's 32 rows of
  // one strip are 512 contiguous bytes (no bank conflicts).  Rows past B fall
  // outside the box's step and are clipped (stores) or read as zero (loads).
  CUtensorMap g, out, outm;
  // 0: no tiles; else G moves through `g`, and bit 0 / bit 1 say that fp32 y
  // (`out`) / the bf16 rows (`outm`) move through their maps
  int tiles;
  // h rows loaded per stage: 128, or round_up(B, 8) when one batch group
  // holds the whole batch (the stage's other rows are never read back: a
  // row of D depends only on the same row of A, and the epilogue skips rows
  // past B)
  int a_rows;
};

struct Ctl {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], wbar, tfull, tfree, mdone, xfull, gbar;
  uint32_t tmem_base;
  int abort;
  int go;   // epilogue: result of the per-step accumulator wait, shared by all its threads
  int go2;  // epilogue: result of the per-step partial-sum wait (K split)
  int g_issued;  // tiled G: loads issued into the G tile (thread 64's count)
  // K split: peer_sent[r] = steps whose partial sums CTA rank r of the
  // cluster sent to this CTA, stored here by rank r itself before the final
  // cluster barrier
  uint32_t peer_sent[4];
};

// KS = CTAs splitting K (a cluster of KS CTAs computes the gate
// pre-activations of 16*KS units for 128 rows; each CTA accumulates its 1/KS
// of K over all 16*KS units, then each finalises 16 of them after the
// partial sums for its units have been exchanged through distributed shared
// memory).
struct Geo {
  int N, nkb, nkbm, stages;
  size_t w_bytes, x_bytes, g_bytes, o_bytes, smem;
};

// tiles (the Maps::tiles mask): reserve the G tile [nG][ar rows][16 units]
// fp32 and the output tiles [ar rows][16 units] of the tiled streams (fp32 y,
// bf16 rows).  ar = the h rows a stage holds (Maps::a_rows): 128, or fewer
// when one batch group holds the whole batch, so that a small batch keeps
// more K blocks in flight.  The MMA still reads 128 rows from each stage
// (M = 128); rows past ar fall on the next stage or on the slack reserved
// after the ring, and only feed accumulator rows the epilogue never uses.
__host__ __device__ inline Geo make_geo(int nG, int K, int KS, int tiles = 0, int ar = BG) {
  Geo g;
  g.N = nG * UNITS * KS;
  g.nkb = ceil_div(K, BK);
  g.nkbm = ceil_div(g.nkb, KS);
  g.w_bytes = (size_t)g.nkbm * g.N * 128;
  // partial sums received from the other KS-1 CTAs: [KS-1][nG][4][128] float4
  g.x_bytes = (size_t)(KS - 1) * nG * 4 * ar * 16;  // (the live rows only)
  g.g_bytes = tiles ? (size_t)nG * ar * UNITS * 4 : 0;
  g.o_bytes = (size_t)((tiles & 1) ? ar * UNITS * 4 : 0) + ((tiles & 2) ? ar * UNITS * 2 : 0);
  const size_t stage = (size_t)ar * BK * 2, slack = (size_t)(BG - ar) * BK * 2;
  const size_t fixed = 1024 + g.w_bytes + g.x_bytes + g.g_bytes + g.o_bytes + 256 + slack;
  int st = (int)((SMEM_LIMIT - (long long)fixed) / (long long)stage);
  g.stages = st > MAX_STAGES ? MAX_STAGES : st;
  g.smem = fixed + (size_t)(g.stages > 0 ? g.stages : 0) * stage;
  return g;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 3D TMA load / store of a box at (x, y, z); the store is committed as a
// bulk group, its shared-memory reads waited for with bulk_wait_read
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(tc::smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(tc::smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *smem_src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(tc::smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Step trace: CTA 0's stamps for every step, and (RCU_ATTR_TRACE = 2) every
// CTA's stamps for a window of steps.  Called by one thread per stamp.
__device__ __forceinline__ void stamp(const RecParams &p, int step, int slot,
                                      unsigned long long v) {
  if (p.trace && blockIdx.x == 0) p.trace[step * 16 + slot] = v;
  if (p.trace_all && (unsigned)(step - TRACE_ALL_S0) < (unsigned)TRACE_ALL_N &&
      blockIdx.x < (unsigned)TRACE_ALL_CTAS)
    p.trace_all[((size_t)(step - TRACE_ALL_S0) * TRACE_ALL_CTAS + blockIdx.x) * 16 + slot] = v;
}
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

// 32 lanes x 4 consecutive 32-bit TMEM columns (no wait)
__device__ __forceinline__ void tmem_ld4_nowait(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// bf16 path activations on the MUFU tanh unit (PTX tanh.approx.f32); the
// logistic function through the identity sigmoid(x) = 1/2 + tanh(x/2)/2
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }

// FULL: every stage and tile strip holds 128 rows (a_rows == 128, known at
// compile time); otherwise maps.a_rows rows (one batch group of fewer rows)
template <int NG, int KS, bool FULL>
__device__ __forceinline__ void rec_tc_body(const Maps &maps, const RecParams &p) {
  static_assert(KS == 1 || KS == 2 || KS == 4, "K is split over 1, 2 or 4 CTAs");
  if (KS > 1 && tc::cluster_nctarank() != (uint32_t)KS) {
    // the K split needs its partner CTA: never address a peer that is not there
    if (threadIdx.x == 0) atomicCAS(p.err, DEV_OK, DEV_CONFIG);
    return;
  }
  constexpr int NTOT = NG * UNITS * KS;
  constexpr uint32_t TCOLS = NTOT <= 64 ? 64 : (NTOT <= 128 ? 128 : 256);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int AR = FULL ? BG : maps.a_rows;    // h rows per stage, rows per tile strip
  const size_t ASTG = (size_t)AR * BK * 2;  // bytes per h stage
  const Geo geo = make_geo(NG, p.Hout, KS, maps.tiles, AR);
  const int N = geo.N, STG = geo.stages;
  uint8_t *sW = smem;                       // resident B operand, nkbm blocks of N x 128 B
  uint8_t *sA = smem + geo.w_bytes;         // ring of STG stages of 128 x 128 B
  float4 *xbuf = reinterpret_cast<float4 *>(sA + (size_t)STG * ASTG);
  float *gtile = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xbuf) + geo.x_bytes);
  uint8_t *otile = reinterpret_cast<uint8_t *>(gtile) + geo.g_bytes;  // fp32 y strips, then
  uint8_t *otile_m = otile + ((maps.tiles & 1) ? AR * UNITS * 4 : 0);   // the bf16 strips
  Ctl *ctl = reinterpret_cast<Ctl *>(otile + geo.o_bytes);

  const int NU = p.NU, NBG = ceil_div(p.B, BG);  // NU = CTAs per (direction, batch group)
  const int d = blockIdx.x / (NBG * NU);
  const int rem = blockIdx.x % (NBG * NU);
  const int bg = rem / NU, cu = rem % NU;
  const int kr = KS > 1 ? cu % KS : 0;          // this CTA's K share (= rank in its cluster)
  const int ugc = cu / KS;                      // unit group of the cluster (16*KS units)
  const int u0 = ugc * UNITS * KS + kr * UNITS, row0 = bg * BG;
  const int kb0 = kr * geo.nkbm;
  const int nk = min(geo.nkb, kb0 + geo.nkbm) - kb0;  // K blocks of this CTA (>= 1)
  const int B = p.B, H = p.H, Kp = p.Kp;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int *abort = &ctl->abort;
  const uint64_t tmo = p.timeout_ns;
  // One step-barrier counter per (d, bg), over all its CTAs.  Every CTA
  // arrives only after it has consumed its peers' partial sums for the step,
  // and a peer starts (and sends for) the next step only after the barrier:
  // that ordering is what lets the partial-sum buffer be reused step after
  // step and bounds the sends in flight to one step.  (Waiting only for the
  // producers of a CTA's own K share would break it.)
  // (each counter on its own 128-byte line, away from the error word)
  unsigned *ctr = p.ctr + (size_t)(d * NBG + bg) * 32 + 16;
  const unsigned n_wait = (unsigned)NU;
  // steps this batch group runs: the longest row of the group (rows sorted by length)
  const int Tg = row0 < B ? p.meta.lens_sorted[row0] : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    tc::mbar_init(&ctl->wbar, 1);
    tc::mbar_init(&ctl->tfull, 1);
    tc::mbar_init(&ctl->tfree, EPI_WARPS);
    tc::mbar_init(&ctl->mdone, 1);
    // partial sums from the peer: this CTA's own arrival with the expected
    // byte count, completed by the peer's asynchronous stores
    tc::mbar_init(&ctl->xfull, 1);
    tc::mbar_init(&ctl->gbar, 1);
    ctl->g_issued = 0;
    ctl->abort = 0;
    for (int i = 0; i < 4; ++i) ctl->peer_sent[i] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, TCOLS);
  tc::tc_fence_before();
  __syncthreads();
  // the partner's barriers exist before any partial-sum store
  if (KS > 1) tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  int x_left = 0;  // K split, thread 64: phases consumed (negated - 1 if one more is armed)
  uint32_t x_sent = 0;  // K split, thread 64: steps whose partial sums this CTA has sent

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&maps.hx);
      tc::prefetch_tmap(&maps.w[d]);
      // resident weights: rows [ugc*N, ugc*N + N) of this direction's packed
      // W_hh (rows past the packed tensor read as zero), K blocks [kb0, kb0+nk)
      tc::mbar_arrive_expect_tx(&ctl->wbar, (uint32_t)(nk * N * 128));
      for (int i = 0; i < nk; ++i)
        tc::tma_load_2d(sW + (size_t)i * N * 128, &maps.w[d], &ctl->wbar, (kb0 + i) * BK, ugc * N);
      int stage = 0;
      uint32_t phase = 0;
      int pend_stage[MAX_STAGES], npend = 0;
      uint32_t pend_phase[MAX_STAGES];
      for (int step = 0; step < Tg; ++step) {
        // wait until every CTA of (d, bg) has published h_{step-1}
        const unsigned target = n_wait * (unsigned)(step + 1);
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
        fence_proxy_async_global();
        if (p.trace) stamp(p, step, 0, globaltimer_ns());
        const int arow = (d * 2 + (step & 1)) * B + row0;
        for (int i = 0; i < nk; ++i) {
          const int kb = kb0 + i;
          if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, p.err, abort, tmo)) goto producer_out;
          tc::mbar_arrive_expect_tx(&ctl->full[stage], (uint32_t)(maps.a_rows * BK * 2));
          tc::tma_load_2d(sA + (size_t)stage * ASTG, &maps.hx, &ctl->full[stage], kb * BK,
                          arow);
          pend_stage[npend % MAX_STAGES] = stage;
          pend_phase[npend % MAX_STAGES] = phase;
          ++npend;
          if (++stage == STG) { stage = 0; phase ^= 1; }
        }
      }
    producer_out:
      if (*abort) {
        // let the copies already issued land before the CTA leaves (bounded
        // waits that ignore the abort flag)
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
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BG, NTOT);
      // The issuing thread is on the critical path: descriptors are built once
      // and advanced by adding (byte offset >> 4) to the start-address field
      // (all shared-memory offsets here stay below 256 KB, so the 14-bit
      // field cannot carry).
      const uint64_t adesc0 = tc::smem_desc_sw128(tc::smem_u32(sA));
      const uint64_t bdesc0 = tc::smem_desc_sw128(tc::smem_u32(sW));
      const uint32_t bstep = (uint32_t)(N * 128) >> 4;
      const bool tr = p.trace != nullptr;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = tc::mbar_wait(&ctl->wbar, 0, p.err, abort, tmo);
      for (int step = 0; ok && step < Tg; ++step) {
        if (!tc::mbar_wait(&ctl->tfree, (step & 1) ^ 1, p.err, abort, tmo)) break;
        tc::tc_fence_after();
        long long cyc_wait = 0, cyc_issue = 0;
        uint64_t bd = bdesc0;
        for (int i = 0; i < nk; ++i, bd += bstep) {
          const long long c0 = tr ? clock64() : 0;
          // the stage's mbarrier (TMA complete_tx) orders its operand bytes for the MMA
          if (!tc::mbar_wait(&ctl->full[stage], phase, p.err, abort, tmo)) { ok = false; break; }
          const long long c1 = tr ? clock64() : 0;
          if (tr) {
            if (i > 0) cyc_wait += c1 - c0;
            if (i == 0) stamp(p, step, 1, globaltimer_ns());
            if (i == nk - 1) {
              stamp(p, step, 8, globaltimer_ns());
              stamp(p, step, 9, cyc_wait);
              stamp(p, step, 10, cyc_issue);
            }
          }
          const uint64_t ad = adesc0 + (uint64_t)((size_t)stage * (ASTG >> 4));
          tc::mma4_bf16_commit(tbase, ad, bd, idesc, i != 0, &ctl->empty[stage]);
          if (tr) cyc_issue += clock64() - c1;
          if (++stage == STG) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(&ctl->tfull);
        if (p.trace) stamp(p, step, 2, globaltimer_ns());
      }
      // drain: every MMA issued above completes before TMEM is released
      tc::mma_commit(&ctl->mdone);
      volatile int never = 0;
      tc::mbar_wait(&ctl->mdone, 0, nullptr, &never, 100000000ull);
    }
  } else {
    // ---------------- epilogue: 16 warps; warp -> (TMEM lane quarter q, 4 units)
    const int q = warp % 4;
    const int part = (warp - 2) / 4;           // units [part*4, part*4+4) of the CTA's 16
    const int r = q * 32 + lane;               // batch row = TMEM lane
    const int s = row0 + r;
    const bool row_ok = s < B;
    const int ldo = p.D * p.Hout;
    __nv_bfloat16 *hx = reinterpret_cast<__nv_bfloat16 *>(p.hx) + (size_t)d * 2 * B * Kp;
    const float *bhn = p.bhn[d];
    const int ub = u0 + part * UPT;            // first unit of this thread
    const int nu = max(0, min(UPT, H - ub));   // valid units of this thread
    // 16-byte vector access only where every address is 16-byte aligned
    const bool vec_g = nu == UPT && (H & 3) == 0;
    const bool vec_y = nu == UPT && (p.Hout & 3) == 0 &&
                       (reinterpret_cast<uintptr_t>(p.y) & 15) == 0;
    // TMEM columns: [owner CTA][gate][16 units]; lane quarter q of the warp
    const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
    const uint32_t own_col = (uint32_t)(kr * NG * UNITS + part * UPT);
    // Peers i = 0..KS-2 are the other ranks in order.  The partial sums for
    // peer pr's units go into pr's buffer, in the slot of this sender (its rank
    // among pr's peers): slot*(NG*4*128) + (g*4 + part)*128 + r, one float4 per
    // (gate, thread).
    constexpr int NP = KS > 1 ? KS - 1 : 1;
    const int SLOT = NG * 4 * AR;  // float4 per slot (rows past AR are never sent)
    uint32_t peer_x[NP], peer_bar[NP], peer_col[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      peer_x[i] = peer_bar[i] = peer_col[i] = 0;
      if (KS > 1) {
        const int pr = i < kr ? i : i + 1;
        const int slot = kr < pr ? kr : kr - 1;
        peer_x[i] = tc::mapa_shared(tc::smem_u32(xbuf + (size_t)slot * SLOT), (uint32_t)pr);
        peer_bar[i] = tc::mapa_shared(tc::smem_u32(&ctl->xfull), (uint32_t)pr);
        peer_col[i] = (uint32_t)(pr * NG * UNITS + part * UPT);
      }
    }
    int x_posted = 0, x_done = 0;  // K split, thread 64: phases armed / completed
    float h[UPT], c[UPT], bn[UPT];
    int b = 0, len = 0;
    if (row_ok) {
      b = p.meta.sorted_idx[s];
      len = p.meta.lens_sorted[s];
    }
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const bool uj = row_ok && j < nu;
      h[j] = (uj && p.h0) ? p.h0[((size_t)d * B + b) * p.Hout + ub + j] : 0.f;
      c[j] = (uj && p.c0 && NG == 4) ? p.c0[((size_t)d * B + b) * H + ub + j] : 0.f;
      bn[j] = (NG == 3 && bhn && j < nu) ? bhn[ub + j] : 0.f;
    }
    if (row_ok) {
      __nv_bfloat16 *dst = hx + (size_t)s * Kp + ub;
#pragma unroll
      for (int j = 0; j < UPT; ++j)
        if (j < nu) dst[j] = __float2bfloat16_rn(h[j]);
    }
    fence_proxy_async_global();
    epi_bar();
    if (threadIdx.x == 64) red_release_gpu_add(ctr, (p.drop_arrival && blockIdx.x == 0) ? 0u : 1u);
    // the input projection G of step st for this thread's row and units
    // (loaded a whole step ahead of its use: right after the previous step's
    // gates, so its latency is off the critical path)
    float gx[NG][UPT];
    auto load_g = [&](int st) {
      if (!(row_ok && st < len)) return;
      const int tg = d == 0 ? st : len - 1 - st;
      const size_t grow = (size_t)p.meta.step_off[tg] + s;
      if (nu == 0) return;  // no unit of this thread exists
      if (!RCU_DCHECK(grow < (size_t)p.T * B &&
                          (size_t)d * NG * H + (size_t)(NG - 1) * H + ub + nu <= (size_t)p.ldG,
                      p.err))
        return;
      const float *gp = p.G + grow * p.ldG + (size_t)d * NG * H + ub;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (vec_g) {
          const float4 f = __ldg(reinterpret_cast<const float4 *>(gp + (size_t)g * H));
          gx[g][0] = f.x; gx[g][1] = f.y; gx[g][2] = f.z; gx[g][3] = f.w;
        } else {
#pragma unroll
          for (int j = 0; j < UPT; ++j) gx[g][j] = j < nu ? __ldg(gp + (size_t)g * H + j) : 0.f;
        }
      }
    };
    // tiled G: thread 64 loads step st's [nG][rows][16 units] tile (every row
    // of a fixed-length batch runs every step, so the step's rows are
    // contiguous), counted on gbar
    const bool tiles = maps.tiles != 0;
    int g_done = 0;  // thread 64: G tiles waited for
    auto issue_g = [&](int st) {
      const int tg = d == 0 ? st : Tg - 1 - st;
      tc::mbar_arrive_expect_tx(&ctl->gbar, (uint32_t)(NG * UNITS * 4 * maps.a_rows));
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int q4 = 0; q4 < UNITS / UPT; ++q4)  // strip [g][q4]: 4 units x rows
          tma_load_3d(gtile + ((size_t)g * (UNITS / UPT) + q4) * AR * UPT, &maps.g, &ctl->gbar,
                      d * NG * H + g * H + u0 + q4 * UPT, row0, tg);
      ++ctl->g_issued;
    };
    if (tiles) {
      if (threadIdx.x == 64 && Tg > 0) issue_g(0);
    } else {
      load_g(0);
    }
    for (int step = 0; step < Tg; ++step) {
      const bool active = row_ok && step < len;
      const int tt = d == 0 ? step : len - 1 - step;
      // one thread waits for the accumulator (and the step's G tile); its
      // result is shared so that all epilogue threads leave the loop together
      if (threadIdx.x == 64) {
        // the output tile is rewritten below: its previous store has read it
        if (tiles) bulk_wait_read();
        bool ok = tc::mbar_wait(&ctl->tfull, step & 1, p.err, abort, tmo);
        if (ok && tiles) {
          ok = tc::mbar_wait(&ctl->gbar, (uint32_t)step & 1u, p.err, abort, tmo);
          if (ok) ++g_done;
        }
        ctl->go = ok;
      }
      epi_bar();
      if (!ctl->go) break;
      if (tiles) {  // (rows past AR read past the strip, in bounds; never used)
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float4 f =
              *reinterpret_cast<const float4 *>(gtile + (((size_t)g * (UNITS / UPT) + part) * AR + r) * UPT);
          gx[g][0] = f.x; gx[g][1] = f.y; gx[g][2] = f.z; gx[g][3] = f.w;
        }
      }
      tc::tc_fence_after();
      if (p.trace && threadIdx.x == 64) stamp(p, step, 3, globaltimer_ns());
      float acc[NG][UPT];
      {
        uint32_t ra[NG][4], rp[NP][KS > 1 ? NG : 1][4];
#pragma unroll
        for (int g = 0; g < NG; ++g) tmem_ld4_nowait(tl + own_col + (uint32_t)(g * UNITS), ra[g]);
        if (KS > 1) {
#pragma unroll
          for (int i = 0; i < NP; ++i)
#pragma unroll
            for (int g = 0; g < NG; ++g)
              tmem_ld4_nowait(tl + peer_col[i] + (uint32_t)(g * UNITS), rp[i][KS > 1 ? g : 0]);
        }
        tmem_wait_ld();
        tc::tc_fence_before();
        if (lane == 0) tc::mbar_arrive(&ctl->tfree);
        if (p.trace && threadIdx.x == 64) stamp(p, step, 12, globaltimer_ns());
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int j = 0; j < UPT; ++j) acc[g][j] = __uint_as_float(ra[g][j]);
        if (KS > 1 && (FULL || r < AR)) {
          // hand each peer its units' partial sums over K blocks [kb0, kb0+nk)
          // (the batch's rows only: the distributed-shared-memory bandwidth
          // is the cost of this exchange)
#pragma unroll
          for (int i = 0; i < NP; ++i)
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              const int gi = KS > 1 ? g : 0;
              tc::st_async_v4(peer_x[i] + (uint32_t)(((g * 4 + part) * AR + r) * 16),
                              __uint_as_float(rp[i][gi][0]), __uint_as_float(rp[i][gi][1]),
                              __uint_as_float(rp[i][gi][2]), __uint_as_float(rp[i][gi][3]),
                              peer_bar[i]);
            }
        }
        // (thread 64 counts the steps sent, whether or not its own row is live)
        if (KS > 1 && threadIdx.x == 64) x_sent = (uint32_t)(step + 1);
      }
      if (p.trace && threadIdx.x == 64) stamp(p, step, 5, globaltimer_ns());
      if (KS > 1) {
        // the peers' partial sums for this CTA's units
        if (threadIdx.x == 64) {
          tc::mbar_arrive_expect_tx(&ctl->xfull, (uint32_t)geo.x_bytes);
          x_posted = step + 1;
          ctl->go2 = tc::mbar_wait_cluster(&ctl->xfull, step & 1, p.err, abort, tmo);
          if (ctl->go2) x_done = step + 1;
        }
        epi_bar();
        if (!ctl->go2) break;
        if (FULL || r < AR) {
#pragma unroll
          for (int i = 0; i < NP; ++i)
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              const float4 v = xbuf[(size_t)i * SLOT + (g * 4 + part) * AR + r];
              acc[g][0] += v.x; acc[g][1] += v.y; acc[g][2] += v.z; acc[g][3] += v.w;
            }
        }
        if (p.trace && threadIdx.x == 64) stamp(p, step, 11, globaltimer_ns());
      }
      if (active) {
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
          if (NG == 4) {
            const float ig = sigmoid_fast(acc[0][j] + gx[0][j]);
            const float fg = sigmoid_fast(acc[1][j] + gx[1][j]);
            const float gg = tanh_fast(acc[2][j] + gx[2][j]);
            const float og = sigmoid_fast(acc[3][j] + gx[3][j]);
            c[j] = fg * c[j] + ig * gg;
            if (p.cclip) c[j] = fminf(fmaxf(c[j], p.cclip_lo), p.cclip_hi);
            h[j] = og * tanh_fast(c[j]);
          } else {
            const float rg = sigmoid_fast(gx[0][j] + acc[0][j]);
            const float zg = sigmoid_fast(gx[1][j] + acc[1][j]);
            const float ng = tanh_fast(gx[2][j] + rg * (acc[NG - 1][j] + bn[j]));
            h[j] = (1.f - zg) * ng + zg * h[j];
          }
        }
      }
      if (p.trace && threadIdx.x == 64) stamp(p, step, 13, globaltimer_ns());
      // exchange buffer for the next step (bf16 MMA operand): on the critical path
      if (active && nu > 0 && RCU_DCHECK(s < B && ub + nu <= Kp, p.err)) {
        __nv_bfloat16 *dst = hx + (size_t)(((step & 1) ^ 1) * B + s) * Kp + ub;
        if (nu == UPT) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(h[0], h[1]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(h[2], h[3]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t *>(&lo);
          pk.y = *reinterpret_cast<uint32_t *>(&hi);
          *reinterpret_cast<uint2 *>(dst) = pk;
        } else {
#pragma unroll
          for (int j = 0; j < UPT; ++j)
            if (j < nu) dst[j] = __float2bfloat16_rn(h[j]);
        }
      }
      if (tiles && row_ok) {
        // the layer output of this row and units, for one TMA store per step
        if (maps.tiles & 2) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(h[0], h[1]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(h[2], h[3]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t *>(&lo);
          pk.y = *reinterpret_cast<uint32_t *>(&hi);
          // bf16 strips of 8 units (16-byte rows): part pairs share one
          *reinterpret_cast<uint2 *>(otile_m + (((size_t)(part >> 1) * AR + r) * 2 * UPT + (part & 1) * UPT) * 2) = pk;
        }
        if (maps.tiles & 1)
          *reinterpret_cast<float4 *>(otile + ((size_t)part * AR + r) * UPT * 4) =
              make_float4(h[0], h[1], h[2], h[3]);
        fence_proxy_async_shared();
      }
      if (p.trace && threadIdx.x == 64) stamp(p, step, 6, globaltimer_ns());
      fence_proxy_async_global();
      epi_bar();
      if (threadIdx.x == 64) {
        if (p.trace) stamp(p, step, 7, globaltimer_ns());
        // release: orders the epilogue's h_t stores (all threads, through the
        // barrier above) before the arrival
        red_release_gpu_add(ctr, 1u);
        if (p.trace) stamp(p, step, 4, globaltimer_ns());
        if (tiles) {
          // off the critical path: the step's output tile, and the next
          // step's G tile (every thread read this step's above)
          if (u0 < p.Hout) {
            // one store per strip: 4 fp32 or 8 bf16 units of every row
            const int ts = d == 0 ? step : Tg - 1 - step;
            if (maps.tiles & 1)
              for (int q4 = 0; q4 < UNITS / UPT; ++q4)
                tma_store_3d(&maps.out, otile + (size_t)q4 * AR * UPT * 4,
                             d * p.Hout + u0 + q4 * UPT, row0, ts);
            if (maps.tiles & 2)
              for (int q8 = 0; q8 < UNITS / (2 * UPT); ++q8)
                tma_store_3d(&maps.outm, otile_m + (size_t)q8 * AR * 2 * UPT * 2,
                             d * p.Hout + u0 + q8 * 2 * UPT, row0, ts);
          }
          if (step + 1 < Tg) issue_g(step + 1);
        }
      }
      // the next step's G: loaded after the release (a release waits for the
      // thread's earlier loads too, and the address needs the step offset
      // table, whose load the h_t store would otherwise wait behind)
      if (!tiles) load_g(step + 1);
      // outputs leave the critical path: written after h_t is published
      if (!tiles && active && p.y && RCU_DCHECK(tt >= 0 && tt < p.T && b >= 0 && b < B, p.err)) {
        float *yo = p.y + ((size_t)tt * B + b) * ldo + (size_t)d * p.Hout + ub;
        if (vec_y) {
          *reinterpret_cast<float4 *>(yo) = make_float4(h[0], h[1], h[2], h[3]);
        } else {
#pragma unroll
          for (int j = 0; j < UPT; ++j)
            if (j < nu) yo[j] = h[j];
        }
      }
      if (!tiles && active && p.ymid &&
          RCU_DCHECK((size_t)p.meta.step_off[tt] + s < (size_t)p.T * B, p.err)) {
        __nv_bfloat16 *ym = reinterpret_cast<__nv_bfloat16 *>(p.ymid) +
                            ((size_t)p.meta.step_off[tt] + s) * ldo + (size_t)d * p.Hout + ub;
#pragma unroll
        for (int j = 0; j < UPT; ++j)
          if (j < nu) ym[j] = __float2bfloat16_rn(h[j]);
      }
    }
    if (row_ok && !*abort) {
#pragma unroll
      for (int j = 0; j < UPT; ++j) {
        if (j >= nu) continue;
        if (p.h_n) p.h_n[((size_t)d * B + b) * p.Hout + ub + j] = h[j];
        if (NG == 4 && p.c_n) p.c_n[((size_t)d * B + b) * H + ub + j] = c[j];
      }
    }
    if (KS > 1) x_left = x_done < x_posted ? -x_done - 1 : x_done;  // < 0: phase x_done armed
    if (tiles && threadIdx.x == 64) {
      // output stores complete, and a G tile still landing lands, before the
      // CTA's shared memory goes away (at most one is outstanding)
      bulk_wait_all();
      if (ctl->g_issued > g_done) {
        volatile int never = 0;
        tc::mbar_wait(&ctl->gbar, (uint32_t)(ctl->g_issued - 1) & 1u, nullptr, &never,
                      100000000ull);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (KS > 1 && threadIdx.x == 64) {
    // Tell every peer how many steps of partial sums it will have received
    // from this CTA.  The count is stored into the peer's shared memory now,
    // while the peer is certain to be resident (it cannot pass the cluster
    // barrier below before this CTA arrives), so that nothing after that
    // barrier touches another CTA's shared memory: a peer may exit as soon as
    // it has passed it.
    for (int pr = 0; pr < KS; ++pr) {
      if (pr == kr) continue;
      const uint32_t dst = tc::mapa_shared(tc::smem_u32(&ctl->peer_sent[kr]), (uint32_t)pr);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(x_sent) : "memory");
    }
  }
  // no member leaves while its partner may still deliver partial sums to it;
  // the barrier's release/acquire also makes the peers' counts visible here
  if (KS > 1) tc::cluster_sync();
  if (KS > 1 && threadIdx.x == 64) {
    // After an early exit a peer may have sent one step more than this CTA
    // consumed (never two: the peer's next step needs this CTA's arrival at
    // the step barrier, made only after consuming).  Those stores land in this
    // CTA's shared memory, so wait for them (bounded) before leaving.  Only
    // this CTA's own shared memory is read here.
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

// K kept whole
template <int NG, bool FULL>
__global__ void __launch_bounds__(NT, 1) rec_tc_kernel(const __grid_constant__ Maps maps,
                                                       const RecParams p) {
  rec_tc_body<NG, 1, FULL>(maps, p);
}
// K split over a CTA pair; the pair is the kernel's own cluster shape
template <int NG, bool FULL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
    rec_tc_pair_kernel(const __grid_constant__ Maps maps, const RecParams p) {
  rec_tc_body<NG, 2, FULL>(maps, p);
}
// K split over 4 CTAs (GRU: the resident weights and the partial-sum buffer
// fit beside a 3-stage h ring)
template <int NG, bool FULL>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(NT, 1)
    rec_tc_quad_kernel(const __grid_constant__ Maps maps, const RecParams p) {
  rec_tc_body<NG, 4, FULL>(maps, p);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [T][rows][cols] (row stride ld elements of esz bytes), box 16 bytes of
// columns x box_rows rows x 1, no swizzle: the tiled G and output streams
bool make_map_steps(CUtensorMap *map, const void *base, bool bf16, int T, int rows, int cols,
                    int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const size_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)ld * esz, (cuuint64_t)ld * esz * rows};
  cuuint32_t box[3] = {(cuuint32_t)(16 / esz), (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap *map, const void *base, long long rows, int cols, int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_map_2d(CUtensorMap *map, const void *base, long long rows, int cols, int ld,
               int box_rows) {
  return make_map(map, base, rows, cols, ld, box_rows);
}

int tc_rec_units() { return UNITS; }

bool tc_rec_packable(int cell, int H, int Hout, int P) {
  if (P > 0) return false;  // projection runs on the portable kernel
  if (H < 1 || Hout < 1) return false;
  const int nG = cell == CELL_LSTM ? 4 : 3;
  return make_geo(nG, Hout, 1).stages >= 2 && encode_fn() != nullptr;
}

bool tc_rec_supported(int cell, int H, int Hout, int P, int nsm, int B, int D) {
  if (!tc_rec_packable(cell, H, Hout, P)) return false;
  const long long ctas = (long long)D * ceil_div(B, BG) * ceil_div(H, UNITS);
  return ctas <= nsm;
}

int tc_rec_counters(int B, int D) {
  return D * ceil_div(B, BG) * 32 + 32;
}

namespace {
bool ks_fits(int nG, int K, int ks);
}

int tc_rec_grid(int cell, int H, int Hout, int B, int D, int ksplit) {
  const int nG = cell == CELL_LSTM ? 4 : 3;
  int ks = ksplit == 0 ? 2 : ksplit;
  while (ks > 1 && !ks_fits(nG, Hout, ks)) ks /= 2;
  const int NU = ks > 1 ? ks * ceil_div(H, ks * UNITS) : ceil_div(H, UNITS);
  return D * ceil_div(B, BG) * NU;
}

void tc_pack_whh(int cell, int H, int Hout, const float *whh, std::vector<uint16_t> &out,
                 uint16_t (*to_bf16)(float)) {
  const int nG = cell == CELL_LSTM ? 4 : 3;
  const int N = nG * UNITS, NU = ceil_div(H, UNITS), Kp = round_up(Hout, 8);
  out.assign((size_t)NU * N * Kp, 0);
  for (int ug = 0; ug < NU; ++ug)
    for (int g = 0; g < nG; ++g)
      for (int j = 0; j < UNITS; ++j) {
        const int u = ug * UNITS + j;
        if (u >= H) continue;
        for (int k = 0; k < Hout; ++k)
          out[((size_t)ug * N + g * UNITS + j) * Kp + k] = to_bf16(whh[(size_t)(g * H + u) * Hout + k]);
      }
}

namespace {

template <int NG, bool FULL>
const void *kernel_for(int ks) {
  if (ks == 4) return (const void *)rec_tc_quad_kernel<NG, FULL>;
  return ks == 2 ? (const void *)rec_tc_pair_kernel<NG, FULL>
                 : (const void *)rec_tc_kernel<NG, FULL>;
}
// a K split over ks CTAs fits: a ring of at least 2 h stages and a K block
// for every CTA
bool ks_fits(int nG, int K, int ks) {
  const Geo g = make_geo(nG, K, ks);
  return g.stages >= 2 && (ks - 1) * g.nkbm < g.nkb;
}

// Cooperative launch of `grid` CTAs of a kernel that declares its cluster
// shape (`cs` CTAs) itself; false (nothing launched) when that cluster grid
// cannot be resident at once.
bool launch_clustered(const void *fn, int grid, int cs, size_t smem, void **args, cudaStream_t s,
                      cudaError_t *err) {
  return tc_launch_clustered(fn, grid, NT, cs, smem, args, s, err);
}

}  // namespace

bool tc_launch_clustered(const void *fn, int grid, int nthreads, int cs, size_t smem, void **args,
                         cudaStream_t s, cudaError_t *err) {
  *err = cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess ||
      (long long)max_clusters * cs < grid) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *err = cudaLaunchKernelExC(&cfg, fn, args);
  return true;
}

cudaError_t launch_tc_recurrent(const TcRecParams &tp, int nsm, cudaStream_t s) {
  (void)nsm;
  RecParams p = tp.base;
  const int nG = p.nG;
  const int NU16 = ceil_div(p.H, UNITS);  // 16-unit tiles in the packed weights
  const int NBG = ceil_div(p.B, BG);
  Maps maps;
  maps.a_rows = NBG == 1 ? round_up(p.B, 8) : BG;
  if (!make_map(&maps.hx, p.hx, (long long)p.D * 2 * p.B, p.Hout, p.Kp, maps.a_rows))
    return cudaErrorInvalidValue;


  // K split over ks CTAs (a cluster): requested (1, 2 or 4), or automatic (a
  // pair); halved until the plan fits shared memory and gives every CTA a K block
  int ks = tp.ksplit;
  if (ks == 0) ks = 2;
  while (ks > 1 && !ks_fits(nG, p.Hout, ks)) ks /= 2;

  // Tiled G and output streams: fixed-length batches (a step's rows are
  // contiguous), 16-byte aligned rows and bases, whole 16-unit tiles of the
  // outputs (fp32 y and / or the bf16 rows of the next layer), and a ring of
  // at least 4 h stages beside the tiles
  const bool y_out = p.y != nullptr, m_out = p.ymid != nullptr;
  const int ldo = p.D * p.Hout;
  auto aligned16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  const bool tiles_ok = tp.fixed_length && (y_out || m_out) && (p.H % 4) == 0 &&
                        (p.Hout % UNITS) == 0 && ((size_t)p.ldG * 4) % 16 == 0 &&
                        ((size_t)ldo * 2) % 16 == 0 && aligned16(p.G) &&
                        (!y_out || aligned16(p.y)) && (!m_out || aligned16(p.ymid));
  const int tmask = (y_out ? 1 : 0) | (m_out ? 2 : 0);

  for (int attempt = 0; attempt < 3; ++attempt) {
    maps.tiles = tiles_ok && make_geo(nG, p.Hout, ks, tmask, maps.a_rows).stages >= 4 ? tmask : 0;
    const Geo geo = make_geo(nG, p.Hout, ks, maps.tiles, maps.a_rows);
    if (maps.tiles &&
        (!make_map_steps(&maps.g, p.G, false, p.T, p.B, p.ldG, p.ldG, maps.a_rows) ||
         (y_out && !make_map_steps(&maps.out, p.y, false, p.T, p.B, ldo, ldo, maps.a_rows)) ||
         (m_out && !make_map_steps(&maps.outm, p.ymid, true, p.T, p.B, ldo, ldo, maps.a_rows))))
      return cudaErrorInvalidValue;
    p.NU = ks > 1 ? ks * ceil_div(p.H, ks * UNITS) : NU16;
    for (int d = 0; d < 2; ++d) {
      const void *w = tp.Wtc[d < p.D ? d : 0];
      if (!make_map(&maps.w[d], w, (long long)NU16 * nG * UNITS, p.Hout, p.Kp, geo.N))
        return cudaErrorInvalidValue;
    }
    const bool full = maps.a_rows == BG;
    const void *fn = nG == 4 ? (full ? kernel_for<4, true>(ks) : kernel_for<4, false>(ks))
                             : (full ? kernel_for<3, true>(ks) : kernel_for<3, false>(ks));
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)geo.smem);
    if (e != cudaSuccess) return e;
    const int grid = p.D * NBG * p.NU;
    void *args[] = {&maps, &p};
    if (ks > 1) {
      if (launch_clustered(fn, grid, ks, geo.smem, args, s, &e)) return e;
      ks /= 2;  // that cluster grid cannot be co-resident: a smaller split
      while (ks > 1 && !ks_fits(nG, p.Hout, ks)) ks /= 2;
      continue;
    }
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(NT), args, geo.smem, s);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace rcu
