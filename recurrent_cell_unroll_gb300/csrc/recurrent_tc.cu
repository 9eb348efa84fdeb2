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

constexpr int UNITS = 16;       // hidden units per CTA
constexpr int BG = 128;         // batch rows per CTA (MMA M)
constexpr int BK = 64;          // K per stage (128 bytes of bf16)
constexpr int A_STAGE = BG * BK * 2;
constexpr int EPI_WARPS = 16;   // 4 per TMEM lane quarter
constexpr int UPT = UNITS / 4;  // units per epilogue thread
constexpr int NT = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int MAX_STAGES = 8;

struct Maps {
  CUtensorMap hx;    // [D*2*B rows][K cols], ld Kp, bf16, box 64 x 128
  CUtensorMap w[2];  // per direction [NU*N rows][K cols], ld Kp, bf16, box 64 x N
};

struct Ctl {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], wbar, tfull, tfree, mdone;
  uint32_t tmem_base;
  int abort;
  int go;  // epilogue: result of the per-step accumulator wait, shared by all 128 threads
};

struct Geo {
  int N, nkb, stages;
  size_t w_bytes, smem;
};

__host__ __device__ inline Geo make_geo(int nG, int K) {
  Geo g;
  g.N = nG * UNITS;
  g.nkb = ceil_div(K, BK);
  g.w_bytes = (size_t)g.nkb * g.N * 128;
  const size_t fixed = 1024 + g.w_bytes + 256;
  int st = (int)((SMEM_LIMIT - (long long)fixed) / A_STAGE);
  g.stages = st > MAX_STAGES ? MAX_STAGES : st;
  g.smem = fixed + (size_t)(g.stages > 0 ? g.stages : 0) * A_STAGE;
  return g;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

// 32 lanes x 4 consecutive 32-bit TMEM columns
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// bf16 path activations on the MUFU tanh unit (PTX tanh.approx.f32); the
// logistic function through the identity sigmoid(x) = 1/2 + tanh(x/2)/2
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }

__device__ __forceinline__ void load16(const float *p, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = __ldg(reinterpret_cast<const float4 *>(p) + i);
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
}

template <int NG>
__global__ void __launch_bounds__(NT, 1) rec_tc_kernel(const __grid_constant__ Maps maps,
                                                       const RecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const Geo geo = make_geo(NG, p.Hout);
  const int N = geo.N, nkb = geo.nkb, STG = geo.stages;
  uint8_t *sW = smem;                       // resident B operand, nkb blocks of N x 128 B
  uint8_t *sA = smem + geo.w_bytes;         // ring of STG stages of 128 x 128 B
  Ctl *ctl = reinterpret_cast<Ctl *>(sA + (size_t)STG * A_STAGE);

  const int NU = p.NU, NBG = ceil_div(p.B, BG);
  const int d = blockIdx.x / (NBG * NU);
  const int rem = blockIdx.x % (NBG * NU);
  const int bg = rem / NU, ug = rem % NU;
  const int u0 = ug * UNITS, row0 = bg * BG;
  const int B = p.B, H = p.H, Kp = p.Kp;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int *abort = &ctl->abort;
  const uint64_t tmo = p.timeout_ns;
  unsigned *ctr = p.ctr + d * NBG + bg;
  // steps this batch group runs: the longest row of the group (rows sorted by length)
  const int Tg = row0 < B ? p.meta.lens_sorted[row0] : 0;
  // cluster of CTAs sharing (d, bg): each issues 1/cs of the h k-blocks as
  // multicast loads into every member; a stage is free again once all
  // members' MMAs have consumed it
  const uint32_t cs = tc::cluster_nctarank(), crank = tc::cluster_ctarank();
  const uint16_t cmask = (uint16_t)((1u << cs) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], cs);
    }
    tc::mbar_init(&ctl->wbar, 1);
    tc::mbar_init(&ctl->tfull, 1);
    tc::mbar_init(&ctl->tfree, EPI_WARPS);
    tc::mbar_init(&ctl->mdone, 1);
    ctl->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, 64);
  tc::tc_fence_before();
  __syncthreads();
  if (cs > 1) tc::cluster_sync();  // peers' barriers exist before any multicast
  tc::tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&maps.hx);
      tc::prefetch_tmap(&maps.w[d]);
      // resident weights: rows [ug*N, ug*N + N) of this direction's packed W_hh
      tc::mbar_arrive_expect_tx(&ctl->wbar, (uint32_t)geo.w_bytes);
      for (int kb = 0; kb < nkb; ++kb)
        tc::tma_load_2d(sW + (size_t)kb * N * 128, &maps.w[d], &ctl->wbar, kb * BK, ug * N);
      int stage = 0;
      uint32_t phase = 0;
      int pend_stage[MAX_STAGES], npend = 0;
      uint32_t pend_phase[MAX_STAGES];
      for (int step = 0; step < Tg; ++step) {
        // wait until every CTA of (d, bg) has published h_{step-1}
        const unsigned target = (unsigned)(NU * (step + 1));
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
        if (p.trace && blockIdx.x == 0) p.trace[step * 16 + 0] = globaltimer_ns();
        const int arow = (d * 2 + (step & 1)) * B + row0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, p.err, abort, tmo)) goto producer_out;
          tc::mbar_arrive_expect_tx(&ctl->full[stage], A_STAGE);
          if (cs == 1) {
            tc::tma_load_2d(sA + (size_t)stage * A_STAGE, &maps.hx, &ctl->full[stage], kb * BK,
                            arow);
          } else if ((uint32_t)kb % cs == crank) {
            tc::tma_load_2d_mc(sA + (size_t)stage * A_STAGE, &maps.hx, &ctl->full[stage],
                               kb * BK, arow, cmask);
          }
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
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BG, NG * UNITS);
      // The issuing thread is on the critical path: descriptors are built once
      // and advanced by adding (byte offset >> 4) to the start-address field
      // (all shared-memory offsets here stay below 256 KB, so the 14-bit
      // field cannot carry).
      const uint64_t adesc0 = tc::smem_desc_sw128(tc::smem_u32(sA));
      const uint64_t bdesc0 = tc::smem_desc_sw128(tc::smem_u32(sW));
      const uint32_t bstep = (uint32_t)(N * 128) >> 4;
      const bool tr = p.trace && blockIdx.x == 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = tc::mbar_wait(&ctl->wbar, 0, p.err, abort, tmo);
      for (int step = 0; ok && step < Tg; ++step) {
        if (!tc::mbar_wait(&ctl->tfree, (step & 1) ^ 1, p.err, abort, tmo)) break;
        tc::tc_fence_after();
        long long cyc_wait = 0, cyc_issue = 0;
        uint64_t bd = bdesc0;
        for (int kb = 0; kb < nkb; ++kb, bd += bstep) {
          const long long c0 = tr ? clock64() : 0;
          // the stage's mbarrier (TMA complete_tx) orders its operand bytes for the MMA
          if (!tc::mbar_wait(&ctl->full[stage], phase, p.err, abort, tmo)) { ok = false; break; }
          const long long c1 = tr ? clock64() : 0;
          if (tr) {
            if (kb > 0) cyc_wait += c1 - c0;
            if (kb == 0) p.trace[step * 16 + 1] = globaltimer_ns();
            if (kb == nkb - 1) {
              p.trace[step * 16 + 8] = globaltimer_ns();
              p.trace[step * 16 + 9] = cyc_wait;
              p.trace[step * 16 + 10] = cyc_issue;
            }
          }
          const uint64_t ad = adesc0 + (uint64_t)(stage * (A_STAGE >> 4));
          if (cs == 1) {
            tc::mma4_bf16_commit(tbase, ad, bd, idesc, kb != 0, &ctl->empty[stage]);
          } else {
            tc::mma_bf16(tbase, ad, bd, idesc, kb != 0);
            tc::mma_bf16(tbase, ad + 2, bd + 2, idesc, 1u);
            tc::mma_bf16(tbase, ad + 4, bd + 4, idesc, 1u);
            tc::mma_bf16(tbase, ad + 6, bd + 6, idesc, 1u);
            tc::mma_commit_mc(&ctl->empty[stage], cmask);
          }
          if (tr) cyc_issue += clock64() - c1;
          if (++stage == STG) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(&ctl->tfull);
        if (p.trace && blockIdx.x == 0) p.trace[step * 16 + 2] = globaltimer_ns();
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
    if (threadIdx.x == 64) {
      red_release_gpu_add(ctr, (p.drop_arrival && blockIdx.x == 0) ? 0u : 1u);
    }
    for (int step = 0; step < Tg; ++step) {
      const bool active = row_ok && step < len;
      const int tt = d == 0 ? step : len - 1 - step;
      float gx[NG][UPT];
      if (active) {
        const size_t grow = (size_t)p.meta.step_off[tt] + s;
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
      }
      // one thread waits for the accumulator; the verdict is shared so that
      // all epilogue threads leave the loop together
      if (threadIdx.x == 64) ctl->go = tc::mbar_wait(&ctl->tfull, step & 1, p.err, abort, tmo);
      epi_bar();
      if (!ctl->go) break;
      tc::tc_fence_after();
      if (p.trace && blockIdx.x == 0 && threadIdx.x == 64) p.trace[step * 16 + 3] = globaltimer_ns();
      float acc[NG][UPT];
#pragma unroll
      for (int g = 0; g < NG; ++g)
        tmem_ld4(tbase + (uint32_t)(g * UNITS + part * UPT) + ((uint32_t)(q * 32) << 16), acc[g]);
      tc::tc_fence_before();
      if (lane == 0) tc::mbar_arrive(&ctl->tfree);
      if (p.trace && blockIdx.x == 0 && threadIdx.x == 64) p.trace[step * 16 + 5] = globaltimer_ns();
      if (active) {
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
          if (NG == 4) {
            const float ig = sigmoid_fast(acc[0][j] + gx[0][j]);
            const float fg = sigmoid_fast(acc[1][j] + gx[1][j]);
            const float gg = tanh_fast(acc[2][j] + gx[2][j]);
            const float og = sigmoid_fast(acc[3][j] + gx[3][j]);
            c[j] = fg * c[j] + ig * gg;
            h[j] = og * tanh_fast(c[j]);
          } else {
            const float rg = sigmoid_fast(gx[0][j] + acc[0][j]);
            const float zg = sigmoid_fast(gx[1][j] + acc[1][j]);
            const float ng = tanh_fast(gx[2][j] + rg * (acc[NG - 1][j] + bn[j]));
            h[j] = (1.f - zg) * ng + zg * h[j];
          }
        }
        // exchange buffer for the next step (bf16 MMA operand): on the critical path
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
      if (p.trace && blockIdx.x == 0 && threadIdx.x == 64) p.trace[step * 16 + 6] = globaltimer_ns();
      fence_proxy_async_global();
      epi_bar();
      if (threadIdx.x == 64) {
        if (p.trace && blockIdx.x == 0) p.trace[step * 16 + 7] = globaltimer_ns();
        red_release_gpu_add(ctr, 1u);  // release: orders the epilogue's h_t stores
        if (p.trace && blockIdx.x == 0) p.trace[step * 16 + 4] = globaltimer_ns();
      }
      // outputs leave the critical path: written after h_t is published
      if (active && p.y) {
        float *yo = p.y + ((size_t)tt * B + b) * ldo + (size_t)d * p.Hout + ub;
        if (vec_y) {
          *reinterpret_cast<float4 *>(yo) = make_float4(h[0], h[1], h[2], h[3]);
        } else {
#pragma unroll
          for (int j = 0; j < UPT; ++j)
            if (j < nu) yo[j] = h[j];
        }
      }
      if (active && p.ymid) {
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
  }
  tc::tc_fence_before();
  __syncthreads();
  // no member leaves while a peer may still deliver loads or arrivals to it
  if (cs > 1) tc::cluster_sync();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, 64);
  }
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

int tc_rec_units() { return UNITS; }

bool tc_rec_packable(int cell, int H, int Hout, int P) {
  if (P > 0) return false;  // projection runs on the portable kernel
  if (H < 1 || Hout < 1) return false;
  const int nG = cell == CELL_LSTM ? 4 : 3;
  return make_geo(nG, Hout).stages >= 2 && encode_fn() != nullptr;
}

bool tc_rec_supported(int cell, int H, int Hout, int P, int nsm, int B, int D) {
  if (!tc_rec_packable(cell, H, Hout, P)) return false;
  const long long ctas = (long long)D * ceil_div(B, BG) * ceil_div(H, UNITS);
  return ctas <= nsm;
}

int tc_rec_counters(int B, int D) { return D * ceil_div(B, BG); }

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

cudaError_t launch_tc_recurrent(const TcRecParams &tp, int nsm, cudaStream_t s) {
  (void)nsm;
  RecParams p = tp.base;
  const int nG = p.nG;
  const Geo geo = make_geo(nG, p.Hout);
  p.NU = ceil_div(p.H, UNITS);
  const int NBG = ceil_div(p.B, BG);
  Maps maps;
  if (!make_map(&maps.hx, p.hx, (long long)p.D * 2 * p.B, p.Hout, p.Kp, BG))
    return cudaErrorInvalidValue;
  for (int d = 0; d < 2; ++d) {
    const void *w = tp.Wtc[d < p.D ? d : 0];
    if (!make_map(&maps.w[d], w, (long long)p.NU * geo.N, p.Hout, p.Kp, geo.N))
      return cudaErrorInvalidValue;
  }
  const void *fn = nG == 4 ? (const void *)rec_tc_kernel<4> : (const void *)rec_tc_kernel<3>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)geo.smem);
  if (e != cudaSuccess) return e;
  const int grid = p.D * NBG * p.NU;
  // cluster size: requested, else the largest of 4, 2 dividing the unit groups
  // Multicast was measured not to pay on GB300 for this kernel (the MMA
  // phase is bound by the tensor pipe's rate on these small-N MMAs, not by
  // L2 requests), so clusters are opt-in.
  int cs = tp.cluster > 0 ? tp.cluster : 1;
  while (cs > 1 && (p.NU % cs) != 0) cs /= 2;
  if (cs > 1) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) { cudaGetLastError(); cs = 1; }
  }
  void *args[] = {&maps, &p};
  if (cs > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = geo.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int max_clusters = 0;
    cudaLaunchConfig_t q = cfg;
    q.numAttrs = 1;  // occupancy query on the cluster shape
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &q) == cudaSuccess &&
        max_clusters * cs >= grid) {
      e = cudaLaunchKernelExC(&cfg, fn, args);
      if (e == cudaSuccess) return cudaSuccess;
    }
    cudaGetLastError();  // fall back to the cluster-free launch
  }
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(NT), args, geo.smem, s);
}

}  // namespace rcu
