// Cluster-resident recurrent kernel (LSTM / GRU without projection) for
// problems whose W_hh fits the shared memory of one thread-block cluster.
//
// A cluster of cs CTAs (16 where the GPU allows it, else 8) keeps one copy
// of a direction's W_hh: CTA `rank` holds the rows of units
// [rank*U, rank*U + U), all gates, in shared memory for the whole sequence.
// Clusters take disjoint slices of Bc sorted batch rows, so they never wait
// for one another; a step needs only the cluster's own hardware barrier.
// Per step each CTA
//   1. computes its rows of h_{t-1} W_hh^T for the active rows of its slice
//      (the "recurrent hidden-hidden dense" of "[TOPI] TE implementation of
//      LSTM using scan", apache/tvm PR 11531): 8 lanes per output row, each
//      taking every 8th 16-byte K chunk, then a 3-level shuffle reduction;
//   2. adds the input projection G (prefetched during the previous step),
//      applies the gates and the cell update (c and h stay in registers, one
//      (row, unit) pair per thread);
//   3. stores h_t into the h buffer of every CTA of the cluster with
//      asynchronous distributed-shared-memory stores (st.async), each
//      signalling its bytes on the receiving CTA's mbarrier for that buffer
//      (double-buffered by step parity).  A CTA starts step t+1 as soon as
//      all bytes of h_t have landed in its own buffer: no cluster-wide
//      barrier and no release fence per step.  A peer can write h_{t+1}
//      into the buffer this CTA reads at step t only after receiving this
//      CTA's h_t, which is sent after that read.
// Rows whose length is exhausted leave the active prefix of the sorted batch
// ("RNN Op Changes", apache/mxnet issue 9543); the backward direction runs
// row s at time len_s - 1 - step.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int KC_MAX = 1024;  // padded K (multiple of 128)
constexpr int SMEM_LIMIT = 227 * 1024;

constexpr int SOFF_MAX = 4096;  // step offsets staged in shared memory up to this T

struct CSmem {
  size_t w, h, pre, lens, soff, bar, total;
};
__host__ __device__ inline CSmem cl_smem(int R, int Kc, int Bc, size_t es, int T) {
  CSmem L;
  size_t o = 0;
  L.w = o;
  o += (size_t)R * Kc * es;
  o = round_up_sz(o, 16);
  L.h = o;
  o += (size_t)2 * Bc * Kc * 4;
  L.pre = o;
  o += (size_t)Bc * R * 4;
  L.lens = o;
  o += (size_t)Bc * 4;
  L.soff = o;
  if (T <= SOFF_MAX) o += (size_t)T * 4;
  o = round_up_sz(o, 8);
  L.bar = o;
  o += 16;  // one mbarrier per h buffer
  L.total = o;
  return L;
}

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_map_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(const void *p, uint32_t rank) {
  return cl_map_addr((uint32_t)__cvta_generic_to_shared(p), rank);
}
// 4-byte asynchronous store into a cluster CTA's shared memory, completing as
// 4 bytes of complete_tx on that CTA's mbarrier
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   addr),
               "r"(__float_as_uint(v)), "r"(bar)
               : "memory");
}

__device__ __forceinline__ float4 wload(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 wload(const __nv_bfloat16 *p) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// KQ4 > 0: the CTA's gate rows (at most 64) stay in registers, warp w owning
// rows 4w..4w+3 over K = 128*KQ4 (lane l takes the 16-byte chunks l, l+32,
// ...); KQ4 == 0: rows stay in shared memory, 8 lanes per row.
template <typename WT, int NG, int KQ4>
__global__ void __launch_bounds__(NT, 1)
    rec_cluster_kernel(const RecParams p, const void *W0, const void *W1, int U, int Kc, int Bc,
                       int NCL, int cs_plan) {
  extern __shared__ __align__(16) unsigned char smem[];
  const uint32_t cs = cl_size(), rank = cl_rank();
  if ((int)cs != cs_plan) {  // units are assigned for cs_plan CTAs per cluster
    if (threadIdx.x == 0) atomicCAS(p.err, DEV_OK, DEV_CONFIG);
    return;
  }
  const int ci = blockIdx.x / cs;
  const int d = ci / NCL, slice = ci % NCL;
  const int B = p.B, H = p.H, Hout = p.Hout;
  const int r0 = slice * Bc;                   // first sorted row of the slice
  const int nrow = max(0, min(Bc, B - r0));    // rows of the slice
  const int u0 = (int)rank * U;
  const int nu = max(0, min(U, H - u0));       // valid units of this CTA
  const int R = NG * U;                        // local row j*NG + g = gate g of unit u0 + j
  const int KQ = Kc / 32;  // 16-byte K chunks per lane of an 8-lane group
  const CSmem L = cl_smem(R, Kc, Bc, sizeof(WT), p.T);
  WT *Ws = reinterpret_cast<WT *>(smem + L.w);
  float *hb = reinterpret_cast<float *>(smem + L.h);     // [2][Bc][Kc]
  float *pre = reinterpret_cast<float *>(smem + L.pre);  // [Bc][R]
  int *slens = reinterpret_cast<int *>(smem + L.lens);   // [Bc] lengths of the slice's rows
  int *ssoff = reinterpret_cast<int *>(smem + L.soff);   // [T] packed row offset of each step
  uint64_t *hbar = reinterpret_cast<uint64_t *>(smem + L.bar);  // [2] h buffer arrivals
  __shared__ int s_ok;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int grp = lane / 8, gl = lane % 8;

  {  // resident weights (16-byte copies; rows past the last unit are zero)
    const size_t n16 = (size_t)R * Kc * sizeof(WT) / 16;
    const size_t v16 = (size_t)nu * NG * Kc * sizeof(WT) / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(d ? W1 : W0) +
                       (size_t)u0 * NG * Kc * sizeof(WT) / 16;
    uint4 *dst = reinterpret_cast<uint4 *>(Ws);
    for (size_t i = threadIdx.x; i < n16; i += NT)
      dst[i] = i < v16 ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < 2 * Bc * Kc; i += NT) hb[i] = 0.f;
    if (threadIdx.x == 0) {
      tc::mbar_init(&hbar[0], 1);
      tc::mbar_init(&hbar[1], 1);
      tc::fence_mbar_init();
    }
  }
  const int32_t *sidx = p.meta.sorted_idx;
  const int32_t *lens = p.meta.lens_sorted;
  // per-step metadata in shared memory, off the step's critical path
  for (int i = threadIdx.x; i < nrow; i += NT) slens[i] = lens[r0 + i];
  const int32_t *soff = p.meta.step_off;
  if (p.T <= SOFF_MAX) {
    for (int i = threadIdx.x; i < p.T; i += NT) ssoff[i] = soff[i];
    soff = ssoff;
  }
  const int Tcl = nrow > 0 ? lens[r0] : 0;  // steps of the slice (rows sorted by length)
  const int ldo = p.D * Hout;

  // this thread's (row, unit) pair
  const int bq = threadIdx.x / U, jq = threadIdx.x % U;
  const bool own = bq < nrow && jq < nu;
  const int s = r0 + bq, u = u0 + jq;
  int len = 0, borig = 0;
  float c = 0.f, hv = 0.f, bn = 0.f;
  if (own) {
    len = lens[s];
    borig = sidx[s];
    hv = p.h0 ? p.h0[((size_t)d * B + borig) * Hout + u] : 0.f;
    if (NG == 4 && p.c0) c = p.c0[((size_t)d * B + borig) * H + u];
    if (NG == 3 && p.bhn[d]) bn = p.bhn[d][u];
  }
  float gx[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) gx[q] = 0.f;
  auto prefetch = [&](int step) {
    if (!own || step >= len) return;
    const int tt = d == 0 ? step : len - 1 - step;
    const float *g = p.G + ((size_t)soff[tt] + s) * p.ldG + (size_t)d * NG * H + u;
#pragma unroll
    for (int q = 0; q < NG; ++q) gx[q] = __ldg(g + (size_t)q * H);
  };
  // every CTA's h buffers are zeroed, its mbarriers initialised (and the
  // metadata staged) before any peer writes into them
  __syncthreads();
  cl_arrive();
  cl_wait();
  // bytes each buffer receives per step: every active row's H units from the
  // whole cluster
  const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&hbar[0]);
  const uint64_t tmo = p.timeout_ns;
  volatile int never = 0;  // no abort source: only the timeout ends a wait
  if (threadIdx.x == 0 && nrow > 0) tc::mbar_arrive_expect_tx(&hbar[0], (uint32_t)(nrow * H * 4));
  if (own) {
    for (uint32_t q = 0; q < cs; ++q)
      st_async_f32(cl_map(hb + (size_t)bq * Kc + u, q), hv, cl_map(&hbar[0], q));
  }
  prefetch(0);

  // register-resident rows (KQ4 > 0): rows 4*warp + i, K chunks 4*lane + 128*m
  float4 wreg[KQ4 > 0 ? 4 : 1][KQ4 > 0 ? KQ4 : 1];
  if (KQ4 > 0) {
#pragma unroll
    for (int i = 0; i < (KQ4 > 0 ? 4 : 1); ++i) {
      const int r = 4 * warp + i;
#pragma unroll
      for (int m = 0; m < (KQ4 > 0 ? KQ4 : 1); ++m)
        wreg[i][m] = r < R ? wload(Ws + (size_t)r * Kc + 4 * lane + 128 * m)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  int nact = nrow;  // active rows: the prefix of the slice with length > step
  int done = 0;     // steps whose input buffer completed
  for (int step = 0; step < Tcl; ++step) {
    const bool tr = p.trace && blockIdx.x == 0 && threadIdx.x == 0;
    while (nact > 0 && slens[nact - 1] <= step) --nact;
    const int cur = step & 1;
    const float *hcur = hb + (size_t)cur * Bc * Kc;
    float *hnxt = hb + (size_t)(cur ^ 1) * Bc * Kc;
    if (threadIdx.x == 0) {
      // arm the next buffer for this step's sends, then wait for h_{t-1}
      tc::mbar_arrive_expect_tx(&hbar[cur ^ 1], (uint32_t)(nact * H * 4));
      s_ok = tc::mbar_wait(&hbar[cur], (uint32_t)(step >> 1) & 1u, p.err, &never, tmo);
    }
    __syncthreads();
    if (!s_ok) break;
    done = step + 1;
    if (tr) p.trace[step * 16 + 0] = globaltimer_ns();
    // ---- h_{t-1} W_hh^T
    if (KQ4 > 0) {
      // 4 register rows per warp; the 4 lane-partial sums are reduced together
      // (reduce-scatter: 2 + 1 shuffles leave lane l with row 2*bit4 + bit3,
      // then 3 more within 8 lanes)
      const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
      for (int b = 0; b < nact; ++b) {
        const float *hrow = hcur + (size_t)b * Kc + 4 * lane;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < (KQ4 > 0 ? KQ4 : 1); ++m) {
          const float4 x = *reinterpret_cast<const float4 *>(hrow + 128 * m);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[i] = fmaf(wreg[i][m].x, x.x, v[i]);
            v[i] = fmaf(wreg[i][m].y, x.y, v[i]);
            v[i] = fmaf(wreg[i][m].z, x.z, v[i]);
            v[i] = fmaf(wreg[i][m].w, x.w, v[i]);
          }
        }
        const float a0 = (hi16 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, hi16 ? v[0] : v[2], 16);
        const float a1 = (hi16 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, hi16 ? v[1] : v[3], 16);
        float a = (hi8 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, hi8 ? a0 : a1, 8);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        const int r = 4 * warp + (hi16 ? 2 : 0) + (hi8 ? 1 : 0);
        if ((lane & 7) == 0 && r < R) pre[(size_t)b * R + r] = a;
      }
    }
    // 8 lanes per output row (4 rows per warp pass); lane l of a group takes
    // the 16-byte K chunks l, l+8, ...
    for (int b = 0; KQ4 == 0 && b < nact; ++b) {
      const float *hrow = hcur + (size_t)b * Kc + 4 * gl;
      for (int rw = warp * 4; rw < R; rw += NW * 4) {
        const int r = rw + grp;
        float a = 0.f;
        if (r < R) {
          const WT *wr = Ws + (size_t)r * Kc + 4 * gl;
#pragma unroll 4
          for (int m = 0; m < KQ; ++m) {
            const float4 w = wload(wr + 32 * m);
            const float4 x = *reinterpret_cast<const float4 *>(hrow + 32 * m);
            a = fmaf(w.x, x.x, a);
            a = fmaf(w.y, x.y, a);
            a = fmaf(w.z, x.z, a);
            a = fmaf(w.w, x.w, a);
          }
        }
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        if (gl == 0 && r < R) pre[(size_t)b * R + r] = a;
      }
    }
    __syncthreads();
    if (tr) p.trace[step * 16 + 3] = globaltimer_ns();
    // ---- gates and cell update; h_t into every CTA's next-step buffer
    const bool act = own && bq < nact;
    if (act) {
      const float *pr = pre + (size_t)bq * R + (size_t)jq * NG;
      if (NG == 4) {
        const float ig = sigmoid_f(pr[0] + gx[0]);
        const float fg = sigmoid_f(pr[1] + gx[1]);
        const float gg = tanh_f(pr[2] + gx[2]);
        const float og = sigmoid_f(pr[3] + gx[3]);
        c = fg * c + ig * gg;
        if (p.cclip) c = fminf(fmaxf(c, p.cclip_lo), p.cclip_hi);
        hv = og * tanh_f(c);
      } else {
        const float rg = sigmoid_f(gx[0] + pr[0]);
        const float zg = sigmoid_f(gx[1] + pr[1]);
        const float ng = tanh_f(gx[2] + rg * (pr[NG - 1] + bn));
        hv = (1.f - zg) * ng + zg * hv;
      }
      if (tr) p.trace[step * 16 + 4] = globaltimer_ns();
      const uint32_t nb = bar0 + (uint32_t)((cur ^ 1) * 8);
      for (uint32_t q = 0; q < cs; ++q)
        st_async_f32(cl_map(hnxt + (size_t)bq * Kc + u, q), hv, cl_map_addr(nb, q));
    }
    if (tr) p.trace[step * 16 + 1] = globaltimer_ns();
    // outputs and the next step's G loads leave the critical path
    if (act) {
      const int tt = d == 0 ? step : len - 1 - step;
      if (p.y) p.y[((size_t)tt * B + borig) * ldo + (size_t)d * Hout + u] = hv;
      if (p.ymid)
        reinterpret_cast<WT *>(p.ymid)[((size_t)soff[tt] + s) * ldo + (size_t)d * Hout + u] =
            Op<WT>::from_f(hv);
    }
    prefetch(step + 1);
  }
  // The last step's h (or, after a failed wait, the pending one) may still
  // be landing here: wait for it (bounded), and leave only when every CTA of
  // the cluster has stopped sending.
  if (threadIdx.x == 0 && Tcl > 0) {
    const int ph = done;  // the step whose input buffer is still armed
    volatile int keep_waiting = 0;  // (a timed-out wait above has set `never`)
    tc::mbar_wait(&hbar[ph & 1], (uint32_t)(ph >> 1) & 1u, nullptr, &keep_waiting, 100000000ull);
  }
  __syncthreads();
  cl_arrive();
  cl_wait();
  if (own) {
    if (p.h_n) p.h_n[((size_t)d * B + borig) * Hout + u] = hv;
    if (NG == 4 && p.c_n) p.c_n[((size_t)d * B + borig) * H + u] = c;
  }
}

// register-resident rows (widened to fp32) when the CTA has at most 64 gate
// rows and K <= 512
int reg_kq4(int R, int Kc, bool wbf16) {
  (void)wbf16;
  return (R <= 4 * NW && Kc <= 512) ? Kc / 128 : 0;
}

template <typename WT, int NG>
const void *cluster_kernel_t(int kq4) {
  switch (kq4) {
    case 1: return (const void *)rec_cluster_kernel<WT, NG, 1>;
    case 2: return (const void *)rec_cluster_kernel<WT, NG, 2>;
    case 3: return (const void *)rec_cluster_kernel<WT, NG, 3>;
    case 4: return (const void *)rec_cluster_kernel<WT, NG, 4>;
    default: return (const void *)rec_cluster_kernel<WT, NG, 0>;
  }
}
const void *cluster_kernel(int nG, bool wbf16, int kq4) {
  if (wbf16)
    return nG == 4 ? cluster_kernel_t<__nv_bfloat16, 4>(kq4) : cluster_kernel_t<__nv_bfloat16, 3>(kq4);
  return nG == 4 ? cluster_kernel_t<float, 4>(kq4) : cluster_kernel_t<float, 3>(kq4);
}

}  // namespace

int cluster_rec_kc(int Hout) { return round_up(Hout, 128); }

bool cluster_rec_packable(int cell, int H, int Hout, int P, bool wbf16) {
  if (P > 0 || H < 1 || Hout < 1) return false;
  const int Kc = cluster_rec_kc(Hout);
  if (Kc > KC_MAX) return false;
  const int nG = cell == CELL_LSTM ? 4 : 3;
  const int U = ceil_div(H, 16);  // the largest cluster
  return cl_smem(nG * U, Kc, 1, wbf16 ? 2 : 4, 1).total <= (size_t)SMEM_LIMIT;
}

void cluster_pack_whh(int cell, int H, int Hout, const float *whh, std::vector<float> &out) {
  const int nG = cell == CELL_LSTM ? 4 : 3, Kc = cluster_rec_kc(Hout);
  out.assign((size_t)H * nG * Kc, 0.f);
  for (int u = 0; u < H; ++u)
    for (int g = 0; g < nG; ++g)
      for (int k = 0; k < Hout; ++k)
        out[((size_t)u * nG + g) * Kc + k] = whh[(size_t)(g * H + u) * Hout + k];
}

bool plan_recurrent_cluster(ClusterRecPlan *cp, int cell, int H, int Hout, int T, int B, int D,
                            bool wbf16, int max_rows) {
  const int nG = cell == CELL_LSTM ? 4 : 3, Kc = cluster_rec_kc(Hout);
  const size_t es = wbf16 ? 2 : 4;
  for (int cs : {16, 8}) {
    const int U = ceil_div(H, cs);
    const void *fn = cluster_kernel(nG, wbf16, reg_kq4(nG * U, Kc, wbf16));
    if (cs > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                      cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    // the batch slice: as many co-resident clusters as the GPU holds, then
    // the smallest slice that covers B
    const size_t smem1 = cl_smem(nG * U, Kc, 1, es, T).total;
    if (smem1 > (size_t)SMEM_LIMIT - 1024) continue;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) !=
        cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(cs);
    q.blockDim = dim3(NT);
    q.dynamicSmemBytes = smem1;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    q.attrs = a;
    q.numAttrs = 1;
    int maxcl = 0;
    if (cudaOccupancyMaxActiveClusters(&maxcl, fn, &q) != cudaSuccess || maxcl < 1) {
      cudaGetLastError();
      continue;
    }
    const int per_dir = std::max(1, maxcl / D);
    const int Bc = ceil_div(std::max(B, 1), per_dir);
    if (Bc > max_rows || Bc * U > NT) continue;
    const size_t smem = cl_smem(nG * U, Kc, Bc, es, T).total;
    if (smem > (size_t)SMEM_LIMIT - 1024) continue;  // room for the kernel's static shared memory
    cp->cs = cs;
    cp->U = U;
    cp->Kc = Kc;
    cp->Bc = Bc;
    cp->NCL = ceil_div(std::max(B, 1), Bc);
    cp->smem = smem;
    return true;
  }
  return false;
}

cudaError_t launch_recurrent_cluster(const RecParams &p, const ClusterRecPlan &cp,
                                     const void *W0, const void *W1, bool wbf16, cudaStream_t s) {
  const void *fn = cluster_kernel(p.nG, wbf16, reg_kq4(p.nG * cp.U, cp.Kc, wbf16));
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)cp.smem);
  if (e != cudaSuccess) return e;
  if (cp.cs > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * cp.NCL * cp.cs);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = cp.smem;
  cfg.stream = s;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = cp.cs;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  RecParams pc = p;
  int U = cp.U, Kc = cp.Kc, Bc = cp.Bc, NCL = cp.NCL, cs = cp.cs;
  void *args[] = {&pc, const_cast<void **>(&W0), const_cast<void **>(&W1), &U, &Kc, &Bc, &NCL,
                  &cs};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace rcu
