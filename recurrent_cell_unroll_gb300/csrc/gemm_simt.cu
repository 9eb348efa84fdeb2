// Portable CUDA-core GEMM for the time-parallel input projection
// G = X W_ih^T + b over all timesteps at once (the "initial input-hidden
// dense" of "[TOPI] TE implementation of LSTM using scan", apache/tvm PR
// 11531).  Used for the fp32 path (fp32 FFMA keeps full single precision)
// and as the portable fallback of the bf16 path.
//
// Tile 128x128x16, 256 threads, 8x8 outputs per thread, double-buffered
// shared memory.  Operands may be fp32 or bf16; accumulation is fp32.
// When the output tiles are too few to fill the GPU (short sequences, small
// batches) K is split over a thread-block cluster of S CTAs along z: each
// parks its partial tile in shared memory and rank z sums rows [z*128/S,
// (z+1)*128/S) of all S partials over distributed shared memory, in rank
// order, so the result does not depend on timing.
#include "common.cuh"
#include "internal.h"

namespace rcu {

namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;

template <typename T>
__device__ __forceinline__ float ldf(const T *p) { return Op<T>::load(p); }

template <typename XT, typename WT>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const XT *__restrict__ X, int ldx,
                                                       const WT *__restrict__ W, int ldw,
                                                       const float *__restrict__ bias,
                                                       float *__restrict__ G, int ldg, int M,
                                                       const int32_t *__restrict__ M_dev, int N,
                                                       int K, int kchunk, int *err) {
  if (gridDim.z > 1) {
    uint32_t ncta;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    if (ncta != gridDim.z) {  // the K slices must share one cluster
      if (err && threadIdx.x == 0) atomicCAS(err, DEV_OK, DEV_CONFIG);
      return;
    }
  }
  if (M_dev) M = *M_dev;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  // every CTA of a K-split cluster shares (m0, n0), so they leave together
  if (m0 >= M) return;
  const int S = gridDim.z, z = blockIdx.z;
  const int kbeg = z * kchunk, kend = min(K, kbeg + kchunk);
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  const int tid = threadIdx.x;
  // loader mapping: 128 rows x 16 k, each thread 8 consecutive k of one row
  const int lr = tid >> 1, lk = (tid & 1) * 8;
  // compute mapping: 16 x 16 threads, each 8 rows (2 groups of 4) x 8 cols
  const int ty = tid >> 4, tx = tid & 15;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  float ra[8], rb[8];
  auto load_regs = [&](int k0) {
    const int am = m0 + lr, bn = n0 + lr;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int k = k0 + lk + q;
      ra[q] = (am < M && k < kend) ? ldf(X + (size_t)am * ldx + k) : 0.f;
      rb[q] = (bn < N && k < kend) ? ldf(W + (size_t)bn * ldw + k) : 0.f;
    }
  };
  auto store_smem = [&](int buf) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      As[buf][lk + q][lr] = ra[q];
      Bs[buf][lk + q][lr] = rb[q];
    }
  };

  const int nk = kend > kbeg ? ceil_div(kend - kbeg, BK) : 0;
  load_regs(kbeg);
  store_smem(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load_regs(kbeg + (kt + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < nk) store_smem(buf ^ 1);
    __syncthreads();
  }

  if (S > 1) {
    extern __shared__ __align__(16) float Ps[];  // [BM][BN + 4] partial tile
    constexpr int LDP = BN + 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4);
      *reinterpret_cast<float4 *>(&Ps[r * LDP + tx * 4]) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4 *>(&Ps[r * LDP + 64 + tx * 4]) =
          make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
    const int rows = BM / S;
    for (int e = tid; e < rows * (BN / 4); e += NT) {
      const int r = z * rows + e / (BN / 4), c = (e % (BN / 4)) * 4;
      const uint32_t local = (uint32_t)__cvta_generic_to_shared(&Ps[r * LDP + c]);
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < S; ++q) {
        uint32_t ra_;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra_) : "r"(local), "r"(q));
        float4 v;
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                     : "r"(ra_)
                     : "memory");
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
      }
      const int m = m0 + r;
      if (m < M) {
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + c + j;
          if (n < N) G[(size_t)m * ldg + n] = av[j] + (bias ? bias[n] : 0.f);
        }
      }
    }
    // no CTA leaves while a peer may still read its partial tile
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
    return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n < N) G[(size_t)m * ldg + n] = acc[i][j] + (bias ? bias[n] : 0.f);
    }
  }
}

}  // namespace

template <typename XT, typename WT>
cudaError_t launch_gemm_simt(const XT *X, int ldx, const WT *W, int ldw, const float *bias,
                             float *G, int ldg, int M, const int32_t *M_dev, int N, int K,
                             cudaStream_t s, int *err) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid(ceil_div(N, BN), ceil_div(M, BM));
  const int tiles = (int)(grid.x * grid.y);
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  // K split: powers of two up to 8 while the grid stays under two CTAs per SM
  // and every slice keeps at least two K tiles
  int S = 1;
  while (S < 8 && tiles * S * 2 <= 2 * nsm && K >= 2 * BK * (S * 2)) S *= 2;
  const void *fn = (const void *)gemm_simt_kernel<XT, WT>;
  if (S > 1) {
    const int kchunk = round_up(ceil_div(K, S), BK);
    const size_t smem = (size_t)BM * (BN + 4) * 4;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid.x, grid.y, S);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = 1;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = S;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int kc = kchunk;
    void *args[] = {&X, &ldx, &W, &ldw, &bias, &G, &ldg, &M, &M_dev, &N, &K, &kc, &err};
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  gemm_simt_kernel<XT, WT><<<grid, NT, 0, s>>>(X, ldx, W, ldw, bias, G, ldg, M, M_dev, N, K, K,
                                                 err);
  return cudaGetLastError();
}

template cudaError_t launch_gemm_simt<float, float>(const float *, int, const float *, int,
                                                    const float *, float *, int, int,
                                                    const int32_t *, int, int, cudaStream_t, int *);
template cudaError_t launch_gemm_simt<__nv_bfloat16, __nv_bfloat16>(
    const __nv_bfloat16 *, int, const __nv_bfloat16 *, int, const float *, float *, int, int,
    const int32_t *, int, int, cudaStream_t, int *);

}  // namespace rcu
