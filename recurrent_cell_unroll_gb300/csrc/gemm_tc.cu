// Time-parallel input projection on the 5th-generation tensor cores:
//   G[m, n] = sum_k X[m, k] * W[n, k] + bias[n]
// for all timesteps at once (the "initial input-hidden dense" that "[TOPI] TE
// implementation of LSTM using scan", apache/tvm PR 11531, names as the first
// of the LSTM's three dense ops).  bf16 operands, fp32 accumulation in TMEM,
// fp32 output with the bias fused into the epilogue.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 128x64 A and 256x64 B tiles (128-byte swizzle)
//               into a 4-stage shared-memory ring (mbarrier expect-tx);
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma (M=128, N=256, K=16) and commits to mbarriers;
//   warps 2..5  epilogue: tcgen05.ld 32x32 blocks of the accumulator, stage
//               them through a swizzled 4 KB shared buffer per warp, add the
//               bias and write fully coalesced 128-byte rows.
// Two accumulators (2 x 256 columns) let the epilogue of tile i overlap the
// MMAs of tile i+1.  Every mbarrier wait is bounded.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int NT = 64 + 32 * EPI_WARPS;
constexpr int STG_FLOATS = 32 * 32;
constexpr size_t SMEM_BYTES =
    1024 /*alignment slack*/ + (size_t)STAGES * STAGE_BYTES + EPI_WARPS * STG_FLOATS * 4 + 256;
constexpr uint32_t TMEM_COLS = 512;

struct Bars {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], mdone;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(NT, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float *__restrict__ bias, float *__restrict__ G, int ldg, int M,
                   const int32_t *__restrict__ M_dev, int N, int K, int *err,
                   uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  float *stg_all = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
  Bars *bars = reinterpret_cast<Bars *>(smem + STAGES * STAGE_BYTES + EPI_WARPS * STG_FLOATS * 4);

  if (M_dev) M = *M_dev;
  const int tiles_n = ceil_div(N, BN);
  const int ntiles = ceil_div(M, BM) * tiles_n;
  const int nkb = ceil_div(K, BK);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int *abort = &bars->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->tfull[b], 1);
      tc::mbar_init(&bars->tempty[b], EPI_WARPS);
    }
    tc::mbar_init(&bars->mdone, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) tc::tmem_alloc(&bars->tmem_base, TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int tm = tile / tiles_n, tn = tile % tiles_n;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(&bars->empty[stage], phase ^ 1, err, abort, timeout_ns)) goto done;
          tc::mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
          tc::tma_load_2d(sA + stage * A_BYTES, &tmA, &bars->full[stage], kb * BK, tm * BM);
          tc::tma_load_2d(sB + stage * B_BYTES, &tmB, &bars->full[stage], kb * BK, tn * BN);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        if (!tc::mbar_wait(&bars->tempty[acc], acc_phase ^ 1, err, abort, timeout_ns)) goto done;
        tc::tc_fence_after();
        const uint32_t d = tbase + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(&bars->full[stage], phase, err, abort, timeout_ns)) goto done;
          tc::tc_fence_after();
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(d, tc::smem_desc_sw128(a0 + kk * 32), tc::smem_desc_sw128(b0 + kk * 32),
                         idesc, (kb | kk) != 0);
          tc::mma_commit(&bars->empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        tc::mma_commit(&bars->tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
    }
  } else {
    const int q = warp % 4;  // TMEM lane quarter this warp may access
    float *stg = stg_all + (warp - 2) * STG_FLOATS;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int cl = lane & 7;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int tm = tile / tiles_n, tn = tile % tiles_n;
      if (!tc::mbar_wait(&bars->tfull[acc], acc_phase, err, abort, timeout_ns)) goto done;
      tc::tc_fence_after();
      const int row0 = tm * BM + q * 32;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int nc = tn * BN + c * 32;
        if (nc >= N) break;  // warp-uniform
        float v[32];
        tc::tmem_ld_32x32b_x32(tbase + (uint32_t)(acc * BN + c * 32) + ((uint32_t)(q * 32) << 16),
                               v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4 *>(stg + lane * 32 + ((j ^ (lane & 7)) * 4)) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        __syncwarp();
        const int n = nc + cl * 4;
        float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias && n < N) b4 = *reinterpret_cast<const float4 *>(bias + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = i * 4 + (lane >> 3);
          float4 f = *reinterpret_cast<const float4 *>(stg + r * 32 + ((cl ^ (r & 7)) * 4));
          f.x += b4.x; f.y += b4.y; f.z += b4.z; f.w += b4.w;
          const int m = row0 + r;
          if (m < M && n < N) *reinterpret_cast<float4 *>(G + (size_t)m * ldg + n) = f;
        }
        __syncwarp();
      }
      tc::tc_fence_before();
      if (lane == 0) tc::mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }
done:
  if (warp == 1 && lane == 0) {
    // drain: every MMA issued completes before TMEM is released
    tc::mma_commit(&bars->mdone);
    volatile int never = 0;
    tc::mbar_wait(&bars->mdone, 0, nullptr, &never, 100000000ull);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tbase, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows][ld] matrix of which the first
// `cols` columns are valid; box = 64 columns x box_rows rows, 128-byte swizzle,
// out-of-range elements read as zero.
bool make_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_gemm_supported(int K, int N) { return K >= 1 && N >= 1 && N % 4 == 0 && encode_fn(); }

cudaError_t launch_tc_gemm(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W, int ldw,
                           const float *bias, float *G, int ldg, int M, const int32_t *M_dev,
                           int N, int K, int nsm, cudaStream_t s, int *err, uint64_t timeout_ns) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if ((ldx % 8) || (ldw % 8) || (ldg % 4) || (reinterpret_cast<uintptr_t>(X) % 16) ||
      (reinterpret_cast<uintptr_t>(W) % 16) || (reinterpret_cast<uintptr_t>(G) % 16))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map(&ma, X, M, K, ldx, BM) || !make_map(&mb, W, N, K, ldw, BN))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute((const void *)gemm_tc_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long tiles = (long long)ceil_div(M, BM) * ceil_div(N, BN);
  const int grid = (int)std::min<long long>(tiles, nsm);
  gemm_tc_kernel<<<grid, NT, SMEM_BYTES, s>>>(ma, mb, bias, G, ldg, M, M_dev, N, K, err,
                                               timeout_ns);
  return cudaGetLastError();
}

}  // namespace rcu
