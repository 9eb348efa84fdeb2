// Time-parallel input projection on the 5th-generation tensor cores:
//   G[m, n] = sum_k X[m, k] * W[n, k] + bias[n]   (or + bias[m])
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
// MMAs of tile i+1.  Every mbarrier wait is bounded.  Tiles are rastered so
// the operand with fewer tiles varies fastest.  The same kernel runs batched
// products (3-D tensor maps) and split-K partials (K cut into chunks, each
// chunk's product to its own output plane, summed afterwards in order).
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

// 3-D TMA load of a box at (x, y, z) (a batch of matrices: z = the batch)
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(tc::smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(tc::smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// BATCH: nb independent products G_b = A_b B_b^T (b < nb, the maps' third
// dimension; G_b at G + b * strideG), their tiles spread over one launch
template <bool BATCH>
__global__ void __launch_bounds__(NT, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float *__restrict__ bias, float *__restrict__ G, int ldg, int M,
                   const int32_t *__restrict__ M_dev, int N, int K, int *err,
                   uint64_t timeout_ns, int nb, long long strideG, int bias_rows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  float *stg_all = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
  Bars *bars = reinterpret_cast<Bars *>(smem + STAGES * STAGE_BYTES + EPI_WARPS * STG_FLOATS * 4);

  if (M_dev) M = *M_dev;
  const int tiles_n = ceil_div(N, BN), tiles_m = ceil_div(M, BM);
  const int ntiles1 = tiles_m * tiles_n;                   // tiles of one product
  // raster: the operand with fewer tiles varies fastest, so that the CTAs
  // running at once share the other operand's tiles and the smaller operand
  // stays in L2 (each tile of the larger one is read once)
  const bool m_fast = tiles_m < tiles_n;
  // without BATCH, nb > 1 cuts K into nb chunks of nkbc blocks: chunk c's
  // product goes to G + c * strideG (a split-K partial)
  const bool ksplit = !BATCH && nb > 1;
  const int ntiles = ntiles1 * (BATCH || ksplit ? nb : 1);
  const int nkb = ceil_div(K, BK);
  const int nkbc = ksplit ? ceil_div(nkb, nb) : nkb;
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
        const int bt = tile / ntiles1, t1 = tile % ntiles1;
        const int tm = m_fast ? t1 % tiles_m : t1 / tiles_n;
        const int tn = m_fast ? t1 / tiles_m : t1 % tiles_n;
        const int kb0 = ksplit ? bt * nkbc : 0, kb1 = ksplit ? min(nkb, kb0 + nkbc) : nkb;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(&bars->empty[stage], phase ^ 1, err, abort, timeout_ns)) goto done;
          tc::mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
          if (BATCH) {
            tma_load_3d(sA + stage * A_BYTES, &tmA, &bars->full[stage], kb * BK, tm * BM, bt);
            tma_load_3d(sB + stage * B_BYTES, &tmB, &bars->full[stage], kb * BK, tn * BN, bt);
          } else {
            tc::tma_load_2d(sA + stage * A_BYTES, &tmA, &bars->full[stage], kb * BK, tm * BM);
            tc::tma_load_2d(sB + stage * B_BYTES, &tmB, &bars->full[stage], kb * BK, tn * BN);
          }
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
        const int bt = tile / ntiles1;
        const int kb0 = ksplit ? bt * nkbc : 0, kb1 = ksplit ? min(nkb, kb0 + nkbc) : nkb;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(&bars->full[stage], phase, err, abort, timeout_ns)) goto done;
          tc::tc_fence_after();
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(d, tc::smem_desc_sw128(a0 + kk * 32), tc::smem_desc_sw128(b0 + kk * 32),
                         idesc, (kb != kb0 || kk != 0));
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
      const int bt = tile / ntiles1, t1 = tile % ntiles1;
      const int tm = m_fast ? t1 % tiles_m : t1 / tiles_n;
      const int tn = m_fast ? t1 / tiles_m : t1 % tiles_n;
      float *Gb = (BATCH || ksplit) ? G + (size_t)bt * strideG : G;
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
        if (bias && !bias_rows && n < N) b4 = *reinterpret_cast<const float4 *>(bias + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = i * 4 + (lane >> 3);
          float4 f = *reinterpret_cast<const float4 *>(stg + r * 32 + ((cl ^ (r & 7)) * 4));
          const int m = row0 + r;
          if (bias_rows && bias && m < M) b4.x = b4.y = b4.z = b4.w = bias[m];
          f.x += b4.x; f.y += b4.y; f.z += b4.z; f.w += b4.w;
          if (m < M && n < N) *reinterpret_cast<float4 *>(Gb + (size_t)m * ldg + n) = f;
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

// The same over a batch of nb such matrices, rstride rows apart (3-D map:
// x = column, y = row, z = batch; box 64 columns x box_rows rows x 1)
bool make_map_batch(CUtensorMap *map, const void *base, int rows, int cols, int ld,
                    long long rstride, int nb, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)rstride * ld * 2};
  cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr() {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute((const void *)gemm_tc_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute((const void *)gemm_tc_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)SMEM_BYTES);
  });
  return attr_err;
}

// nb products G_b = X_b W_b^T (X_b: rows [b*rsx, b*rsx + M) of X, W_b: rows
// [b*rsw, b*rsw + N) of W; G_b at G + b*strideG), no bias, in one launch
cudaError_t launch_tc_gemm_batched(const __nv_bfloat16 *X, int ldx, long long rsx,
                                   const __nv_bfloat16 *W, int ldw, long long rsw, float *G,
                                   int ldg, long long strideG, int M, int N, int K, int nb,
                                   int nsm, cudaStream_t s, int *err, uint64_t timeout_ns) {
  if (M <= 0 || N <= 0 || nb <= 0) return cudaSuccess;
  if ((ldx % 8) || (ldw % 8) || (ldg % 4) || (strideG % 4) ||
      (reinterpret_cast<uintptr_t>(X) % 16) || (reinterpret_cast<uintptr_t>(W) % 16) ||
      (reinterpret_cast<uintptr_t>(G) % 16))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map_batch(&ma, X, M, K, ldx, rsx, nb, BM) ||
      !make_map_batch(&mb, W, N, K, ldw, rsw, nb, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr();
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)ceil_div(M, BM) * ceil_div(N, BN) * nb;
  const int grid = (int)std::min<long long>(tiles, nsm);
  gemm_tc_kernel<true><<<grid, NT, SMEM_BYTES, s>>>(ma, mb, nullptr, G, ldg, M, nullptr, N, K,
                                                    err, timeout_ns, nb, strideG, 0);
  return cudaGetLastError();
}

}  // namespace

bool tc_gemm_supported(int K, int N) { return K >= 1 && N >= 1 && N % 4 == 0 && encode_fn(); }

namespace {
// Three-term bf16 split of an fp32 matrix R x C (row stride ld) into six
// K segments of kp columns per row (dst row stride 6*kp), in the order that
// pairs operand A's terms with operand B's: products a1b2, a2b1, a1b3, a2b2,
// a3b1, then a1b1 (pattern 0 = A: x1 x2 x1 x2 x3 x1; pattern 1 = B: x2 x1
// x3 x2 x1 x1).  The five small products come first, while the accumulator
// is still small, so their additions round at their own scale and the sum
// carries the rounding of the K large additions only, as an FFMA loop does.
// x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2): both residuals
// are exact in fp32, so x - (x1 + x2 + x3) is within 2^-24 |x|.  Columns past
// a chunk's width are written as zero.
// One launch splits every K chunk of an operand: chunk c = blockIdx.y takes
// columns [c*kc, min(K, c*kc + kc)) of rows r < R into dst + (c*Rr + r)*6*kp.
// Each thread splits 8 consecutive columns and writes each of the six
// segments as one 16-byte store (kp is a multiple of 8).
__global__ void split3_kernel(const float *__restrict__ src, int R, int K, int ld, int kc,
                              int Rr, __nv_bfloat16 *__restrict__ dst, int kp, int pattern) {
  const int ch = blockIdx.y, k0 = ch * kc, kw = min(kc, K - k0);
  const bool v4 = (ld % 4) == 0 && (k0 % 4) == 0 && (reinterpret_cast<uintptr_t>(src) % 16) == 0;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const float *sr = src + (size_t)r * ld + k0;
    __nv_bfloat16 *o = dst + ((size_t)ch * Rr + r) * 6 * kp;
    for (int c8 = threadIdx.x * 8; c8 < kp; c8 += blockDim.x * 8) {
      float x[8];
      if (v4 && c8 + 8 <= kw) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(sr + c8));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(sr + c8 + 4));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = c8 + q < kw ? sr[c8 + q] : 0.f;
      }
      uint4 t1, t2, t3;
      uint32_t *p1 = reinterpret_cast<uint32_t *>(&t1), *p2 = reinterpret_cast<uint32_t *>(&t2),
               *p3 = reinterpret_cast<uint32_t *>(&t3);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __nv_bfloat16 a1[2], a2[2], a3[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float v = x[2 * q + h];
          a1[h] = __float2bfloat16_rn(v);
          const float r1 = v - __bfloat162float(a1[h]);
          a2[h] = __float2bfloat16_rn(r1);
          a3[h] = __float2bfloat16_rn(r1 - __bfloat162float(a2[h]));
        }
        p1[q] = (uint32_t)__bfloat16_as_ushort(a1[0]) | ((uint32_t)__bfloat16_as_ushort(a1[1]) << 16);
        p2[q] = (uint32_t)__bfloat16_as_ushort(a2[0]) | ((uint32_t)__bfloat16_as_ushort(a2[1]) << 16);
        p3[q] = (uint32_t)__bfloat16_as_ushort(a3[0]) | ((uint32_t)__bfloat16_as_ushort(a3[1]) << 16);
      }
      uint4 *ov = reinterpret_cast<uint4 *>(o + c8);
      const size_t sg = (size_t)kp / 8;  // one segment, in 16-byte units
      if (pattern == 0) {
        ov[0] = t1; ov[sg] = t2; ov[2 * sg] = t1; ov[3 * sg] = t2; ov[4 * sg] = t3; ov[5 * sg] = t1;
      } else {
        ov[0] = t2; ov[sg] = t1; ov[2 * sg] = t3; ov[3 * sg] = t2; ov[4 * sg] = t1; ov[5 * sg] = t1;
      }
    }
  }
}
// C[m][n] = sum over the nch chunk partials P[c][m][n] (row stride ldp) in
// chunk order, plus bias[n]
__global__ void sum_parts_kernel(const float *__restrict__ P, int nch, int M, int N, int ldp,
                                 const float *__restrict__ bias, float *__restrict__ C, int ldc) {
  const size_t plane = (size_t)M * ldp;
  for (int m = blockIdx.x; m < M; m += gridDim.x)
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      float a = bias ? bias[n] : 0.f;
      for (int c = 0; c < nch; ++c) a += P[c * plane + (size_t)m * ldp + n];
      C[(size_t)m * ldc + n] = a;
    }
}
}  // namespace

// Reductions longer than this are cut into chunks whose partial products
// are summed in fp32 afterwards (blocked summation: the tensor cores
// accumulate a chunk in one fp32 accumulator, and a 32,000-term reduction in
// one accumulator measured 4e-5 relative against FFMA's blocked 9e-7)
constexpr int F32X6_KCHUNK = 4096;

bool f32x6_supported(int N, int ldc, const void *C) {
  return N >= 1 && N % 4 == 0 && ldc % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0 &&
         encode_fn();
}

size_t f32x6_scratch_bytes(int M, int N, int K) {
  const int nch = ceil_div(K, F32X6_KCHUNK);
  const size_t kp = (size_t)round_up(nch > 1 ? F32X6_KCHUNK : K, 8);
  size_t b = (size_t)nch * ((size_t)round_up(M, 8) + (size_t)round_up(N, 8)) * 6 * kp * 2 + 256;
  if (nch > 1) b += (size_t)nch * M * round_up(N, 4) * 4 + 256;  // the chunk partials
  return b;
}

int f32x6_launches(int K) {
  const int nch = ceil_div(K, F32X6_KCHUNK);
  return nch > 1 ? 4 : 3;
}

cudaError_t launch_gemm_f32x6(const float *A, int lda, const float *B, int ldb, const float *bias,
                              float *C, int ldc, int M, const int32_t *M_dev, int N, int K,
                              void *scratch, int nsm, cudaStream_t s, int *err,
                              uint64_t timeout_ns) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int nch = ceil_div(K, F32X6_KCHUNK);
  if (nch > 1 && M_dev) return cudaErrorInvalidValue;  // (a device-side M: short K only)
  const int kc = nch > 1 ? F32X6_KCHUNK : K, kp = round_up(kc, 8);
  const long long Mr = round_up(M, 8), Nr = round_up(N, 8);
  // chunk c's splits: As rows [c*Mr, c*Mr + M), Bs rows [c*Nr, c*Nr + N)
  __nv_bfloat16 *As = reinterpret_cast<__nv_bfloat16 *>(scratch);
  __nv_bfloat16 *Bs = As + (size_t)nch * Mr * 6 * kp;
  {
    const int thr = std::min(256, round_up(kp / 8, 32));
    split3_kernel<<<dim3(std::min(M, 65535), nch), thr, 0, s>>>(A, M, K, lda, kc, (int)Mr, As, kp, 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    split3_kernel<<<dim3(std::min(N, 65535), nch), thr, 0, s>>>(B, N, K, ldb, kc, (int)Nr, Bs, kp, 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (nch == 1)
    return launch_tc_gemm(As, 6 * kp, Bs, 6 * kp, bias, C, ldc, M, M_dev, N, 6 * kp, nsm, s, err,
                          timeout_ns);
  // the chunks' products side by side in one launch (a long reduction over a
  // small output has too few tiles to fill the GPU on its own), then their
  // fp32 sum in chunk order
  const int ldp = round_up(N, 4);
  float *P = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(Bs + (size_t)nch * Nr * 6 * kp) + 255) & ~uintptr_t(255));
  cudaError_t e = launch_tc_gemm_batched(As, 6 * kp, Mr, Bs, 6 * kp, Nr, P, ldp,
                                         (long long)M * ldp, M, N, 6 * kp, nch, nsm, s, err,
                                         timeout_ns);
  if (e != cudaSuccess) return e;
  sum_parts_kernel<<<std::min(M, 65535), 256, 0, s>>>(P, nch, M, N, ldp, bias, C, ldc);
  return cudaGetLastError();
}

// K chunks for a long reduction over few output tiles: the count (at most
// 4) that minimises the waves of tiles times the chunk length, the smallest
// on a tie; 1 when the tiles fill the GPU or K is short
int tc_gemm_splitk_chunks(int M, int N, int K, int nsm) {
  const long long tiles = (long long)ceil_div(M, BM) * ceil_div(N, BN);
  const int nkb = ceil_div(K, BK);
  if (nsm < 1 || tiles >= nsm || nkb < 64) return 1;
  int best = 1;
  double best_cost = (double)ceil_div(tiles, (long long)nsm);
  for (int c = 2; c <= 4; ++c) {
    const int nkbc = ceil_div(nkb, c);
    if ((c - 1) * nkbc >= nkb) break;  // every chunk holds K blocks
    const double cost = (double)ceil_div(tiles * c, (long long)nsm) * nkbc / nkb;
    if (cost < best_cost - 1e-9) { best = c; best_cost = cost; }
  }
  return best;
}

size_t tc_gemm_splitk_scratch_floats(int M, int N, int K, int nsm) {
  const int c = tc_gemm_splitk_chunks(M, N, K, nsm);
  return c > 1 ? (size_t)c * M * round_up(N, 4) : 0;
}

cudaError_t launch_tc_gemm_splitk(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W,
                                  int ldw, const float *bias, float *G, int ldg, int M, int N,
                                  int K, float *scratch, int nsm, cudaStream_t s, int *err,
                                  uint64_t timeout_ns, int *launches) {
  const int c = tc_gemm_splitk_chunks(M, N, K, nsm);
  if (c == 1) {
    if (launches) *launches = 1;
    return launch_tc_gemm(X, ldx, W, ldw, bias, G, ldg, M, nullptr, N, K, nsm, s, err,
                          timeout_ns);
  }
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int ldp = round_up(N, 4);
  if ((ldx % 8) || (ldw % 8) || (reinterpret_cast<uintptr_t>(X) % 16) ||
      (reinterpret_cast<uintptr_t>(W) % 16) || (reinterpret_cast<uintptr_t>(scratch) % 16))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map(&ma, X, M, K, ldx, BM) || !make_map(&mb, W, N, K, ldw, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr();
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)ceil_div(M, BM) * ceil_div(N, BN) * c;
  const int grid = (int)std::min<long long>(tiles, nsm);
  gemm_tc_kernel<false><<<grid, NT, SMEM_BYTES, s>>>(ma, mb, nullptr, scratch, ldp, M, nullptr,
                                                      N, K, err, timeout_ns, c,
                                                      (long long)M * ldp, 0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sum_parts_kernel<<<std::min(M, 65535), 256, 0, s>>>(scratch, c, M, N, ldp, bias, G, ldg);
  if (launches) *launches = 2;
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W, int ldw,
                           const float *bias, float *G, int ldg, int M, const int32_t *M_dev,
                           int N, int K, int nsm, cudaStream_t s, int *err, uint64_t timeout_ns,
                           bool bias_rows) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if ((ldx % 8) || (ldw % 8) || (ldg % 4) || (reinterpret_cast<uintptr_t>(X) % 16) ||
      (reinterpret_cast<uintptr_t>(W) % 16) || (reinterpret_cast<uintptr_t>(G) % 16))
    return cudaErrorInvalidValue;
  // the epilogue stores 4 columns at a time: a ragged N needs its row padded
  // to a multiple of 4 and no per-column bias to read past N
  if (N % 4 && (ldg < N + (4 - N % 4) || (bias && !bias_rows))) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map(&ma, X, M, K, ldx, BM) || !make_map(&mb, W, N, K, ldw, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr();
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)ceil_div(M, BM) * ceil_div(N, BN);
  const int grid = (int)std::min<long long>(tiles, nsm);
  gemm_tc_kernel<false><<<grid, NT, SMEM_BYTES, s>>>(ma, mb, bias, G, ldg, M, M_dev, N, K, err,
                                                      timeout_ns, 1, 0, bias_rows ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace rcu
