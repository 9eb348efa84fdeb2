// Tensor-core (tcgen05 / TMEM / TMA) kernels of the bf16 path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include <cuda.h>

#include "internal.h"

namespace rcu {

// ---- gemm_tc.cu: G[m, n] = sum_k X[m, k] W[n, k] + bias[n], bf16 operands,
// fp32 accumulate in TMEM, fp32 output.  ldx, ldw in elements (multiples of 8).
// bias_rows: + bias[m] instead (then N needs no multiple of 4 when ldg holds
// N rounded up to one).
bool tc_gemm_supported(int K, int N);
cudaError_t launch_tc_gemm(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W, int ldw,
                           const float *bias, float *G, int ldg, int M, const int32_t *M_dev,
                           int N, int K, int nsm, cudaStream_t s, int *err, uint64_t timeout_ns,
                           bool bias_rows = false);

// The same product with K cut into chunks when the output tiles alone cannot
// fill the GPU (a weight gradient: a long reduction over a small output):
// the chunks' fp32 partials go to scratch (tc_gemm_splitk_scratch_floats)
// and are summed in chunk order, plus bias[n].  *launches = kernels launched.
int tc_gemm_splitk_chunks(int M, int N, int K, int nsm);
size_t tc_gemm_splitk_scratch_floats(int M, int N, int K, int nsm);
cudaError_t launch_tc_gemm_splitk(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W,
                                  int ldw, const float *bias, float *G, int ldg, int M, int N,
                                  int K, float *scratch, int nsm, cudaStream_t s, int *err,
                                  uint64_t timeout_ns, int *launches);

// fp32-accurate C = A B^T + bias on the tensor cores for fp32 operands (row
// strides lda, ldb): each operand is split into three bf16 terms and the six
// products whose terms carry at least 2^-24 of the result are summed in one
// bf16 GEMM over a six-segment K, after "Leveraging the bfloat16 artificial
// intelligence datatype for higher-precision computations" (Henry, Tang,
// Heinecke, ARITH 2019), the five small products first.  Reductions longer
// than 4096 are cut into chunks whose fp32 partials are summed afterwards in
// a fixed order.  It needs f32x6_scratch_bytes of device scratch and
// f32x6_launches kernels (the two operands' splits, the GEMM, and with
// several chunks the ordered sum).
bool f32x6_supported(int N, int ldc, const void *C);
size_t f32x6_scratch_bytes(int M, int N, int K);
int f32x6_launches(int K);
cudaError_t launch_gemm_f32x6(const float *A, int lda, const float *B, int ldb, const float *bias,
                              float *C, int ldc, int M, const int32_t *M_dev, int N, int K,
                              void *scratch, int nsm, cudaStream_t s, int *err,
                              uint64_t timeout_ns);

// ---- recurrent_tc.cu: persistent recurrent kernel with the per-step
// h W_hh^T on tcgen05.
struct TcRecParams {
  RecParams base;
  const void *Wtc[2];  // tensor-core packed W_hh per direction (tc_pack_whh)
  int ksplit = 0;      // CTAs splitting K: 0 = automatic (2), 1 = none, 2 or 4 = a cluster
  bool fixed_length = false;  // no lengths: every row runs every step (tiled G and outputs)
};
// weights can be packed for the tensor-core kernel (shape only)
bool tc_rec_packable(int cell, int H, int Hout, int P);
// the kernel can run this forward (co-resident grid for B rows, D directions)
bool tc_rec_supported(int cell, int H, int Hout, int P, int nsm, int B, int D);
// barrier counter words one layer needs (each counter on its own 128-byte line)
int tc_rec_counters(int B, int D);
// CTAs of the kernel's first-choice plan (K split as requested or automatic)
int tc_rec_grid(int cell, int H, int Hout, int B, int D, int ksplit);
void tc_pack_whh(int cell, int H, int Hout, const float *whh, std::vector<uint16_t> &out,
                 uint16_t (*to_bf16)(float));
cudaError_t launch_tc_recurrent(const TcRecParams &p, int nsm, cudaStream_t s);

// Shared host helpers of the tcgen05 kernels: a 2D bf16 tensor map with
// 128-byte swizzle (box 64 columns x box_rows rows; row stride ld elements,
// a multiple of 8), and a cooperative launch of `grid` CTAs of a kernel that
// declares its own cluster shape of `cs` CTAs (false, nothing launched, when
// that cluster grid cannot be resident at once).
bool tc_map_2d(CUtensorMap *map, const void *base, long long rows, int cols, int ld, int box_rows);
bool tc_launch_clustered(const void *fn, int grid, int nthreads, int cs, size_t smem, void **args,
                         cudaStream_t s, cudaError_t *err);

// ---- bwd_tc.cu: the reverse-time recurrence of the GRU backward pass with
// the per-step W_hh^T dR_t on tcgen05 (bf16 handles, fixed-length batches).
// Per reverse step t it forms dh_t = dy_t + z_{t+1} dh_{t+1} + W_hh^T dR_{t+1}
// (dh_{T-1} = dy_{T-1} + dh_n), the gate gradients of step t (DA: input side,
// DR: hidden side, fp32, every row), publishes dR_t as the next step's bf16
// MMA operand, and finally dh0 = z_0 dh_0 + W_hh^T dR_0.
struct TcBwdParams {
  int T, B, H;
  // the per-step inputs, transposed (column t*B + b, row stride ldz, a
  // multiple of 4 >= T*B) so that a warp's 32 batch rows are 128 contiguous
  // bytes of one row
  const float *zin;    // [3H][ldz]: input-side pre-activations (X W_ih^T + b_ih)^T
  const float *zh;     // [3H][ldz]: hidden-side pre-activations (H_prev W_hh^T + b_hh)^T
  const float *hp;     // [H][ldz]: h_{t-1}^T
  const float *dy;     // [H][ldz]: dy^T
  int ldz;
  const float *dhn;    // [B][H] or NULL
  float *DA, *DR;      // [T*B][3H] fp32, or NULL
  // the same gradients as the tensor-core GEMMs after the loop read them, or
  // NULL: DA^T and DR^T in bf16 ([3H][ldt], ldt a multiple of 8 >= T*B; the
  // weight-gradient operands), DA in bf16 ([T*B][ldab]; the input-gradient
  // operand), and the column sums of DA and DR over each batch group's rows
  // ([2][ceil(B/128)][3H] fp32, in a fixed order: the bias gradients)
  __nv_bfloat16 *dat, *drt;
  int ldt;
  __nv_bfloat16 *dab;
  int ldab;
  float *bsum;
  float *dh0;          // [B][H] or NULL
  __nv_bfloat16 *xdr;  // [2][B][Kx]: dR_t exchange, bf16 (buffer t & 1)
  int Kx;              // its row stride (a multiple of 8, >= 3H)
  const __nv_bfloat16 *wt;  // [H][Kx]: W_hh^T, bf16
  unsigned *ctr;       // step counters (tc_bwd_counters words, zeroed)
  int *err;
  uint64_t timeout_ns;
  int drop_arrival;
  unsigned long long *trace;  // NULL, or [T+1][16] global-timer stamps of CTA 0
};
bool tc_bwd_supported(int H, int B, int nsm);
int tc_bwd_counters(int B);
cudaError_t launch_tc_bwd(const TcBwdParams &p, int nsm, cudaStream_t s);

}  // namespace rcu
