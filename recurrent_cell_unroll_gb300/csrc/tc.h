// Tensor-core (tcgen05 / TMEM / TMA) kernels of the bf16 path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "internal.h"

namespace rcu {

// ---- gemm_tc.cu: G[m, n] = sum_k X[m, k] W[n, k] + bias[n], bf16 operands,
// fp32 accumulate in TMEM, fp32 output.  ldx, ldw in elements (multiples of 8).
bool tc_gemm_supported(int K, int N);
cudaError_t launch_tc_gemm(const __nv_bfloat16 *X, int ldx, const __nv_bfloat16 *W, int ldw,
                           const float *bias, float *G, int ldg, int M, const int32_t *M_dev,
                           int N, int K, int nsm, cudaStream_t s, int *err, uint64_t timeout_ns);

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

}  // namespace rcu
