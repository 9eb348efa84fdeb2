// Helpers of the projected-LSTM (LSTMP) tensor-core path.
//
// With a projection, the recurrent input is h_{t-1} = W_hr m_{t-1}
// ("Integrating CuDNN API for LSTMs with projections", pytorch/pytorch issue
// 46213: the projection is one more matmul on the cell's hidden output), so
//     W_hh h_{t-1} = (W_hh W_hr) m_{t-1}.
// The tensor-core path keeps the product W' = W_hh W_hr resident and runs the
// recurrence on m; the projection of every m_t then happens after the
// sequential loop as one large GEMM.  What remains are two small kernels:
// the initial state's contribution W_hh h0 to the first step's gate
// pre-activations, and the final projected state h_n.
#include "common.cuh"
#include "internal.h"

namespace rcu {

namespace {

// G[row(s), d*4H + r] += sum_k W_hh[r, k] * h0[s, k] for the row of each
// sequence's first step (forward: t = 0; backward: t = T-1); no lengths.
__global__ void h0_gate_kernel(float *G, int ldG, const float *Whh, const float *h0, int B, int T,
                               int H4, int P, int d) {
  const int s = blockIdx.y;
  const int t = d == 0 ? 0 : T - 1;
  const float *hv = h0 + (size_t)s * P;
  float *g = G + ((size_t)t * B + s) * ldG + (size_t)d * H4;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < H4; r += gridDim.x * blockDim.x) {
    const float *w = Whh + (size_t)r * P;
    float a = 0.f;
    for (int k = 0; k < P; ++k) a = fmaf(w[k], hv[k], a);
    g[r] += a;
  }
}

// h_n[d, b, :] = Y[t_last * B + b, d*P : d*P + P] (forward t_last = T-1,
// backward t_last = 0); no lengths.
__global__ void last_h_kernel(const float *Y, int ldY, float *h_n, int B, int T, int P, int d) {
  const int b = blockIdx.x;
  const int t = d == 0 ? T - 1 : 0;
  for (int k = threadIdx.x; k < P; k += blockDim.x)
    h_n[(size_t)b * P + k] = Y[((size_t)t * B + b) * ldY + (size_t)d * P + k];
}

}  // namespace

cudaError_t launch_h0_gates(float *G, int ldG, const float *Whh, const float *h0, int B, int T,
                            int H4, int P, int d, cudaStream_t s) {
  dim3 grid((H4 + 255) / 256, B);
  h0_gate_kernel<<<grid, 256, 0, s>>>(G, ldG, Whh, h0, B, T, H4, P, d);
  return cudaGetLastError();
}

cudaError_t launch_last_h(const float *Y, int ldY, float *h_n, int B, int T, int P, int d,
                          cudaStream_t s) {
  last_h_kernel<<<B, 128, 0, s>>>(Y, ldY, h_n, B, T, P, d);
  return cudaGetLastError();
}

}  // namespace rcu
