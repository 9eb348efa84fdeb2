// One-layer fp32 LSTM forward that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code running inside a host framework
// that owns the device heap and hands out no allocator, processes whose
// device-memory budget is fixed up front, or latency-critical loops where an
// allocation (which may synchronise the device or fail under memory
// pressure) is not acceptable.  rnn_lstm_forward_noalloc serves them: the
// caller passes inputs, weights and outputs, and every piece of temporary
// memory comes from the file-scope device array below, which each GPU that
// loads this library holds until the process exits.
//
// Scratch layout (floats): summed bias [4H] | input projection G [T*B*4H] |
// exchange h [2*B*H] | state h [B*H] | state c [B*H] | control (counter,
// error word).  Every call overwrites it; calls that overlap on the GPU
// (for example on two streams at once) race on it.
#include <cstdio>
#include <mutex>

#include "rcu.h"
#include "common.cuh"
#include "internal.h"

namespace rcu {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RCU_NOALLOC_SCRATCH_BYTES];

constexpr int NT = 256;
constexpr int MAX_DEVICES = 64;

// Host-side cache of the array's device address, one per device.  In host
// code the array's name is only a stand-in; the address must come from
// cudaGetSymbolAddress with the device current.
std::mutex g_mu;
void *g_addr[MAX_DEVICES] = {};

cudaError_t scratch_address(int dev, void **out) {
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

__global__ void bias_sum_kernel(const float *b_ih, const float *b_hh, float *bias, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    bias[i] = (b_ih ? b_ih[i] : 0.f) + (b_hh ? b_hh[i] : 0.f);
}

struct NoallocParams {
  int T, B, H, U, NU, CB;
  const float *G;        // [T*B][4H], biases included
  const float *W_hh;     // [4H][H] caller layout
  const float *h0, *c0;  // [B][H] or NULL
  float *y, *h_n, *c_n;  // [T][B][H], [B][H], [B][H] (h_n, c_n may be NULL)
  float *hx, *hst, *cst; // scratch
  unsigned *ctr;
  int *err;
  uint64_t timeout_ns;
};

// Same scheme as the library's portable persistent kernel, reduced to one
// unidirectional fp32 LSTM layer without length masking: CTA ug owns units
// [ug*U, ug*U+U) and keeps their W_hh rows (k-major) in shared memory.
__global__ void __launch_bounds__(NT, 1) lstm_noalloc_kernel(const NoallocParams p) {
  extern __shared__ __align__(16) float sm[];
  const int H = p.H, U = p.U, R = 4 * U, CB = p.CB, B = p.B;
  const int u0 = blockIdx.x * U;
  float *Ws = sm;                    // [H][R]
  float *hs = Ws + (size_t)H * R;    // [H][CB]
  float *acc = hs + (size_t)H * CB;  // [CB][R]
  for (int e = threadIdx.x; e < H * R; e += NT) {
    const int k = e / R, r = e % R, g = r / U, u = u0 + r % U;
    Ws[e] = u < H ? p.W_hh[(size_t)(g * H + u) * H + k] : 0.f;
  }
  for (int e = threadIdx.x; e < B * U; e += NT) {
    const int s = e / U, u = u0 + e % U;
    if (u >= H) continue;
    const float h = p.h0 ? p.h0[(size_t)s * H + u] : 0.f;
    p.hst[(size_t)s * H + u] = h;
    p.cst[(size_t)s * H + u] = p.c0 ? p.c0[(size_t)s * H + u] : 0.f;
    p.hx[(size_t)s * H + u] = h;
  }
  unsigned nbar = 0;
  if (!group_barrier(p.ctr, ++nbar * p.NU, p.err, p.timeout_ns)) return;
  for (int t = 0; t < p.T; ++t) {
    const float *hcur = p.hx + (size_t)(t & 1) * B * H;
    float *hnxt = p.hx + (size_t)((t & 1) ^ 1) * B * H;
    for (int cb = 0; cb < B; cb += CB) {
      const int nr = min(CB, B - cb);
      __syncthreads();
      for (int e = threadIdx.x; e < H * CB; e += NT) {
        const int i = e % CB, k = e / CB;
        hs[e] = i < nr ? __ldcg(hcur + (size_t)(cb + i) * H + k) : 0.f;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < CB * R; e += NT) {
        const int i = e / R, r = e % R;
        float a = 0.f;
        for (int k = 0; k < H; ++k) a = fmaf(hs[k * CB + i], Ws[k * R + r], a);
        acc[e] = a;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < nr * U; e += NT) {
        const int i = e / U, j = e % U, u = u0 + j;
        if (u >= H) continue;
        const int s = cb + i;
        const float *g = p.G + ((size_t)t * B + s) * 4 * H + u;
        const float ig = sigmoid_f(acc[i * R + 0 * U + j] + g[0 * H]);
        const float fg = sigmoid_f(acc[i * R + 1 * U + j] + g[1 * H]);
        const float gg = tanh_f(acc[i * R + 2 * U + j] + g[2 * H]);
        const float og = sigmoid_f(acc[i * R + 3 * U + j] + g[3 * H]);
        const float c = fg * p.cst[(size_t)s * H + u] + ig * gg;
        const float h = og * tanh_f(c);
        p.cst[(size_t)s * H + u] = c;
        p.hst[(size_t)s * H + u] = h;
        hnxt[(size_t)s * H + u] = h;
        p.y[((size_t)t * B + s) * H + u] = h;
      }
    }
    if (!group_barrier(p.ctr, ++nbar * p.NU, p.err, p.timeout_ns)) return;
  }
  for (int e = threadIdx.x; e < B * U; e += NT) {
    const int s = e / U, u = u0 + e % U;
    if (u >= H) continue;
    if (p.h_n) p.h_n[(size_t)s * H + u] = p.hst[(size_t)s * H + u];
    if (p.c_n) p.c_n[(size_t)s * H + u] = p.cst[(size_t)s * H + u];
  }
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace
}  // namespace rcu

using namespace rcu;

extern "C" int rnn_lstm_forward_noalloc(int T, int B, int in_dim, int hidden, const float *x,
                                        const float *W_ih, const float *W_hh, const float *b_ih,
                                        const float *b_hh, const float *h0, const float *c0,
                                        float *y, float *h_n, float *c_n, void *stream) {
  if (T < 0 || B < 0 || in_dim < 1 || hidden < 1)
    return set_error(RCU_ERR_INVALID, "rnn_lstm_forward_noalloc: bad dimensions");
  if (T == 0 || B == 0) return RCU_OK;
  if (!x || !W_ih || !W_hh || !y)
    return set_error(RCU_ERR_INVALID, "rnn_lstm_forward_noalloc: x, W_ih, W_hh, y required");
  const int H = hidden;
  const size_t G_elems = (size_t)T * B * 4 * H;
  const size_t need = align256((size_t)4 * H * 4) + align256(G_elems * 4) +
                      align256((size_t)2 * B * H * 4) + 2 * align256((size_t)B * H * 4) + 256;
  if (need > RCU_NOALLOC_SCRATCH_BYTES) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "rnn_lstm_forward_noalloc: this problem needs %zu bytes of scratch; the fixed "
             "scratch holds %u bytes (T*B*hidden must be smaller)",
             need, (unsigned)RCU_NOALLOC_SCRATCH_BYTES);
    return set_error(RCU_ERR_UNSUPPORTED, msg);
  }
  int dev = 0, nsm = 1;
  if (cudaGetDevice(&dev) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, "rnn_lstm_forward_noalloc: no current device");
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  void *base = nullptr;
  cudaError_t e = scratch_address(dev, &base);
  if (e != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  char *cur = (char *)base;
  auto carve = [&](size_t bytes) { char *r = cur; cur += align256(bytes); return r; };
  float *bias = (float *)carve((size_t)4 * H * 4);
  float *G = (float *)carve(G_elems * 4);
  float *hx = (float *)carve((size_t)2 * B * H * 4);
  float *hst = (float *)carve((size_t)B * H * 4);
  float *cst = (float *)carve((size_t)B * H * 4);
  unsigned *ctl = (unsigned *)carve(256);
  cudaStream_t s = (cudaStream_t)stream;

  NoallocParams p{};
  p.T = T; p.B = B; p.H = H;
  const int budget = nsm < 128 ? nsm : 128;
  p.U = (H + budget - 1) / budget;
  p.NU = (H + p.U - 1) / p.U;
  const int R = 4 * p.U;
  p.CB = B < 32 ? B : 32;
  auto smem_of = [&](int cb) { return ((size_t)H * R + (size_t)H * cb + (size_t)cb * R) * 4; };
  // dynamic shared memory may use what the device allows a block by opt-in,
  // less the kernel's own static shared memory (the step barrier's flag)
  int optin = 0;
  cudaFuncAttributes fa{};
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
          cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, (const void *)lstm_noalloc_kernel)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  const size_t smem_cap = (size_t)optin > fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
  while (p.CB > 1 && smem_of(p.CB) > smem_cap) --p.CB;
  if (smem_of(p.CB) > smem_cap)
    return set_error(RCU_ERR_UNSUPPORTED, "rnn_lstm_forward_noalloc: hidden too large");
  p.G = G; p.W_hh = W_hh; p.h0 = h0; p.c0 = c0; p.y = y; p.h_n = h_n; p.c_n = c_n;
  p.hx = hx; p.hst = hst; p.cst = cst;
  p.ctr = ctl;
  p.err = (int *)(ctl + 16);
  p.timeout_ns = 2000000000ull;

  // counter and error word start at zero on every call
  if ((e = cudaMemsetAsync(ctl, 0, 256, s)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  bias_sum_kernel<<<(4 * H + 255) / 256, 256, 0, s>>>(b_ih, b_hh, bias, 4 * H);
  if ((e = cudaGetLastError()) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  if ((e = launch_gemm_simt<float, float>(x, in_dim, W_ih, in_dim, bias, G, 4 * H, T * B,
                                           nullptr, 4 * H, in_dim, s, p.err)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  const size_t smem = smem_of(p.CB);
  if ((e = cudaFuncSetAttribute((const void *)lstm_noalloc_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  void *args[] = {&p};
  if ((e = cudaLaunchCooperativeKernel((const void *)lstm_noalloc_kernel, dim3(p.NU), dim3(NT),
                                       args, smem, s)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  // synchronous: the device status of this call is known on return
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  int dstat = 0;
  if ((e = cudaMemcpy(&dstat, p.err, sizeof dstat, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return set_error(RCU_ERR_CUDA, cudaGetErrorString(e));
  switch (dstat) {
    case DEV_OK: return RCU_OK;
    case DEV_TIMEOUT:
      return set_error(RCU_ERR_TIMEOUT, "rnn_lstm_forward_noalloc: a step barrier timed out");
    case DEV_CONFIG:
      return set_error(RCU_ERR_CUDA,
                       "rnn_lstm_forward_noalloc: a cluster kernel ran without its cluster shape");
    default: {
      char msg[96];
      snprintf(msg, sizeof msg, "rnn_lstm_forward_noalloc: device error code %d", dstat);
      return set_error(RCU_ERR_CUDA, msg);
    }
  }
}
