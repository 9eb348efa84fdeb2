// Shared device/host helpers for the recurrent-cell unroll kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rcu {

// Device-side error words (one int per handle workspace).
// DEV_CONFIG: a kernel that exchanges data between the CTAs of a thread-block
// cluster found itself launched with another cluster shape, and returned
// before touching any peer's shared memory.
// DEV_BOUNDS: a device bounds check of the RCU_DEBUG build failed (the
// access was skipped).
enum DevErr : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_LENGTHS = 2, DEV_CONFIG = 3, DEV_BOUNDS = 4 };

// Device bounds checks, compiled only into the debug build of the library
// (-DRCU_DEBUG: recurrent_cell_unroll_gb300._build.build(debug=True)), the
// stand-in for a memory checker.  RCU_DCHECK(cond, err) is true when `cond`
// holds; otherwise it records DEV_BOUNDS in the error word `err` (first error
// wins) and is false, so `if (RCU_DCHECK(...)) access;` skips the access.  In
// the normal build it is the constant true and costs nothing.
#ifdef RCU_DEBUG
#define RCU_DCHECK(cond, err) \
  ((cond) ? true : (atomicCAS((err), (int)::rcu::DEV_OK, (int)::rcu::DEV_BOUNDS), false))
#else
#define RCU_DCHECK(cond, err) true
#endif

enum Cell : int { CELL_LSTM = 0, CELL_GRU = 1 };

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int round_up(int a, int b) { return ceil_div(a, b) * b; }
__host__ __device__ inline size_t round_up_sz(size_t a, size_t b) { return (a + b - 1) / b * b; }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_volatile_int(const int *p) {
  return *reinterpret_cast<const volatile int *>(p);
}

// Precise activations on the fp32 path (library expf/tanhf).
__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }
__device__ __forceinline__ float tanh_f(float v) { return tanhf(v); }

// Operand storage helpers: fp32 or bf16 values in memory, fp32 in registers.
template <typename T> struct Op;
template <> struct Op<float> {
  __device__ __forceinline__ static float load(const float *p) { return *p; }
  __device__ __forceinline__ static float to_f(float v) { return v; }
  __device__ __forceinline__ static float from_f(float v) { return v; }
};
template <> struct Op<__nv_bfloat16> {
  __device__ __forceinline__ static float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Split form of group_barrier (below): group_arrive publishes the CTA's
// writes made so far; work placed between the two calls (output stores,
// loads of the next step's inputs) is not waited for by this arrival's
// release.  group_wait is bounded exactly like group_barrier.
__device__ __forceinline__ void group_arrive(unsigned *ctr, bool skip_arrive = false) {
  __syncthreads();
  if (threadIdx.x == 0 && !skip_arrive) red_release_gpu_add(ctr, 1u);
}
__device__ __forceinline__ bool group_wait(unsigned *ctr, unsigned target, int *err,
                                           uint64_t timeout_ns) {
  __shared__ int s_ok2;
  if (threadIdx.x == 0) {
    const uint64_t deadline_ns = globaltimer_ns() + timeout_ns;
    int ok = 1;
    unsigned spins = 0;
    while (ld_acquire_gpu(ctr) < target) {
      if (ld_volatile_int(err) != DEV_OK) { ok = 0; break; }
      if ((++spins & 63u) == 0 && globaltimer_ns() > deadline_ns) {
        atomicCAS(err, DEV_OK, DEV_TIMEOUT);
        ok = 0;
        break;
      }
    }
    s_ok2 = ok && ld_volatile_int(err) == DEV_OK;
  }
  __syncthreads();
  return s_ok2 != 0;
}

// Bounded group barrier over `n` CTAs sharing counter `ctr` (monotone; the
// k-th barrier waits for k*n arrivals).  Every wait is bounded by
// `timeout_ns` on the global timer and by the shared error word: a CTA that
// times out records DEV_TIMEOUT and every CTA then leaves its step loop.
// Returns false when the kernel must stop.
// Ordering: the CTA's writes precede thread 0's arrival through
// __syncthreads, and the arrival is a release at GPU scope (cumulative), so
// no separate full fence is needed; the waiting side reads with acquire and
// passes the ordering on through __syncthreads.  Data exchanged this way is
// read with L1-bypassing loads.
__device__ __forceinline__ bool group_barrier(unsigned *ctr, unsigned target, int *err,
                                              uint64_t timeout_ns, bool skip_arrive = false) {
  __syncthreads();
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    const uint64_t deadline_ns = globaltimer_ns() + timeout_ns;
    if (!skip_arrive) red_release_gpu_add(ctr, 1u);
    int ok = 1;
    unsigned spins = 0;
    while (ld_acquire_gpu(ctr) < target) {
      if (ld_volatile_int(err) != DEV_OK) { ok = 0; break; }
      if ((++spins & 63u) == 0 && globaltimer_ns() > deadline_ns) {
        atomicCAS(err, DEV_OK, DEV_TIMEOUT);
        ok = 0;
        break;
      }
    }
    s_ok = ok && ld_volatile_int(err) == DEV_OK;
  }
  __syncthreads();
  return s_ok != 0;
}

}  // namespace rcu
