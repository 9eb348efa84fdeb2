// Length sort, packing metadata, packed gather and zero tails for
// variable-length batches.  The sort-by-length-then-pack scheme is the one
// "RNN Op Changes (was: Variable Length Support for cuDNN RNN)"
// (apache/mxnet issue 9543) describes for cuDNN, done here on the device
// and hidden inside the forward call.  Ties keep ascending row order.
#include "common.cuh"
#include "internal.h"

namespace rcu {

namespace {

constexpr int kMetaThreads = 1024;

__global__ void __launch_bounds__(kMetaThreads) meta_kernel(const int32_t *__restrict__ lengths,
                                                            int B, int T, Meta m, int *err) {
  __shared__ int s_part[kMetaThreads];
  const int tid = threadIdx.x;
  // 1. rank of every row: rows with a longer length, or equal length and a
  //    smaller index, come first (stable descending sort).
  for (int b = tid; b < B; b += blockDim.x) {
    int lb = lengths ? lengths[b] : T;
    if (lb < 1 || lb > T) {
      atomicCAS(err, DEV_OK, DEV_LENGTHS);
      lb = lb < 1 ? 1 : T;
    }
    int pos = 0;
    if (lengths) {
      for (int o = 0; o < B; ++o) {
        int lo = lengths[o];
        lo = lo < 1 ? 1 : (lo > T ? T : lo);
        pos += (lo > lb) || (lo == lb && o < b);
      }
    } else {
      pos = b;
    }
    m.sorted_idx[pos] = b;
    m.unsorted_idx[b] = pos;
    m.lens_sorted[pos] = lb;
  }
  // 2. batch_sizes[t] = #{b : len_b > t}
  for (int t = tid; t < T; t += blockDim.x) {
    int n = 0;
    if (lengths) {
      for (int b = 0; b < B; ++b) {
        int lb = lengths[b];
        lb = lb < 1 ? 1 : (lb > T ? T : lb);
        n += lb > t;
      }
    } else {
      n = B;
    }
    m.batch_sizes[t] = n;
  }
  __syncthreads();
  // 3. step_off = exclusive prefix sum of batch_sizes (blocked scan).
  const int per = ceil_div(T, blockDim.x);
  const int t0 = tid * per, t1 = min(T, t0 + per);
  int sum = 0;
  for (int t = t0; t < t1; ++t) sum += m.batch_sizes[t];
  // block-wide exclusive scan of the per-thread sums: inclusive scan inside
  // each warp by shuffles, then of the warp totals by warp 0
  const int lane = tid & 31, wid = tid >> 5, nw = (int)blockDim.x >> 5;
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) s_part[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? s_part[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < nw) s_part[lane] = w;  // inclusive warp totals
    if (lane == nw - 1) m.step_off[T] = w;
  }
  __syncthreads();
  int run = inc - sum + (wid > 0 ? s_part[wid - 1] : 0);
  for (int t = t0; t < t1; ++t) {
    m.step_off[t] = run;
    run += m.batch_sizes[t];
  }
}

template <typename OT>
__device__ __forceinline__ OT cvt(float v);
template <>
__device__ __forceinline__ float cvt<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 8 consecutive values to 16-byte aligned storage
__device__ __forceinline__ void store8(float *d, float4 a, float4 b) {
  reinterpret_cast<float4 *>(d)[0] = a;
  reinterpret_cast<float4 *>(d)[1] = b;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *d, float4 a, float4 b) {
  const __nv_bfloat162 v0 = __floats2bfloat162_rn(a.x, a.y), v1 = __floats2bfloat162_rn(a.z, a.w),
                       v2 = __floats2bfloat162_rn(b.x, b.y), v3 = __floats2bfloat162_rn(b.z, b.w);
  uint4 o;
  o.x = *reinterpret_cast<const uint32_t *>(&v0);
  o.y = *reinterpret_cast<const uint32_t *>(&v1);
  o.z = *reinterpret_cast<const uint32_t *>(&v2);
  o.w = *reinterpret_cast<const uint32_t *>(&v3);
  *reinterpret_cast<uint4 *>(d) = o;
}

// One warp per (t, s) row; lanes stride the columns.  vec8: in and ld_out
// multiples of 8, x and out 16-byte aligned (each lane then moves 8 values
// per iteration with 16-byte accesses)
template <typename OT>
__global__ void pack_rows_kernel(const float *__restrict__ x, int T, int B, int in, Meta m,
                                 OT *__restrict__ out, int ld_out, int vec8) {
  const int warps = blockDim.x / 32, lane = threadIdx.x % 32;
  const long long nrows = (long long)T * B;
  for (long long r = (long long)blockIdx.x * warps + threadIdx.x / 32; r < nrows;
       r += (long long)gridDim.x * warps) {
    const int t = (int)(r / B), s = (int)(r % B);
    if (s >= m.batch_sizes[t]) continue;
    const int b = m.sorted_idx[s];
    const float *src = x + ((size_t)t * B + b) * in;
    OT *dst = out + (size_t)(m.step_off[t] + s) * ld_out;
    if (vec8) {
      for (int k = 8 * lane; k < in; k += 256)
        store8(dst + k, __ldg(reinterpret_cast<const float4 *>(src + k)),
               __ldg(reinterpret_cast<const float4 *>(src + k + 4)));
    } else {
      for (int k = lane; k < in; k += 32) dst[k] = cvt<OT>(__ldg(src + k));
    }
    for (int k = in + lane; k < ld_out; k += 32) dst[k] = cvt<OT>(0.f);
  }
}

__global__ void zero_tail_kernel(float *__restrict__ y, const int32_t *__restrict__ lengths,
                                 int T, int B, int width) {
  const int warps = blockDim.x / 32;
  const long long nrows = (long long)T * B;
  for (long long r = (long long)blockIdx.x * warps + threadIdx.x / 32; r < nrows;
       r += (long long)gridDim.x * warps) {
    const int t = (int)(r / B), b = (int)(r % B);
    int lb = lengths[b];
    lb = lb < 1 ? 1 : (lb > T ? T : lb);
    if (t < lb) continue;
    float *dst = y + (size_t)r * width;
    if ((width & 3) == 0 && ((uintptr_t)dst & 15) == 0) {
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = (threadIdx.x % 32) * 4; k < width; k += 128)
        *reinterpret_cast<float4 *>(dst + k) = z;
    } else {
      for (int k = threadIdx.x % 32; k < width; k += 32) dst[k] = 0.f;
    }
  }
}

template <typename OT>
__global__ void convert_kernel(const float *__restrict__ src, OT *__restrict__ dst, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = cvt<OT>(src[i]);
}

int grid_for(long long work, int per_block) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return (int)g;
}

}  // namespace

cudaError_t launch_meta(const int32_t *lengths, int B, int T, Meta m, int *err, cudaStream_t s) {
  meta_kernel<<<1, kMetaThreads, 0, s>>>(lengths, B, T, m, err);
  return cudaGetLastError();
}

template <typename OT>
cudaError_t launch_pack_rows(const float *x, int T, int B, int in, Meta m, OT *out, int ld_out,
                             cudaStream_t s) {
  const int vec8 = (in % 8 == 0 && ld_out % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(out) & 15) == 0) ? 1 : 0;
  pack_rows_kernel<OT><<<grid_for((long long)T * B, 8), 256, 0, s>>>(x, T, B, in, m, out, ld_out,
                                                                     vec8);
  return cudaGetLastError();
}
template cudaError_t launch_pack_rows<float>(const float *, int, int, int, Meta, float *, int,
                                             cudaStream_t);
template cudaError_t launch_pack_rows<__nv_bfloat16>(const float *, int, int, int, Meta,
                                                     __nv_bfloat16 *, int, cudaStream_t);

cudaError_t launch_zero_tail(float *y, const int32_t *lengths, int T, int B, int width, int *err,
                             cudaStream_t s) {
  (void)err;
  zero_tail_kernel<<<grid_for((long long)T * B, 8), 256, 0, s>>>(y, lengths, T, B, width);
  return cudaGetLastError();
}

template <typename OT>
cudaError_t launch_convert(const float *src, OT *dst, size_t n, cudaStream_t s) {
  convert_kernel<OT><<<grid_for((long long)n, 256), 256, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}
template cudaError_t launch_convert<float>(const float *, float *, size_t, cudaStream_t);
template cudaError_t launch_convert<__nv_bfloat16>(const float *, __nv_bfloat16 *, size_t,
                                                   cudaStream_t);

}  // namespace rcu
