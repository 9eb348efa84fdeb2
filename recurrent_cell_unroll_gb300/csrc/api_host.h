// Host-side pieces shared by the two halves of the C ABI (api.cu: the stacked
// LSTM / GRU / LSTMP networks; api_rssm.cu: the RSSM prior): failure
// reporting, device buffers, host-buffer staging, device status codes and
// opt-in event timing.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "rcu.h"
#include "common.cuh"

namespace rcu_api {

// Record the message of a failure (read back by rcu_last_error on the same
// host thread) and return `code`.
int fail(int code, const char *fmt, ...);

#define CU(expr)                                                                        \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(RCU_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                                  \
  } while (0)

inline float bf2f(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// fp32 -> bf16 bits, round to nearest even (NaN kept quiet).
inline uint16_t f2bf(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0x7fffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

inline int device_sm_count(int *dev) {
  cudaGetDevice(dev);
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
  return n > 0 ? n : 1;
}

// Copy a device fp32 tensor to the host (synchronous on `s`).
inline cudaError_t fetch(std::vector<float> &dst, const float *src, size_t n, cudaStream_t s) {
  dst.assign(n, 0.f);
  if (!src || n == 0) return cudaSuccess;
  cudaError_t e = cudaMemcpyAsync(dst.data(), src, n * sizeof(float), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

struct DevBuf {
  void *p = nullptr;
  size_t n = 0;
  ~DevBuf() { if (p) cudaFree(p); }
  cudaError_t ensure(size_t bytes) {
    if (bytes <= n) return cudaSuccess;
    if (p) { cudaFree(p); p = nullptr; n = 0; }
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e == cudaSuccess) n = bytes;
    return e;
  }
  // upload host bytes (synchronous)
  cudaError_t upload(const void *src, size_t bytes) {
    cudaError_t e = ensure(bytes);
    if (e != cudaSuccess) return e;
    return cudaMemcpy(p, src, bytes, cudaMemcpyHostToDevice);
  }
};

// ---- host buffers of the *_host entry points
//
// A host buffer that is page-locked and registered with CUDA (cudaHostAlloc,
// cudaHostRegister, torch's pin_memory) has a device address: the kernels
// read or write it in place over the coherent CPU-GPU link, so its copy
// happens inside the kernel that touches it.  A pageable buffer is staged
// through a device buffer with cudaMemcpyAsync.  Device (or managed) memory
// passed here is used as it is.
inline const void *device_address(const void *p) {
  if (!p) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost && a.devicePointer) return a.devicePointer;
  return nullptr;  // pageable
}

struct HostIO {
  cudaStream_t s;
  struct Back { void *host; const void *dev; size_t bytes; };
  std::vector<Back> back;
  // input: in place when `in_place` and mapped, else copied to `stage`
  cudaError_t in(const void *host, size_t bytes, DevBuf &stage, bool in_place, const void **out,
                 bool *placed = nullptr) {
    *out = nullptr;
    if (placed) *placed = false;
    if (!host || bytes == 0) return cudaSuccess;
    if (in_place) {
      if (const void *d = device_address(host)) {
        *out = d;
        if (placed) *placed = true;
        return cudaSuccess;
      }
    }
    cudaError_t e = stage.ensure(bytes);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(stage.p, host, bytes, cudaMemcpyDefault, s);
    *out = stage.p;
    return e;
  }
  // output: in place when `in_place` and mapped, else staged and copied back by finish()
  cudaError_t out(void *host, size_t bytes, DevBuf &stage, bool in_place, void **dst) {
    *dst = nullptr;
    if (!host || bytes == 0) return cudaSuccess;
    if (in_place) {
      if (const void *d = device_address(host)) {
        *dst = const_cast<void *>(d);
        return cudaSuccess;
      }
    }
    cudaError_t e = stage.ensure(bytes);
    if (e != cudaSuccess) return e;
    back.push_back({host, stage.p, bytes});
    *dst = stage.p;
    return cudaSuccess;
  }
  cudaError_t finish() {
    for (auto &b : back) {
      cudaError_t e = cudaMemcpyAsync(b.host, b.dev, b.bytes, cudaMemcpyDefault, s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
};

inline int status_from_dev(int v) {
  switch (v) {
    case rcu::DEV_OK: return RCU_OK;
    case rcu::DEV_TIMEOUT: return fail(RCU_ERR_TIMEOUT, "device step barrier timed out");
    case rcu::DEV_LENGTHS: return fail(RCU_ERR_LENGTHS, "a length was outside [1, T]");
    case rcu::DEV_CONFIG: return fail(RCU_ERR_CUDA, "a cluster kernel ran without its cluster shape");
    case rcu::DEV_BOUNDS: return fail(RCU_ERR_CUDA, "a device bounds check (debug build) failed");
    default: return fail(RCU_ERR_CUDA, "unknown device status %d", v);
  }
}

// Opt-in timing of named spans of launches (one kernel, or a group) with CUDA
// events recorded on the launching stream (RCU_ATTR_PROFILE); totals per name
// are read with *_profile_entry.
struct EventProfiler {
  bool profile = false;
  struct Pending { const char *name; cudaEvent_t a, b; };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
  std::vector<std::pair<std::string, std::pair<double, long>>> totals;
  const char *open_name = nullptr;
  cudaEvent_t open_ev = nullptr;
  cudaEvent_t get_event() {
    if (!pool.empty()) { cudaEvent_t e = pool.back(); pool.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void prof_begin(const char *name, cudaStream_t s) {
    if (!profile) return;
    open_name = name;
    open_ev = get_event();
    cudaEventRecord(open_ev, s);
  }
  void prof_end(cudaStream_t s) {
    if (!profile || !open_ev) return;
    cudaEvent_t b = get_event();
    cudaEventRecord(b, s);
    pending.push_back({open_name, open_ev, b});
    open_ev = nullptr;
  }
  void collect() {
    for (auto &p : pending) {
      cudaEventSynchronize(p.b);
      float ms = 0.f;
      cudaEventElapsedTime(&ms, p.a, p.b);
      bool found = false;
      for (auto &t : totals)
        if (t.first == p.name) { t.second.first += ms; t.second.second += 1; found = true; break; }
      if (!found) totals.push_back({p.name, {ms, 1L}});
      pool.push_back(p.a);
      pool.push_back(p.b);
    }
    pending.clear();
  }
  int entry(int i, const char **name, double *total_ms, int64_t *count) {
    collect();
    if (i < 0 || i >= (int)totals.size()) return fail(RCU_ERR_INVALID, "no profile entry %d", i);
    if (name) *name = totals[i].first.c_str();
    if (total_ms) *total_ms = totals[i].second.first;
    if (count) *count = totals[i].second.second;
    return RCU_OK;
  }
  void reset() {
    collect();
    totals.clear();
  }
  ~EventProfiler() {
    for (auto &p : pending) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
    if (open_ev) cudaEventDestroy(open_ev);
    for (auto e : pool) cudaEventDestroy(e);
  }
};

}  // namespace rcu_api
