// Persistent recurrent kernel, CUDA-core version (fp32 path and portable
// fallback of the bf16 path).
//
// One cooperative launch runs every timestep of one layer (both directions
// at once).  CTA (d, ug) owns hidden units [ug*U, ug*U+U) of direction d and
// keeps the matching rows of W_hh (all gates of those units) resident in
// shared memory for the whole sequence.  Per step it
//   1. reads h_{t-1} of the active rows (the packed prefix) from the
//      exchange buffer in L2,
//   2. computes its slice of h_{t-1} W_hh^T (the "recurrent hidden-hidden
//      dense" of "[TOPI] TE implementation of LSTM using scan",
//      apache/tvm PR 11531) with fp32 FFMA: for fp32 exchange rows, K split
//      over the 16 lanes of a half-warp and summed by shuffles (8 x 8 or
//      fewer register tiles), else 8x4 or 4x4 register tiles with K split
//      over at most 8 thread groups,
//   3. adds the input projection G (loaded for the step before the previous
//      step's barrier, so its HBM latency is off the critical path), applies
//      the gate nonlinearities and the cell update, and writes h_t (exchange
//      buffer, output); h/c state stays in shared memory when it fits,
//   4. for LSTMP, a second phase computes h_t = W_hr m_t (the
//      "hidden-projection dense"; projection rows also resident),
//   5. crosses the step with a bounded group barrier over the CTAs of its
//      direction.
// Rows whose length is exhausted drop out of the active prefix (rows are
// sorted by length), so padding costs nothing ("RNN Op Changes",
// apache/mxnet issue 9543).  The backward direction runs row s at time
// len_s - 1 - step.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace rcu {

namespace {

constexpr int NT = 512;
constexpr int KS_MAX = 8;
constexpr int STATE_SMEM_MAX = 8192;  // B*U entries kept in shared memory (per array)
constexpr int BSZ_SMEM_MAX = 4096;    // batch_sizes staged in shared memory up to this T

__device__ __forceinline__ void load4(const float *p, float (&w)[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(p);
  w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&w)[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  w[0] = fa.x; w[1] = fa.y; w[2] = fb.x; w[3] = fb.y;
}
// 4 consecutive exchange values from L2 (bypassing L1: written by other CTAs)
__device__ __forceinline__ void ldcg4(const float *p, float (&w)[4]) {
  const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
  w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
}
__device__ __forceinline__ void ldcg4(const __nv_bfloat16 *p, float (&w)[4]) {
  const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(p));
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  w[0] = fa.x; w[1] = fa.y; w[2] = fb.x; w[3] = fb.y;
}

struct Split {
  int tiles, ks, kc;
};
__host__ __device__ inline Split make_split(int CB, int Rx, int Kx) {
  Split s;
  s.tiles = (CB / 4) * (Rx / 4);
  int ks = s.tiles > 0 ? NT / s.tiles : 1;
  if (ks > KS_MAX) ks = KS_MAX;
  if (ks > Kx / 4) ks = Kx / 4;
  if (ks < 1) ks = 1;
  s.ks = ks;
  s.kc = ceil_div(Kx / 4, ks) * 4;
  return s;
}

// 8 x 4 register tiles for the row-major h rows (below): twice the rows per
// h load of the 4 x 4 tiles.  K slices: up to 8 (the gates sum them), and no
// more than let the partial sums [ks][CB][Rx] fit in the h rows' buffer,
// which they overwrite once the products are done.  tiles = 0: not
// applicable.
constexpr int KS8_MAX = 8;
__host__ __device__ inline Split make_split8(int CB, int Rx, int Kx) {
  Split s{0, 0, 0};
  if (CB % 8 != 0 || Rx % 4 != 0 || Rx == 0) return s;
  const int tiles = (CB / 8) * (Rx / 4);
  if (tiles == 0 || tiles > NT) return s;
  int ks = NT / tiles;
  if (ks > KS8_MAX) ks = KS8_MAX;
  if (ks > Kx / 4) ks = Kx / 4;
  if (ks > (Kx + 4) / Rx) ks = (Kx + 4) / Rx;
  if (ks < 1) return s;
  s.tiles = tiles;
  s.ks = ks;
  s.kc = ceil_div(Kx / 4, ks) * 4;
  return s;
}

// red[ks][i][r] = sum over this thread's k range of hs[k][i] * Wsm[k][r]
template <typename WT>
__device__ __forceinline__ void chunk_matmul(const WT *Wsm, int Rx, int Kx, const float *hs,
                                             int CB, float *red, Split sp) {
  const int tid = threadIdx.x;
  if (tid >= sp.tiles * sp.ks) return;
  const int tile = tid % sp.tiles, ks = tid / sp.tiles;
  const int nrt = Rx / 4;
  const int ir = tile % nrt, ii = tile / nrt;
  const int k0 = ks * sp.kc, k1 = min(Kx, k0 + sp.kc);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const float *hp = hs + ii * 4;
  const WT *wp = Wsm + ir * 4;
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    const float4 hv = *reinterpret_cast<const float4 *>(hp + (size_t)k * CB);
    float w[4];
    load4(wp + (size_t)k * Rx, w);
    const float h[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(h[i], w[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4 *>(red + ((size_t)(ks * CB + ii * 4 + i)) * Rx + ir * 4) = v;
  }
}

// Row-major variant (fp32 exchange): hs[i][k] with row stride HS = Kx + 4
// floats (the 16-byte pad puts 8 consecutive rows on distinct banks), filled
// by bulk asynchronous copies.  A thread's 4 rows are ii, ii + CB/4, ...,
// so the lanes of one load touch consecutive rows.  red as in chunk_matmul.
template <typename WT>
__device__ __forceinline__ void chunk_matmul_rm(const WT *Wsm, int Rx, int Kx, const float *hs,
                                                int HS, int CB, float *red, Split sp) {
  const int tid = threadIdx.x;
  if (tid >= sp.tiles * sp.ks) return;
  const int tile = tid % sp.tiles, ks = tid / sp.tiles;
  const int nrt = Rx / 4;
  const int ir = tile % nrt, ii = tile / nrt;
  const int k0 = ks * sp.kc, k1 = min(Kx, k0 + sp.kc);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int rs = CB / 4;  // row stride between a thread's rows
  const float *hp = hs + (size_t)ii * HS;
  const WT *wp = Wsm + ir * 4;
#pragma unroll 2
  for (int k = k0; k < k1; k += 4) {
    float4 hv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      hv[i] = *reinterpret_cast<const float4 *>(hp + (size_t)i * rs * HS + k);
    float w[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) load4(wp + (size_t)(k + q) * Rx, w[q]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float h4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(h4[q], w[q][j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4 *>(red + ((size_t)(ks * CB + ii + i * rs)) * Rx + ir * 4) = v;
  }
}

// The same with 8 x 4 tiles (rows ii + i * CB/8), where red aliases hs: every
// thread of the CTA calls it (a barrier separates the last read of hs from
// the first store of red).
template <typename WT>
__device__ __forceinline__ void chunk_matmul_rm8(const WT *Wsm, int Rx, int Kx, const float *hs,
                                                 int HS, int CB, float *red, Split sp) {
  const int tid = threadIdx.x;
  const bool act = tid < sp.tiles * sp.ks;
  const int tile = tid % sp.tiles, ks = tid / sp.tiles;
  const int nrt = Rx / 4;
  const int ir = tile % nrt, ii = tile / nrt;
  const int rs = CB / 8;  // row stride between a thread's rows
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  if (act) {
    const int k0 = ks * sp.kc, k1 = min(Kx, k0 + sp.kc);
    const float *hp = hs + (size_t)ii * HS;
    const WT *wp = Wsm + ir * 4;
#pragma unroll 2
    for (int k = k0; k < k1; k += 4) {
      float4 hv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        hv[i] = *reinterpret_cast<const float4 *>(hp + (size_t)i * rs * HS + k);
      float w[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) load4(wp + (size_t)(k + q) * Rx, w[q]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float h4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(h4[q], w[q][j], acc[i][j]);
      }
    }
  }
  __syncthreads();  // hs is dead: red takes its place
  if (act) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4 *>(red + ((size_t)(ks * CB + ii + i * rs)) * Rx + ir * 4) = v;
    }
  }
}

// The same product with W_hh kept [Rx][Kx] (gate row r's K columns
// contiguous) and K split over the 16 lanes of a half-warp (lane l: columns
// 4l, 4l + 64, ...: consecutive 16-byte words of one row across the lanes).
// Half-warp g takes a tile of 8 batch rows x TC = Rx / 4 gate rows (the rows
// in CB / 8 row tiles, the gate rows in 4 column tiles), reduce-scatters its
// tile over the 16 lanes by shuffles, and after a CTA barrier (hs is dead)
// writes the whole sums over the h rows: red[i * Rx + r] (one K slice).
// Every thread of the CTA calls it.
template <int TC>
__device__ __forceinline__ void chunk_matmul_sl(const float *Wr, int Rx, int Kx, const float *hs,
                                                int HS, int CB, float *red) {
  constexpr int TR = 8, SL = 16, NV = TR * TC;
  constexpr int PER0 = (NV + SL - 1) / SL;
  constexpr int PER = PER0 <= 1 ? 1 : (PER0 <= 2 ? 2 : (PER0 <= 4 ? 4 : 8));  // sums per lane
  constexpr int NVP = SL * PER;
  const int tid = threadIdx.x, g = tid / SL, l = tid % SL, lane = tid & 31;
  const bool act = g < (CB / TR) * 4;  // (warp-uniform: an even number of tiles)
  const int tr = g / 4, tcol = g % 4;
  float acc[TR][TC];
#pragma unroll
  for (int r = 0; r < TR; ++r)
#pragma unroll
    for (int c = 0; c < TC; ++c) acc[r][c] = 0.f;
  if (act) {
    const float *hp = hs + (size_t)tr * TR * HS;
    const float *wp = Wr + (size_t)tcol * TC * Kx;
    for (int k = 4 * l; k < Kx; k += 4 * SL) {
      float4 w[TC];
#pragma unroll
      for (int c = 0; c < TC; ++c) w[c] = *reinterpret_cast<const float4 *>(wp + (size_t)c * Kx + k);
#pragma unroll
      for (int r = 0; r < TR; ++r) {
        const float4 h = *reinterpret_cast<const float4 *>(hp + (size_t)r * HS + k);
#pragma unroll
        for (int c = 0; c < TC; ++c)
          acc[r][c] = fmaf(h.x, w[c].x, fmaf(h.y, w[c].y, fmaf(h.z, w[c].z, fmaf(h.w, w[c].w, acc[r][c]))));
      }
    }
  }
  float v[NVP];
#pragma unroll
  for (int i = 0; i < NVP; ++i) v[i] = i < NV ? acc[i / TC][i % TC] : 0.f;
  // each step keeps half of the values (the upper half on lanes with bit m
  // set) plus the partner lane's same half: lane l ends with entries
  // PER*l .. PER*l + PER - 1 summed over its 16 lanes
#pragma unroll
  for (int h = NVP / 2, m = SL / 2; m >= 1; h >>= 1, m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  __syncthreads();  // hs is dead: red takes its place
  if (act) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = PER * l + i;
      if (idx < NV)
        red[(size_t)(tr * TR + idx / TC) * Rx + tcol * TC + idx % TC] = v[i];
    }
  }
}

// hs[k][i] = src[(row0 + i) * ld + k] for i < nr (0 for i >= nr), k < Kx.
// Loads are issued LB at a time into registers before any store, so their L2
// latencies overlap.
template <typename WT>
__device__ __forceinline__ void load_chunk_T(const WT *src, int ld, int row0, int nr, int Kx,
                                             int CB, float *hs) {
  constexpr int LB = 8;
  const int n = CB * (Kx / 4);
  for (int base = threadIdx.x; base < n; base += NT * LB) {
    float v[LB][4];
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      const int e = base + u * NT;
      const int i = e % CB, k = (e / CB) * 4;
      v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.f;
      if (e < n && i < nr) ldcg4(src + (size_t)(row0 + i) * ld + k, v[u]);
    }
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      const int e = base + u * NT;
      if (e >= n) break;
      const int i = e % CB, k = (e / CB) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) hs[(size_t)(k + q) * CB + i] = v[u][q];
    }
  }
}

__device__ __forceinline__ float red_sum(const float *red, int ks, int CB, int Rx, int i, int r) {
  float a = 0.f;
  for (int q = 0; q < ks; ++q) a += red[((size_t)(q * CB + i)) * Rx + r];
  return a;
}

struct Smem {
  size_t ws, wr, hs, red, st, bsz, mbar, total;
};
// fp32 exchange without projection: h rows arrive by bulk copy, row-major
__host__ __device__ inline bool rowmajor_h(const RecParams &p, size_t wsz) {
  return wsz == 4 && p.proj == 0;
}
// ... multiplied with K split over half-warps and summed by shuffles (W_hh
// kept [Rp][Kp]), the sums written over the h buffer
__host__ __device__ inline bool rowmajor_hsl(const RecParams &p, size_t wsz) {
  return rowmajor_h(p, wsz) && p.CB % 8 == 0 && p.Rp % 4 == 0 && p.Rp >= 4 && p.Rp <= 32 &&
         (p.CB / 8) * 4 * 16 <= NT && p.Rp <= p.Kp + 4;
}
// ... else in 8 x 4 tiles whose partial sums reuse the h buffer
__host__ __device__ inline bool rowmajor_h8(const RecParams &p, size_t wsz) {
  return rowmajor_h(p, wsz) && !rowmajor_hsl(p, wsz) && make_split8(p.CB, p.Rp, p.Kp).tiles > 0;
}
__host__ __device__ inline Smem smem_layout(const RecParams &p, size_t wsz) {
  const bool proj = p.proj > 0;
  Smem L;
  size_t o = 0;
  L.ws = o;
  o += (size_t)p.Kp * p.Rp * wsz;
  L.wr = o;
  if (proj) o += (size_t)p.Hp * p.Pcp * wsz;
  o = round_up_sz(o, 16);
  L.hs = o;
  const int Kh = p.Kp > (proj ? p.Hp : 0) ? p.Kp : p.Hp;
  if (rowmajor_h(p, wsz))
    o += (size_t)p.CB * (p.Kp + 4) * 4;
  else
    o += (size_t)Kh * p.CB * 4;
  L.red = o;
  const Split s1 = make_split(p.CB, p.Rp, p.Kp);
  size_t red = (size_t)s1.ks * p.CB * p.Rp;
  if (rowmajor_h8(p, wsz) || rowmajor_hsl(p, wsz)) {
    L.red = L.hs;  // (the sums overwrite the h rows)
    red = 0;
  }
  if (proj) {
    const Split s2 = make_split(p.CB, p.Pcp, p.Hp);
    red = red > (size_t)s2.ks * p.CB * p.Pcp ? red : (size_t)s2.ks * p.CB * p.Pcp;
  }
  o += red * 4;
  L.st = o;
  if (!proj && (size_t)p.B * p.U <= STATE_SMEM_MAX) o += (size_t)2 * p.B * p.U * 4;
  L.bsz = o;
  if (p.T <= BSZ_SMEM_MAX) o += (size_t)p.T * 4;
  o = round_up_sz(o, 8);
  L.mbar = o;
  o += 16;
  L.total = o;
  return L;
}

template <typename WT>
__global__ void __launch_bounds__(NT, 1) rec_simt_kernel(const RecParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = blockIdx.x / p.NU;
  const int ug = blockIdx.x % p.NU;
  const int u0 = ug * p.U;
  const int B = p.B, H = p.H, Hout = p.Hout, Kp = p.Kp, Hp = p.Hp, U = p.U, CB = p.CB;
  const int nG = p.nG;
  const bool lstm = p.cell == CELL_LSTM;
  const bool proj = p.proj > 0;
  const bool prow = proj && ug < p.NP;  // owns projection rows
  const int pr0 = ug * p.Pc;
  const Smem L = smem_layout(p, sizeof(WT));

  WT *Ws = reinterpret_cast<WT *>(smem + L.ws);
  WT *Wr = reinterpret_cast<WT *>(smem + L.wr);
  float *hs = reinterpret_cast<float *>(smem + L.hs);
  float *red = reinterpret_cast<float *>(smem + L.red);
  const bool rm = rowmajor_h(p, sizeof(WT));
  uint64_t *hbar = reinterpret_cast<uint64_t *>(smem + L.mbar);
  __shared__ int s_abort, s_ok;
  uint32_t hphase = 0;
  if (threadIdx.x == 0) {
    s_abort = 0;
    if (rm) {
      tc::mbar_init(hbar, 1);
      tc::fence_mbar_init();
    }
  }

  {  // resident weights
    const WT *gW = reinterpret_cast<const WT *>(p.Whh[d]) + (size_t)ug * Kp * p.Rp;
    if (rowmajor_hsl(p, sizeof(WT))) {
      // [Kp][Rp] -> [Rp][Kp]
      for (int i = threadIdx.x; i < Kp * p.Rp; i += NT)
        Ws[(size_t)(i % p.Rp) * Kp + i / p.Rp] = gW[i];
    } else {
      for (int i = threadIdx.x; i < Kp * p.Rp; i += NT) Ws[i] = gW[i];
    }
    if (prow) {
      const WT *gR = reinterpret_cast<const WT *>(p.Whr[d]) + (size_t)ug * Hp * p.Pcp;
      for (int i = threadIdx.x; i < Hp * p.Pcp; i += NT) Wr[i] = gR[i];
    }
  }
  const float *bhn = p.bhn[d];
  WT *hx = reinterpret_cast<WT *>(p.hx) + (size_t)d * 2 * B * Kp;
  WT *mx = reinterpret_cast<WT *>(p.mx) + (size_t)d * B * Hp;
  // h/c of the owned (row, unit) entries: shared memory [B][U] when it fits,
  // else the global state arrays [D][B][H]
  const bool st_smem = !proj && (size_t)B * U <= STATE_SMEM_MAX;
  float *hS, *cS;
  int sld, soff0;
  if (st_smem) {
    hS = reinterpret_cast<float *>(smem + L.st);
    cS = hS + (size_t)B * U;
    sld = U;
    soff0 = 0;
  } else {
    hS = p.hst + (size_t)d * B * Hout;
    cS = p.cst + (size_t)d * B * H;
    sld = -1;  // global: index with the unit
    soff0 = u0;
  }
  auto hidx = [&](int s, int j) -> size_t {
    return sld > 0 ? (size_t)s * sld + j : (size_t)s * Hout + soff0 + j;
  };
  auto cidx = [&](int s, int j) -> size_t {
    return sld > 0 ? (size_t)s * sld + j : (size_t)s * H + soff0 + j;
  };
  float *hst_g = p.hst + (size_t)d * B * Hout;  // projected h (LSTMP phase 2)
  const int32_t *sidx = p.meta.sorted_idx;
  const int32_t *lens = p.meta.lens_sorted;
  const int32_t *bsz = p.meta.batch_sizes;
  if (p.T <= BSZ_SMEM_MAX) {  // the step's active-row count, off the critical path
    int *sb = reinterpret_cast<int *>(smem + L.bsz);
    for (int i = threadIdx.x; i < p.T; i += NT) sb[i] = bsz[i];
    bsz = sb;
    __syncthreads();
  }
  const int32_t *soff = p.meta.step_off;
  const int ldo = p.D * Hout;

  // initial state of the entries this CTA owns
  for (int e = threadIdx.x; e < B * U; e += NT) {
    const int s = e / U, j = e % U, u = u0 + j;
    if (u >= H) continue;
    const int b = sidx[s];
    if (lstm) cS[cidx(s, j)] = p.c0 ? p.c0[((size_t)d * B + b) * H + u] : 0.f;
    if (!proj) {
      const float h = p.h0 ? p.h0[((size_t)d * B + b) * Hout + u] : 0.f;
      hS[hidx(s, j)] = h;
      hx[(size_t)s * Kp + u] = Op<WT>::from_f(h);
    }
  }
  if (prow) {
    for (int e = threadIdx.x; e < B * p.Pc; e += NT) {
      const int s = e / p.Pc, q = pr0 + e % p.Pc;
      if (q >= Hout) continue;
      const float h = p.h0 ? p.h0[((size_t)d * B + sidx[s]) * Hout + q] : 0.f;
      hst_g[(size_t)s * Hout + q] = h;
      hx[(size_t)s * Kp + q] = Op<WT>::from_f(h);
    }
  }

  // G of the next step for this thread's (row, unit) pair, loaded before the
  // barrier that precedes the step (single-chunk steps with one pair per thread)
  float gpre[4] = {0.f, 0.f, 0.f, 0.f};
  bool have_pre = false;
  auto prefetch = [&](int step) {
    have_pre = false;
    if (step >= p.T) return;
    const int nn = bsz[step];
    if (nn <= 0 || nn > CB || nn * U > NT) return;
    const int e = threadIdx.x;
    if (e < nn * U) {
      const int i = e / U, j = e % U, u = u0 + j;
      if (u < H) {
        const int tt = d == 0 ? step : lens[i] - 1 - step;
        const float *g = p.G + ((size_t)soff[tt] + i) * p.ldG + (size_t)d * nG * H + u;
        if (RCU_DCHECK(tt >= 0 && tt < p.T && (size_t)soff[tt] + i < (size_t)p.T * p.B, p.err))
          for (int q = 0; q < nG; ++q) gpre[q] = __ldg(g + (size_t)q * H);
      }
    }
    have_pre = true;
  };

  prefetch(0);
  unsigned nbar = 0;
  unsigned *ctr = p.ctr + d;
  const bool drop = p.drop_arrival && blockIdx.x == 0;
  if (!group_barrier(ctr, ++nbar * p.NU, p.err, p.timeout_ns, drop)) return;

  const bool rm8 = rowmajor_h8(p, sizeof(WT)), rmsl = rowmajor_hsl(p, sizeof(WT));
  const Split sp1 = rmsl ? Split{(CB / 8) * 4, 1, Kp}
                         : (rm8 ? make_split8(CB, p.Rp, Kp) : make_split(CB, p.Rp, Kp));
  const Split sp2 = proj ? make_split(CB, p.Pcp, Hp) : Split{0, 0, 0};

  for (int step = 0; step < p.T; ++step) {
    const int nact = bsz[step];
    const bool tr = p.trace && blockIdx.x == 0 && threadIdx.x == 0;
    if (tr) p.trace[step * 16 + 0] = globaltimer_ns();
    if (nact <= 0) break;
    const WT *hcur = hx + (size_t)(step & 1) * B * Kp;
    WT *hnxt = hx + (size_t)((step & 1) ^ 1) * B * Kp;
    // one (row, unit) pair per thread: its output store is deferred (non-LSTMP)
    const bool one = !proj && nact <= CB && nact * U <= NT;
    float yv = 0.f;
    size_t y_at = SIZE_MAX, ym_at = SIZE_MAX;

    // ---- phase 1: gates and cell update for this CTA's units
    for (int cb = 0; cb < nact; cb += CB) {
      const int nr = min(CB, nact - cb);
      __syncthreads();
      if (rm) {
        // rows [cb, cb+nr) of h_{t-1} by bulk copy (the exchange buffer was
        // written through the generic proxy and acquired at the step barrier)
        if (threadIdx.x < 32) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          if (threadIdx.x == 0) tc::mbar_arrive_expect_tx(hbar, (uint32_t)(nr * Kp * 4));
          __syncwarp();
          for (int i = threadIdx.x; i < nr; i += 32)
            tc::bulk_load(hs + (size_t)i * (Kp + 4), hcur + (size_t)(cb + i) * Kp,
                          (uint32_t)(Kp * 4), hbar);
        }
        if (threadIdx.x == 0)
          s_ok = tc::mbar_wait(hbar, hphase & 1u, p.err, &s_abort, p.timeout_ns);
        ++hphase;
        __syncthreads();
        if (!s_ok) {
          // let the copies land before the CTA leaves (bounded, ignores the abort)
          if (threadIdx.x == 0) {
            volatile int never = 0;
            tc::mbar_wait(hbar, (hphase - 1) & 1u, nullptr, &never, 100000000ull);
          }
          __syncthreads();
          return;
        }
        if (tr && cb == 0) p.trace[step * 16 + 3] = globaltimer_ns();
        if (rmsl) {
          const float *Wf = reinterpret_cast<const float *>(Ws);
          switch (p.Rp / 4) {
            case 1: chunk_matmul_sl<1>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 2: chunk_matmul_sl<2>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 3: chunk_matmul_sl<3>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 4: chunk_matmul_sl<4>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 5: chunk_matmul_sl<5>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 6: chunk_matmul_sl<6>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            case 7: chunk_matmul_sl<7>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
            default: chunk_matmul_sl<8>(Wf, p.Rp, Kp, hs, Kp + 4, CB, red); break;
          }
        } else if (rm8) {
          chunk_matmul_rm8(Ws, p.Rp, Kp, hs, Kp + 4, CB, red, sp1);
        } else {
          chunk_matmul_rm(Ws, p.Rp, Kp, hs, Kp + 4, CB, red, sp1);
        }
      } else {
        load_chunk_T(hcur, Kp, cb, nr, Kp, CB, hs);
        __syncthreads();
        chunk_matmul(Ws, p.Rp, Kp, hs, CB, red, sp1);
      }
      __syncthreads();
      if (tr && cb == 0) p.trace[step * 16 + 4] = globaltimer_ns();
      const bool pre = have_pre && cb == 0;
      for (int e = threadIdx.x; e < nr * U; e += NT) {
        const int i = e / U, j = e % U, u = u0 + j;
        if (u >= H) continue;
        const int s = cb + i;
        const int tt = d == 0 ? step : lens[s] - 1 - step;
        const size_t row = (size_t)soff[tt] + s;
        float gx[4];
        if (pre) {
          gx[0] = gpre[0]; gx[1] = gpre[1]; gx[2] = gpre[2]; gx[3] = gpre[3];
        } else {
          const float *g = p.G + row * p.ldG + (size_t)d * nG * H + u;
          if (RCU_DCHECK(tt >= 0 && tt < p.T && row < (size_t)p.T * B, p.err))
            for (int q = 0; q < nG; ++q) gx[q] = __ldg(g + (size_t)q * H);
        }
        float hv;
        if (lstm) {
          const float ai = red_sum(red, sp1.ks, CB, p.Rp, i, 0 * U + j) + gx[0];
          const float af = red_sum(red, sp1.ks, CB, p.Rp, i, 1 * U + j) + gx[1];
          const float ag = red_sum(red, sp1.ks, CB, p.Rp, i, 2 * U + j) + gx[2];
          const float ao = red_sum(red, sp1.ks, CB, p.Rp, i, 3 * U + j) + gx[3];
          const float ig = sigmoid_f(ai), fg = sigmoid_f(af), gg = tanh_f(ag), og = sigmoid_f(ao);
          float c = cS[cidx(s, j)];
          c = fg * c + ig * gg;
          if (p.cclip) c = fminf(fmaxf(c, p.cclip_lo), p.cclip_hi);
          cS[cidx(s, j)] = c;
          hv = og * tanh_f(c);
          if (proj) {
            mx[(size_t)s * Hp + u] = Op<WT>::from_f(hv);
            continue;
          }
        } else {
          const float hr = red_sum(red, sp1.ks, CB, p.Rp, i, 0 * U + j);
          const float hz = red_sum(red, sp1.ks, CB, p.Rp, i, 1 * U + j);
          const float hn = red_sum(red, sp1.ks, CB, p.Rp, i, 2 * U + j) + (bhn ? bhn[u] : 0.f);
          const float rg = sigmoid_f(gx[0] + hr);
          const float zg = sigmoid_f(gx[1] + hz);
          const float ng = tanh_f(gx[2] + rg * hn);
          const float hprev = hS[hidx(s, j)];
          hv = (1.f - zg) * ng + zg * hprev;
        }
        hS[hidx(s, j)] = hv;
        hnxt[(size_t)s * Kp + u] = Op<WT>::from_f(hv);
        const size_t yo = ((size_t)tt * B + sidx[s]) * ldo + (size_t)d * Hout + u;
        const size_t ymo = row * ldo + (size_t)d * Hout + u;
        const bool out_ok = RCU_DCHECK(yo < (size_t)p.T * B * ldo && ymo < (size_t)p.T * B * ldo,
                                       p.err);
        if (one && out_ok) {  // written after the step's arrival
          yv = hv;
          y_at = yo;
          ym_at = ymo;
        } else if (out_ok) {
          if (p.y) p.y[yo] = hv;
          if (p.ymid) reinterpret_cast<WT *>(p.ymid)[ymo] = Op<WT>::from_f(hv);
        }
      }
    }
    if (tr) p.trace[step * 16 + 1] = globaltimer_ns();
    // h_t is read by bulk copies (async proxy) in the next step
    if (rm) asm volatile("fence.proxy.async.global;" ::: "memory");
    // publish h_t first; the outputs and the next step's G loads follow the
    // arrival, so its release does not wait for them
    group_arrive(ctr);
    if (one && y_at != SIZE_MAX) {
      if (p.y) p.y[y_at] = yv;
      if (p.ymid) reinterpret_cast<WT *>(p.ymid)[ym_at] = Op<WT>::from_f(yv);
    }
    if (!proj) prefetch(step + 1);
    if (!group_wait(ctr, ++nbar * p.NU, p.err, p.timeout_ns)) return;
    if (tr) p.trace[step * 16 + 2] = globaltimer_ns();

    // ---- phase 2 (LSTMP): h_t = W_hr m_t for this CTA's projection rows
    if (proj) {
      if (prow) {
        for (int cb = 0; cb < nact; cb += CB) {
          const int nr = min(CB, nact - cb);
          __syncthreads();
          load_chunk_T(mx, Hp, cb, nr, Hp, CB, hs);
          __syncthreads();
          chunk_matmul(Wr, p.Pcp, Hp, hs, CB, red, sp2);
          __syncthreads();
          for (int e = threadIdx.x; e < nr * p.Pc; e += NT) {
            const int i = e / p.Pc, j = e % p.Pc, q = pr0 + j;
            if (q >= Hout) continue;
            const int s = cb + i;
            const int tt = d == 0 ? step : lens[s] - 1 - step;
            const size_t row = (size_t)soff[tt] + s;
            float hv = red_sum(red, sp2.ks, CB, p.Pcp, i, j);
            if (p.pclip) hv = fminf(fmaxf(hv, p.pclip_lo), p.pclip_hi);
            hst_g[(size_t)s * Hout + q] = hv;
            hnxt[(size_t)s * Kp + q] = Op<WT>::from_f(hv);
            if (p.y) p.y[((size_t)tt * B + sidx[s]) * ldo + (size_t)d * Hout + q] = hv;
            if (p.ymid)
              reinterpret_cast<WT *>(p.ymid)[row * ldo + (size_t)d * Hout + q] =
                  Op<WT>::from_f(hv);
          }
        }
      }
      prefetch(step + 1);
      if (!group_barrier(ctr, ++nbar * p.NU, p.err, p.timeout_ns)) return;
    }
  }

  // final state of each row = state after its last processed step
  __syncthreads();
  for (int e = threadIdx.x; e < B * U; e += NT) {
    const int s = e / U, j = e % U, u = u0 + j;
    if (u >= H) continue;
    const int b = sidx[s];
    if (lstm && p.c_n) p.c_n[((size_t)d * B + b) * H + u] = cS[cidx(s, j)];
    if (!proj && p.h_n) p.h_n[((size_t)d * B + b) * Hout + u] = hS[hidx(s, j)];
  }
  if (prow && p.h_n) {
    for (int e = threadIdx.x; e < B * p.Pc; e += NT) {
      const int s = e / p.Pc, q = pr0 + e % p.Pc;
      if (q >= Hout) continue;
      p.h_n[((size_t)d * B + sidx[s]) * Hout + q] = hst_g[(size_t)s * Hout + q];
    }
  }
}

}  // namespace

size_t recurrent_simt_smem(const RecParams &p, bool wbf16) {
  return smem_layout(p, wbf16 ? 2 : 4).total;
}

bool plan_recurrent_simt(RecParams &p, bool wbf16) {
  int CB = std::min(64, round_up(std::max(p.B, 1), 4));
  for (;;) {
    p.CB = CB;
    const bool tiles_ok = (CB / 4) * (p.Rp / 4) <= NT &&
                          (p.proj == 0 || (CB / 4) * (p.Pcp / 4) <= NT);
    if (tiles_ok && recurrent_simt_smem(p, wbf16) <= 227 * 1024) return true;
    if (CB <= 4) return false;
    CB -= 4;
  }
}

cudaError_t launch_recurrent_simt(const RecParams &p, bool wbf16, int nsm, cudaStream_t s) {
  (void)nsm;
  const size_t smem = recurrent_simt_smem(p, wbf16);
  const void *fn = wbf16 ? (const void *)rec_simt_kernel<__nv_bfloat16>
                         : (const void *)rec_simt_kernel<float>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  RecParams pc = p;
  void *args[] = {&pc};
  return cudaLaunchCooperativeKernel(fn, dim3(p.D * p.NU), dim3(NT), args, smem, s);
}

}  // namespace rcu
