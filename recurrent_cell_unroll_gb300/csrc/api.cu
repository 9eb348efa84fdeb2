// Host side of the C ABI declared in include/rcu.h: handles, weight packing,
// workspace, planning and launch sequencing.  Every step of the forward pass
// runs in this library's kernels; nothing falls back to the host.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "rcu.h"
#include "common.cuh"
#include "internal.h"
#include "tc.h"
#include "api_host.h"


using namespace rcu;
using namespace rcu_api;

namespace rcu_api {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

}  // namespace rcu_api

// ---------------------------------------------------------------------------
// network handle

struct LayerDirW {
  DevBuf whh, whr, bhn;  // SIMT-packed recurrent weights, projection, GRU b_hn
  DevBuf tc_whh;         // tensor-core packed recurrent weights (bf16 path)
  DevBuf cl_whh;         // cluster-resident layout [H*nG][Kc] (small W_hh, no projection)
  // bf16 LSTMP tensor-core path: packed W_hh W_hr, fp32 copy of the rounded
  // W_hh (initial-state term) and bf16 W_hr [P][round_up(H, 8)] (projection GEMM)
  DevBuf fold_w, whh_f32, whr_bf;
  // fp32 handles, for the backward pass: plain W_hh [nG*H][round_up(Hout, 8)],
  // b_ih, b_hh (zeros when NULL), and W_hr [P][H] with a projection
  DevBuf whh_plain, bih_plain, bhh_plain, whr_plain;
  bool set = false;
};

struct rcu_rnn_s : EventProfiler {
  int cell, layers, D, in_dim, H, P, Hout, nG, dtype;
  int device, nsm;
  // SIMT plan
  int U, NU, Rp, Kp, Hp, Pc, Pcp, NP;
  std::vector<int> in_l;         // GEMM K per layer
  std::vector<DevBuf> wih;       // [D*nG*H][ldk] per layer (dtype), ldk = round_up(in_l, 8)
  std::vector<DevBuf> wih_f32;   // bf16 handles: the same, fp32 of the rounded values (backward)
  std::vector<DevBuf> gbias;     // [D*nG*H] fp32 per layer
  std::vector<std::vector<float>> host_bias; // staging: per layer, filled by set_weights
  std::vector<LayerDirW> lw;     // layers*D
  // workspace
  DevBuf ctl;   // err word + counters
  DevBuf ws;
  Meta meta{};
  int ws_T = -1, ws_B = -1;
  // (T, B, stream) whose fixed-length metadata (identity sort, full batch
  // sizes) h->meta holds, so a repeated fixed-length forward skips the sort
  int meta_T = -1, meta_B = -1;
  cudaStream_t meta_s = nullptr;
  int last_T = -1, last_B = -1;
  char *xp = nullptr, *g = nullptr, *ymid = nullptr, *hx = nullptr, *mx = nullptr;
  char *mbuf = nullptr, *hx2 = nullptr;  // LSTMP tensor-core path
  float *ytmp = nullptr;
  float *hst = nullptr, *cst = nullptr;
  int64_t timeout_ns = 2000000000LL;
  int drop_arrival = 0;
  int force_path = 0;
  int tc_ksplit = 0;   // CTAs splitting K in the tensor-core recurrent kernel (0 = automatic)
  // LSTM clipping (rnn_set_clip)
  int cclip = 0, pclip = 0;
  float cclip_lo = 0.f, cclip_hi = 0.f, pclip_lo = 0.f, pclip_hi = 0.f;
  int launches = 0;
  bool used_tc_gemm = false, used_tc_rec = false;
  // rnn_forward_host: staging buffers, and x read in place from host memory
  // (then always through the packing kernel's plain loads)
  DevBuf io_x, io_len, io_h0, io_c0, io_y, io_hn, io_cn;
  bool x_in_place = false;
  // what the last rnn_forward_host did (rnn_host_plan)
  int plan_chunks = 0, plan_x_in_place = 0, plan_y_in_place = 0;
  // rnn_forward_host over chunks of steps: two copy streams, double-buffered
  // x / y chunks, ping-pong per-layer state, events
  int host_chunks = 0;  // RCU_ATTR_HOST_CHUNKS
  cudaStream_t cp_in = nullptr, cp_out = nullptr;
  std::vector<cudaEvent_t> chunk_ev;
  DevBuf io_xc[2], io_yc[2], io_st[2], io_ct[2];
  // layer-pipelined forward: one stream per layer past the first,
  // events between them, per-(layer, chunk) step counters, per-layer
  // exchange buffers and chunk-boundary states, chunk metadata
  std::vector<cudaStream_t> lp_streams;
  std::vector<cudaEvent_t> lp_events;
  DevBuf lp_ctl, lp_hx, lp_state, lp_meta;
  int layer_pipeline = 1;  // RCU_ATTR_LAYER_PIPELINE
  // rnn_backward: workspace, per-layer weight gradients of the last call, and
  // the forward's per-layer outputs (layer l < L-1 written to keep_out + l*T*B*Hout)
  DevBuf bw;
  DevBuf bwb;  // bf16 handles: the bf16 operands of the backward's tensor-core GEMMs
  DevBuf f32x;  // the split bf16 operands of the fp32 GEMMs on the tensor cores
  std::vector<DevBuf> gw;
  bool grads_ready = false;
  float *keep_out = nullptr;
  // opt-in per-step trace of the first layer's recurrent kernel
  int trace = 0;  // RCU_ATTR_TRACE: 1 = CTA 0 every step, 2 = also every CTA for a window
  DevBuf trace_buf;
  int trace_T = 0;
  void begin(const char *name, cudaStream_t s) { prof_begin(name, s); }
  void end(cudaStream_t s) {
    ++launches;
    prof_end(s);
  }
  ~rcu_rnn_s() {
    for (auto e : chunk_ev) cudaEventDestroy(e);
    for (auto e : lp_events) cudaEventDestroy(e);
    for (auto st : lp_streams) cudaStreamDestroy(st);
    if (cp_in) cudaStreamDestroy(cp_in);
    if (cp_out) cudaStreamDestroy(cp_out);
  }
};

static size_t esize(int dtype) { return dtype == RCU_BF16 ? 2 : 4; }
// control block: error word at 0, then 4 barrier counters per layer from byte 64
static size_t ctl_bytes(int layers) { return 64 + 16 * (size_t)layers + 64; }

extern "C" const char *rcu_last_error(void) { return g_last_error.c_str(); }

int rcu::set_error(int code, const char *msg) { return fail(code, "%s", msg); }
extern "C" const char *rcu_version(void) { return "rcu 0.1 (sm_103a)"; }

static void plan_simt(rcu_rnn_s *h) {
  const int budget = std::max(1, h->nsm / h->D);
  int U = ceil_div(h->H, budget);
  h->U = U;
  h->NU = ceil_div(h->H, U);
  h->Rp = round_up(h->nG * U, 4);
  h->Kp = round_up(h->Hout, 8);
  h->Hp = round_up(h->H, 8);
  if (h->P > 0) {
    h->Pc = ceil_div(h->P, h->NU);
    h->Pcp = round_up(h->Pc, 4);
    h->NP = ceil_div(h->P, h->Pc);
  } else {
    h->Pc = h->Pcp = h->NP = 0;
  }
}

extern "C" int rnn_create(rcu_rnn_t *out, int cell, int layers, int in_dim, int hidden, int proj,
                          int dtype) {
  if (!out) return fail(RCU_ERR_INVALID, "rnn_create: out is NULL");
  *out = nullptr;
  const int base = cell & 0xff;
  const bool bidir = (cell & RCU_BIDIR) != 0;
  if ((cell & ~(0xff | RCU_BIDIR)) != 0 || (base != RCU_LSTM && base != RCU_GRU))
    return fail(RCU_ERR_INVALID, "rnn_create: unknown cell %d", cell);
  if (layers < 1 || in_dim < 1 || hidden < 1 || proj < 0)
    return fail(RCU_ERR_INVALID, "rnn_create: layers, in_dim, hidden must be >= 1, proj >= 0");
  if (proj > 0 && base != RCU_LSTM)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_create: projection is only defined for LSTM");
  if (proj >= hidden && proj > 0)
    return fail(RCU_ERR_INVALID, "rnn_create: proj must be smaller than hidden");
  if (dtype != RCU_F32 && dtype != RCU_BF16)
    return fail(RCU_ERR_INVALID, "rnn_create: unknown dtype %d", dtype);
  auto *h = new rcu_rnn_s();
  h->cell = base;
  h->layers = layers;
  h->D = bidir ? 2 : 1;
  h->in_dim = in_dim;
  h->H = hidden;
  h->P = proj;
  h->Hout = proj > 0 ? proj : hidden;
  h->nG = base == RCU_LSTM ? 4 : 3;
  h->dtype = dtype;
  h->nsm = device_sm_count(&h->device);
  plan_simt(h);
  h->in_l.resize(layers);
  h->wih.resize(layers);
  h->wih_f32.resize(layers);
  h->gbias.resize(layers);
  h->host_bias.resize(layers);
  h->lw.resize((size_t)layers * h->D);
  for (int l = 0; l < layers; ++l) {
    h->in_l[l] = l == 0 ? in_dim : h->D * h->Hout;
    h->host_bias[l].assign((size_t)h->D * h->nG * h->H, 0.f);
  }
  cudaError_t e = h->ctl.ensure(ctl_bytes(layers));
  if (e != cudaSuccess) {
    delete h;
    return fail(RCU_ERR_CUDA, "rnn_create: cudaMalloc failed: %s", cudaGetErrorString(e));
  }
  cudaMemset(h->ctl.p, 0, ctl_bytes(layers));
  *out = h;
  return RCU_OK;
}

extern "C" int rnn_set_clip(rcu_rnn_t h, int what, int enable, double lo, double hi) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_set_clip: NULL handle");
  if (what != RCU_CLIP_CELL && what != RCU_CLIP_PROJ)
    return fail(RCU_ERR_INVALID, "rnn_set_clip: unknown target %d", what);
  if (h->cell != RCU_LSTM)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_set_clip: clipping applies to LSTM cells");
  if (what == RCU_CLIP_PROJ && h->P == 0)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_set_clip: projection clipping needs proj > 0");
  if (enable && !(lo <= hi))  // also rejects NaN bounds
    return fail(RCU_ERR_INVALID, "rnn_set_clip: need lo <= hi");
  if (what == RCU_CLIP_CELL) {
    h->cclip = enable != 0;
    h->cclip_lo = (float)lo;
    h->cclip_hi = (float)hi;
  } else {
    h->pclip = enable != 0;
    h->pclip_lo = (float)lo;
    h->pclip_hi = (float)hi;
  }
  return RCU_OK;
}

extern "C" int rnn_set_attr(rcu_rnn_t h, int attr, int64_t value) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_set_attr: NULL handle");
  switch (attr) {
    case RCU_ATTR_BARRIER_TIMEOUT_NS:
      if (value <= 0) return fail(RCU_ERR_INVALID, "timeout must be > 0");
      h->timeout_ns = value;
      return RCU_OK;
    case RCU_ATTR_TEST_DROP_ARRIVAL:
      if (value < 0 || value > 2) return fail(RCU_ERR_INVALID, "drop arrival must be 0, 1 or 2");
      h->drop_arrival = (int)value;
      return RCU_OK;
    case RCU_ATTR_PROFILE:
      h->profile = value != 0;
      return RCU_OK;
    case RCU_ATTR_TC_KSPLIT:
      if (value != 0 && value != 1 && value != 2 && value != 4)
        return fail(RCU_ERR_INVALID, "K split must be 0, 1, 2 or 4");
      h->tc_ksplit = (int)value;
      return RCU_OK;
    case RCU_ATTR_TRACE:
      if (value < 0 || value > 2) return fail(RCU_ERR_INVALID, "trace must be 0, 1 or 2");
      h->trace = (int)value;
      return RCU_OK;
    case RCU_ATTR_LAYER_PIPELINE:
      if (value != 0 && value != 1) return fail(RCU_ERR_INVALID, "layer pipeline must be 0 or 1");
      h->layer_pipeline = (int)value;
      return RCU_OK;
    case RCU_ATTR_FORCE_PATH:
      if (value < 0 || value > 3) return fail(RCU_ERR_INVALID, "force_path must be 0, 1, 2 or 3");
      h->force_path = (int)value;
      return RCU_OK;
    case RCU_ATTR_HOST_CHUNKS:
      if (value < 0 || value > RCU_MAX_HOST_CHUNKS)
        return fail(RCU_ERR_INVALID, "host chunks must be 0 .. %d", RCU_MAX_HOST_CHUNKS);
      h->host_chunks = (int)value;
      return RCU_OK;
    default: return fail(RCU_ERR_INVALID, "rnn_set_attr: unknown attribute %d", attr);
  }
}

extern "C" int rnn_set_weights(rcu_rnn_t h, int layer, int dir, const float *W_ih,
                               const float *W_hh, const float *b_ih, const float *b_hh,
                               const float *W_hr, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_set_weights: NULL handle");
  if (layer < 0 || layer >= h->layers || dir < 0 || dir >= h->D)
    return fail(RCU_ERR_INVALID, "rnn_set_weights: layer %d / dir %d out of range", layer, dir);
  if (!W_ih || !W_hh) return fail(RCU_ERR_INVALID, "rnn_set_weights: W_ih and W_hh are required");
  if ((h->P > 0) != (W_hr != nullptr))
    return fail(RCU_ERR_INVALID, "rnn_set_weights: W_hr must be given iff proj > 0");
  cudaStream_t s = (cudaStream_t)stream;
  const int H = h->H, nG = h->nG, Hout = h->Hout, P = h->P, D = h->D;
  const int in = h->in_l[layer];
  const int ldk = round_up(in, 8);
  std::vector<float> wih, whh, bih, bhh, whr;
  CU(fetch(wih, W_ih, (size_t)nG * H * in, s));
  CU(fetch(whh, W_hh, (size_t)nG * H * Hout, s));
  CU(fetch(bih, b_ih, (size_t)nG * H, s));
  CU(fetch(bhh, b_hh, (size_t)nG * H, s));
  if (P > 0) CU(fetch(whr, W_hr, (size_t)P * H, s));
  const bool bf = h->dtype == RCU_BF16;
  const size_t es = esize(h->dtype);
  auto put = [&](std::vector<unsigned char> &buf, size_t idx, float v) {
    if (bf) {
      uint16_t b = f2bf(v);
      std::memcpy(&buf[idx * 2], &b, 2);
    } else {
      std::memcpy(&buf[idx * 4], &v, 4);
    }
  };

  // --- GEMM weights: rows [dir*nG*H, +nG*H) of the layer's [D*nG*H][ldk] matrix
  DevBuf &gw = h->wih[layer];
  const size_t gw_bytes = (size_t)D * nG * H * ldk * es;
  if (gw.n < gw_bytes) {
    CU(gw.ensure(gw_bytes));
    CU(cudaMemset(gw.p, 0, gw_bytes));
  }
  {
    std::vector<unsigned char> buf((size_t)nG * H * ldk * es, 0);
    for (int r = 0; r < nG * H; ++r)
      for (int k = 0; k < in; ++k) put(buf, (size_t)r * ldk + k, wih[(size_t)r * in + k]);
    CU(cudaMemcpy((char *)gw.p + (size_t)dir * nG * H * ldk * es, buf.data(), buf.size(),
                  cudaMemcpyHostToDevice));
    if (bf) {  // fp32 of the rounded weights, for the backward pass's GEMMs
      DevBuf &gf = h->wih_f32[layer];
      const size_t gf_bytes = (size_t)D * nG * H * ldk * 4;
      if (gf.n < gf_bytes) {
        CU(gf.ensure(gf_bytes));
        CU(cudaMemset(gf.p, 0, gf_bytes));
      }
      std::vector<float> fb((size_t)nG * H * ldk, 0.f);
      for (int r = 0; r < nG * H; ++r)
        for (int k = 0; k < in; ++k) fb[(size_t)r * ldk + k] = bf2f(f2bf(wih[(size_t)r * in + k]));
      CU(cudaMemcpy((char *)gf.p + (size_t)dir * nG * H * ldk * 4, fb.data(), fb.size() * 4,
                    cudaMemcpyHostToDevice));
    }
  }
  // --- GEMM bias: LSTM b_ih + b_hh; GRU r,z: b_ih + b_hh, n: b_ih (b_hn stays with r*(.))
  {
    std::vector<float> &hb = h->host_bias[layer];
    for (int r = 0; r < nG * H; ++r) {
      const bool gru_n = h->cell == RCU_GRU && r >= 2 * H;
      hb[(size_t)dir * nG * H + r] = bih[r] + (gru_n ? 0.f : bhh[r]);
    }
    CU(h->gbias[layer].upload(hb.data(), hb.size() * sizeof(float)));
  }
  LayerDirW &lw = h->lw[(size_t)layer * D + dir];
  // --- recurrent weights, SIMT layout [NU][Kp][Rp]: row g*U + j = gate g of unit ug*U + j
  {
    const int U = h->U, NU = h->NU, Kp = h->Kp, Rp = h->Rp;
    std::vector<unsigned char> buf((size_t)NU * Kp * Rp * es, 0);
    for (int ug = 0; ug < NU; ++ug)
      for (int g = 0; g < nG; ++g)
        for (int j = 0; j < U; ++j) {
          const int u = ug * U + j;
          if (u >= H) continue;
          for (int k = 0; k < Hout; ++k)
            put(buf, ((size_t)ug * Kp + k) * Rp + g * U + j, whh[(size_t)(g * H + u) * Hout + k]);
        }
    CU(lw.whh.upload(buf.data(), buf.size()));
  }
  if (P > 0) {  // projection rows, layout [NP][Hp][Pcp]
    const int Pc = h->Pc, NP = h->NP, Hp = h->Hp, Pcp = h->Pcp;
    std::vector<unsigned char> buf((size_t)NP * Hp * Pcp * es, 0);
    for (int pg = 0; pg < NP; ++pg)
      for (int j = 0; j < Pc; ++j) {
        const int q = pg * Pc + j;
        if (q >= P) continue;
        for (int k = 0; k < H; ++k) put(buf, ((size_t)pg * Hp + k) * Pcp + j, whr[(size_t)q * H + k]);
      }
    CU(lw.whr.upload(buf.data(), buf.size()));
  }
  if (h->cell == RCU_GRU) {
    std::vector<float> bn(H);
    for (int j = 0; j < H; ++j) bn[j] = bhh[2 * H + j];
    CU(lw.bhn.upload(bn.data(), bn.size() * sizeof(float)));
  }
  // --- tensor-core layout (bf16 path only)
  if (bf && tc_rec_packable(h->cell, H, Hout, P)) {
    std::vector<uint16_t> packed;
    tc_pack_whh(h->cell, H, Hout, whh.data(), packed, f2bf);
    CU(lw.tc_whh.upload(packed.data(), packed.size() * 2));
  }
  // --- cluster-resident layout (LSTM/GRU without projection whose W_hh fits
  //     one thread-block cluster's shared memory)
  if (cluster_rec_packable(h->cell, H, Hout, P, bf)) {
    std::vector<float> cw;
    cluster_pack_whh(h->cell, H, Hout, whh.data(), cw);
    std::vector<unsigned char> buf(cw.size() * es);
    for (size_t i = 0; i < cw.size(); ++i) put(buf, i, cw[i]);
    CU(lw.cl_whh.upload(buf.data(), buf.size()));
  }
  // --- LSTMP on the tensor cores: recurrent weight W_hh W_hr over m (from the
  //     bf16-rounded factors, product accumulated in fp32, rounded to bf16)
  if (bf && P > 0 && tc_rec_packable(RCU_LSTM, H, H, 0)) {
    const int G4 = nG * H, ldH = round_up(H, 8);
    std::vector<float> whh_r((size_t)G4 * P), whr_r((size_t)P * H), wp((size_t)G4 * H, 0.f);
    for (size_t i = 0; i < whh_r.size(); ++i) whh_r[i] = bf2f(f2bf(whh[i]));
    for (size_t i = 0; i < whr_r.size(); ++i) whr_r[i] = bf2f(f2bf(whr[i]));
    for (int r = 0; r < G4; ++r) {
      float *dst = &wp[(size_t)r * H];
      for (int q = 0; q < P; ++q) {
        const float a = whh_r[(size_t)r * P + q];
        const float *src = &whr_r[(size_t)q * H];
        for (int k = 0; k < H; ++k) dst[k] += a * src[k];
      }
    }
    std::vector<uint16_t> packed;
    tc_pack_whh(RCU_LSTM, H, H, wp.data(), packed, f2bf);
    CU(lw.fold_w.upload(packed.data(), packed.size() * 2));
    CU(lw.whh_f32.upload(whh_r.data(), whh_r.size() * 4));
    std::vector<uint16_t> hr((size_t)P * ldH, 0);
    for (int q = 0; q < P; ++q)
      for (int k = 0; k < H; ++k) hr[(size_t)q * ldH + k] = f2bf(whr[(size_t)q * H + k]);
    CU(lw.whr_bf.upload(hr.data(), hr.size() * 2));
  }
  // --- plain fp32 copies for the backward pass (bf16 handles: of the rounded
  //     weight matrices; biases stay fp32 as in the forward)
  {
    auto rw = [&](float v) { return bf ? bf2f(f2bf(v)) : v; };
    const int ldo = round_up(Hout, 8);
    std::vector<float> wp((size_t)nG * H * ldo, 0.f);
    for (int r = 0; r < nG * H; ++r)
      for (int k = 0; k < Hout; ++k) wp[(size_t)r * ldo + k] = rw(whh[(size_t)r * Hout + k]);
    CU(lw.whh_plain.upload(wp.data(), wp.size() * 4));
    CU(lw.bih_plain.upload(bih.data(), (size_t)nG * H * 4));
    CU(lw.bhh_plain.upload(bhh.data(), (size_t)nG * H * 4));
    if (P > 0) {
      std::vector<float> hr((size_t)P * H);
      for (size_t q = 0; q < hr.size(); ++q) hr[q] = rw(whr[q]);
      CU(lw.whr_plain.upload(hr.data(), hr.size() * 4));
    }
  }
  lw.set = true;
  return RCU_OK;
}

// Workspace for T, B (grows on demand).
static int ensure_ws(rcu_rnn_s *h, int T, int B) {
  if (T <= h->ws_T && B <= h->ws_B && h->ws.p) {
    // reuse; pointers were laid out for (ws_T, ws_B) and stay valid for smaller shapes
  } else {
    const int Tm = std::max(T, h->ws_T), Bm = std::max(B, h->ws_B);
    const size_t M = (size_t)Tm * Bm;
    const size_t es = esize(h->dtype);
    const int N = h->D * h->nG * h->H;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t r = off; off = round_up_sz(off + bytes, 256); return r; };
    const size_t o_meta = take(((size_t)3 * Bm + 2 * Tm + 1) * 4);
    const size_t o_xp = take(M * round_up(h->in_dim, 8) * es);
    const size_t o_g = take(M * N * 4);
    const size_t o_ymid = h->layers > 1 ? take(M * h->D * h->Hout * es) : 0;
    const size_t o_hx = take((size_t)h->D * 2 * Bm * h->Kp * es);
    const size_t o_mx = take((size_t)h->D * Bm * h->Hp * es);
    const size_t o_hst = take((size_t)h->D * Bm * h->Hout * 4);
    const size_t o_cst = take((size_t)h->D * Bm * h->H * 4);
    // LSTMP tensor-core path: m_t of every step (bf16), its exchange buffer,
    // and the fp32 projected outputs of the non-final layers
    const bool fold = h->P > 0 && h->dtype == RCU_BF16;
    const size_t ldH = round_up(h->H, 8);
    const size_t o_mbuf = fold ? take(M * h->D * h->H * 2) : 0;
    const size_t o_hx2 = fold ? take((size_t)h->D * 2 * Bm * ldH * 2) : 0;
    const size_t o_ytmp = (fold && h->layers > 1) ? take(M * h->D * h->P * 4) : 0;
    cudaError_t e = h->ws.ensure(off);
    if (e != cudaSuccess)
      return fail(RCU_ERR_CUDA, "workspace allocation of %zu bytes failed: %s", off,
                  cudaGetErrorString(e));
    char *base = (char *)h->ws.p;
    int32_t *mi = (int32_t *)(base + o_meta);
    h->meta.sorted_idx = mi;
    h->meta.unsorted_idx = mi + Bm;
    h->meta.lens_sorted = mi + 2 * Bm;
    h->meta.batch_sizes = mi + 3 * Bm;
    h->meta.step_off = mi + 3 * Bm + Tm;
    h->xp = base + o_xp;
    h->g = base + o_g;
    h->ymid = h->layers > 1 ? base + o_ymid : nullptr;
    h->hx = base + o_hx;
    h->mx = base + o_mx;
    h->hst = (float *)(base + o_hst);
    h->cst = (float *)(base + o_cst);
    h->mbuf = fold ? base + o_mbuf : nullptr;
    h->hx2 = fold ? base + o_hx2 : nullptr;
    h->ytmp = (fold && h->layers > 1) ? (float *)(base + o_ytmp) : nullptr;
    h->ws_T = Tm;
    h->ws_B = Bm;
    h->meta_T = h->meta_B = -1;  // the metadata moved
  }
  return RCU_OK;
}

// ---------------------------------------------------------------------------
// Layer-pipelined forward of a stacked unidirectional LSTMP on the tensor-core
// path.  A layer's recurrence on the tensor cores holds one batch group of
// B <= 128 rows on a fraction of the GPU (64 CTAs for H = 1024), so layer l+1
// can run steps [t0, t1) while layer l runs the next steps.  The sequence is
// cut into chunks of steps; layer l runs its chunks in order on its own
// stream, each chunk a launch of the folded recurrence that starts from the
// previous chunk's final m and c (fp32) and reads the chunk's G rows.
// Between layer l's chunk c and layer l+1's chunk c, on layer l+1's stream:
// the projection of chunk c (h = W_hr m), its conversion to the next layer's
// bf16 operand and the next layer's input GEMM for the chunk.  Every row of
// these GEMMs depends only on its own inputs and every recurrent step starts
// from the same bf16(m_{t-1}) and fp32 c_{t-1} as without chunks, so the
// results equal the unpipelined ones.  The GEMMs that run beside a
// recurrence use the SMs it leaves free.
// fp32 C = A B^T + bias (row strides lda, ldb, ldc): on the tensor cores as a
// three-term bf16 split of both operands (launch_gemm_f32x6: fp32-accurate,
// small products first, long reductions in chunks) when the product is
// large enough to pay for the split passes, else the FFMA GEMM.
// RCU_ATTR_FORCE_PATH = 1 keeps the FFMA GEMM, 2 takes the split one at any
// size.  *n counts the kernels launched.
static constexpr double F32X6_MIN_MACS = 2.0e8;
static bool use_f32x6(rcu_rnn_t h, int M, const int32_t *M_dev, int N, int K, int ldc,
                      const void *C) {
  const bool big = (double)M * N * K >= F32X6_MIN_MACS || h->force_path == 2;
  return h->force_path != 1 && big && (!M_dev || K <= 4096) && f32x6_supported(N, ldc, C);
}
static cudaError_t gemm_f32(rcu_rnn_t h, const float *A, int lda, const float *B, int ldb,
                            const float *bias, float *C, int ldc, int M, const int32_t *M_dev,
                            int N, int K, cudaStream_t s, int *err, int *n) {
  if (use_f32x6(h, M, M_dev, N, K, ldc, C)) {
    cudaError_t e = h->f32x.ensure(f32x6_scratch_bytes(M, N, K));
    if (e != cudaSuccess) return e;
    *n += f32x6_launches(K);
    return launch_gemm_f32x6(A, lda, B, ldb, bias, C, ldc, M, M_dev, N, K, h->f32x.p, h->nsm, s,
                             err, (uint64_t)h->timeout_ns);
  }
  *n += 1;
  return launch_gemm_simt<float, float>(A, lda, B, ldb, bias, C, ldc, M, M_dev, N, K, s, err);
}

static int lp_chunks(int T) { return std::min(32, std::max(2, T / 64)); }

static bool layer_pipeline_ok(rcu_rnn_t h, int T, int B, bool varlen, bool bf) {
  if (!h->layer_pipeline || !bf || h->D != 1 || h->layers < 2 || varlen || h->pclip ||
      h->force_path == 1 || h->trace || T < 128)
    return false;
  const int H = h->H, P = h->P;
  if ((H % 8) != 0) return false;
  if (P > 0) {
    if (!h->mbuf || !tc_rec_supported(RCU_LSTM, H, H, 0, h->nsm, B, 1) || !tc_gemm_supported(H, P))
      return false;
    for (int l = 0; l < h->layers; ++l)
      if (!h->lw[l].fold_w.p || !tc_gemm_supported(h->in_l[l], h->nG * H)) return false;
    // two recurrences side by side, and room beside one of them for the GEMMs
    const int rg = tc_rec_grid(RCU_LSTM, H, H, B, 1, h->tc_ksplit);
    return 2 * rg <= h->nsm && h->nsm - rg >= 16;
  }
  // No projection: only where the layer-by-layer forward would take the
  // tensor-core recurrence, and without the training pass's kept outputs.
  if (h->force_path == 3 || h->keep_out || !tc_rec_supported(h->cell, H, H, 0, h->nsm, B, 1))
    return false;
  ClusterRecPlan cp{};
  if (h->force_path == 0 && h->lw[0].cl_whh.p &&
      plan_recurrent_cluster(&cp, h->cell, H, H, T, B, 1, bf, 16))
    return false;
  for (int l = 0; l < h->layers; ++l)
    if (!h->lw[l].tc_whh.p || !tc_gemm_supported(h->in_l[l], h->nG * H)) return false;
  // Only where two layers' recurrences fit side by side (as for LSTMP): a
  // recurrence that fills the GPU (the 3-layer GRU's 128 CTAs) gains ~1 %
  // from chunking, since the next layer's GEMM then runs on the few SMs left
  // and its memory traffic slows the latency-bound steps beside it.
  const int rg = tc_rec_grid(h->cell, H, H, B, 1, h->tc_ksplit);
  return 2 * rg <= h->nsm && h->nsm - rg >= 16;
}

static int forward_layer_pipelined(rcu_rnn_t h, int T, int B, const void *X0, int ldx0,
                                   const float *h0, const float *c0, float *y, float *h_n,
                                   float *c_n, int *err, cudaStream_t s) {
  const int L = h->layers, H = h->H, P = h->P, nG = h->nG, G4 = nG * H;
  // proj: LSTMP, whose recurrence runs on m with W_hh W_hr folded, each
  // chunk's projection a GEMM; otherwise the layer's own recurrence writes
  // the next layer's bf16 input (or y) directly
  const bool proj = P > 0;
  const int rcell = proj ? RCU_LSTM : h->cell, Ho = proj ? P : H;
  const int ldH = round_up(H, 8);
  const int n = lp_chunks(T);
  const int Tc = ceil_div(T, n), nch = ceil_div(T, Tc), Tl = T - (nch - 1) * Tc;
  const int rg = tc_rec_grid(rcell, H, H, B, 1, h->tc_ksplit);
  const int gemm_sms = std::max(16, h->nsm - rg);
  const int cstride = std::max(4, tc_rec_counters(B, 1));
  // resources
  while ((int)h->lp_streams.size() < L - 1) {
    cudaStream_t st;
    CU(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
    h->lp_streams.push_back(st);
  }
  const int nev = L * nch + L;
  while ((int)h->lp_events.size() < nev) {
    cudaEvent_t e;
    CU(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    h->lp_events.push_back(e);
  }
  CU(h->lp_ctl.ensure((size_t)L * nch * cstride * 4));
  CU(h->lp_hx.ensure((size_t)L * 2 * B * ldH * 2));
  // per layer: m and c at the chunk boundaries, ping-pong [2][B][H] each
  CU(h->lp_state.ensure((size_t)L * 4 * B * H * 4));
  // chunk metadata for lengths Tc and Tl (identity order)
  const size_t meta_ints = (size_t)3 * B + 2 * (size_t)Tc + 1;
  CU(h->lp_meta.ensure(2 * meta_ints * 4));
  Meta mc[2];
  for (int i = 0; i < 2; ++i) {
    int32_t *mi = (int32_t *)h->lp_meta.p + i * meta_ints;
    mc[i].sorted_idx = mi;
    mc[i].unsorted_idx = mi + B;
    mc[i].lens_sorted = mi + 2 * B;
    mc[i].batch_sizes = mi + 3 * B;
    mc[i].step_off = mi + 3 * B + Tc;
  }
  CU(cudaMemsetAsync(h->lp_ctl.p, 0, (size_t)L * nch * cstride * 4, s));
  CU(cudaMemsetAsync(h->lp_hx.p, 0, (size_t)L * 2 * B * ldH * 2, s));
  for (int i = 0; i < 2; ++i) {
    h->begin("meta_sort", s);
    CU(launch_meta(nullptr, B, i == 0 ? Tc : Tl, mc[i], err, s));
    h->end(s);
  }
  // every layer's stream starts after the work already on s
  cudaEvent_t *ev = h->lp_events.data();  // ev[l*nch + c]: layer l finished chunk c
  cudaEvent_t *ev_done = ev + L * nch;     // ev_done[l]: layer l's stream is done
  CU(cudaEventRecord(ev_done[0], s));
  for (int l = 1; l < L; ++l) CU(cudaStreamWaitEvent(h->lp_streams[l - 1], ev_done[0], 0));
  auto stream_of = [&](int l) { return l == 0 ? s : h->lp_streams[l - 1]; };

  float *G = (float *)h->g;
  __nv_bfloat16 *mbuf = (__nv_bfloat16 *)h->mbuf;
  // layer 0's input projection for all steps at once (nothing runs beside it yet)
  h->begin("input_gemm_tc", s);
  {
    cudaError_t e = launch_tc_gemm((const __nv_bfloat16 *)X0, ldx0,
                                   (const __nv_bfloat16 *)h->wih[0].p, round_up(h->in_l[0], 8),
                                   (const float *)h->gbias[0].p, G, G4, T * B, nullptr, G4,
                                   h->in_l[0], h->nsm, s, err, (uint64_t)h->timeout_ns);
    if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc gemm: %s", cudaGetErrorString(e));
  }
  h->end(s);
  for (int c = 0; c < nch; ++c) {
    const int t0 = c * Tc, tc = c + 1 < nch ? Tc : Tl;
    const size_t r0 = (size_t)t0 * B;  // first packed row of the chunk
    for (int l = 0; l < L; ++l) {
      cudaStream_t sl = stream_of(l);
      const bool last = l == L - 1;
      if (l > 0) {
        // layer l-1 finished chunk c: project it and convert (LSTMP), and
        // form this layer's gate pre-activations for the chunk
        CU(cudaStreamWaitEvent(sl, ev[(l - 1) * nch + c], 0));
      }
      if (l > 0 && proj) {
        float *Yp = h->keep_out ? h->keep_out + (size_t)(l - 1) * T * B * P : h->ytmp;
        h->begin("projection_gemm_tc", sl);
        cudaError_t e = launch_tc_gemm(mbuf + r0 * H, H, (const __nv_bfloat16 *)h->lw[l - 1].whr_bf.p,
                                       ldH, nullptr, Yp + r0 * P, P, tc * B, nullptr, P, H,
                                       gemm_sms, sl, err, (uint64_t)h->timeout_ns);
        h->end(sl);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "projection gemm: %s", cudaGetErrorString(e));
        if (c == nch - 1 && h_n) {
          h->begin("last_h", sl);
          CU(launch_last_h(Yp, P, h_n + (size_t)(l - 1) * B * P, B, T, P, 0, sl));
          h->end(sl);
        }
        h->begin("convert_bf16", sl);
        CU(launch_convert<__nv_bfloat16>(Yp + r0 * P, (__nv_bfloat16 *)h->ymid + r0 * P,
                                         (size_t)tc * B * P, sl));
        h->end(sl);
      }
      if (l > 0) {
        // (rows [r0, r0 + tc*B) of ymid hold layer l-1's output for the chunk;
        // this layer's recurrence overwrites them only after this GEMM)
        h->begin("input_gemm_tc", sl);
        cudaError_t e = launch_tc_gemm((const __nv_bfloat16 *)h->ymid + r0 * Ho, Ho,
                                       (const __nv_bfloat16 *)h->wih[l].p, round_up(h->in_l[l], 8),
                                       (const float *)h->gbias[l].p, G + r0 * G4, G4, tc * B,
                                       nullptr, G4, h->in_l[l], gemm_sms, sl, err,
                                       (uint64_t)h->timeout_ns);
        h->end(sl);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc gemm: %s", cudaGetErrorString(e));
      }
      // the layer's initial projected state enters as W_hh h0 in the first step's G
      if (proj && c == 0 && h0) {
        h->begin("h0_gates", sl);
        CU(launch_h0_gates(G, G4, (const float *)h->lw[l].whh_f32.p, h0 + (size_t)l * B * P, B,
                           tc, G4, P, 0, sl));
        h->end(sl);
      }
      float *st = (float *)h->lp_state.p + (size_t)l * 4 * B * H;  // [m0, m1, c0, c1][B][H]
      float *m_in = st + (size_t)((c + 1) & 1) * B * H, *m_out = st + (size_t)(c & 1) * B * H;
      float *c_in = st + (size_t)(2 + ((c + 1) & 1)) * B * H;
      float *c_out = st + (size_t)(2 + (c & 1)) * B * H;
      RecParams pf{};
      pf.T = tc; pf.B = B; pf.H = H; pf.Hout = H; pf.Kp = ldH; pf.Hp = h->Hp; pf.nG = nG; pf.D = 1;
      pf.cell = rcell; pf.proj = 0;
      pf.U = h->U; pf.NU = h->NU; pf.Rp = h->Rp;
      pf.meta = mc[c + 1 < nch ? 0 : 1];
      pf.G = G + r0 * G4;
      pf.ldG = G4;
      pf.bhn[0] = proj ? nullptr : (const float *)h->lw[l].bhn.p;
      pf.bhn[1] = nullptr;
      // LSTMP: m_{-1} does not enter the first chunk (W_hh h0 is in G).  Later
      // chunks start from the previous chunk's state (m or h, and c), rounded
      // to bf16 by the kernel as every step's exchange is.
      const float *h0l = (!proj && h0) ? h0 + (size_t)l * B * H : nullptr;
      pf.h0 = c == 0 ? h0l : m_in;
      if (nG == 4) {
        pf.c0 = c == 0 ? (c0 ? c0 + (size_t)l * B * H : nullptr) : c_in;
        pf.c_n = (c == nch - 1 && c_n) ? c_n + (size_t)l * B * H : c_out;
      }
      pf.h_n = (!proj && c == nch - 1 && h_n) ? h_n + (size_t)l * B * H : m_out;
      if (proj) {
        pf.y = nullptr;
        pf.ymid = mbuf + r0 * H;
      } else {
        pf.y = last ? y + r0 * H : nullptr;
        pf.ymid = last ? nullptr : (__nv_bfloat16 *)h->ymid + r0 * H;
      }
      pf.hx = (char *)h->lp_hx.p + (size_t)l * 2 * B * ldH * 2;
      pf.mx = h->mx; pf.hst = h->hst; pf.cst = h->cst;
      pf.ctr = (unsigned *)h->lp_ctl.p + ((size_t)l * nch + c) * cstride;
      pf.err = err;
      pf.timeout_ns = (uint64_t)h->timeout_ns;
      pf.drop_arrival = h->drop_arrival == 1 && l == 0 && c == 0;
      pf.cclip = h->cclip; pf.cclip_lo = h->cclip_lo; pf.cclip_hi = h->cclip_hi;
      TcRecParams tp;
      tp.base = pf;
      tp.ksplit = h->tc_ksplit;
      tp.fixed_length = true;
      tp.Wtc[0] = tp.Wtc[1] = proj ? h->lw[l].fold_w.p : h->lw[l].tc_whh.p;
      h->begin(proj ? "recurrent_tc_lstmp" : "recurrent_tc", sl);
      cudaError_t e = launch_tc_recurrent(tp, h->nsm, sl);
      h->end(sl);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc recurrent: %s", cudaGetErrorString(e));
      CU(cudaEventRecord(ev[l * nch + c], sl));
      if (last && proj) {
        // the last layer's projection of the chunk, straight into y
        h->begin("projection_gemm_tc", sl);
        e = launch_tc_gemm(mbuf + r0 * H, H, (const __nv_bfloat16 *)h->lw[l].whr_bf.p, ldH,
                           nullptr, y + r0 * P, P, tc * B, nullptr, P, H, gemm_sms, sl, err,
                           (uint64_t)h->timeout_ns);
        h->end(sl);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "projection gemm: %s", cudaGetErrorString(e));
        if (c == nch - 1 && h_n) {
          h->begin("last_h", sl);
          CU(launch_last_h(y, P, h_n + (size_t)l * B * P, B, T, P, 0, sl));
          h->end(sl);
        }
      }
    }
  }
  // the call is complete on s once every layer's stream is
  for (int l = 1; l < L; ++l) {
    CU(cudaEventRecord(ev_done[l], h->lp_streams[l - 1]));
    CU(cudaStreamWaitEvent(s, ev_done[l], 0));
  }
  return RCU_OK;
}

extern "C" int rnn_forward(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                           const float *h0, const float *c0, const float *eps, float *y,
                           float *h_n, float *c_n, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_forward: NULL handle");
  h->launches = 0;
  if (T < 0 || B < 0) return fail(RCU_ERR_INVALID, "rnn_forward: T and B must be >= 0");
  if (eps) return fail(RCU_ERR_INVALID, "rnn_forward: eps is reserved and must be NULL");
  if (h->cell == RCU_GRU && (c0 || c_n))
    return fail(RCU_ERR_INVALID, "rnn_forward: c0/c_n are LSTM-only");
  for (auto &w : h->lw)
    if (!w.set) return fail(RCU_ERR_STATE, "rnn_forward: weights missing for some layer/direction");
  if (T == 0 || B == 0) return RCU_OK;
  if (!x || !y) return fail(RCU_ERR_INVALID, "rnn_forward: x and y are required");
  if ((size_t)T * B > (size_t)INT32_MAX / 4)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_forward: T*B too large");
  if (int rc = ensure_ws(h, T, B)) return rc;
  h->last_T = T;
  h->last_B = B;
  cudaStream_t s = (cudaStream_t)stream;
  const bool bf = h->dtype == RCU_BF16;
  const size_t es = esize(h->dtype);
  const int D = h->D, H = h->H, Hout = h->Hout, nG = h->nG;
  const int N = D * nG * H;
  const bool varlen = lengths != nullptr;
  // control block: error word, then per layer `cstride` barrier counters
  const int cstride = std::max(4, tc_rec_counters(B, D));
  const size_t cbytes = 64 + (size_t)h->layers * cstride * 4 + 64;
  CU(h->ctl.ensure(std::max(cbytes, ctl_bytes(h->layers))));
  int *err = (int *)h->ctl.p;
  unsigned *ctr = (unsigned *)((char *)h->ctl.p + 64);

  CU(cudaMemsetAsync(h->ctl.p, 0, std::max(cbytes, ctl_bytes(h->layers)), s));
  CU(cudaMemsetAsync(h->hx, 0, (size_t)D * 2 * B * h->Kp * es, s));
  if (h->trace) {
    const size_t rows = (size_t)T + (h->trace == 2 ? (size_t)TRACE_ALL_N * TRACE_ALL_CTAS : 0);
    CU(h->trace_buf.ensure(rows * 16 * 8));
    CU(cudaMemsetAsync(h->trace_buf.p, 0, rows * 16 * 8, s));
    h->trace_T = (int)rows;
  }
  if (h->P > 0) CU(cudaMemsetAsync(h->mx, 0, (size_t)D * B * h->Hp * es, s));
  if (varlen || T != h->meta_T || B != h->meta_B || s != h->meta_s) {
    h->begin("meta_sort", s);
    CU(launch_meta(lengths, B, T, h->meta, err, s));
    h->end(s);
    h->meta_T = varlen ? -1 : T;
    h->meta_B = varlen ? -1 : B;
    h->meta_s = s;
  }
  if (varlen) {
    h->begin("zero_tail", s);
    CU(launch_zero_tail(y, lengths, T, B, D * Hout, err, s));
    h->end(s);
  }

  // layer-0 GEMM operand
  const void *X = x;
  int ldx = h->in_dim;
  const int32_t *M_dev = varlen ? h->meta.step_off + T : nullptr;
  const int Mmax = T * B;
  if (varlen || bf || h->x_in_place) {
    ldx = round_up(h->in_dim, 8);
    h->begin("pack_rows", s);
    if (bf)
      CU(launch_pack_rows<__nv_bfloat16>(x, T, B, h->in_dim, h->meta, (__nv_bfloat16 *)h->xp,
                                         ldx, s));
    else
      CU(launch_pack_rows<float>(x, T, B, h->in_dim, h->meta, (float *)h->xp, ldx, s));
    h->end(s);
    X = h->xp;
  }
  h->used_tc_gemm = h->used_tc_rec = false;
  if (layer_pipeline_ok(h, T, B, varlen, bf)) {
    h->used_tc_gemm = h->used_tc_rec = true;
    return forward_layer_pipelined(h, T, B, X, ldx, h0, c0, y, h_n, c_n, err, s);
  }
  for (int l = 0; l < h->layers; ++l) {
    const int K = h->in_l[l];
    const int ldw = round_up(K, 8);
    float *G = (float *)h->g;
    bool done = false;
    // TMA needs 16-byte row strides: the tensor-core GEMM takes rows of a multiple of 8
    const bool tc_gemm = bf && h->force_path != 1 && (ldx % 8) == 0 && tc_gemm_supported(K, N);
    h->begin(tc_gemm ? "input_gemm_tc"
                     : (!bf && use_f32x6(h, Mmax, M_dev, N, K, N, G)) ? "input_gemm_f32x6"
                                                                      : "input_gemm_simt",
             s);
    if (tc_gemm) {
      cudaError_t e = launch_tc_gemm((const __nv_bfloat16 *)X, ldx, (const __nv_bfloat16 *)h->wih[l].p,
                                     ldw, (const float *)h->gbias[l].p, G, N, Mmax, M_dev, N, K,
                                     h->nsm, s, err, (uint64_t)h->timeout_ns);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc gemm: %s", cudaGetErrorString(e));
      done = true;
      h->used_tc_gemm = true;
    }
    if (!done) {
      int nk = 0;
      cudaError_t e = bf ? launch_gemm_simt<__nv_bfloat16, __nv_bfloat16>(
                               (const __nv_bfloat16 *)X, ldx, (const __nv_bfloat16 *)h->wih[l].p,
                               ldw, (const float *)h->gbias[l].p, G, N, Mmax, M_dev, N, K, s, err)
                         : gemm_f32(h, (const float *)X, ldx, (const float *)h->wih[l].p, ldw,
                                    (const float *)h->gbias[l].p, G, N, Mmax, M_dev, N, K, s, err,
                                    &nk);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "gemm: %s", cudaGetErrorString(e));
      if (nk > 1) h->launches += nk - 1;  // (the profile range counts one)
    }
    h->end(s);

    const bool last = l == h->layers - 1;
    RecParams p{};
    p.T = T; p.B = B; p.H = H; p.Hout = Hout; p.Kp = h->Kp; p.Hp = h->Hp; p.nG = nG; p.D = D;
    p.cell = h->cell; p.proj = h->P;
    p.U = h->U; p.NU = h->NU; p.Rp = h->Rp;
    p.Pc = h->Pc; p.Pcp = h->Pcp; p.NP = h->NP;
    p.meta = h->meta;
    p.G = G; p.ldG = N;
    for (int d = 0; d < D; ++d) {
      LayerDirW &lw = h->lw[(size_t)l * D + d];
      p.Whh[d] = lw.whh.p;
      p.Whr[d] = lw.whr.p;
      p.bhn[d] = (const float *)lw.bhn.p;
    }
    p.h0 = h0 ? h0 + (size_t)l * D * B * Hout : nullptr;
    p.c0 = c0 ? c0 + (size_t)l * D * B * H : nullptr;
    p.h_n = h_n ? h_n + (size_t)l * D * B * Hout : nullptr;
    p.c_n = c_n ? c_n + (size_t)l * D * B * H : nullptr;
    p.y = last ? y : (h->keep_out ? h->keep_out + (size_t)l * T * B * D * Hout : nullptr);
    p.ymid = last ? nullptr : h->ymid;
    p.hx = h->hx; p.mx = h->mx; p.hst = h->hst; p.cst = h->cst;
    p.ctr = ctr + (size_t)cstride * l;  // fresh counters per layer (zeroed above)
    p.err = err;
    p.timeout_ns = (uint64_t)h->timeout_ns;
    p.drop_arrival = h->drop_arrival == 1 && l == 0;
    p.trace = (h->trace && l == 0) ? (unsigned long long *)h->trace_buf.p : nullptr;
    p.trace_all = (h->trace == 2 && l == 0) ? (unsigned long long *)h->trace_buf.p + (size_t)T * 16
                                            : nullptr;
    p.cclip = h->cclip;
    p.cclip_lo = h->cclip_lo;
    p.cclip_hi = h->cclip_hi;
    p.pclip = h->pclip;
    p.pclip_lo = h->pclip_lo;
    p.pclip_hi = h->pclip_hi;

    // ---- LSTMP on the tensor cores: recurrence on m with W_hh W_hr resident,
    //      then the projection of every step as one GEMM
    const int P = h->P, ldH = round_up(H, 8);
    // (a projection clip is applied to h_t before it feeds the next step, so
    // the recurrence cannot be folded onto m)
    const bool folded = bf && P > 0 && !varlen && !h->pclip && h->force_path != 1 && h->mbuf &&
                        h->lw[(size_t)l * D].fold_w.p && (H % 8) == 0 && ((D * H) % 8) == 0 &&
                        tc_rec_supported(RCU_LSTM, H, H, 0, h->nsm, B, D) &&
                        tc_gemm_supported(H, P);
    if (folded) {
      if (h0) {
        h->begin("h0_gates", s);
        for (int d = 0; d < D; ++d)
          CU(launch_h0_gates(G, N, (const float *)h->lw[(size_t)l * D + d].whh_f32.p,
                             h0 + ((size_t)l * D + d) * B * P, B, T, nG * H, P, d, s));
        h->end(s);
      }
      RecParams pf = p;
      pf.Hout = H;
      pf.Kp = ldH;
      pf.proj = 0;
      pf.hx = h->hx2;
      pf.y = nullptr;
      pf.ymid = h->mbuf;  // m_t, packed rows, bf16 [T*B][D*H]
      pf.h0 = nullptr;    // m_{-1} does not enter: the h0 term is in G already
      pf.h_n = nullptr;
      CU(cudaMemsetAsync(h->hx2, 0, (size_t)D * 2 * B * ldH * 2, s));
      TcRecParams tp;
      tp.base = pf;
      tp.ksplit = h->tc_ksplit;
      tp.fixed_length = !varlen;
      for (int d = 0; d < D; ++d) tp.Wtc[d] = h->lw[(size_t)l * D + d].fold_w.p;
      h->begin("recurrent_tc_lstmp", s);
      cudaError_t e = launch_tc_recurrent(tp, h->nsm, s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc recurrent: %s", cudaGetErrorString(e));
      h->end(s);
      h->used_tc_rec = true;
      // projection h_t = W_hr m_t for all steps and directions
      float *Y = last ? y : (h->keep_out ? h->keep_out + (size_t)l * T * B * D * Hout : h->ytmp);
      h->begin("projection_gemm_tc", s);
      for (int d = 0; d < D; ++d) {
        e = launch_tc_gemm((const __nv_bfloat16 *)h->mbuf + (size_t)d * H, D * H,
                           (const __nv_bfloat16 *)h->lw[(size_t)l * D + d].whr_bf.p, ldH, nullptr,
                           Y + (size_t)d * P, D * P, Mmax, nullptr, P, H, h->nsm, s, err,
                           (uint64_t)h->timeout_ns);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "projection gemm: %s", cudaGetErrorString(e));
      }
      h->end(s);
      if (h_n) {
        h->begin("last_h", s);
        for (int d = 0; d < D; ++d)
          CU(launch_last_h(Y, D * P, h_n + ((size_t)l * D + d) * B * P, B, T, P, d, s));
        h->end(s);
      }
      if (!last) {
        h->begin("convert_bf16", s);
        CU(launch_convert<__nv_bfloat16>(Y, (__nv_bfloat16 *)h->ymid, (size_t)Mmax * D * P,
                                         s));
        h->end(s);
      }
      X = h->ymid;
      ldx = D * Hout;
      continue;
    }

    bool rec_done = false;
    // small problems first: the cluster-resident kernel (automatic when W_hh
    // fits one cluster and the batch slices have at most 16 rows), else the
    // tensor-core grid for bf16, else the SIMT grid
    ClusterRecPlan cp{};
    const bool cl_rec = (h->force_path == 0 || h->force_path == 3) &&
                        h->lw[(size_t)l * D].cl_whh.p &&
                        plan_recurrent_cluster(&cp, h->cell, H, Hout, T, B, D, bf,
                                               h->force_path == 3 ? (1 << 30) : 16);
    const bool tc_rec = !cl_rec && bf && (h->force_path == 0 || h->force_path == 2) &&
                        tc_rec_supported(h->cell, H, Hout, h->P, h->nsm, B, D) &&
                        h->lw[(size_t)l * D].tc_whh.p;
    h->begin(tc_rec ? "recurrent_tc" : cl_rec ? "recurrent_cluster" : "recurrent_simt", s);
    if (tc_rec) {
      TcRecParams tp;
      tp.base = p;
      tp.ksplit = h->tc_ksplit;
      tp.fixed_length = !varlen;
      for (int d = 0; d < D; ++d) tp.Wtc[d] = h->lw[(size_t)l * D + d].tc_whh.p;
      cudaError_t e = launch_tc_recurrent(tp, h->nsm, s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "tc recurrent: %s", cudaGetErrorString(e));
      rec_done = true;
      h->used_tc_rec = true;
    } else if (cl_rec) {
      cudaError_t e = launch_recurrent_cluster(p, cp, h->lw[(size_t)l * D].cl_whh.p,
                                               h->lw[(size_t)l * D + (D - 1)].cl_whh.p, bf, s);
      if (e != cudaSuccess)
        return fail(RCU_ERR_CUDA, "cluster recurrent kernel: %s", cudaGetErrorString(e));
      rec_done = true;
    }
    if (!rec_done) {
      // the batch chunk is shrunk until the shared-memory plan fits
      if (!plan_recurrent_simt(p, bf))
        return fail(RCU_ERR_UNSUPPORTED, "recurrent kernel: resident weights do not fit");
      cudaError_t e = launch_recurrent_simt(p, bf, h->nsm, s);
      if (e != cudaSuccess)
        return fail(RCU_ERR_CUDA, "recurrent kernel launch: %s", cudaGetErrorString(e));
    }
    h->end(s);
    // next layer reads this layer's packed output
    X = h->ymid;
    ldx = D * Hout;
  }
  (void)es;
  return RCU_OK;
}


// rnn_forward_host over n chunks of steps.  A forward over steps [t0, t1)
// needs only those steps' x and every layer's state at t0 (its h_n / c_n
// after the previous chunk), so each chunk is one rnn_forward with the
// per-layer state carried in fp32 device buffers: the results are the
// unchunked ones.  Copy stream cp_in moves x chunk c+2 in while chunk c+1
// computes, cp_out moves y chunk c out meanwhile; only the first chunk's x
// and the last chunk's y are not hidden behind compute, so those two chunks
// are a quarter of the others' length.
static int forward_host_chunked(rcu_rnn_t h, int T, int B, int n, const float *x,
                                const float *h0, const float *c0, float *y, float *h_n,
                                float *c_n, cudaStream_t s) {
  // chunk starts: q, then n-2 equal chunks, then q steps (q = a quarter chunk)
  int t_at[RCU_MAX_HOST_CHUNKS + 1];
  {
    const int q = n >= 3 ? std::max(1, T / (4 * (n - 2) + 2)) : 0;
    const int mid = n >= 3 ? n - 2 : n, span = T - 2 * q;
    t_at[0] = 0;
    int c = 0;
    if (q > 0) t_at[++c] = q;
    for (int i = 1; i <= mid; ++i) t_at[++c] = q + (int)((long long)span * i / mid);
    if (q > 0) t_at[++c] = T;
    n = c;
  }
  int Tc = 0;
  for (int c = 0; c < n; ++c) Tc = std::max(Tc, t_at[c + 1] - t_at[c]);
  const size_t in_row = (size_t)B * h->in_dim, out_row = (size_t)B * h->D * h->Hout;
  const size_t LDB = (size_t)h->layers * h->D * B;
  const bool lstm = h->cell == RCU_LSTM;
  if (!h->cp_in) CU(cudaStreamCreateWithFlags(&h->cp_in, cudaStreamNonBlocking));
  if (!h->cp_out) CU(cudaStreamCreateWithFlags(&h->cp_out, cudaStreamNonBlocking));
  while ((int)h->chunk_ev.size() < 3 * RCU_MAX_HOST_CHUNKS + 1) {
    cudaEvent_t e;
    CU(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    h->chunk_ev.push_back(e);
  }
  cudaEvent_t *ev_in = h->chunk_ev.data(), *ev_comp = ev_in + RCU_MAX_HOST_CHUNKS,
              *ev_out = ev_comp + RCU_MAX_HOST_CHUNKS, ev_entry = ev_out[RCU_MAX_HOST_CHUNKS];
  for (int i = 0; i < 2; ++i) {
    CU(h->io_xc[i].ensure((size_t)Tc * in_row * 4));
    CU(h->io_yc[i].ensure((size_t)Tc * out_row * 4));
    CU(h->io_st[i].ensure(LDB * h->Hout * 4));
    if (lstm) CU(h->io_ct[i].ensure(LDB * h->H * 4));
  }
  HostIO io{s, {}};
  const void *dh0, *dc0;
  CU(io.in(h0, LDB * h->Hout * 4, h->io_h0, false, &dh0));
  CU(io.in(c0, LDB * h->H * 4, h->io_c0, false, &dc0));
  // an early return (an error) must not leave copies of the caller's host
  // buffers in flight on the handle's streams
  struct DrainOnError {
    cudaStream_t a, b;
    bool armed = true;
    ~DrainOnError() {
      if (armed) {
        cudaStreamSynchronize(a);
        cudaStreamSynchronize(b);
      }
    }
  } drain{h->cp_in, h->cp_out};
  // the copy streams start after the work already on s
  CU(cudaEventRecord(ev_entry, s));
  CU(cudaStreamWaitEvent(h->cp_in, ev_entry, 0));
  CU(cudaStreamWaitEvent(h->cp_out, ev_entry, 0));
  auto steps_of = [&](int c) { return t_at[c + 1] - t_at[c]; };
  auto copy_in = [&](int c) -> cudaError_t {
    cudaError_t e = cudaMemcpyAsync(h->io_xc[c & 1].p, x + (size_t)t_at[c] * in_row,
                                    (size_t)steps_of(c) * in_row * 4, cudaMemcpyDefault,
                                    h->cp_in);
    return e != cudaSuccess ? e : cudaEventRecord(ev_in[c], h->cp_in);
  };
  for (int c = 0; c < std::min(n, 2); ++c) CU(copy_in(c));
  int launches = 0;
  for (int c = 0; c < n; ++c) {
    const int k = c & 1;
    CU(cudaStreamWaitEvent(s, ev_in[c], 0));
    if (c >= 2) CU(cudaStreamWaitEvent(s, ev_out[c - 2], 0));  // y buffer k is free again
    const float *sh = c == 0 ? (const float *)dh0 : (const float *)h->io_st[k ^ 1].p;
    const float *sc = c == 0 ? (const float *)dc0 : (lstm ? (const float *)h->io_ct[k ^ 1].p : nullptr);
    const int rc = rnn_forward(h, steps_of(c), B, (const float *)h->io_xc[k].p, nullptr, sh, sc,
                               nullptr, (float *)h->io_yc[k].p, (float *)h->io_st[k].p,
                               lstm ? (float *)h->io_ct[k].p : nullptr, s);
    if (rc != RCU_OK) return rc;
    launches += h->launches;
    CU(cudaEventRecord(ev_comp[c], s));
    CU(cudaStreamWaitEvent(h->cp_out, ev_comp[c], 0));
    CU(cudaMemcpyAsync(y + (size_t)t_at[c] * out_row, h->io_yc[k].p,
                       (size_t)steps_of(c) * out_row * 4, cudaMemcpyDefault, h->cp_out));
    CU(cudaEventRecord(ev_out[c], h->cp_out));
    if (c + 2 < n) {  // x buffer k is free once chunk c has computed
      CU(cudaStreamWaitEvent(h->cp_in, ev_comp[c], 0));
      CU(copy_in(c + 2));
    }
  }
  // the call is complete on s once the last y chunk has landed
  CU(cudaStreamWaitEvent(s, ev_out[n - 1], 0));
  const int kl = (n - 1) & 1;
  if (h_n) CU(cudaMemcpyAsync(h_n, h->io_st[kl].p, LDB * h->Hout * 4, cudaMemcpyDefault, s));
  if (c_n) CU(cudaMemcpyAsync(c_n, h->io_ct[kl].p, LDB * h->H * 4, cudaMemcpyDefault, s));
  drain.armed = false;  // s now waits for every copy
  h->launches = launches;
  return RCU_OK;
}

extern "C" int rnn_forward_host(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                                const float *h0, const float *c0, float *y, float *h_n,
                                float *c_n, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_forward_host: NULL handle");
  h->launches = 0;
  if (T < 0 || B < 0) return fail(RCU_ERR_INVALID, "rnn_forward_host: T and B must be >= 0");
  if (T == 0 || B == 0) return rnn_forward(h, T, B, x, lengths, h0, c0, nullptr, y, h_n, c_n, stream);
  if (!x || !y) return fail(RCU_ERR_INVALID, "rnn_forward_host: x and y are required");
  if (h->cell == RCU_GRU && (c0 || c_n))
    return fail(RCU_ERR_INVALID, "rnn_forward_host: c0/c_n are LSTM-only");
  for (auto &w : h->lw)
    if (!w.set) return fail(RCU_ERR_STATE, "rnn_forward_host: weights missing for some layer/direction");
  const size_t TB = (size_t)T * B, LDB = (size_t)h->layers * h->D * B;
  const size_t x_bytes = TB * h->in_dim * 4, y_bytes = TB * h->D * h->Hout * 4;
  // chunked pipeline: unidirectional, no lengths, no projection (the folded
  // LSTMP path takes an initial state through a separate fp32 term, which
  // would round differently from the recurrence it replaces), x and y
  // page-locked (so the copies are asynchronous); automatic for transfers of
  // 64 MB and more, one chunk per 64 steps up to 6
  int n = h->host_chunks;
  if (n == 0) n = x_bytes + y_bytes >= ((size_t)64 << 20) ? std::min(6, T / 64) : 1;
  n = std::min(n, T);
  if (n > 1 && h->D == 1 && h->P == 0 && !lengths && device_address(x) && device_address(y)) {
    h->plan_chunks = n;
    h->plan_x_in_place = h->plan_y_in_place = 0;
    return forward_host_chunked(h, T, B, n, x, h0, c0, y, h_n, c_n, (cudaStream_t)stream);
  }

  HostIO io{(cudaStream_t)stream, {}};
  const void *dx, *dlen, *dh0, *dc0;
  void *dy, *dhn, *dcn;
  bool x_placed = false;
  // x read and y written in place when page-locked; the small buffers staged
  CU(io.in(x, x_bytes, h->io_x, true, &dx, &x_placed));
  CU(io.in(lengths, (size_t)B * 4, h->io_len, false, &dlen));
  CU(io.in(h0, LDB * h->Hout * 4, h->io_h0, false, &dh0));
  CU(io.in(c0, LDB * h->H * 4, h->io_c0, false, &dc0));
  CU(io.out(y, y_bytes, h->io_y, true, &dy));
  CU(io.out(h_n, LDB * h->Hout * 4, h->io_hn, false, &dhn));
  CU(io.out(c_n, LDB * h->H * 4, h->io_cn, false, &dcn));
  h->x_in_place = x_placed;
  h->plan_chunks = 1;
  h->plan_x_in_place = x_placed ? 1 : 0;
  h->plan_y_in_place = dy == device_address(y) ? 1 : 0;
  const int rc = rnn_forward(h, T, B, (const float *)dx, (const int32_t *)dlen,
                             (const float *)dh0, (const float *)dc0, nullptr, (float *)dy,
                             (float *)dhn, (float *)dcn, stream);
  h->x_in_place = false;
  if (rc != RCU_OK) return rc;
  CU(io.finish());
  return RCU_OK;
}

// Backward pass through time (fp32 handles, unidirectional, no lengths or
// clipping; LSTM optionally with projection).  Recompute design: the forward
// is run again keeping every layer's output, which makes all of h_{t-1}
// known, so the layer's pre-activations are two GEMMs over all steps and the
// LSTM cell sequence one elementwise scan; only the hidden-state gradient
// runs step by step (bwd_rec_kernel).  Weight and input gradients are GEMMs
// over all T*B rows.
// With a projection h = W_hr m the step recurrence is
//   dh_t = dy_t + W_hh^T dz_{t+1} (width P),  dm_t = W_hr^T dh_t (width H),
// so dm_t = W_hr^T dy_t + (W_hh W_hr)^T dz_{t+1}: the same kernel runs it with
// W_hh W_hr in place of W_hh and A = dy W_hr (one GEMM, dh_n folded into the
// last step) in place of dy; dh_t, dh0 and dW_hr follow from GEMMs.
extern "C" int rnn_backward(rcu_rnn_t h, int T, int B, const float *x, const int32_t *lengths,
                            const float *h0, const float *c0, const float *dy, const float *dh_n,
                            const float *dc_n, float *dx, float *dh0, float *dc0, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_backward: NULL handle");
  h->launches = 0;
  for (auto &w : h->lw)
    if (!w.set) return fail(RCU_ERR_STATE, "rnn_backward: weights missing for some layer/direction");
  if (h->pclip)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_backward: projection clipping (cell clipping is supported)");
  if (T < 1 || B < 1 || !x || !dy) return fail(RCU_ERR_INVALID, "rnn_backward: need T, B >= 1, x and dy");
  if (h->cell == RCU_GRU && (c0 || dc_n || dc0))
    return fail(RCU_ERR_INVALID, "rnn_backward: c0/dc_n/dc0 are LSTM-only");
  if ((size_t)T * B > (size_t)INT32_MAX / 8)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_backward: T*B too large");
  const int L = h->layers, D = h->D, H = h->H, nG = h->nG, G = nG * H, cell = h->cell;
  const int P = h->P, Ho = h->Hout, DHo = D * Ho;
  if (bwd_units_per_cta(H, B, nG, h->nsm) < 1)
    return fail(RCU_ERR_UNSUPPORTED, "rnn_backward: W_hh columns do not fit one SM per unit group");
  cudaStream_t s = (cudaStream_t)stream;
  const int M = T * B;
  const size_t TBH = (size_t)M * H, TBO = (size_t)M * Ho, TBY = (size_t)M * DHo,
               TBG = (size_t)M * G;
  // transposed per-step streams ([rows][ldm8], column t*B + b)
  const int ldm8 = round_up(M, 8);
  const bool gru16 = h->dtype == RCU_BF16 && cell == RCU_GRU;
  // the tcgen05 GRU reverse-time kernel can run (its transposed inputs)
  const bool tcb_any = gru16 && P == 0 && !lengths && h->force_path != 1 &&
                       tc_bwd_supported(H, B, h->nsm);
  const int ldh = round_up(H, 8), ldo = round_up(Ho, 8);
  int kmax = std::max(H, DHo);
  for (int l = 0; l < L; ++l) kmax = std::max(kmax, h->in_l[l]);
  const size_t TBK = (size_t)M * kmax;
  // ---- workspace (floats; every piece 256-byte aligned)
  size_t off = 0;
  auto take = [&](size_t n) { size_t r = off; off += (n + 63) & ~size_t(63); return r; };
  const size_t o_keep = take((size_t)L * TBY), o_hp = take(TBO),
               // [M][G], or transposed [G][ldm8] for the tcgen05 GRU kernel
               o_zin = take((size_t)G * ldm8), o_zh = take((size_t)G * ldm8),
               // that kernel's h_{t-1}^T and dy^T
               o_hpt = take(tcb_any ? (size_t)Ho * ldm8 : 0),
               o_dyt = take(tcb_any ? (size_t)Ho * ldm8 : 0),
               o_cs = take(cell == RCU_LSTM ? TBH : 0), o_da = take(TBG),
               o_dr = take(cell == RCU_GRU ? TBG : 0), o_dya = take(TBY), o_dyb = take(TBY),
               o_t1 = take(TBG), o_t2 = take(TBK), o_t3 = take(cell == RCU_GRU ? TBG : 0),
               o_t4 = take(TBO), o_wt = take((size_t)kmax * G),
               o_cs2 = take(colsum_scratch_floats(M, G)),
               // projection only
               o_ms = take(P ? TBH : 0), o_dyp = take(P ? TBO : 0), o_a = take(P ? TBH : 0),
               o_f = take(P ? (size_t)G * ldh : 0), o_whrt = take(P ? (size_t)H * P : 0),
               o_whht = take(P ? (size_t)Ho * G : 0), o_r = take(P ? TBO : 0),
               o_t5 = take(P ? TBH : 0), o_t6 = take(P ? TBO : 0),
               // bidirectional only: processing-order copies of one direction
               o_xr = take(D > 1 ? TBK : 0), o_yd = take(D > 1 ? TBO : 0),
               o_dyd = take(D > 1 ? TBO : 0), o_dxr = take(D > 1 ? TBK : 0),
               o_tmp = take(D > 1 ? TBK : 0),
               // variable lengths: dy of one direction, zero past each row's end
               o_dym = take(lengths ? TBO : 0),
               // cell clipping: the unclamped cell state of every step
               o_cr = take(cell == RCU_LSTM && h->cclip ? TBH : 0),
               o_xm = take(lengths ? (size_t)M * h->in_l[0] : 0),
               // the tcgen05 GRU reverse-time kernel's bias sums [2][batch groups][G]
               o_bs = take(gru16 ? 2 * (size_t)ceil_div(B, 128) * G : 0),
               o_ctl = take((size_t)std::max(64, tc_bwd_counters(B))),
               // split-K partials of the tensor-core weight-gradient GEMMs (at most 4 chunks)
               o_wsk = take(h->dtype == RCU_BF16 ? 4 * (size_t)G * round_up(std::max(kmax, Ho), 4) : 0);
  // a bidirectional layer whose two directions' reverse-time recurrences
  // share one launch: the second direction's copies of the pieces that live
  // from its recompute to its recurrence
  const size_t n2 = D > 1 ? 1 : 0;
  const size_t o_zin1 = take(n2 * G * ldm8), o_zh1 = take(n2 * G * ldm8),
               o_cs1 = take(n2 * (cell == RCU_LSTM ? TBH : 0)), o_da1 = take(n2 * TBG),
               o_dr1 = take(n2 * (cell == RCU_GRU ? TBG : 0)), o_hp1 = take(n2 * TBO),
               o_dym1 = take(n2 * (lengths ? TBO : 0)),
               o_cr1 = take(n2 * (cell == RCU_LSTM && h->cclip ? TBH : 0)),
               o_yd1 = take(n2 * TBO), o_dyd1 = take(n2 * TBO),
               o_ctl1 = take(n2 * std::max(64, tc_bwd_counters(B)));
  CU(h->bw.ensure(off * 4));
  float *wsf = (float *)h->bw.p;
  float *keep = wsf + o_keep, *hp = wsf + o_hp, *zin = wsf + o_zin, *zh = wsf + o_zh;
  float *cs = cell == RCU_LSTM ? wsf + o_cs : nullptr, *DA = wsf + o_da;
  float *DR = cell == RCU_GRU ? wsf + o_dr : DA;
  float *dYa = wsf + o_dya, *dYb = wsf + o_dyb, *T1 = wsf + o_t1, *T2 = wsf + o_t2;
  float *T3 = cell == RCU_GRU ? wsf + o_t3 : T1, *T4 = wsf + o_t4;
  float *WT = wsf + o_wt, *csum = wsf + o_cs2;
  float *ms = P ? wsf + o_ms : nullptr, *dYp = wsf + o_dyp, *Aw = wsf + o_a, *Fw = wsf + o_f;
  float *WhrT = wsf + o_whrt, *WhhT = wsf + o_whht, *Rw = wsf + o_r, *T5 = wsf + o_t5,
        *T6 = wsf + o_t6;
  float *XR = wsf + o_xr, *YD = wsf + o_yd, *DYD = wsf + o_dyd, *DXR = wsf + o_dxr,
        *TMP = wsf + o_tmp, *DYM = wsf + o_dym, *XM = wsf + o_xm;
  float *CR = (cell == RCU_LSTM && h->cclip) ? wsf + o_cr : nullptr;
  float *BS = wsf + o_bs, *HPT = wsf + o_hpt, *DYT = wsf + o_dyt, *WSK = wsf + o_wsk;
  unsigned *ctr = (unsigned *)(wsf + o_ctl);
  // the pieces that live from a direction's recompute to its reverse-time
  // recurrence, by slot: 0 (every layer's first direction, and every
  // direction run on its own) and 1 (a bidirectional layer's second direction
  // when both recurrences share one launch); run_dir picks them by slot
  float *const zin_0 = zin, *const zh_0 = zh, *const cs_0 = cs, *const DA_0 = DA, *const DR_0 = DR,
              *const hp_0 = hp, *const DYM_0 = DYM, *const CR_0 = CR;
  unsigned *const ctr_0 = ctr;
  float *const zin_1 = wsf + o_zin1, *const zh_1 = wsf + o_zh1,
              *const cs_1 = cell == RCU_LSTM ? wsf + o_cs1 : nullptr, *const DA_1 = wsf + o_da1,
              *const DR_1 = cell == RCU_GRU ? wsf + o_dr1 : DA_1, *const hp_1 = wsf + o_hp1,
              *const DYM_1 = wsf + o_dym1, *const CR_1 = CR ? wsf + o_cr1 : nullptr,
              *const YD_1 = wsf + o_yd1, *const DYD_1 = wsf + o_dyd1;
  unsigned *const ctr_1 = (unsigned *)(wsf + o_ctl1);
  // bf16 handles: the backward's GEMMs run on the tensor cores like the
  // forward's, on operands rounded to bf16 (the precision of every forward
  // MMA operand: x, h, W) with fp32 accumulation.  fp32 handles, and
  // RCU_ATTR_FORCE_PATH = 1, keep the fp32 FFMA GEMMs.  bf16 workspace,
  // elements (every piece 256-byte aligned):
  const bool tcg = h->dtype == RCU_BF16 && h->force_path != 1 && tc_gemm_supported(8, 8);
  const int g8 = round_up(G, 8), k8 = round_up(kmax, 8);
  size_t boff = 0;
  auto btake = [&](size_t n) { size_t r = boff; boff += (n + 127) & ~size_t(127); return r; };
  const size_t b_x = btake(tcg ? (size_t)M * k8 : 0),        // x rows
      b_hp = btake(tcg ? (size_t)M * ldo : 0),                  // h_{t-1} rows
      b_whh = btake(tcg ? (size_t)G * ldo : 0),                 // W_hh rows
      b_t1 = btake(tcg ? (size_t)G * ldm8 : 0),                 // DA^T
      b_t2 = btake(tcg ? (size_t)kmax * ldm8 : 0),              // X^T
      b_t3 = btake(tcg && cell == RCU_GRU ? (size_t)G * ldm8 : 0),  // DR^T
      b_t4 = btake(tcg ? (size_t)Ho * ldm8 : 0),                // H_prev^T
      b_da = btake(tcg ? (size_t)M * g8 : 0),                   // DA rows
      b_wt = btake(tcg ? (size_t)kmax * g8 : 0),                // W_ih^T
      b_wth = btake(tcg && cell == RCU_GRU ? (size_t)H * g8 : 0),        // W_hh^T
      b_xdr = btake(tcg && cell == RCU_GRU ? 2 * (size_t)B * g8 : 0);    // dR_t exchange
  if (tcg) CU(h->bwb.ensure(boff * 2));
  __nv_bfloat16 *bws = (__nv_bfloat16 *)h->bwb.p;
  auto aligned16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  if ((int)h->gw.size() < L * D) h->gw.resize((size_t)L * D);
  h->grads_ready = false;
  int launches = 0;
  // ---- forward again, keeping every layer's output sequence.  With variable
  // lengths the forward writes no step past a row's end: those entries of the
  // inner layers' outputs are zeroed first, and x is read through a copy zero
  // there, so every operand past a row's end is 0 (its gradient terms vanish)
  if (lengths && L > 1) CU(cudaMemsetAsync(keep, 0, (size_t)(L - 1) * TBY * 4, s));
  h->keep_out = keep;
  int rc = rnn_forward(h, T, B, x, lengths, h0, c0, nullptr, keep + (size_t)(L - 1) * TBY,
                       nullptr, nullptr, stream);
  h->keep_out = nullptr;
  if (rc != RCU_OK) return rc;
  launches += h->launches;
  // the handle's error word (cleared by the forward above), read by rnn_get_status
  int *err = (int *)h->ctl.p;

  // One (layer, direction) i = l*D + d, on inputs in its processing order (the
  // reverse direction's sequences are time-reversed copies, so it is an
  // ordinary forward recurrence): X [M][K], its output sequence Y [M][Ho],
  // dY [M][Ho]; writes dX [M][K] (may be NULL) and the weight gradients.
  // the tcgen05 GRU reverse-time kernel (below) activates the gates itself
  // and reads its per-step inputs transposed
  const bool tcb_all = tcg && cell == RCU_GRU && P == 0 && !lengths && tc_bwd_supported(H, B, h->nsm);
  // stage 0: everything; 1: up to the reverse-time recurrence, whose
  // arguments go to *rec_out (not launched); 2: what follows it.  slot 1: the
  // second direction's copies of the pieces that live across the recurrence.
  auto run_dir = [&](int l, int d, const float *X, int K, const float *Y, const float *dYdir,
                     float *dX, int stage = 0, int slot = 0, BwdRecArgs *rec_out = nullptr) -> int {
    float *const zin = slot ? zin_1 : zin_0, *const zh = slot ? zh_1 : zh_0,
                *const cs = slot ? cs_1 : cs_0, *const DA = slot ? DA_1 : DA_0,
                *const DR = slot ? DR_1 : DR_0, *const hp = slot ? hp_1 : hp_0,
                *const DYM = slot ? DYM_1 : DYM_0, *const CR = slot ? CR_1 : CR_0;
    unsigned *const ctr = slot ? ctr_1 : ctr_0;
    const bool pre = stage != 2;
    const int i = l * D + d, ldk = round_up(K, 8);
    const LayerDirW &lw = h->lw[(size_t)i];
    // fp32 W_ih (bf16 handles: of the rounded weights the forward used)
    const float *Wih = (const float *)(h->dtype == RCU_BF16 ? h->wih_f32[l].p : h->wih[l].p) +
                       (size_t)d * G * ldk;
    const float *dhnl = dh_n ? dh_n + (size_t)i * B * Ho : nullptr;
    // variable lengths: dy zero past each row's end, dh_n added at its last
    // step (h_n is the state there); the recurrence then carries no dh_n
    if (lengths) {
      if (pre) {
        h->begin("bwd_mask", s);
        cudaError_t e = launch_mask_steps(dYdir, Ho, T, B, lengths, dhnl, DYM, s);
        h->end(s);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: mask: %s", cudaGetErrorString(e));
        ++launches;
      }
      dYdir = DYM;
      dhnl = nullptr;
    }
    const bool tcb = tcb_all;
    // h_{t-1} for t = 0 .. T-1 as one [M][Ho] sequence: h0's rows, then Y's
    // first T-1 steps.  The tcgen05 path reads the two parts where they are
    // (its bf16 rows and transposes are written from h0 and Y directly) and
    // copies them only if a later step needs the sequence itself.
    const float *h0i = h0 ? h0 + (size_t)i * B * Ho : nullptr;
    bool hp_ready = !pre;  // (stage 2: filled by stage 1)
    auto ensure_hp = [&]() -> cudaError_t {
      if (hp_ready) return cudaSuccess;
      hp_ready = true;
      cudaError_t e0 = h0i ? cudaMemcpyAsync(hp, h0i, (size_t)B * Ho * 4, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(hp, 0, (size_t)B * Ho * 4, s);
      if (e0 == cudaSuccess && T > 1)
        e0 = cudaMemcpyAsync(hp + (size_t)B * Ho, Y, (size_t)(T - 1) * B * Ho * 4,
                             cudaMemcpyDeviceToDevice, s);
      return e0;
    };
    if (!tcb && pre) CU(ensure_hp());
    // pre-activations of every step
    const bool tcr = tcg && tc_gemm_supported(K, G) && tc_gemm_supported(Ho, G);
    int nl = 0;  // kernels launched by this (layer, direction)
    if (pre) h->begin("bwd_recompute_gemm", s);
    cudaError_t e = cudaSuccess;
    if (!pre) {
    } else if (tcb) {
      // (W_ih X^T + b_ih) and (W_hh H_prev^T + b_hh): the same products with
      // the operands' roles swapped, the biases added per output row
      __nv_bfloat16 *Xb = bws + b_x, *Hb = bws + b_hp, *Wb = bws + b_whh;
      e = launch_convert_rows_bf16(X, M, K, K, Xb, ldk, s);
      if (e == cudaSuccess)
        e = launch_tc_gemm((const __nv_bfloat16 *)h->wih[l].p + (size_t)d * G * ldk, ldk, Xb, ldk,
                           (const float *)lw.bih_plain.p, zin, ldm8, G, nullptr, M, K, h->nsm, s,
                           err, (uint64_t)h->timeout_ns, true);
      // bf16 h_{t-1} rows: h0's (or zeros), then Y's first T-1 steps
      if (e == cudaSuccess)
        e = h0i ? launch_convert_rows_bf16(h0i, B, Ho, Ho, Hb, ldo, s)
                : cudaMemsetAsync(Hb, 0, (size_t)B * ldo * 2, s);
      if (e == cudaSuccess && T > 1)
        e = launch_convert_rows_bf16(Y, M - B, Ho, Ho, Hb + (size_t)B * ldo, ldo, s);
      if (e == cudaSuccess)
        e = launch_convert_rows_bf16((const float *)lw.whh_plain.p, G, Ho, ldo, Wb, ldo, s);
      if (e == cudaSuccess)
        e = launch_tc_gemm(Wb, ldo, Hb, ldo, (const float *)lw.bhh_plain.p, zh, ldm8, G, nullptr,
                           M, Ho, h->nsm, s, err, (uint64_t)h->timeout_ns, true);
      nl += 4 + (h0i ? 1 : 0) + (T > 1 ? 1 : 0);
    } else if (tcr) {
      // the forward's own operands: bf16 x (or the previous layer's bf16
      // output), bf16 h_{t-1}, the bf16 weights
      __nv_bfloat16 *Xb = bws + b_x, *Hb = bws + b_hp, *Wb = bws + b_whh;
      e = launch_convert_rows_bf16(X, M, K, K, Xb, ldk, s);
      if (e == cudaSuccess)
        e = launch_tc_gemm(Xb, ldk, (const __nv_bfloat16 *)h->wih[l].p + (size_t)d * G * ldk, ldk,
                           (const float *)lw.bih_plain.p, zin, G, M, nullptr, G, K, h->nsm, s, err,
                           (uint64_t)h->timeout_ns);
      if (e == cudaSuccess) e = launch_convert_rows_bf16(hp, M, Ho, Ho, Hb, ldo, s);
      if (e == cudaSuccess)
        e = launch_convert_rows_bf16((const float *)lw.whh_plain.p, G, Ho, ldo, Wb, ldo, s);
      if (e == cudaSuccess)
        e = launch_tc_gemm(Hb, ldo, Wb, ldo, (const float *)lw.bhh_plain.p, zh, G, M, nullptr, G,
                           Ho, h->nsm, s, err, (uint64_t)h->timeout_ns);
      nl += 5;
    } else {
      e = gemm_f32(h, X, K, Wih, ldk, (const float *)lw.bih_plain.p, zin, G, M, nullptr, G, K, s,
                   err, &nl);
      if (e == cudaSuccess)
        e = gemm_f32(h, hp, Ho, (const float *)lw.whh_plain.p, ldo, (const float *)lw.bhh_plain.p,
                     zh, G, M, nullptr, G, Ho, s, err, &nl);
    }
    if (pre) h->end(s);
    const float *c0l = c0 ? c0 + (size_t)i * B * H : nullptr;
    if (!tcb && pre) {
      h->begin("bwd_prep", s);
      if (e == cudaSuccess)
        e = launch_bwd_prep(T, B, H, cell, zin, zh, c0l, cs, ms, s, CR, h->cclip_lo, h->cclip_hi);
      h->end(s);
      nl += 1;
    }
    if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: recompute: %s", cudaGetErrorString(e));
    // projection: dy' = dy (+ dh_n at the last step), A = dy' W_hr, F = W_hh W_hr
    const float *rec_dy = dYdir, *rec_W = (const float *)lw.whh_plain.p;
    int rec_ldw = ldo;
    if (P > 0) {
      h->begin("bwd_proj_fold", s);
      CU(cudaMemcpyAsync(dYp, dYdir, TBO * 4, cudaMemcpyDeviceToDevice, s));
      if (dhnl) e = launch_add(dYp + (size_t)(T - 1) * B * Ho, dhnl, (size_t)B * Ho, s);
      if (e == cudaSuccess) e = launch_transpose((const float *)lw.whr_plain.p, P, H, H, WhrT, P, s);
      int pn = 0;
      if (e == cudaSuccess)
        e = gemm_f32(h, dYp, Ho, WhrT, P, nullptr, Aw, H, M, nullptr, H, P, s, err, &pn);
      if (e == cudaSuccess)
        e = gemm_f32(h, (const float *)lw.whh_plain.p, ldo, WhrT, P, nullptr, Fw, ldh, G, nullptr,
                     H, P, s, err, &pn);
      nl += pn - 2;  // (counted with the projection's fixed launches below)
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: projection: %s", cudaGetErrorString(e));
      rec_dy = Aw;
      rec_W = Fw;
      rec_ldw = ldh;
    }
    // the reverse-time recurrence: on the tensor cores for the GRU of a bf16
    // handle over fixed-length rows (W_hh^T dR_{t+1} with bf16 operands, as
    // every MMA of its forward), else the FFMA kernel
    if (pre) CU(cudaMemsetAsync(ctr, 0, (size_t)std::max(64, tc_bwd_counters(B)) * 4, s));
    DevBuf &g = h->gw[(size_t)i];
    CU(g.ensure(((size_t)G * K + (size_t)G * Ho + 2 * (size_t)G + (size_t)P * H) * 4));
    float *gWih = (float *)g.p, *gWhh = gWih + (size_t)G * K, *gbih = gWhh + (size_t)G * Ho,
          *gbhh = gbih + G, *gWhr = gbhh + G;
    // the weight and input gradients on the tensor cores (below)
    const bool tw = tcg && (K % 4) == 0 && (Ho % 4) == 0 && (G % 4) == 0 && aligned16(gWih) &&
                    aligned16(gWhh) && (!dX || aligned16(dX));
    // with both, the reverse-time kernel writes the gate gradients straight
    // in the forms those GEMMs read (DA^T, DR^T and DA in bf16, the bias sums
    // per batch group): no fp32 DA / DR, transposes or column sums of them
    const bool tcd = tcb && tw;
    __nv_bfloat16 *T1b = bws + b_t1, *T2b = bws + b_t2, *T4b = bws + b_t4;
    __nv_bfloat16 *T3b = cell == RCU_GRU ? bws + b_t3 : T1b, *DAb = bws + b_da;
    const int nbg = ceil_div(B, 128);
    if (tcb) {
      __nv_bfloat16 *WTh = bws + b_wth, *XDR = bws + b_xdr;
      // h_{t-1}^T and dy^T for the kernel (and with the weight GEMMs on the
      // tensor cores, H_prev^T in bf16 from the same pass)
      h->begin("bwd_transpose", s);
      // (columns [0, B) from h0, or zeros; columns [B, M) from Y)
      if (h0i) {
        e = launch_transpose_dual(h0i, B, Ho, Ho, HPT, tw ? T4b : nullptr, ldm8, s);
      } else {
        e = cudaMemset2DAsync(HPT, (size_t)ldm8 * 4, 0, (size_t)B * 4, Ho, s);
        if (e == cudaSuccess && tw)
          e = cudaMemset2DAsync(T4b, (size_t)ldm8 * 2, 0, (size_t)B * 2, Ho, s);
      }
      if (e == cudaSuccess && T > 1)
        e = launch_transpose_dual(Y, M - B, Ho, Ho, HPT + B, tw ? T4b + B : nullptr, ldm8, s);
      if (e == cudaSuccess) e = launch_transpose_dual(rec_dy, M, Ho, Ho, DYT, nullptr, ldm8, s);
      h->end(s);
      nl += 1 + (h0i ? 1 : 0) + (T > 1 ? 1 : 0);
      h->begin("bwd_recurrent_tc", s);
      if (e == cudaSuccess)
        e = launch_transpose_bf16((const float *)lw.whh_plain.p, G, H, ldo, WTh, g8, s);
      TcBwdParams q{};
      q.T = T; q.B = B; q.H = H;
      q.zin = zin; q.zh = zh; q.hp = HPT; q.dy = DYT; q.ldz = ldm8;
      q.dhn = dhnl;
      if (tcd) {
        q.dat = T1b; q.drt = T3b; q.ldt = ldm8;
        q.dab = dX ? DAb : nullptr; q.ldab = g8;
        q.bsum = BS;
      } else {
        q.DA = DA; q.DR = DR;
      }
      q.dh0 = dh0 ? dh0 + (size_t)i * B * H : nullptr;
      q.xdr = XDR; q.Kx = g8; q.wt = WTh;
      q.ctr = ctr; q.err = err; q.timeout_ns = (uint64_t)h->timeout_ns;
      q.drop_arrival = h->drop_arrival == 2 && l == L - 1 && d == 0;
      if (h->trace && l == 0 && d == 0 && e == cudaSuccess) {
        // the last reverse-time launch (layer 0) replaces the forward's stamps
        const size_t rows = (size_t)T + 1;
        e = h->trace_buf.ensure(rows * 16 * 8);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->trace_buf.p, 0, rows * 16 * 8, s);
        h->trace_T = (int)rows;
        q.trace = (unsigned long long *)h->trace_buf.p;
      }
      if (e == cudaSuccess) e = launch_tc_bwd(q, h->nsm, s);
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: recurrence: %s", cudaGetErrorString(e));
      nl += 2;
    }
    BwdRecArgs a{};
    a.T = T; a.B = B; a.H = H; a.cell = cell;
    a.Whh = rec_W; a.ldw = rec_ldw;
    a.gates = zin; a.zh = zh; a.cs = cs; a.c0 = c0l; a.hp = hp; a.dy = rec_dy;
    a.dhn = P > 0 ? nullptr : dhnl;
    a.dcn = dc_n ? dc_n + (size_t)i * B * H : nullptr;
    a.lengths = lengths;
    a.cr = CR; a.clo = h->cclip_lo; a.chi = h->cclip_hi;
    a.DA = DA; a.DR = DR;
    a.dh0 = (P > 0 || !dh0) ? nullptr : dh0 + (size_t)i * B * H;
    a.dc0 = dc0 ? dc0 + (size_t)i * B * H : nullptr;
    a.ctr = ctr; a.err = err; a.timeout_ns = (uint64_t)h->timeout_ns;
    a.drop_arrival = h->drop_arrival == 2 && l == L - 1 && d == 0;
    if (!tcb && pre && h->trace && l == 0 && d == 0) {
      // the last reverse-time launch (layer 0) replaces the forward's stamps
      const size_t rows = (size_t)T + 1;
      CU(h->trace_buf.ensure(rows * 16 * 8));
      CU(cudaMemsetAsync(h->trace_buf.p, 0, rows * 16 * 8, s));
      h->trace_T = (int)rows;
      a.trace = (unsigned long long *)h->trace_buf.p;
    }
    if (!tcb && stage == 1) {  // launched with the other direction's
      if (rec_out) *rec_out = a;
      launches += nl;
      return RCU_OK;
    }
    if (!tcb && stage == 0) {
      h->begin("bwd_recurrent", s);
      e = launch_bwd_rec(a, h->nsm, s);
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: recurrence: %s", cudaGetErrorString(e));
      nl += 1;
    }
    // projection: R = DZ W_hh (R_t = W_hh^T dz_t), dh0 = R_0, dh_t = dy'_t + R_{t+1},
    // dW_hr = sum_t dh_t m_t^T
    if (P > 0) {
      h->begin("bwd_proj_grad", s);
      e = launch_transpose((const float *)lw.whh_plain.p, G, Ho, ldo, WhhT, G, s);
      int pn = 0;
      if (e == cudaSuccess) e = gemm_f32(h, DA, G, WhhT, G, nullptr, Rw, Ho, M, nullptr, Ho, G, s, err, &pn);
      if (e == cudaSuccess && dh0)
        e = cudaMemcpyAsync(dh0 + (size_t)i * B * Ho, Rw, (size_t)B * Ho * 4, cudaMemcpyDeviceToDevice, s);
      if (e == cudaSuccess && T > 1) e = launch_add(dYp, Rw + (size_t)B * Ho, (size_t)(T - 1) * B * Ho, s);
      if (e == cudaSuccess) e = launch_transpose(dYp, M, Ho, Ho, T6, M, s);
      if (e == cudaSuccess) e = launch_transpose(ms, M, H, H, T5, M, s);
      if (e == cudaSuccess) e = gemm_f32(h, T6, M, T5, M, nullptr, gWhr, H, P, nullptr, H, M, s, err, &pn);
      nl += pn - 2;
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: projection gradients: %s", cudaGetErrorString(e));
    }
    // weight gradients: dW_ih = DA^T X, dW_hh = DR^T H_prev (through transposes
    // to K-contiguous operands), db = column sums; input gradient dX = DA W_ih
    h->begin("bwd_transpose", s);
    if (tcd) {
      // (H_prev^T came with the reverse-time kernel's inputs)
      e = launch_transpose_bf16(X, M, K, K, T2b, ldm8, s);
      nl += 1;
    } else if (tw) {
      e = launch_transpose_bf16(DA, M, G, G, T1b, ldm8, s);
      if (e == cudaSuccess) e = launch_transpose_bf16(X, M, K, K, T2b, ldm8, s);
      if (e == cudaSuccess && cell == RCU_GRU) e = launch_transpose_bf16(DR, M, G, G, T3b, ldm8, s);
      if (e == cudaSuccess) e = launch_transpose_bf16(hp, M, Ho, Ho, T4b, ldm8, s);
      nl += cell == RCU_GRU ? 4 : 3;
    } else {
      e = ensure_hp();
      if (e == cudaSuccess) e = launch_transpose(DA, M, G, G, T1, M, s);
      if (e == cudaSuccess) e = launch_transpose(X, M, K, K, T2, M, s);
      if (e == cudaSuccess && cell == RCU_GRU) e = launch_transpose(DR, M, G, G, T3, M, s);
      if (e == cudaSuccess) e = launch_transpose(hp, M, Ho, Ho, T4, M, s);
      if (e == cudaSuccess) e = launch_transpose(Wih, G, K, ldk, WT, G, s);
      nl += cell == RCU_GRU ? 5 : 4;
    }
    h->end(s);
    h->begin("bwd_weight_gemm", s);
    if (tw) {
      // (a reduction over all T*B rows into a small output: K split into
      // chunks summed in order where the output tiles cannot fill the GPU)
      int n1 = 1, n2 = 1;
      if (e == cudaSuccess)
        e = launch_tc_gemm_splitk(T1b, ldm8, T2b, ldm8, nullptr, gWih, K, G, K, M, WSK, h->nsm, s,
                                  err, (uint64_t)h->timeout_ns, &n1);
      if (e == cudaSuccess)
        e = launch_tc_gemm_splitk(T3b, ldm8, T4b, ldm8, nullptr, gWhh, Ho, G, Ho, M, WSK, h->nsm,
                                  s, err, (uint64_t)h->timeout_ns, &n2);
      nl += n1 + n2 - 2;
    } else {
      if (e == cudaSuccess)
        e = gemm_f32(h, T1, M, T2, M, nullptr, gWih, K, G, nullptr, K, M, s, err, &nl);
      if (e == cudaSuccess)
        e = gemm_f32(h, T3, M, T4, M, nullptr, gWhh, Ho, G, nullptr, Ho, M, s, err, &nl);
      nl -= 2;
    }
    nl += 2;
    h->end(s);
    h->begin("bwd_colsum", s);
    // (with the kernel's per-batch-group sums, over nbg rows instead of M)
    if (e == cudaSuccess) e = launch_colsum(tcd ? BS : DA, tcd ? nbg : M, G, csum, gbih, s);
    if (!tcd && DR == DA) {
      // LSTM: both biases enter the same pre-activations, db_hh = db_ih
      if (e == cudaSuccess) e = cudaMemcpyAsync(gbhh, gbih, (size_t)G * 4, cudaMemcpyDeviceToDevice, s);
      nl += 2;
    } else {
      if (e == cudaSuccess)
        e = launch_colsum(tcd ? BS + (size_t)nbg * G : DR, tcd ? nbg : M, G, csum, gbhh, s);
      nl += 4;
    }
    h->end(s);
    h->begin("bwd_dx_gemm", s);
    if (e == cudaSuccess && dX) {
      if (tw) {
        __nv_bfloat16 *WTb = bws + b_wt;
        if (!tcd) {
          e = launch_convert_rows_bf16(DA, M, G, G, DAb, g8, s);
          nl += 1;
        }
        if (e == cudaSuccess) e = launch_transpose_bf16(Wih, G, K, ldk, WTb, g8, s);
        if (e == cudaSuccess)
          e = launch_tc_gemm(DAb, g8, WTb, g8, nullptr, dX, K, M, nullptr, K, G, h->nsm, s, err,
                             (uint64_t)h->timeout_ns);
        nl += 2;
      } else {
        e = gemm_f32(h, DA, G, WT, G, nullptr, dX, K, M, nullptr, K, G, s, err, &nl);
      }
    }
    h->end(s);
    if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: gradients: %s", cudaGetErrorString(e));
    // projection: 3 GEMMs, 4 transposes, up to 2 adds
    launches += nl + (P > 0 ? 7 + (dhnl ? 1 : 0) + (T > 1 ? 1 : 0) : 0);
    return RCU_OK;
  };

  if (lengths) {
    h->begin("bwd_mask", s);
    cudaError_t e = launch_mask_steps(x, h->in_l[0], T, B, lengths, nullptr, XM, s);
    h->end(s);
    if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: mask: %s", cudaGetErrorString(e));
    ++launches;
  }
  const float *dYcur = dy;
  for (int l = L - 1; l >= 0; --l) {
    const int K = h->in_l[l];
    const float *Xl = l == 0 ? (lengths ? XM : x) : keep + (size_t)(l - 1) * TBY;
    const float *Yl = keep + (size_t)l * TBY;
    float *dXl = l == 0 ? dx : (dYcur == dYa ? dYb : dYa);
    if (l > 0 && !dXl) return fail(RCU_ERR_INVALID, "rnn_backward: internal");
    // both directions' reverse-time recurrences in one launch, each on half
    // of the SMs (FFMA kernel, no projection), when that plan fits
    const bool conc = D == 2 && P == 0 && !tcb_all &&
                      bwd_units_per_cta(H, B, nG, h->nsm / 2) >= 1;
    if (D == 1) {
      if (int r = run_dir(l, 0, Xl, K, Yl, dYcur, dXl)) return r;
    } else if (conc) {
      h->begin("bwd_reorder", s);
      cudaError_t e = launch_gather_steps(Yl, DHo, 0, Ho, T, B, false, lengths, YD, s);
      if (e == cudaSuccess) e = launch_gather_steps(dYcur, DHo, 0, Ho, T, B, false, lengths, DYD, s);
      if (e == cudaSuccess) e = launch_gather_steps(Yl, DHo, Ho, Ho, T, B, true, lengths, YD_1, s);
      if (e == cudaSuccess)
        e = launch_gather_steps(dYcur, DHo, Ho, Ho, T, B, true, lengths, DYD_1, s);
      if (e == cudaSuccess) e = launch_gather_steps(Xl, K, 0, K, T, B, true, lengths, XR, s);
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: reorder: %s", cudaGetErrorString(e));
      launches += 5;
      BwdRecArgs a0{}, a1{};
      if (int r = run_dir(l, 0, Xl, K, YD, DYD, dXl, 1, 0, &a0)) return r;
      if (int r = run_dir(l, 1, XR, K, YD_1, DYD_1, dXl ? DXR : nullptr, 1, 1, &a1)) return r;
      h->begin("bwd_recurrent", s);
      e = launch_bwd_rec(a0, h->nsm, s, &a1);
      h->end(s);
      if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: recurrence: %s", cudaGetErrorString(e));
      launches += 1;
      if (int r = run_dir(l, 0, Xl, K, YD, DYD, dXl, 2, 0)) return r;
      if (int r = run_dir(l, 1, XR, K, YD_1, DYD_1, dXl ? DXR : nullptr, 2, 1)) return r;
      if (dXl) {  // dX of the layer input: the forward one plus the reversed backward one
        h->begin("bwd_reorder", s);
        e = launch_gather_steps(DXR, K, 0, K, T, B, true, lengths, TMP, s);
        if (e == cudaSuccess) e = launch_add(dXl, TMP, (size_t)M * K, s);
        h->end(s);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: reorder: %s", cudaGetErrorString(e));
        launches += 2;
      }
    } else {
      for (int d = 0; d < 2; ++d) {
        // direction d's sequences in its processing order
        h->begin("bwd_reorder", s);
        cudaError_t e = launch_gather_steps(Yl, DHo, d * Ho, Ho, T, B, d == 1, lengths, YD, s);
        if (e == cudaSuccess)
          e = launch_gather_steps(dYcur, DHo, d * Ho, Ho, T, B, d == 1, lengths, DYD, s);
        if (e == cudaSuccess && d == 1)
          e = launch_gather_steps(Xl, K, 0, K, T, B, true, lengths, XR, s);
        h->end(s);
        if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: reorder: %s", cudaGetErrorString(e));
        launches += d == 1 ? 3 : 2;
        float *dXd = dXl ? (d == 0 ? dXl : DXR) : nullptr;
        if (int r = run_dir(l, d, d == 1 ? XR : Xl, K, YD, DYD, dXd)) return r;
        if (d == 1 && dXl) {  // dX of the layer input: the forward one plus the reversed backward one
          h->begin("bwd_reorder", s);
          e = launch_gather_steps(DXR, K, 0, K, T, B, true, lengths, TMP, s);
          if (e == cudaSuccess) e = launch_add(dXl, TMP, (size_t)M * K, s);
          h->end(s);
          if (e != cudaSuccess) return fail(RCU_ERR_CUDA, "rnn_backward: reorder: %s", cudaGetErrorString(e));
          launches += 2;
        }
      }
    }
    dYcur = dXl;
  }
  h->grads_ready = true;
  h->launches = launches;
  return RCU_OK;
}

extern "C" int rnn_get_weight_grads(rcu_rnn_t h, int layer, int dir, float *dW_ih, float *dW_hh,
                                    float *db_ih, float *db_hh, float *dW_hr, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_get_weight_grads: NULL handle");
  if (!h->grads_ready) return fail(RCU_ERR_STATE, "rnn_get_weight_grads: no rnn_backward has run");
  if (layer < 0 || layer >= h->layers || dir < 0 || dir >= h->D)
    return fail(RCU_ERR_INVALID, "rnn_get_weight_grads: layer %d / dir %d out of range", layer, dir);
  if (dW_hr && h->P == 0) return fail(RCU_ERR_INVALID, "rnn_get_weight_grads: no projection");
  cudaStream_t s = (cudaStream_t)stream;
  const int G = h->nG * h->H, K = h->in_l[layer], Ho = h->Hout, P = h->P, H = h->H;
  const float *g = (const float *)h->gw[(size_t)layer * h->D + dir].p;
  const size_t o1 = (size_t)G * K, o2 = o1 + (size_t)G * Ho, o3 = o2 + G, o4 = o3 + G;
  const float *src[5] = {g, g + o1, g + o2, g + o3, g + o4};
  float *dst[5] = {dW_ih, dW_hh, db_ih, db_hh, dW_hr};
  const size_t n[5] = {(size_t)G * K, (size_t)G * Ho, (size_t)G, (size_t)G, (size_t)P * H};
  for (int i = 0; i < 5; ++i)
    if (dst[i] && n[i]) CU(cudaMemcpyAsync(dst[i], src[i], n[i] * 4, cudaMemcpyDefault, s));
  return RCU_OK;
}

extern "C" int rnn_get_pack(rcu_rnn_t h, int32_t *sorted_idx, int32_t *unsorted_idx,
                            int32_t *batch_sizes, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_get_pack: NULL handle");
  if (h->last_B < 0) return fail(RCU_ERR_STATE, "rnn_get_pack: no forward has run");
  cudaStream_t s = (cudaStream_t)stream;
  const size_t nb = (size_t)h->last_B * 4, nt = (size_t)h->last_T * 4;
  if (sorted_idx)
    CU(cudaMemcpyAsync(sorted_idx, h->meta.sorted_idx, nb, cudaMemcpyDeviceToDevice, s));
  if (unsorted_idx)
    CU(cudaMemcpyAsync(unsorted_idx, h->meta.unsorted_idx, nb, cudaMemcpyDeviceToDevice, s));
  if (batch_sizes)
    CU(cudaMemcpyAsync(batch_sizes, h->meta.batch_sizes, nt, cudaMemcpyDeviceToDevice, s));
  return RCU_OK;
}

extern "C" int rnn_get_status(rcu_rnn_t h, void *stream) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_get_status: NULL handle");
  cudaStream_t s = (cudaStream_t)stream;
  CU(cudaStreamSynchronize(s));
  CU(cudaGetLastError());
  int v = 0;
  CU(cudaMemcpy(&v, h->ctl.p, sizeof v, cudaMemcpyDeviceToHost));
  CU(cudaMemset(h->ctl.p, 0, sizeof v));
  return status_from_dev(v);
}

extern "C" int rnn_last_launch_count(rcu_rnn_t h) { return h ? h->launches : -1; }

extern "C" int rnn_host_plan(rcu_rnn_t h, int *chunks, int *x_in_place, int *y_in_place) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_host_plan: NULL handle");
  if (chunks) *chunks = h->plan_chunks;
  if (x_in_place) *x_in_place = h->plan_x_in_place;
  if (y_in_place) *y_in_place = h->plan_y_in_place;
  return RCU_OK;
}

extern "C" int rnn_profile_entry(rcu_rnn_t h, int i, const char **name, double *total_ms,
                                 int64_t *count) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_profile_entry: NULL handle");
  return h->entry(i, name, total_ms, count);
}

extern "C" int rnn_get_trace(rcu_rnn_t h, int64_t *host_out, int n_steps, void *stream) {
  if (!h || !host_out || n_steps < 0) return fail(RCU_ERR_INVALID, "rnn_get_trace: bad arguments");
  if (!h->trace_buf.p) return fail(RCU_ERR_STATE, "rnn_get_trace: no traced forward");
  const int n = std::min(n_steps, h->trace_T);
  CU(cudaStreamSynchronize((cudaStream_t)stream));
  CU(cudaMemcpy(host_out, h->trace_buf.p, (size_t)n * 16 * 8, cudaMemcpyDeviceToHost));
  return RCU_OK;
}

extern "C" int rnn_profile_reset(rcu_rnn_t h) {
  if (!h) return fail(RCU_ERR_INVALID, "rnn_profile_reset: NULL handle");
  h->reset();
  return RCU_OK;
}

extern "C" int rnn_destroy(rcu_rnn_t h) {
  if (!h) return RCU_OK;
  cudaDeviceSynchronize();
  delete h;
  return RCU_OK;
}
