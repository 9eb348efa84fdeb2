// Internal launchers shared by the host API (api.cu) and the kernel files.
#pragma once

#include <vector>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rcu {

// Packing metadata for one forward (device int32 arrays inside the workspace).
struct Meta {
  int32_t *sorted_idx;   // [B] original row at sorted position s
  int32_t *unsorted_idx; // [B] sorted position of original row b
  int32_t *lens_sorted;  // [B] length of the row at sorted position s
  int32_t *batch_sizes;  // [T] rows with length > t
  int32_t *step_off;     // [T+1] exclusive prefix of batch_sizes; step_off[T] = packed rows
};

// ---- api.cu: record `msg` as this host thread's last error; returns `code`
int set_error(int code, const char *msg);

// ---- pack.cu -------------------------------------------------------------
// Build Meta from lengths (NULL = every row has length T).  Lengths outside
// [1, T] raise DEV_LENGTHS in *err and are clamped so later kernels stay in bounds.
cudaError_t launch_meta(const int32_t *lengths, int B, int T, Meta m, int *err, cudaStream_t s);
// Gather x [T,B,in] (fp32) into packed order (step_off[t] + s) and convert to OT.
template <typename OT>
cudaError_t launch_pack_rows(const float *x, int T, int B, int in, Meta m, OT *out, int ld_out,
                             cudaStream_t s);
// Zero y[t, b, :] for t >= lengths[b] (varlen only).
cudaError_t launch_zero_tail(float *y, const int32_t *lengths, int T, int B, int width,
                             int *err, cudaStream_t s);
// Convert fp32 [n] to OT (weights / bias preparation).
template <typename OT>
cudaError_t launch_convert(const float *src, OT *dst, size_t n, cudaStream_t s);

// ---- gemm_simt.cu ----------------------------------------------------------
// G[m, n] = sum_k X[m, k] * W[n, k] + bias[n] for m < *M_dev (or M when M_dev
// is NULL).  Row-major; ldx/ldw/ldg are row strides in elements.
template <typename XT, typename WT>
// err: device error word (DEV_CONFIG if a K-split cluster launch ran with
// another cluster shape), or NULL.
cudaError_t launch_gemm_simt(const XT *X, int ldx, const WT *W, int ldw, const float *bias,
                             float *G, int ldg, int M, const int32_t *M_dev, int N, int K,
                             cudaStream_t s, int *err);

// ---- recurrent_simt.cu -------------------------------------------------------
// all-CTA step trace window (RCU_ATTR_TRACE = 2)
constexpr int TRACE_ALL_S0 = 16, TRACE_ALL_N = 8, TRACE_ALL_CTAS = 1024;
struct RecParams {
  int T, B, H, Hout, Kp, Hp, nG, D, cell, proj;
  int U, NU, Rp;   // units per CTA, unit groups per direction, padded gate rows per CTA
  int Pc, Pcp, NP; // projection rows per CTA (padded), CTAs with projection rows
  int CB;          // batch rows per chunk (multiple of 4, <= 32)
  Meta meta;
  const float *G;
  int ldG;                // G row stride; direction d's gates start at column d*nG*H
  const void *Whh[2];     // [NU][Kp][Rp] per direction, WT
  const void *Whr[2];     // [NP][Hp][Pcp] per direction, WT (projection only)
  const float *bhn[2];    // GRU hidden-side n-gate bias [H] (NULL = zero)
  const float *h0, *c0;   // [D][B][Hout], [D][B][H] original row order (NULL = zero)
  float *h_n, *c_n;       // [D][B][Hout], [D][B][H] or NULL
  float *y;               // last layer: [T][B][D*Hout] original order, or NULL
  void *ymid;             // other layers: packed [M][D*Hout] (OT), or NULL
  void *hx;               // exchange [D][2][B][Kp] (OT)
  void *mx;               // projection input exchange [D][B][Hp] (OT)
  float *hst, *cst;       // fp32 state [D][B][Hout], [D][B][H]
  unsigned *ctr;          // [D] barrier counters (zeroed before launch)
  int *err;
  uint64_t timeout_ns;
  int drop_arrival;
  unsigned long long *trace;  // NULL, or [T][16] global-timer stamps written by CTA 0
  // NULL, or stamps of every CTA for steps [TRACE_ALL_S0, TRACE_ALL_S0 + TRACE_ALL_N):
  // row (step - TRACE_ALL_S0) * TRACE_ALL_CTAS + blockIdx.x, 16 slots (tensor-core kernel)
  unsigned long long *trace_all;
  // LSTM clipping: c_t clamped to [cclip_lo, cclip_hi] when updated (cclip != 0);
  // projected h_t clamped to [pclip_lo, pclip_hi] when formed (pclip != 0)
  int cclip, pclip;
  float cclip_lo, cclip_hi, pclip_lo, pclip_hi;
};
// wbf16: weights stored bf16 (operands bf16) vs fp32.
cudaError_t launch_recurrent_simt(const RecParams &p, bool wbf16, int nsm, cudaStream_t s);
size_t recurrent_simt_smem(const RecParams &p, bool wbf16);
// choose the batch chunk p.CB so that the shared-memory plan fits; false if none does
bool plan_recurrent_simt(RecParams &p, bool wbf16);

// ---- recurrent_cluster.cu: cluster-resident kernel for a W_hh that fits one
// thread-block cluster (LSTM / GRU without projection)
struct ClusterRecPlan {
  int cs, U, Kc, Bc, NCL;  // cluster size, units per CTA, padded K, rows per cluster, clusters per direction
  size_t smem;
};
int cluster_rec_kc(int Hout);
bool cluster_rec_packable(int cell, int H, int Hout, int P, bool wbf16);
// rows u*nG + g (gate g of unit u), Kc = cluster_rec_kc(Hout) columns, zero padded
void cluster_pack_whh(int cell, int H, int Hout, const float *whh, std::vector<float> &out);
// false when no cluster plan fits, or the batch slice would exceed max_rows
bool plan_recurrent_cluster(ClusterRecPlan *cp, int cell, int H, int Hout, int T, int B, int D,
                            bool wbf16, int max_rows);
cudaError_t launch_recurrent_cluster(const RecParams &p, const ClusterRecPlan &cp,
                                     const void *W0, const void *W1, bool wbf16, cudaStream_t s);

// ---- lstmp_fold.cu -------------------------------------------------------------
// G rows of each sequence's first step (direction d) += W_hh h0 (W_hh fp32 [4H][P]).
cudaError_t launch_h0_gates(float *G, int ldG, const float *Whh, const float *h0, int B, int T,
                            int H4, int P, int d, cudaStream_t s);
// h_n (direction d, [B][P]) from the projected outputs Y [T*B][ldY].
cudaError_t launch_last_h(const float *Y, int ldY, float *h_n, int B, int T, int P, int d,
                          cudaStream_t s);

// ---- rssm.cu -----------------------------------------------------------------
struct RssmParams {
  int S, A, Hd, RH, T, B;
  const float *W1, *b1, *Wih, *Whh, *bih, *bhh, *W2, *b2, *W3, *b3; // PyTorch layout, fp32
  const float *state0, *belief0, *actions, *eps;
  float *means, *stds, *states, *beliefs;
  unsigned long long *trace;  // NULL, or [T][16] stamps written by CTA 0 (see rssm_get_trace)
  int *err;                   // device error word (DEV_TIMEOUT when a bounded wait gave up)
  uint64_t timeout_ns;        // bound on each wait for a broadcast vector
  int drop_send;              // testing: the first CTA of cluster 0 skips its step-0 state send
  // unroll variant 2: Wa1 != NULL computes each step's action as
  // tanh(Wa2 ELU(Wa1 [state, belief] + ba1) + ba2) (Wa1 [Hx, S+RH], Wa2 [A, Hx]);
  // actions_out [T,B,A] receives them (may be NULL); `actions` is unused
  int Hx;
  const float *Wa1, *ba1, *Wa2, *ba2;
  float *actions_out;
};
cudaError_t launch_rssm(const RssmParams &p, int nsm, cudaStream_t s, int *clusters_used);

// Reverse-time chain of the RSSM backward pass (given actions) in one launch:
// per step ds_t -> dp -> dv -> dh_t -> gate gradients -> du -> ds_{t-1} and
// dh_{t-1}, the transposed weights resident in a thread-block cluster.
struct RssmBwdChainParams {
  int S, A, Hd, RH, T, B;
  const float *W1, *Wih, *Whh, *W2, *W3;              // PyTorch layout, fp32
  const float *dmeans, *dstds, *dstates, *dbeliefs;   // [T][B][S] / [T][B][RH], NULL = 0
  const float *eps;                                   // [T][B][S]
  const float *p;                                     // head outputs [T*B][2S]
  const float *v, *u;                                 // pre-ELU W2 h + b2, W1 [s, a] + b1 [T*B][Hd]
  const float *gates;                                 // activated r, z, n [T*B][3RH]
  const float *zh;                                    // hidden-side pre-activations [T*B][3RH]
  const float *hp;                                    // h_{t-1} [T*B][RH]
  float *DP, *DV, *DA, *DR, *DU;                      // [T*B][2S], [Hd], [3RH], [3RH], [Hd]
  float *cs_out;                                      // [B][S]: ds_{-1} (dstate0)
  float *gh_out;                                      // [B][RH]: dh_{-1} (dbelief0)
  int *err;
  uint64_t timeout_ns;
};
// false (nothing launched) when the resident plan does not fit
bool rssm_bwd_chain_supported(int S, int A, int Hd, int RH);
cudaError_t launch_rssm_bwd_chain(const RssmBwdChainParams &p, int nsm, cudaStream_t s);
// the weights (and, with Hx > 0, the actor's) fit one cluster's shared memory
bool rssm_supported(int S, int A, int Hd, int RH, int Hx = 0);

// ---- backward.cu: backward pass through time (fp32, unidirectional) ---------
// zin: X W_ih^T + b_ih in, activated gates out; zh: H_prev W_hh^T + b_hh;
// cs: LSTM cell sequence out; ms: m_t = o tanh(c_t) out (projection) or NULL.
// cr: LSTM cell clipping, the unclamped c_t out (c_t itself clamped to
// [clo, chi]), or NULL.  Parallel over B*H, sequential over T.
cudaError_t launch_bwd_prep(int T, int B, int H, int cell, float *zin, const float *zh,
                            const float *c0, float *cs, float *ms, cudaStream_t s,
                            float *cr = nullptr, float clo = 0.f, float chi = 0.f);
// dst[i] += src[i], i < n
cudaError_t launch_add(float *dst, const float *src, size_t n, cudaStream_t s);
// out[s][b][0..w) = in[t][b][col0 .. col0+w) with t = s, or, reversed,
// t = len_b-1-s for s < len_b and t = s past the row's end (len_b = T without
// lengths); the map is its own inverse.  in: row stride ldi per (t, b);
// out: contiguous [T][B][w]
cudaError_t launch_gather_steps(const float *in, int ldi, int col0, int w, int T, int B,
                                bool reverse, const int32_t *lengths, float *out,
                                cudaStream_t s);
// out[t][b][:] = in[t][b][:] for t < len_b, plus dhn[b][:] (NULL: none) at
// t = len_b - 1, and 0 for t >= len_b; [T][B][w] contiguous, out may be in
cudaError_t launch_mask_steps(const float *in, int w, int T, int B, const int32_t *lengths,
                              const float *dhn, float *out, cudaStream_t s);
// ---- rssm_backward.cu: RSSM backward pieces ---------------------------------
// in [T*B][S+A] = [s_{t-1}, a_t] (s_{-1} = state0, NULL: 0)
cudaError_t launch_rssm_inputs(int T, int B, int S, int A, const float *state0,
                               const float *states, const float *actions, float *in,
                               cudaStream_t s);
// post = ELU(pre); out = g * ELU'(pre)  (n elements)
cudaError_t launch_elu(const float *pre, float *post, size_t n, cudaStream_t s);
cudaError_t launch_elu_grad(const float *g, const float *pre, float *out, size_t n,
                            cudaStream_t s);
// out = g * (1 - y^2)  (y = tanh of something; n elements)
cudaError_t launch_tanh_grad(const float *g, const float *y, float *out, size_t n, cudaStream_t s);
// step t: dp (rows t*B..) of the sample and head from dmeans/dstds/dstates
// (NULL = 0), eps, the head output p [T*B][2S] and cs [B][S] (ds from t+1)
cudaError_t launch_rssm_sample_grad(int t, int B, int S, const float *dmeans, const float *dstds,
                                    const float *dstates, const float *eps, const float *p,
                                    const float *cs, float *dp, cudaStream_t s);
// step t: GRU gate gradients (DA, DR rows t*B..) from dh = dbeliefs_t + dhq +
// gh + dhz ([B][RH] each); dhz <- z_t * dh
cudaError_t launch_rssm_gru_grad(int t, int B, int RH, const float *dbeliefs, const float *dhq,
                                 const float *gh, float *dhz, const float *gates, const float *zh,
                                 const float *hp, float *DA, float *DR, cudaStream_t s);

// Weight and bias gradients of up to WG_MAX_GROUPS layers over M rows in two
// launches: dW [nz][ny] = dZ^T Y and db [nz] = column sums of dZ, from
// row-major dZ [M][nz] and Y [M][ny]; the rows are summed in chunks of
// WG_ROWS_PER_CHUNK whose partials are added in a fixed order.  scratch:
// wgrad_scratch_floats(groups, n, M) floats.  (tile0 and off are set by the
// launcher.)
constexpr int WG_MAX_GROUPS = 8, WG_ROWS_PER_CHUNK = 160;
struct WgradGroup {
  const float *dz;
  int nz;
  const float *y;
  int ny;
  float *dW, *db;
  int tile0;
  size_t off;
};
struct WgradParams {
  int ngroups, M, S, mchunk;
  size_t total;
  float *part;
  WgradGroup g[WG_MAX_GROUPS];
};
size_t wgrad_scratch_floats(const WgradGroup *g, int n, int M);
cudaError_t launch_wgrad(const WgradGroup *groups, int n, int M, float *scratch, cudaStream_t s);

struct BwdRecArgs {
  int T, B, H, cell;
  const float *Whh;  // [nG*H][ldw]
  int ldw;
  const float *gates, *zh, *cs, *c0, *hp, *dy, *dhn, *dcn;
  // [B] or NULL: steps t >= lengths[b] get zero gate gradients and pass the
  // carried gradients through (dh_n must then come in through dy, dhn NULL)
  const int32_t *lengths;
  // LSTM cell clipping: the unclamped c_t [T*B][H] (NULL: none) and its bounds
  const float *cr;
  float clo, chi;
  float *DA, *DR, *dh0, *dc0;
  unsigned *ctr;  // zeroed before the launch
  int *err;
  uint64_t timeout_ns;
  int drop_arrival;  // testing: CTA 0 skips its first step arrival (the wait must run out)
  unsigned long long *trace;  // NULL, or [T+1][16] global-timer stamps of CTA 0
};
// hidden units per CTA of the reverse-time kernel, 0 if W_hh^T does not fit
int bwd_units_per_cta(int H, int B, int nG, int nsm);
// a2: a second problem of the same T, B, H and cell (the other direction of a
// bidirectional layer, with its own buffers and counters) in the same launch,
// each on half of the SMs
cudaError_t launch_bwd_rec(const BwdRecArgs &a, int nsm, cudaStream_t s,
                           const BwdRecArgs *a2 = nullptr);
cudaError_t launch_transpose(const float *in, int R, int C, int ldi, float *out, int ldo,
                             cudaStream_t s);
// the same, rounded to bf16 (a tensor-core GEMM operand), and a row-wise
// fp32 -> bf16 copy with its own row strides
cudaError_t launch_transpose_bf16(const float *in, int R, int C, int ldi, __nv_bfloat16 *out,
                                  int ldo, cudaStream_t s);
cudaError_t launch_convert_rows_bf16(const float *in, int R, int C, int ldi, __nv_bfloat16 *out,
                                     int ldo, cudaStream_t s);
// the fp32 transpose, and its bf16 rounding too when outb is given (same ldo)
cudaError_t launch_transpose_dual(const float *in, int R, int C, int ldi, float *out,
                                  __nv_bfloat16 *outb, int ldo, cudaStream_t s);
size_t colsum_scratch_floats(int M, int N);
cudaError_t launch_colsum(const float *A, int M, int N, float *scratch, float *out,
                          cudaStream_t s);

}  // namespace rcu
