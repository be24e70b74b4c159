// Argument blocks and launchers of the non-GEMM kernels.
#pragma once

#include <cuda.h>

#include "internal.h"

namespace dlite {

struct StageArgs {
  const void* hidden = nullptr;  // [B, m, D] (f32 or bf16)
  const int32_t* anchor = nullptr;  // [B, G]: the local token group, the anchor last
  const void* E = nullptr;       // [V, D] in the weight dtype (anchor row lookup)
  int E_tiled = 0;               // E stored in the tiled layout (bf16 weights)
  const float* e_depth = nullptr;
  const float* g_stage = nullptr;
  const float* e_ph = nullptr;
  const float* g_attn0 = nullptr;
  int B = 0, m = 0, K = 0, D = 0, V = 0, G = 1;
  float eps = 1e-6f;
  bf16* z[2] = {nullptr, nullptr};
  int nz = 1;
  float* x = nullptr;            // [B*(G+K), D]
  bf16* y[2] = {nullptr, nullptr};
  int ny = 1;
  float* tap_z = nullptr;
  int* status = nullptr;
};

struct AttnArgs {
  const float* part_loc = nullptr;  // [splits][B*(K+1)][qd + 2 kvd]
  Splits sp_loc;
  const float* part_ctx = nullptr;  // [splits][ctx_rows][ldc]: row ctx_row0 + b m + j, columns ctx_col0 ..
  Splits sp_ctx;
  int ctx_row0 = 0, ctx_col0 = 0, ldc = 0, ctx_rows = 0;  // ldc = 0: 2 kvd; ctx_rows = 0: B m
  int loc_rows = 0;  // rows of a local partial plane (0: B (K+1))
  const float* rope_cos = nullptr;  // [K+1][d_h/2]
  const float* rope_sin = nullptr;
  int B = 0, m = 0, K = 0, n_q = 0, n_kv = 0, d_h = 0;
  int K1 = 0;  // local rows per request (G + K; 0: K + 1)
  int hq = 1;  // query heads per CTA (divides n_q / n_kv): attention_heads_per_cta
  float scale = 1.f;
  int round_bf16 = 0;
  bf16* o[2] = {nullptr, nullptr};  // [B*(K+1), n_q*d_h]
  int no = 1;
  // history mode (bf16 values): instead of attending, hand the rotated block to
  // the history kernels: queries [B][n_kv][(n_q/n_kv) K1][d_h] (row hh K1 + i);
  // block keys / values (context rows, then local rows) at rows
  // (b n_kv + g) hist_ld + hist_off + j of the layer's key / value tensors
  bf16* hist_q = nullptr;
  bf16* hist_k = nullptr;
  bf16* hist_v = nullptr;
  int hist_ld = 0, hist_off = 0;
};

struct ResNormArgs {
  const float* part = nullptr;  // [splits][rows][D]
  Splits sp;
  int rows = 0, D = 0;
  float* x = nullptr;           // [rows, D], updated in place
  const float* g = nullptr;
  float eps = 1e-6f;
  bf16* y[2] = {nullptr, nullptr};
  int ny = 1;
  int final_mode = 0;
  int K1 = 0;                   // rows per request (final mode)
  int G = 1;                    // leading group rows per request, dropped in final mode
  float* bout = nullptr;        // [B*K, D] (final mode)
  bf16* bp[2] = {nullptr, nullptr};
  float* tap_x = nullptr;
  float* tap_b = nullptr;
};

struct ChainArgs {
  const float* part = nullptr;  // [S][B*K][2Rp]: c at [0, R), e at [Rp, Rp + R)
  int S = 1, rows = 0;
  const float* Mt = nullptr;    // M = Q_h P in the chain's register image (launch_head_matrix)
  int B = 0, K = 0, R = 0;
  float* t = nullptr;           // [B*K, R]
  bf16* tp[2] = {nullptr, nullptr};  // [B*K, ldt] planes (columns R..ldt stay zero)
  int ldt = 0;
  int Bg = 1;                   // requests per cluster (chain_group_size)
  int Rp = 0;                   // R padded to 64
};

struct VerifyArgs {
  int B = 0, K = 0, V = 0, D = 0;
  const int32_t* cand = nullptr;
  const int32_t* tgt = nullptr;        // greedy
  const dlite_qstats* qs = nullptr;    // sampling
  const float* hs = nullptr;           // [B*K, D]
  const float* probs = nullptr;        // [B, K+1, V]
  const bf16* Eb = nullptr;            // E rows for q(v) (bf16 weights, tiled layout)
  const float* Ef = nullptr;           // ... or fp32 weights
  unsigned long long* resid = nullptr; // [B, V] fallback scratch (fixed-point residual)
  unsigned long long* counters = nullptr;  // [4]: residual draws, proposals, fallbacks, bonus
  double T = 0.0;
  uint32_t k0 = 0, k1 = 0;
  const int64_t* pos = nullptr;
  int32_t* accepted = nullptr;
  int32_t* commits = nullptr;
  int32_t* n_commit = nullptr;
  int32_t* next_anchor = nullptr;
  int* status = nullptr;
  int kv = -1;                         // candidates verified (the first kv of K; -1: all K)
  int32_t* tsamp = nullptr;            // match mode: the target's samples [B, K+1]
};

// The gated token-feedback head's per-step state (gated.cu).
struct GatedArgs {
  int B = 0, K = 0, R = 0, G = 1, V = 0;
  const int32_t* anchor = nullptr;   // [B, G]: d_0 is the last
  int32_t* cand_tmp = nullptr;       // [B] this step's choice (written by the LM merge)
  dlite_qstats* qs_tmp = nullptr;    // [B]
  int32_t* cand = nullptr;           // [B, K]
  dlite_qstats* qs = nullptr;        // [B, K] or null
  const int64_t* pos = nullptr;      // [B] or null
  int64_t* pos_i = nullptr;          // [B] pos + i - 1 (the LM head's positions at step i)
  const float* ER = nullptr;         // [V, R] fp32
  const float* bs = nullptr;         // [2R]
  const float* bh = nullptr;         // [R]
  const float* hu = nullptr;         // [B*K, R] W_h[:, R:] u_i
  float* s = nullptr;                // [2][B, R] state, double-buffered by step parity
  const bf16* Ws[2] = {nullptr, nullptr};   // W_s [2R, 2R], tiled bf16 planes
  const bf16* Whs[2] = {nullptr, nullptr};  // W_h[:, :R] [R, R], tiled bf16 planes
  int np = 1;                               // weight planes
  float* r_all = nullptr;            // [B*K, R]
  float* r_step = nullptr;           // [B, R]
  bf16* rp = nullptr;                // [B, R] bf16(r) (the vocabulary product's activation)
  int* status = nullptr;
  int warm = 0;                      // s_0 from a warm-up step on the token before the anchor
};
// fused: the step's r in the same launch (one weight plane; a cluster of R / 32
// CTAs per group of 4 requests). gated_step_clusters: how many such clusters
// the device runs at once (0: the fused form is unavailable)
cudaError_t launch_gated_state(const GatedArgs& a, int i, bool fused, cudaStream_t s);
cudaError_t launch_gated_r(const GatedArgs& a, int i, cudaStream_t s);
int gated_step_clusters(const GatedArgs& a);
cudaError_t launch_gated_sum(const float* part, const Splits& sp, int rows, int cols, float* out,
                             cudaStream_t s);
cudaError_t launch_gated_final(const GatedArgs& a, cudaStream_t s);

cudaError_t launch_stage(const StageArgs& a, bool f32, cudaStream_t s);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);
size_t attention_smem(int K1, int m, int d_h, int G);  // K1 local rows per request
int attention_heads_per_cta(int n_q, int n_kv, int B);
cudaError_t launch_resnorm(const ResNormArgs& a, cudaStream_t s);
cudaError_t launch_swiglu_interleaved(const float* part, const Splits& sp, int rows, int F, bf16* const* o, int no,
                                      cudaStream_t s);
cudaError_t launch_head_chain(const ChainArgs& a, cudaStream_t s);
int chain_group_size(int R, int B);
size_t chain_smem_bytes(int R, int K, int Bg);
cudaError_t launch_head_out(const float* part, int S, int rows, int D, const float* b, float* hs,
                            bf16* const* hp, float* tap, cudaStream_t s);
cudaError_t launch_split(const float* src, size_t n, bf16* const* pl, float* copy, cudaStream_t s);
cudaError_t launch_verify_greedy(const VerifyArgs& a, cudaStream_t s);
cudaError_t launch_verify_sample(const VerifyArgs& a, cudaStream_t s);
// match mode, step 1: the target's own samples t_j ~ p_j for j = 0..kv into a.tsamp
// (step 2 is launch_verify_greedy with a.tgt = a.tsamp)
cudaError_t launch_match_sample(const VerifyArgs& a, cudaStream_t s);
cudaError_t launch_advance(int B, const int32_t* n_commit, int64_t* pos, cudaStream_t s);
// Bounded-wait probe: result[0] / result[1] = 1 when the warp-wide / single-thread wait on a
// barrier nobody arrives at gave up after limit_ns (flagging the timeout bit in *status);
// result[2] = 1 when a following kernel sees that bit at entry and skips its work.
cudaError_t launch_wait_probe(uint64_t limit_ns, int* status, int32_t* result, cudaStream_t s);
cudaError_t launch_shift_group(int B, int G, int K1, const int32_t* commits, const int32_t* n_commit,
                               int32_t* group, cudaStream_t s);
cudaError_t launch_repack(const void* src, bool src_f32, int rows, int cols, int src_ld,
                          int src_off, bf16* p0, bf16* p1, int np, float* f32, int dst_ld,
                          cudaStream_t s);
cudaError_t launch_repack_gate_up(const void* Wg, const void* Wu, bool src_f32, int F, int D, bf16* p0, bf16* p1,
                                  int np, cudaStream_t s);
cudaError_t launch_head_matrix(const void* Q, const void* P, bool f32, int D, int R, float* Mt,
                               cudaStream_t s);

// ---------------------------------------------------------------- history-KV control
// Per layer one key and one value tensor of `rows` rows x d_h bf16: row
// (b n_kv + g) Hx + t holds ring slot t < H of request slot b, head g, and
// rows H .. H + m + G + K - 1 behind it the current block's rows (so a head's
// keys are one contiguous run); rows past B_max n_kv Hx are padding.
struct HistFillArgs {
  bf16* k = nullptr;  // [L][rows][d_h]
  bf16* v = nullptr;
  int* cursor = nullptr;  // [B_max], zeroed
  int L = 0, Bm = 0, n_kv = 0, H = 0, Hx = 0, d_h = 0;
  size_t rows = 0;
};
struct HistAttnArgs {
  const bf16* q = nullptr;   // [B][n_kv][QR][d_h] the block's rotated queries
  int B = 0, n_kv = 0, H = 0, Hx = 0, Tk = 0, QR = 0;
  int sub_per_chunk = 1, nchunk = 1;  // 64-key sub-tiles per chunk; chunks
  float scale_log2 = 1.f;             // softmax scale x log2(e)
  float* part_o = nullptr;            // [B][n_kv][nchunk][KS][QR][d_h] (KS = hist_key_splits(QR))
  float* part_ml = nullptr;           // [B][n_kv][nchunk][KS][QR][2]: running max (log2 domain), sum
  int* status = nullptr;              // copy timeouts
};
struct HistCombineArgs {
  const float* part_o = nullptr;
  const float* part_ml = nullptr;
  int B = 0, n_q = 0, n_kv = 0, d_h = 0, QR = 0, K1 = 0, m = 0, H = 0, Hx = 0;
  int nchunk = 1;             // partials per row: chunks x key splits
  bf16* o = nullptr;          // [B K1][n_q d_h]
  bf16* kc = nullptr;         // this layer's key / value tensors (block rows appended into the ring)
  bf16* vc = nullptr;
  const int* cursor = nullptr;
};
struct HistPlan {
  int sub_per_chunk = 1, nchunk = 1;
};
size_t hist_attn_smem(int d_h, int QR);
int hist_key_splits(int QR);           // key halves per tile (partials per chunk)
long long hist_max_ctas(int num_sms);  // bound on chunks x heads x requests (partial buffer sizing)
HistPlan hist_plan(int B, int n_kv, int H, int Tk, int QR, int d_h, int num_sms);
cudaError_t launch_hist_fill(const HistFillArgs& a, cudaStream_t s);
cudaError_t launch_hist_attn(const CUtensorMap* mk, const CUtensorMap* mv, const HistAttnArgs& a, int d_h,
                             cudaStream_t s);
cudaError_t launch_hist_combine(const HistCombineArgs& a, cudaStream_t s);
cudaError_t launch_hist_advance(int* cursor, int B, int n, int H, cudaStream_t s);

}  // namespace dlite
