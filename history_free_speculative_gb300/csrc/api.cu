// C ABI of the DLite round: handle lifetime, weight preparation, workspace
// layout and the launch sequences of draft / verify.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "kernels.h"
#include "tc_gemm.h"

using namespace dlite;

struct LayerW {
  const bf16* Wqkv[2];  // [qd + 2 kvd, D] = [Wq; Wk; Wv]
  const bf16* Wo[2];    // [D, qd]
  const bf16* Wgu[2];   // [2F, D]: gate and up rows interleaved in blocks of 32 (fused SwiGLU)
  const bf16* Wd[2];    // [D, F]
  float* g_attn;
  float* g_ffn;
};

// A one-CTA-engine product shape and the plan chosen for it by timing at create.
struct TunedPlan {
  int rows, outs, K, xp, wp, act, skip_row0, skip_cols;
  tc::Plan pl;
};

struct MapEntry {
  const void* base;
  int rows, K, box;
  bool tiled;
  CUtensorMap map;
};

// Map of fp32 split-K partials [S][rows][outs] (bulk-store epilogue).
struct OutMapEntry {
  const void* base;
  int S, rows, outs;
  CUtensorMap map;
};

struct dlite_handle {
  dlite_config cfg;
  bool f32 = false;
  int np = 1;  // planes of the weights (2 for fp32 weights)
  int xp = 1;  // planes of the backbone activations (2: fp32-class, cfg.act_planes or fp32 weights)
  int qd = 0, kvd = 0;
  int Rp = 0;                       // R padded to a multiple of 64 (GEMM k extent)
  int Lcap = 0, Ccap = 0, Hcap = 0;  // activation row capacities (multiples of 128)
  int num_sms = 0;  // SMs of the device (persistent LM-head grid)
  std::vector<void*> allocs;
  std::vector<MapEntry> maps;
  std::vector<OutMapEntry> out_maps;
  std::vector<TunedPlan> tuned;  // plans of the B_max products, chosen by timing (tune_products)
  size_t part_cap = 0;           // floats in part

  // weights
  float *e_depth = nullptr, *g_stage = nullptr, *e_ph = nullptr, *g_final = nullptr;
  const void* E_src = nullptr;  // E in the weight dtype (anchor lookup, q(v) rows)
  const bf16* E[2] = {nullptr, nullptr};
  LayerW layer[DLITE_MAX_LAYERS];
  const bf16* Wce[2] = {nullptr, nullptr};  // [2R, D] = [Q_b; Q_h]
  const bf16* P[2] = {nullptr, nullptr};    // [D, R]
  float* Mt = nullptr;                      // [R, R] Q_h P in the chain's register image
  // gated token-feedback head (head_type 1)
  bool gated = false;
  int gated_clusters = 0;  // fused-step clusters (R / 32 CTAs, 4 requests each) the device runs at once
  const bf16 *Ws[2] = {nullptr, nullptr}, *Whs[2] = {nullptr, nullptr}, *Whu[2] = {nullptr, nullptr},
             *Wo[2] = {nullptr, nullptr};     // tiled planes: [2R, 2R], [R, R], [R, D], [Vp, R]
  float *ER32 = nullptr, *bs32 = nullptr, *bh32 = nullptr, *Wo32 = nullptr;  // fp32 (Wo32: fp32 drafters)
  int Bcap = 0;                             // B_max padded to 128 (rows of the vocabulary product's r operand)
  float *g_s = nullptr, *g_hu = nullptr, *g_r = nullptr, *g_rstep = nullptr;
  bf16* g_rp = nullptr;
  int32_t* g_cand = nullptr;
  dlite_qstats* g_qs = nullptr;
  int64_t* g_pos = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr;
  // history-KV control (cfg.history = H > 0)
  int H = 0, hQR = 0, hTk = 0, hHx = 0;  // Hx = H + m + G + K rows per (request, head)
  size_t hrows = 0;                       // rows of one layer's key (value) tensor
  bf16 *hk_ring = nullptr, *hv_ring = nullptr;   // [L_D][hrows][d_h]: ring, then the block's rows
  CUtensorMap hmap_k[DLITE_MAX_LAYERS], hmap_v[DLITE_MAX_LAYERS];  // 64-row x 64-column boxes
  int* hcursor = nullptr;                        // [B_max]
  bf16* hst_q = nullptr;                         // the rotated block queries of one layer
  float *hpart_o = nullptr, *hpart_ml = nullptr;  // chunk partials

  // workspace
  float* x = nullptr;
  bf16 *y[2] = {nullptr, nullptr}, *z[2] = {nullptr, nullptr}, *o[2] = {nullptr, nullptr},
       *a[2] = {nullptr, nullptr};
  float* b = nullptr;
  bf16* bp[2] = {nullptr, nullptr};
  float* t = nullptr;
  bf16* tp[2] = {nullptr, nullptr};
  float* hs = nullptr;
  bf16* hp[2] = {nullptr, nullptr};
  float *part = nullptr, *part2 = nullptr;
  LmRec* lmrec = nullptr;
  unsigned long long* resid = nullptr;
  int32_t* tsamp = nullptr;                 // [B_max, K+1] the target's samples (match verification)
  unsigned long long* counters = nullptr;
  int Vp = 0;  // V padded to a multiple of 64 (tiled LM-head weight rows)
  int* status = nullptr;

  // per-kernel event recording (dlite_stage_times)
  cudaEvent_t prof_ev[128];
  const char* prof_name[128];
  int prof_n = -1;  // -1: not recording
  bool prof_events_made = false;
  cudaStream_t prof_stream = nullptr;

  // staging for dlite_round_host
  void* d_hidden = nullptr;
  int32_t *d_anchor = nullptr, *d_tgt = nullptr, *d_cand = nullptr, *d_acc = nullptr,
          *d_commits = nullptr, *d_ncommit = nullptr, *d_next = nullptr;
  int64_t* d_pos = nullptr;
  float* d_probs = nullptr;
  dlite_qstats* d_qs = nullptr;
  // dlite_round_host copies the target rows on its own stream, under the draft
  cudaStream_t cstream = nullptr;
  cudaEvent_t ev_in = nullptr, ev_cp = nullptr;
};

namespace {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

#define CK(call)                     \
  do {                               \
    cudaError_t e_ = (call);         \
    if (e_ != cudaSuccess) {         \
      g_last_cuda_error = e_;        \
      return DLITE_ERR_CUDA;         \
    }                                \
  } while (0)

// Record an event after a launch when the handle is in profiling mode.
void mark(dlite_handle* h, const char* name) {
  if (h->prof_n < 0 || h->prof_n >= 127) return;
  h->prof_name[h->prof_n] = name;
  cudaEventRecord(h->prof_ev[++h->prof_n], h->prof_stream);
}

template <typename T>
int alloc(dlite_handle* h, T** p, size_t n) {
  void* q = nullptr;
  if (n == 0) n = 1;
  if (cudaMalloc(&q, n * sizeof(T)) != cudaSuccess) return DLITE_ERR_OOM;
  h->allocs.push_back(q);
  *p = (T*)q;
  return DLITE_OK;
}

#define AL(ptr, n)                          \
  do {                                      \
    int r_ = alloc(h, &(ptr), (size_t)(n)); \
    if (r_) return r_;                      \
  } while (0)

// local token group (anchor_group 0 or 1: the anchor alone)
static int group_of(const dlite_config* c) { return c->anchor_group > 1 ? c->anchor_group : 1; }

int check_config(const dlite_config* c) {
  if (!c) return DLITE_ERR_INVALID_ARG;
  if (c->dtype != DLITE_F32 && c->dtype != DLITE_BF16) return DLITE_ERR_INVALID_ARG;
  if (c->B_max < 1 || c->K < 1 || c->K > 31 || c->m < 1 || c->anchor_group < 0 || c->anchor_group > 8 ||
      c->m + c->K + group_of(c) > 32)
    return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->L_D < 1 || c->L_D > DLITE_MAX_LAYERS) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->n_q < 1 || c->n_kv < 1 || c->n_q % c->n_kv) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->d_h != 64 && c->d_h != 128) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->D > 16384) return DLITE_ERR_UNSUPPORTED_SHAPE;  // row kernels: 4 float4 per thread
  if (c->D % 64 || c->F % 64 || c->R % 32 || c->R > 512 || c->V < 8 || c->V % 8 || c->V > 262144)
    return DLITE_ERR_UNSUPPORTED_SHAPE;
  if ((c->n_q * c->d_h) % 64) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (attention_smem(group_of(c) + c->K, c->m, c->d_h, c->n_q / c->n_kv) > 200 * 1024)
    return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->R < 32 || chain_smem_bytes(c->R, c->K, chain_group_size(c->R, c->B_max)) > 200 * 1024)
    return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return DLITE_ERR_INVALID_ARG;
  if (c->head_type != DLITE_HEAD_RNN && c->head_type != DLITE_HEAD_GATED) return DLITE_ERR_INVALID_ARG;
  if (c->head_type == DLITE_HEAD_GATED && c->R % 64) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (c->act_planes < 0 || c->act_planes > 2) return DLITE_ERR_INVALID_ARG;
  if (c->act_planes == 2 && c->history > 0) return DLITE_ERR_UNSUPPORTED_SHAPE;  // the history kernels are bf16
  if (c->head_warmup < 0 || c->head_warmup > 1) return DLITE_ERR_INVALID_ARG;
  if (c->head_warmup && (c->head_type != DLITE_HEAD_GATED || group_of(c) < 2))
    return DLITE_ERR_UNSUPPORTED_SHAPE;  // the warm-up token is the group's second-to-last
  if (c->history < 0) return DLITE_ERR_INVALID_ARG;
  if (c->history > 0 && (c->dtype != DLITE_BF16 || c->history < group_of(c) + c->K || c->history > (1 << 20) ||
                         (c->n_q / c->n_kv) * (group_of(c) + c->K) > 128))
    return DLITE_ERR_UNSUPPORTED_SHAPE;
  return DLITE_OK;
}

// Copy a [rows, cols] slice of a weight (row stride src_ld, column offset off)
// into bf16 planes and / or fp32.
int repack(dlite_handle* h, const void* src, int rows, int cols, int src_ld, int off,
           const bf16** planes_out, float** f32_out) {
  bf16* p0 = nullptr;
  bf16* p1 = nullptr;
  const size_t n = (size_t)rows * cols;
  if (planes_out) {
    AL(p0, n);
    if (h->np == 2) AL(p1, n);
    planes_out[0] = p0;
    planes_out[1] = p1;
  }
  float* f = nullptr;
  if (f32_out) {
    AL(f, n);
    *f32_out = f;
  }
  // planes feed the tensor-core products: tiled layout (rows here are multiples of 64)
  CK(launch_repack(src, h->f32, rows, cols, src_ld, off, p0, p1, planes_out ? h->np : 0, f, -cols, 0));
  return DLITE_OK;
}

// Stack several [rows_i, cols] weights into one planes buffer.
int stack(dlite_handle* h, const void* const* srcs, const int* rows, int n, int cols,
          const bf16** planes_out) {
  int total = 0;
  for (int i = 0; i < n; ++i) total += rows[i];
  bf16* p0 = nullptr;
  bf16* p1 = nullptr;
  AL(p0, (size_t)total * cols);
  if (h->np == 2) AL(p1, (size_t)total * cols);
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    // every piece has a multiple of 64 rows, so the tiled pieces concatenate
    CK(launch_repack(srcs[i], h->f32, rows[i], cols, cols, 0, p0 + off, p1 ? p1 + off : nullptr,
                     h->np, nullptr, -cols, 0));
    off += (size_t)rows[i] * cols;
  }
  planes_out[0] = p0;
  planes_out[1] = p1;
  return DLITE_OK;
}

// A GEMM operand: one or two bf16 planes of a row-major [rows, K] buffer.
struct Operand {
  const bf16* p[2];
  int n;     // planes
  int rows;  // rows of the buffer (tensor-map extent)
  int K;     // k extent = row length
};

Operand opnd(const bf16* const* p, int n, int rows, int K) {
  Operand o;
  o.p[0] = p[0];
  o.p[1] = n == 2 ? p[1] : nullptr;
  o.n = n;
  o.rows = rows;
  o.K = K;
  return o;
}

const CUtensorMap* get_map(dlite_handle* h, const void* base, int rows, int K, int box,
                           bool tiled = false) {
  for (const MapEntry& e : h->maps)
    if (e.base == base && e.rows == rows && e.K == K && e.box == box && e.tiled == tiled) return &e.map;
  MapEntry e;
  e.base = base;
  e.rows = rows;
  e.K = K;
  e.box = box;
  e.tiled = tiled;
  if (!(tiled ? tc::make_map_tiled(&e.map, base, rows, K, box) : tc::make_map(&e.map, base, rows, K, box)))
    return nullptr;
  h->maps.push_back(e);
  return &h->maps.back().map;
}

const CUtensorMap* get_out_map(dlite_handle* h, const void* base, int S, int rows, int outs) {
  for (const OutMapEntry& e : h->out_maps)
    if (e.base == base && e.S == S && e.rows == rows && e.outs == outs) return &e.map;
  OutMapEntry e;
  e.base = base;
  e.S = S;
  e.rows = rows;
  e.outs = outs;
  if (!tc::make_out_map(&e.map, base, S, rows, outs)) return nullptr;
  h->out_maps.push_back(e);
  return &h->out_maps.back().map;
}

// One launch of the one-CTA engine with plan pl (partials, or the SwiGLU output when act is set).
int launch_onecta(dlite_handle* h, const tc::Plan& pl, const Operand& X, const Operand& W, int rows, int outs,
                  float* part, cudaStream_t s, bf16* const* act, int act_planes, int skip_row0, int skip_cols) {
  const int xb = tc::x_box_rows(rows);
  h->maps.reserve(h->maps.size() + 4);
  const CUtensorMap* x0 = get_map(h, X.p[0], X.rows, X.K, xb);
  const CUtensorMap* x1 = X.n == 2 ? get_map(h, X.p[1], X.rows, X.K, xb) : nullptr;
  const CUtensorMap* w0 = get_map(h, W.p[0], W.rows, W.K, pl.N, true);
  const CUtensorMap* w1 = W.n == 2 ? get_map(h, W.p[1], W.rows, W.K, pl.N, true) : nullptr;
  if (!x0 || !w0 || (X.n == 2 && !x1) || (W.n == 2 && !w1)) return DLITE_ERR_CUDA;
  tc::TcParams prm;
  prm.rows = rows;
  prm.outs = outs;
  prm.K = X.K;
  prm.xplanes = X.n;
  prm.wplanes = W.n;
  prm.mode = 0;
  prm.x_box = xb;
  prm.part = part;
  prm.status = h->status;
  prm.skip_row0 = skip_row0;
  prm.skip_cols = skip_cols;
  const CUtensorMap* out = nullptr;
  if (act) {
    prm.mode = 2;
    prm.act[0] = act[0];
    prm.act[1] = act_planes == 2 ? act[1] : nullptr;
    prm.act_planes = act_planes;
  } else {
    out = get_out_map(h, part, pl.S, rows, outs);  // partials leave through bulk tensor stores
    if (!out) return DLITE_ERR_CUDA;
  }
  CK(tc::launch(pl, x0, x1, w0, w1, prm, s, out));
  return DLITE_OK;
}

#define RUN(call)          \
  do {                     \
    int r_ = (call);       \
    if (r_) return r_;     \
  } while (0)

// part[z][r][o] = sum over split z of X[r, :] . W[o, :], r < rows, o < outs.
// With act != nullptr the product is the gate / up one (columns interleaved in
// blocks of 32): on the one-CTA engine the epilogue writes a = silu(gate) * up
// to the act planes directly and *fused is set; otherwise the partials are
// written as usual and the caller runs the SwiGLU kernel.
int gemm(dlite_handle* h, const char* name, const Operand& X, const Operand& W, int rows, int outs,
         float* part, Splits* sp_out, cudaStream_t s, bf16* const* act = nullptr, int act_planes = 1,
         bool* fused = nullptr, int skip_row0 = 0, int skip_cols = 0) {
  if (fused) *fused = false;
  const bool skipping = skip_row0 > 0;  // tiles to skip: the one-CTA engine
  if (!skipping && tc::use_pair_engine(rows, X.n, W.n)) {  // 2-SM MMAs
    const tc::PairPlan pp = tc::pair_plan(rows, outs, X.K, h->num_sms);
    if (pp.ok) {
      h->maps.reserve(h->maps.size() + 4);
      const CUtensorMap* x0 = get_map(h, X.p[0], X.rows, X.K, 128);
      const CUtensorMap* w0 = get_map(h, W.p[0], W.rows, W.K, 128, true);
      if (!x0 || !w0) return DLITE_ERR_CUDA;
      tc::PairParams prm;
      prm.rows = rows;
      prm.outs = outs;
      prm.part = part;
      prm.status = h->status;
      if (sp_out) *sp_out = tc::pair_splits(pp);
      CK(tc::launch_pair(pp, x0, w0, prm, s));
      mark(h, name);
      return DLITE_OK;
    }
  }
  tc::Plan pl = tc::plan(rows, outs, X.K, X.n, W.n, false, act != nullptr, skip_row0, skip_cols);
  for (const TunedPlan& t : h->tuned)
    if (t.rows == rows && t.outs == outs && t.K == X.K && t.xp == X.n && t.wp == W.n && t.act == (act != nullptr) &&
        t.skip_row0 == skip_row0 && t.skip_cols == skip_cols) {
      pl = t.pl;
      break;
    }
  if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (act && fused) *fused = true;
  if (sp_out) *sp_out = uniform_splits(pl.S);
  RUN(launch_onecta(h, pl, X, W, rows, outs, part, s, act, act_planes, skip_row0, skip_cols));
  mark(h, name);
  return DLITE_OK;
}

void seed_key(uint64_t seed, uint32_t* k0, uint32_t* k1) {
  *k0 = (uint32_t)(seed & 0xffffffffu);
  *k1 = (uint32_t)(seed >> 32);
}

// ---------------------------------------------------------------- stages

// LM head: one bf16 plane of h and of E; the merge re-scores the finalists exactly.
tc::Plan lm_plan(dlite_handle* h, int rows) {
  return tc::plan(rows, h->cfg.V, h->cfg.D, 1, 1, true);
}

// The gated head's fused step (state and r in one launch) when every one of its
// clusters (4 requests each) is resident at once.
static bool gated_fused(const dlite_handle* h, int B) {
  return h->gated_clusters > 0 && (B + 3) / 4 <= h->gated_clusters;
}

// bf16 drafters store the context rows z behind the local rows y in one
// buffer, and a single product [y; z] W_qkv^T on the one-CTA engine serves
// both, one launch instead of two: its tiles of context rows x query columns
// are skipped. fp32-class drafters run two products.
static bool fuse_ctx(const dlite_handle* h, int B) {
  const dlite_config& c = h->cfg;
  const int rows = B * (group_of(&c) + c.K) + B * c.m;
  if (h->np != 1 || h->xp != 1) return false;
  return tc::plan(rows, h->qd + 2 * h->kvd, c.D, 1, 1, false, false, B * (group_of(&c) + c.K), h->qd).ok;
}

// History-KV control, layer l: split-KV attention of the block's queries over
// the ring and the block, then the merge into h->o and the ring append.
int run_history_attention(dlite_handle* h, int B, int l, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  const HistPlan hp = hist_plan(B, c.n_kv, h->H, h->hTk, h->hQR, c.d_h, h->num_sms);
  const size_t ring_l = (size_t)l * h->hrows * c.d_h;
  HistAttnArgs ha;
  ha.q = h->hst_q;
  ha.B = B;
  ha.n_kv = c.n_kv;
  ha.H = h->H;
  ha.Hx = h->hHx;
  ha.Tk = h->hTk;
  ha.QR = h->hQR;
  ha.sub_per_chunk = hp.sub_per_chunk;
  ha.nchunk = hp.nchunk;
  ha.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.d_h));
  ha.part_o = h->hpart_o;
  ha.part_ml = h->hpart_ml;
  ha.status = h->status;
  CK(launch_hist_attn(&h->hmap_k[l], &h->hmap_v[l], ha, c.d_h, s));
  mark(h, "hist_attn");
  HistCombineArgs hc;
  hc.part_o = h->hpart_o;
  hc.part_ml = h->hpart_ml;
  hc.B = B;
  hc.n_q = c.n_q;
  hc.n_kv = c.n_kv;
  hc.d_h = c.d_h;
  hc.QR = h->hQR;
  hc.K1 = group_of(&c) + c.K;
  hc.m = c.m;
  hc.H = h->H;
  hc.Hx = h->hHx;
  hc.nchunk = hp.nchunk * hist_key_splits(h->hQR);
  hc.o = h->o[0];
  hc.kc = h->hk_ring + ring_l;
  hc.vc = h->hv_ring + ring_l;
  hc.cursor = h->hcursor;
  CK(launch_hist_combine(hc, s));
  mark(h, "hist_combine");
  return DLITE_OK;
}

int run_backbone(dlite_handle* h, int B, const void* hidden, const int32_t* anchor,
                 const dlite_taps* taps, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  const int G = group_of(&c), L = B * (G + c.K), C = B * c.m;
  const bool fused_ctx = fuse_ctx(h, B);
  StageArgs st;
  st.hidden = hidden;
  st.anchor = anchor;
  st.E = h->E_src;
  st.E_tiled = h->f32 ? 0 : 1;
  st.e_depth = h->e_depth;
  st.g_stage = h->g_stage;
  st.e_ph = h->e_ph;
  st.g_attn0 = h->layer[0].g_attn;
  st.B = B;
  st.m = c.m;
  st.K = c.K;
  st.G = G;
  st.D = c.D;
  st.V = c.V;
  st.eps = c.rms_eps;
  st.z[0] = fused_ctx ? h->y[0] + (size_t)L * c.D : h->z[0];
  st.z[1] = h->z[1];
  st.nz = h->xp;
  st.x = h->x;
  st.y[0] = h->y[0];
  st.y[1] = h->y[1];
  st.ny = h->xp;
  st.tap_z = taps ? taps->z : nullptr;
  st.status = h->status;
  CK(launch_stage(st, h->f32, s));
  mark(h, "stage");

  for (int l = 0; l < c.L_D; ++l) {
    const LayerW& w = h->layer[l];
    Splits S1, S2;
    AttnArgs at;
    if (fused_ctx) {
      RUN(gemm(h, "gemm_qkv", opnd(h->y, h->xp, h->Lcap + h->Ccap, c.D),
               opnd(w.Wqkv, h->np, h->qd + 2 * h->kvd, c.D), L + C, h->qd + 2 * h->kvd, h->part, &S1, s,
               nullptr, 1, nullptr, L, h->qd));
      at.part_ctx = h->part;
      at.sp_ctx = S1;
      at.ctx_row0 = L;
      at.ctx_col0 = h->qd;
      at.ldc = h->qd + 2 * h->kvd;
      at.ctx_rows = L + C;
      at.loc_rows = L + C;
    } else {
      // local rows: y -> [q | k | v]; context rows: z -> [k | v] with the same bytes
      RUN(gemm(h, "gemm_qkv", opnd(h->y, h->xp, h->Lcap, c.D), opnd(w.Wqkv, h->np, h->qd + 2 * h->kvd, c.D),
               L, h->qd + 2 * h->kvd, h->part, &S1, s));
      const bf16* wkv[2] = {w.Wqkv[0] + (size_t)h->qd * c.D,
                            w.Wqkv[1] ? w.Wqkv[1] + (size_t)h->qd * c.D : nullptr};
      RUN(gemm(h, "gemm_ctx_kv", opnd(h->z, h->xp, h->Ccap, c.D), opnd(wkv, h->np, 2 * h->kvd, c.D), C,
               2 * h->kvd, h->part2, &S2, s));
      at.part_ctx = h->part2;
      at.sp_ctx = S2;
    }
    at.part_loc = h->part;
    at.sp_loc = S1;
    at.rope_cos = h->rope_cos;
    at.rope_sin = h->rope_sin;
    at.B = B;
    at.m = c.m;
    at.K = c.K;
    at.K1 = G + c.K;
    at.n_q = c.n_q;
    at.n_kv = c.n_kv;
    at.d_h = c.d_h;
    at.hq = attention_heads_per_cta(c.n_q, c.n_kv, B);
    at.scale = (float)(1.0 / sqrt((double)c.d_h));
    at.round_bf16 = h->xp == 1 ? 1 : 0;
    at.o[0] = h->o[0];
    at.o[1] = h->o[1];
    at.no = h->xp;
    if (h->H) {
      at.hist_q = h->hst_q;
      at.hist_k = h->hk_ring + (size_t)l * h->hrows * c.d_h;
      at.hist_v = h->hv_ring + (size_t)l * h->hrows * c.d_h;
      at.hist_ld = h->hHx;
      at.hist_off = h->H;
    }
    CK(launch_attention(at, s));
    mark(h, "attention");
    if (h->H) RUN(run_history_attention(h, B, l, s));
    // O projection + residual, then the FFN pre-norm
    RUN(gemm(h, "gemm_o", opnd(h->o, h->xp, h->Lcap, h->qd), opnd(w.Wo, h->np, c.D, h->qd), L, c.D,
             h->part, &S1, s));
    ResNormArgs rn;
    rn.part = h->part;
    rn.sp = S1;
    rn.rows = L;
    rn.D = c.D;
    rn.x = h->x;
    rn.g = w.g_ffn;
    rn.eps = c.rms_eps;
    rn.y[0] = h->y[0];
    rn.y[1] = h->y[1];
    rn.ny = h->xp;
    CK(launch_resnorm(rn, s));
    mark(h, "resnorm");
    // gate/up + SwiGLU
    bool fused = false;
    RUN(gemm(h, "gemm_gate_up", opnd(h->y, h->xp, h->Lcap, c.D), opnd(w.Wgu, h->np, 2 * c.F, c.D), L,
             2 * c.F, h->part, &S1, s, h->a, h->xp, &fused));
    if (!fused) {
      CK(launch_swiglu_interleaved(h->part, S1, L, c.F, h->a, h->xp, s));
      mark(h, "swiglu");
    }
    // down + residual, then the next layer's pre-norm (or the final norm)
    RUN(gemm(h, "gemm_down", opnd(h->a, h->xp, h->Lcap, c.F), opnd(w.Wd, h->np, c.D, c.F), L, c.D,
             h->part, &S1, s));
    ResNormArgs r2 = rn;
    r2.sp = S1;
    r2.tap_x = (taps && taps->x) ? taps->x + (size_t)l * L * c.D : nullptr;
    if (l + 1 < c.L_D) {
      r2.g = h->layer[l + 1].g_attn;
    } else {
      r2.g = h->g_final;
      r2.final_mode = 1;
      r2.K1 = G + c.K;
      r2.G = G;
      r2.bout = h->b;
      r2.bp[0] = h->bp[0];
      r2.bp[1] = h->bp[1];
      r2.tap_b = taps ? taps->b : nullptr;
    }
    CK(launch_resnorm(r2, s));
    mark(h, "resnorm");
  }
  if (h->H) {  // the round's rows are in every layer's ring: move the cursors on
    CK(launch_hist_advance(h->hcursor, B, G + c.K, h->H, s));
    mark(h, "hist_advance");
  }
  return DLITE_OK;
}

// out32 = res + X W^T on the one-CTA engine with one k split, written as fp32
// and as two bf16 planes by the product's epilogue (no partials, no second
// kernel); DLITE_ERR_UNSUPPORTED_SHAPE when no single-split plan fits.
int gemm_residual(dlite_handle* h, const char* name, const Operand& X, const Operand& W, int rows, int outs,
                  const float* res, float* out32, bf16* const* planes, float* tap, cudaStream_t s) {
  if (outs % 16) return DLITE_ERR_UNSUPPORTED_SHAPE;
  const tc::Plan pl = tc::plan(rows, outs, X.K, X.n, W.n, false, true);
  if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
  const int xb = tc::x_box_rows(rows);
  h->maps.reserve(h->maps.size() + 4);
  const CUtensorMap* x0 = get_map(h, X.p[0], X.rows, X.K, xb);
  const CUtensorMap* x1 = X.n == 2 ? get_map(h, X.p[1], X.rows, X.K, xb) : nullptr;
  const CUtensorMap* w0 = get_map(h, W.p[0], W.rows, W.K, pl.N, true);
  const CUtensorMap* w1 = W.n == 2 ? get_map(h, W.p[1], W.rows, W.K, pl.N, true) : nullptr;
  if (!x0 || !w0 || (X.n == 2 && !x1) || (W.n == 2 && !w1)) return DLITE_ERR_CUDA;
  tc::TcParams prm;
  prm.rows = rows;
  prm.outs = outs;
  prm.K = X.K;
  prm.xplanes = X.n;
  prm.wplanes = W.n;
  prm.mode = 3;
  prm.x_box = xb;
  prm.res = res;
  prm.out32 = out32;
  prm.tap32 = tap;
  prm.act[0] = planes[0];
  prm.act[1] = planes[1];
  prm.act_planes = 2;
  prm.status = h->status;
  CK(tc::launch(pl, x0, x1, w0, w1, prm, s));
  mark(h, name);
  return DLITE_OK;
}

// b (h->b, h->bp) -> hs (h->hs, h->hp)
int run_seq_head(dlite_handle* h, int B, float* tap_hs, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  const int rows = B * c.K;
  Splits S;
  RUN(gemm(h, "gemm_head_ce", opnd(h->bp, 2, h->Hcap, c.D), opnd(h->Wce, h->np, 2 * h->Rp, c.D), rows,
           2 * h->Rp, h->part, &S, s));
  ChainArgs ch;
  ch.part = h->part;
  ch.S = S.S;  // the head products run on the one-CTA engine (uniform splits)
  ch.rows = rows;
  ch.Mt = h->Mt;
  ch.B = B;
  ch.K = c.K;
  ch.R = c.R;
  ch.t = h->t;
  ch.tp[0] = h->tp[0];
  ch.tp[1] = h->tp[1];
  ch.ldt = h->Rp;
  ch.Rp = h->Rp;
  ch.Bg = chain_group_size(c.R, B);
  CK(launch_head_chain(ch, s));
  mark(h, "head_chain");
  // few rows: h = b + t P^T straight from the product's epilogue (fp32 and the bf16
  // planes of the LM head); with more rows a single k split leaves too few CTAs
  const int rc = rows > 64 ? DLITE_ERR_UNSUPPORTED_SHAPE : gemm_residual(h, "gemm_head_p", opnd(h->tp, 2, h->Hcap, h->Rp), opnd(h->P, h->np, c.D, h->Rp),
                               rows, c.D, h->b, h->hs, h->hp, tap_hs, s);
  if (rc != DLITE_ERR_UNSUPPORTED_SHAPE) return rc;
  RUN(gemm(h, "gemm_head_p", opnd(h->tp, 2, h->Hcap, h->Rp), opnd(h->P, h->np, c.D, h->Rp), rows, c.D,
           h->part, &S, s));
  CK(launch_head_out(h->part, S.S, rows, c.D, h->b, h->hs, h->hp, tap_hs, s));
  mark(h, "head_out");
  return DLITE_OK;
}

// The vocabulary projection with the fused choice: logits = W x for `rows`
// rows of the bf16 activation x [x_cap rows, Kd] (tiled weight w [Vp, Kd]);
// records, then the merge re-scores the finalists with the fp32 vectors vec
// [rows, Kd] against the weight (bf16 tiled w, or w32 fp32 row-major) and
// writes cand / qs per row. Row r draws its noise at position
// pos[r / K_draft] + r % K_draft + 1.
struct LmOperands {
  const bf16* x;
  int x_cap, Kd;
  const bf16* w;
  const float* w32;
  const float* vec;
  int K_draft;
};

int run_lm_core(dlite_handle* h, int rows, const LmOperands& op, float temperature, uint64_t seed,
                const int64_t* pos, int32_t* cand, dlite_qstats* qs, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  const float inv_T = temperature > 0.f ? 1.f / temperature : 0.f;
  uint32_t k0 = 0, k1 = 0;
  seed_key(seed, &k0, &k1);
  int n_tiles = 0;
  const tc::LmPlan lp = tc::lm_plan_persistent(rows, c.V, op.Kd, h->num_sms);
  if (lp.ok) {  // persistent kernel, epilogue overlapped with the E stream
    h->maps.reserve(h->maps.size() + 4);
    const CUtensorMap* x0 = get_map(h, op.x, op.x_cap, op.Kd, lp.x_box0);
    const CUtensorMap* x1 = lp.paired ? get_map(h, op.x, op.x_cap, op.Kd, lp.x_box1) : nullptr;
    // a pair's CTAs each load half of every slab
    const CUtensorMap* w0 = get_map(h, op.w, h->Vp, op.Kd, lp.paired ? lp.N / 2 : lp.N, true);
    if (!x0 || !w0 || (lp.paired && !x1)) return DLITE_ERR_CUDA;
    tc::LmParams prm;
    prm.rows = rows;
    prm.outs = c.V;
    prm.rec = h->lmrec;
    prm.inv_T = inv_T;
    prm.k0 = k0;
    prm.k1 = k1;
    prm.pos = pos;
    prm.K_draft = op.K_draft;
    prm.status = h->status;
    CK(tc::launch_lm_persistent(lp, x0, x1, w0, prm, s));
    n_tiles = lp.n_units;  // one record per walk and row
  } else {  // one slab per CTA
    const tc::Plan pl = tc::plan(rows, c.V, op.Kd, 1, 1, true);
    if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
    const int xb = tc::x_box_rows(rows);
    h->maps.reserve(h->maps.size() + 4);
    const CUtensorMap* x0 = get_map(h, op.x, op.x_cap, op.Kd, xb);
    const CUtensorMap* w0 = get_map(h, op.w, h->Vp, op.Kd, pl.N, true);
    if (!x0 || !w0) return DLITE_ERR_CUDA;
    tc::TcParams prm;
    prm.rows = rows;
    prm.outs = c.V;
    prm.K = op.Kd;
    prm.xplanes = 1;
    prm.wplanes = 1;
    prm.mode = 1;
    prm.x_box = xb;
    prm.rec = h->lmrec;
    prm.inv_T = inv_T;
    prm.k0 = k0;
    prm.k1 = k1;
    prm.pos = pos;
    prm.K_draft = op.K_draft;
    prm.status = h->status;
    CK(tc::launch(pl, x0, nullptr, w0, nullptr, prm, s));
    n_tiles = (c.V + pl.N - 1) / pl.N * tc::kGemmEpiGroups;
  }
  mark(h, "lm_head");
  LmMergeArgs mg;
  mg.rec = h->lmrec;
  mg.n_tiles = n_tiles;
  mg.rows = rows;
  mg.K = op.K_draft;
  mg.D = op.Kd;
  mg.V = c.V;
  mg.inv_T = inv_T;
  mg.T = (double)temperature;
  mg.k0 = k0;
  mg.k1 = k1;
  mg.pos = pos;
  mg.h = op.vec;
  if (op.w32)
    mg.Ef = op.w32;
  else
    mg.Eb = op.w;
  mg.cand = cand;
  mg.qs = qs;
  mg.counters = h->counters;
  CK(launch_lm_merge(mg, s));
  mark(h, "lm_merge");
  return DLITE_OK;
}

int run_lm_head(dlite_handle* h, int B, float temperature, uint64_t seed, const int64_t* pos,
                int32_t* cand, dlite_qstats* qs, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  LmOperands op;
  op.x = h->hp[0];
  op.x_cap = h->Hcap;
  op.Kd = c.D;
  op.w = h->E[0];
  op.w32 = h->f32 ? (const float*)h->E_src : nullptr;
  op.vec = h->hs;
  op.K_draft = c.K;
  return run_lm_core(h, B * c.K, op, temperature, seed, pos, cand, qs, s);
}

// The gated token-feedback head after the backbone (b, h->bp): per step i the
// input [s_{i-1}; E_R[d_{i-1}]], the state product and gate, the r product,
// then the vocabulary projection over W_o with the fused choice, whose token
// the next step feeds back. r [B, K, R] stays in h->g_r (verification's q(v)).
int run_gated_head(dlite_handle* h, int B, const int32_t* anchor, float temperature, uint64_t seed,
                   const int64_t* pos, int32_t* cand, dlite_qstats* qs, float* tap_r, cudaStream_t s) {
  const dlite_config& c = h->cfg;
  const int R = c.R, K = c.K;
  Splits S;
  RUN(gemm(h, "gemm_gated_hu", opnd(h->bp, 2, h->Hcap, c.D), opnd(h->Whu, h->np, R, c.D), B * K, R, h->part,
           &S, s));
  CK(launch_gated_sum(h->part, S, B * K, R, h->g_hu, s));
  mark(h, "gated_hu");
  GatedArgs g;
  g.B = B;
  g.K = K;
  g.R = R;
  g.G = group_of(&c);
  g.V = c.V;
  g.anchor = anchor;
  g.cand_tmp = h->g_cand;
  g.qs_tmp = qs ? h->g_qs : nullptr;
  g.cand = cand;
  g.qs = qs;
  g.pos = pos;
  g.pos_i = h->g_pos;
  g.ER = h->ER32;
  g.bs = h->bs32;
  g.bh = h->bh32;
  g.hu = h->g_hu;
  g.s = h->g_s;
  g.Ws[0] = h->Ws[0];
  g.Ws[1] = h->Ws[1];
  g.Whs[0] = h->Whs[0];
  g.Whs[1] = h->Whs[1];
  g.np = h->np;
  g.r_all = h->g_r;
  g.r_step = h->g_rstep;
  g.rp = h->g_rp;
  g.status = h->status;
  LmOperands op;
  op.x = h->g_rp;
  op.x_cap = h->Bcap;
  op.Kd = R;
  op.w = h->Wo[0];
  op.w32 = h->f32 ? h->Wo32 : nullptr;
  op.vec = h->g_rstep;
  op.K_draft = 1;
  g.warm = c.head_warmup;
  if (c.head_warmup) {  // s_0: one state update from zero on the token before the anchor, no output
    CK(launch_gated_state(g, 0, false, s));
    mark(h, "gated_state");
  }
  // the step's r in the state kernel's launch when all its clusters run at
  // once (in waves they were slower than the two launches: 0.96 vs 0.90 ms
  // per round at B = 32)
  const bool fused = gated_fused(h, B);
  for (int i = 1; i <= K; ++i) {
    CK(launch_gated_state(g, i, fused, s));
    mark(h, "gated_state");
    if (!fused) {
      CK(launch_gated_r(g, i, s));
      mark(h, "gated_r");
    }
    RUN(run_lm_core(h, B, op, temperature, seed, pos ? h->g_pos : nullptr, h->g_cand, qs ? h->g_qs : nullptr, s));
  }
  CK(launch_gated_final(g, s));
  mark(h, "gated_final");
  if (tap_r) CK(cudaMemcpyAsync(tap_r, h->g_r, (size_t)B * K * R * 4, cudaMemcpyDeviceToDevice, s));
  return DLITE_OK;
}

int check_round_args(dlite_handle* h, int B, const void* hidden, const int32_t* anchor,
                     float temperature, const int64_t* pos, int32_t* cand, dlite_qstats* qs) {
  if (!h || !hidden || !anchor || !cand) return DLITE_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || isinf(temperature)) return DLITE_ERR_INVALID_ARG;
  if (temperature > 0.f && (!pos || !qs)) return DLITE_ERR_INVALID_ARG;
  return DLITE_OK;
}

}  // namespace

// ================================================================ C ABI

extern "C" {

const char* dlite_status_string(int st) {
  switch (st) {
    case DLITE_OK: return "ok";
    case DLITE_ERR_INVALID_ARG: return "invalid argument";
    case DLITE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case DLITE_ERR_CUDA: return "CUDA runtime error";
    case DLITE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case DLITE_ERR_BOUNDS: return "id out of range on the device";
    case DLITE_ERR_OOM: return "device allocation failed";
    default: return "unknown status";
  }
}

const char* dlite_last_cuda_error(void) {
  static thread_local char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s", cudaGetErrorName(g_last_cuda_error),
           cudaGetErrorString(g_last_cuda_error));
  return buf;
}

void dlite_destroy(dlite_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->prof_events_made)
    for (int i = 0; i < 128; ++i) cudaEventDestroy(h->prof_ev[i]);
  if (h->ev_in) cudaEventDestroy(h->ev_in);
  if (h->ev_cp) cudaEventDestroy(h->ev_cp);
  if (h->cstream) cudaStreamDestroy(h->cstream);
  for (void* p : h->allocs) cudaFree(p);
  delete h;
}

// Plans of the one-CTA-engine products at B = B_max, chosen by timing every
// feasible plan on the device (CUDA events; before each launch L2 is flushed
// and the activation operand rewritten, so that as in a round the weights
// stream from HBM and the activations sit in L2; best of two). Other batch sizes
// keep the analytical planner's choice. bf16 drafters only.
static int tune_products(dlite_handle* h) {
  const dlite_config& c = h->cfg;
  if (h->np != 1 || h->xp != 1) return DLITE_OK;
  const int B = c.B_max, L = B * (group_of(&c) + c.K), C = B * c.m, Hr = B * c.K;
  struct Site {
    Operand X, W;
    int rows, outs;
    bf16* const* act;
    int skip_row0, skip_cols;
  };
  std::vector<Site> sites;
  const LayerW& w = h->layer[0];
  const int qkv = h->qd + 2 * h->kvd;
  if (fuse_ctx(h, B))
    sites.push_back({opnd(h->y, 1, h->Lcap + h->Ccap, c.D), opnd(w.Wqkv, 1, qkv, c.D), L + C, qkv, nullptr, L, h->qd});
  sites.push_back({opnd(h->o, 1, h->Lcap, h->qd), opnd(w.Wo, 1, c.D, h->qd), L, c.D, nullptr, 0, 0});
  sites.push_back({opnd(h->y, 1, h->Lcap, c.D), opnd(w.Wgu, 1, 2 * c.F, c.D), L, 2 * c.F, h->a, 0, 0});
  sites.push_back({opnd(h->a, 1, h->Lcap, c.F), opnd(w.Wd, 1, c.D, c.F), L, c.D, nullptr, 0, 0});
  if (!h->gated)
    sites.push_back({opnd(h->bp, 2, h->Hcap, c.D), opnd(h->Wce, 1, 2 * h->Rp, c.D), Hr, 2 * h->Rp, nullptr, 0, 0});
  const size_t flush_bytes = (size_t)256 << 20;  // twice the L2
  void* flush = nullptr;
  if (cudaMalloc(&flush, flush_bytes) != cudaSuccess) {
    cudaGetLastError();
    return DLITE_OK;  // no room to time: the analytical plans stay
  }
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int rc = DLITE_OK;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess)
    rc = DLITE_ERR_CUDA;
  for (const Site& st : sites) {
    if (rc) break;
    const bool skipping = st.skip_row0 > 0;
    const bool pair = !skipping && tc::use_pair_engine(st.rows, st.X.n, st.W.n) &&
                      tc::pair_plan(st.rows, st.outs, st.X.K, h->num_sms).ok;
    if (pair) continue;  // the pair engine serves this product
    TunedPlan best;
    float best_ms = 1e30f, model_ms = 1e30f;
    // the analytical plan stays unless a timed one beats it clearly: one cold
    // launch per candidate is noisy, and near-equal tilings flipped from one
    // handle to the next
    const tc::Plan model = tc::plan(st.rows, st.outs, st.X.K, st.X.n, st.W.n, false, st.act != nullptr,
                                    st.skip_row0, st.skip_cols);
    for (const tc::Plan& pl : tc::plan_candidates(st.rows, st.outs, st.X.K, st.X.n, st.W.n, st.act != nullptr)) {
      if (!st.act && (size_t)pl.S * st.rows * st.outs > h->part_cap) continue;
      float t = 1e30f;
      for (int rep = 0; rep < 3 && !rc; ++rep) {
        float ms = 0.f;
        // weights from HBM, activations L2-resident (as written by the previous kernel of a round)
        bool ok = cudaMemsetAsync(flush, rep, flush_bytes, s) == cudaSuccess;
        for (int pl_i = 0; pl_i < st.X.n && ok; ++pl_i)
          ok = cudaMemsetAsync((void*)st.X.p[pl_i], 0, (size_t)st.rows * st.X.K * sizeof(bf16), s) == cudaSuccess;
        if (!ok || cudaEventRecord(e0, s) != cudaSuccess) {
          rc = DLITE_ERR_CUDA;
          break;
        }
        rc = launch_onecta(h, pl, st.X, st.W, st.rows, st.outs, h->part, s, st.act, 1, st.skip_row0, st.skip_cols);
        if (rc || cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
          rc = rc ? rc : DLITE_ERR_CUDA;
          break;
        }
        t = std::min(t, ms);
      }
      if (!rc && model.ok && pl.N == model.N && pl.S == model.S && pl.n_mt == model.n_mt && pl.groups == model.groups)
        model_ms = t;
      if (!rc && t < best_ms) {
        best_ms = t;
        best = {st.rows, st.outs, st.X.K, st.X.n, st.W.n, st.act != nullptr, st.skip_row0, st.skip_cols, pl};
      }
    }
    if (!rc && best_ms < 1e29f && best_ms < 0.97f * model_ms) h->tuned.push_back(best);
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (s) cudaStreamDestroy(s);
  cudaFree(flush);
  if (!rc) {  // a timed launch must not have tripped a bounded wait
    int st = 0;
    if (cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DLITE_ERR_CUDA;
    if (st) return DLITE_ERR_DEVICE_TIMEOUT;
  }
  return rc;
}

static int create_impl(dlite_handle* h, const dlite_weights* w) {
  const dlite_config& c = h->cfg;
  const int D = c.D, F = c.F, R = c.R, V = c.V;
  // ---- weights
  RUN(repack(h, w->e_depth, c.m, D, D, 0, nullptr, &h->e_depth));
  RUN(repack(h, w->g_stage, 1, D, D, 0, nullptr, &h->g_stage));
  RUN(repack(h, w->e_ph, 1, D, D, 0, nullptr, &h->e_ph));
  RUN(repack(h, w->g_final, 1, D, D, 0, nullptr, &h->g_final));
  {  // E planes padded to Vp rows (zero rows past V) for the LM-head tiles
    bf16* p0 = nullptr;
    bf16* p1 = nullptr;
    AL(p0, (size_t)h->Vp * D);
    CK(cudaMemset(p0, 0, (size_t)h->Vp * D * 2));
    if (h->np == 2) {
      AL(p1, (size_t)h->Vp * D);
      CK(cudaMemset(p1, 0, (size_t)h->Vp * D * 2));
    }
    float* e32 = nullptr;
    if (h->f32) AL(e32, (size_t)V * D);
    CK(launch_repack(w->E, h->f32, V, D, D, 0, p0, p1, h->np, e32, -D, 0));
    h->E[0] = p0;
    h->E[1] = p1;
    h->E_src = h->f32 ? (const void*)e32 : (const void*)p0;
  }
  for (int l = 0; l < c.L_D; ++l) {
    const dlite_layer_weights& lw = w->layer[l];
    LayerW& L = h->layer[l];
    if (!lw.g_attn || !lw.Wq || !lw.Wk || !lw.Wv || !lw.Wo || !lw.g_ffn || !lw.Wg || !lw.Wu || !lw.Wd)
      return DLITE_ERR_INVALID_ARG;
    const void* qkv[3] = {lw.Wq, lw.Wk, lw.Wv};
    const int qkv_rows[3] = {h->qd, h->kvd, h->kvd};
    RUN(stack(h, qkv, qkv_rows, 3, D, L.Wqkv));
    RUN(repack(h, lw.Wo, D, h->qd, h->qd, 0, L.Wo, nullptr));
    {
      bf16* p0 = nullptr;
      bf16* p1 = nullptr;
      AL(p0, (size_t)2 * F * D);
      if (h->np == 2) AL(p1, (size_t)2 * F * D);
      CK(launch_repack_gate_up(lw.Wg, lw.Wu, h->f32, F, D, p0, p1, h->np, 0));
      L.Wgu[0] = p0;
      L.Wgu[1] = p1;
    }
    RUN(repack(h, lw.Wd, D, F, F, 0, L.Wd, nullptr));
    RUN(repack(h, lw.g_attn, 1, D, D, 0, nullptr, &L.g_attn));
    RUN(repack(h, lw.g_ffn, 1, D, D, 0, nullptr, &L.g_ffn));
  }
  {  // Wce = [Q_b; 0; Q_h; 0] = [Q[:, :D] padded to Rp rows; Q[:, D:] padded to Rp rows], tiled
    bf16* p0 = nullptr;
    bf16* p1 = nullptr;
    const size_t n = (size_t)2 * h->Rp * D;
    AL(p0, n);
    CK(cudaMemset(p0, 0, n * 2));
    if (h->np == 2) {
      AL(p1, n);
      CK(cudaMemset(p1, 0, n * 2));
    }
    const size_t half = (size_t)h->Rp * D;  // Rp rows: a whole number of 64-row tile rows
    CK(launch_repack(w->Q, h->f32, R, D, 2 * D, 0, p0, p1, h->np, nullptr, -D, 0));
    CK(launch_repack(w->Q, h->f32, R, D, 2 * D, D, p0 + half, p1 ? p1 + half : nullptr, h->np, nullptr,
                     -D, 0));
    h->Wce[0] = p0;
    h->Wce[1] = p1;
  }
  {  // P as [D, Rp] with zero columns R..Rp (the GEMM k extent is a multiple of 64)
    bf16* p0 = nullptr;
    bf16* p1 = nullptr;
    AL(p0, (size_t)D * h->Rp);
    CK(cudaMemset(p0, 0, (size_t)D * h->Rp * 2));
    if (h->np == 2) {
      AL(p1, (size_t)D * h->Rp);
      CK(cudaMemset(p1, 0, (size_t)D * h->Rp * 2));
    }
    CK(launch_repack(w->P, h->f32, D, R, R, 0, p0, p1, h->np, nullptr, -h->Rp, 0));
    h->P[0] = p0;
    h->P[1] = p1;
  }
  if (h->gated) {  // the gated token-feedback head's weights (R is a multiple of 64)
    RUN(repack(h, w->gated.W_s, 2 * R, 2 * R, 2 * R, 0, h->Ws, nullptr));
    RUN(repack(h, w->gated.W_h, R, R, R + D, 0, h->Whs, nullptr));
    RUN(repack(h, w->gated.W_h, R, D, R + D, R, h->Whu, nullptr));
    RUN(repack(h, w->gated.E_R, V, R, R, 0, nullptr, &h->ER32));
    RUN(repack(h, w->gated.b_s, 1, 2 * R, 2 * R, 0, nullptr, &h->bs32));
    RUN(repack(h, w->gated.b_h, 1, R, R, 0, nullptr, &h->bh32));
    bf16* p0 = nullptr;
    bf16* p1 = nullptr;
    AL(p0, (size_t)h->Vp * R);
    CK(cudaMemset(p0, 0, (size_t)h->Vp * R * 2));
    if (h->np == 2) {
      AL(p1, (size_t)h->Vp * R);
      CK(cudaMemset(p1, 0, (size_t)h->Vp * R * 2));
    }
    if (h->f32) AL(h->Wo32, (size_t)V * R);
    CK(launch_repack(w->gated.W_o, h->f32, V, R, R, 0, p0, p1, h->np, h->Wo32, -R, 0));
    h->Wo[0] = p0;
    h->Wo[1] = p1;
  }
  AL(h->Mt, (size_t)R * R);
  CK(launch_head_matrix(w->Q, w->P, h->f32, D, R, h->Mt, 0));
  {  // RoPE table for local positions 0..G+K-1 (float64 on the host)
    const int half = c.d_h / 2, npos = group_of(&c) + c.K;
    std::vector<float> cs((size_t)npos * half), sn((size_t)npos * half);
    for (int p = 0; p < npos; ++p)
      for (int j = 0; j < half; ++j) {
        const double ang = p * pow((double)c.rope_theta, -2.0 * j / c.d_h);
        cs[(size_t)p * half + j] = (float)cos(ang);
        sn[(size_t)p * half + j] = (float)sin(ang);
      }
    AL(h->rope_cos, cs.size());
    AL(h->rope_sin, sn.size());
    CK(cudaMemcpy(h->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(h->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
  }
  // ---- workspace (sized for B_max; GEMM A operands padded to 128-row multiples)
  const int Bm = c.B_max;
  const size_t Lr = (size_t)h->Lcap, Cr = (size_t)h->Ccap, Hr = (size_t)h->Hcap;
  AL(h->x, Lr * D);
  for (int p = 0; p < h->xp; ++p) {
    AL(h->y[p], (Lr + Cr) * D);  // context rows behind the local rows when fused (fuse_ctx)
    AL(h->z[p], Cr * D);
    AL(h->o[p], Lr * h->qd);
    AL(h->a[p], Lr * F);
  }
  AL(h->b, Hr * D);
  AL(h->t, Hr * R);
  AL(h->hs, Hr * D);
  for (int p = 0; p < 2; ++p) {
    AL(h->bp[p], Hr * D);
    AL(h->tp[p], Hr * h->Rp);
    CK(cudaMemset(h->tp[p], 0, Hr * h->Rp * 2));
    AL(h->hp[p], Hr * D);
  }
  size_t pe = 0, pe2 = 0, lme = 0;
  for (int B = 1; B <= Bm; ++B) {
    const int L = B * (group_of(&c) + c.K), C = B * c.m, H = B * c.K;
    const int sites[7][4] = {{L, h->qd + 2 * h->kvd, D, h->xp}, {L, D, h->qd, h->xp},
                             {L, 2 * F, D, h->xp},               {L, D, F, h->xp},
                             {H, 2 * h->Rp, D, 2},               {H, D, h->Rp, 2},
                             {H, h->Rp, D, 2}};  // the gated head's W_h u product (sized whatever the head type)
    for (auto& st : sites) {
      const tc::Plan pl = tc::plan(st[0], st[1], st[2], st[3], h->np, false);
      if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
      const size_t v = (size_t)pl.S * st[0] * st[1];
      pe = v > pe ? v : pe;
      const tc::PairPlan pp = tc::pair_plan(st[0], st[1], st[2], h->num_sms);
      if (pp.ok && tc::use_pair_engine(st[0], st[3], h->np)) pe = (size_t)pp.S * st[0] * st[1] > pe ? (size_t)pp.S * st[0] * st[1] : pe;  // planes
    }
    if (fuse_ctx(h, B)) {
      const tc::Plan pf = tc::plan(L + C, h->qd + 2 * h->kvd, D, 1, 1, false, false, L, h->qd);
      pe = std::max(pe, (size_t)pf.S * (L + C) * (h->qd + 2 * h->kvd));
    }
    const tc::Plan pc = tc::plan(C, 2 * h->kvd, D, h->xp, h->np, false);
    if (!pc.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
    const size_t v2 = (size_t)pc.S * C * 2 * h->kvd;
    pe2 = v2 > pe2 ? v2 : pe2;
    const tc::PairPlan pc2 = tc::pair_plan(C, 2 * h->kvd, D, h->num_sms);
    if (pc2.ok && tc::use_pair_engine(C, h->xp, h->np)) pe2 = (size_t)pc2.S * C * 2 * h->kvd > pe2 ? (size_t)pc2.S * C * 2 * h->kvd : pe2;
    const tc::Plan pl = lm_plan(h, H);
    if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
    const size_t v3 = (size_t)((V + pl.N - 1) / pl.N) * tc::kGemmEpiGroups * H;
    lme = v3 > lme ? v3 : lme;
    const tc::LmPlan lp = tc::lm_plan_persistent(H, V, D, h->num_sms);
    if (lp.ok) {
      const size_t v4 = (size_t)lp.n_units * H;
      lme = v4 > lme ? v4 : lme;
    }
  }
  {  // the timed plan selection at B_max may pick up to 4 splits for the layer products
    const int L = Bm * (group_of(&c) + c.K), C = Bm * c.m;
    pe = std::max(pe, (size_t)4 * L * std::max(h->qd + 2 * h->kvd, D));
    if (fuse_ctx(h, Bm)) pe = std::max(pe, (size_t)4 * (L + C) * (h->qd + 2 * h->kvd));
  }
  AL(h->part, pe);
  h->part_cap = pe;
  AL(h->part2, pe2);
  AL(h->lmrec, lme);
  AL(h->resid, (size_t)Bm * V);
  AL(h->tsamp, (size_t)Bm * (c.K + 1));
  if (h->gated) {
    const size_t Bc = (size_t)h->Bcap;
    AL(h->g_s, (size_t)2 * Bm * R);
    AL(h->g_hu, (size_t)Bm * c.K * R);
    AL(h->g_r, (size_t)Bm * c.K * R);
    AL(h->g_rstep, (size_t)Bm * R);
    AL(h->g_rp, Bc * R);
    CK(cudaMemset(h->g_rp, 0, Bc * R * 2));
    AL(h->g_cand, (size_t)Bm);
    AL(h->g_qs, (size_t)Bm);
    AL(h->g_pos, (size_t)Bm);
  }
  AL(h->counters, 8);
  CK(cudaMemset(h->counters, 0, 8 * sizeof(unsigned long long)));
  AL(h->status, 1);
  CK(cudaMemset(h->status, 0, sizeof(int)));
  for (int i = 0; i < 128; ++i) CK(cudaEventCreate(&h->prof_ev[i]));
  h->prof_events_made = true;
  // ---- staging for dlite_round_host
  {
    void* q = nullptr;
    if (cudaMalloc(&q, (size_t)Bm * c.m * D * (h->f32 ? 4 : 2)) != cudaSuccess) return DLITE_ERR_OOM;
    h->allocs.push_back(q);
    h->d_hidden = q;
  }
  AL(h->d_anchor, (size_t)Bm * group_of(&c));
  AL(h->d_pos, Bm);
  AL(h->d_tgt, (size_t)Bm * (c.K + 1));
  AL(h->d_probs, (size_t)Bm * (c.K + 1) * V);
  AL(h->d_cand, Hr);
  AL(h->d_qs, Hr);
  AL(h->d_acc, Bm);
  AL(h->d_commits, (size_t)Bm * (c.K + 1));
  AL(h->d_ncommit, Bm);
  AL(h->d_next, Bm);
  CK(cudaStreamCreateWithFlags(&h->cstream, cudaStreamNonBlocking));
  CK(cudaEventCreateWithFlags(&h->ev_in, cudaEventDisableTiming));
  CK(cudaEventCreateWithFlags(&h->ev_cp, cudaEventDisableTiming));
  if (c.history > 0) {  // the conventional drafter's draft KV and the history kernels' buffers
    const int K1 = group_of(&c) + c.K;
    h->H = c.history;
    h->hQR = (c.n_q / c.n_kv) * K1;
    h->hTk = c.m + K1;
    h->hHx = h->H + h->hTk;
    h->hrows = std::max<size_t>((size_t)Bm * c.n_kv * h->hHx, 64);
    const size_t ring = (size_t)c.L_D * h->hrows * c.d_h;
    AL(h->hk_ring, ring);
    AL(h->hv_ring, ring);
    for (int l = 0; l < c.L_D; ++l)
      if (!tc::make_map(&h->hmap_k[l], h->hk_ring + (size_t)l * h->hrows * c.d_h, (int)h->hrows, c.d_h, 64) ||
          !tc::make_map(&h->hmap_v[l], h->hv_ring + (size_t)l * h->hrows * c.d_h, (int)h->hrows, c.d_h, 64))
        return DLITE_ERR_CUDA;
    AL(h->hcursor, Bm);
    AL(h->hst_q, (size_t)Bm * c.n_kv * h->hQR * c.d_h);
    const size_t prow =
        (size_t)(hist_max_ctas(h->num_sms) + (long long)Bm * c.n_kv) * hist_key_splits(h->hQR) * h->hQR;
    AL(h->hpart_o, prow * c.d_h);
    AL(h->hpart_ml, prow * 2);
    RUN(dlite_history_reset(h, nullptr));
  }
  if (h->gated) {  // the fused step needs a co-resident cluster of R / 32 CTAs
    GatedArgs ga;
    ga.B = c.B_max;
    ga.R = c.R;
    ga.np = h->np;
    h->gated_clusters = gated_step_clusters(ga);
  }
  CK(cudaDeviceSynchronize());
  RUN(tune_products(h));
  CK(cudaDeviceSynchronize());
  return DLITE_OK;
}

int dlite_create(const dlite_config* cfg, const dlite_weights* w, dlite_handle** out) {
  if (!out || !w) return DLITE_ERR_INVALID_ARG;
  *out = nullptr;
  const int rc = check_config(cfg);
  if (rc) return rc;
  if (cfg->head_type == DLITE_HEAD_GATED &&
      (!w->gated.E_R || !w->gated.W_s || !w->gated.b_s || !w->gated.W_h || !w->gated.b_h || !w->gated.W_o))
    return DLITE_ERR_INVALID_ARG;
  if (!w->e_depth || !w->g_stage || !w->e_ph || !w->E || !w->g_final || !w->Q || !w->P)
    return DLITE_ERR_INVALID_ARG;
  dlite_handle* h = new dlite_handle();
  h->cfg = *cfg;
  h->f32 = cfg->dtype == DLITE_F32;
  h->np = h->f32 ? 2 : 1;
  h->xp = (h->f32 || cfg->act_planes == 2) ? 2 : 1;
  h->qd = cfg->n_q * cfg->d_h;
  h->kvd = cfg->n_kv * cfg->d_h;
  h->Rp = (cfg->R + 63) / 64 * 64;
  h->Vp = (cfg->V + 63) / 64 * 64;
  h->Lcap = (cfg->B_max * (group_of(cfg) + cfg->K) + 127) / 128 * 128;
  h->Ccap = (cfg->B_max * cfg->m + 127) / 128 * 128;
  h->Hcap = (cfg->B_max * cfg->K + 127) / 128 * 128;
  h->Bcap = (cfg->B_max + 127) / 128 * 128;
  h->gated = cfg->head_type == DLITE_HEAD_GATED;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        h->num_sms < 1) {
      delete h;
      return DLITE_ERR_CUDA;
    }
  }
  const int r = create_impl(h, w);
  if (r) {
    dlite_destroy(h);
    return r;
  }
  *out = h;
  return DLITE_OK;
}

int dlite_draft_round_taps(dlite_handle* h, int B, const void* hidden, const int32_t* anchor,
                           float temperature, uint64_t seed, const int64_t* pos, int32_t* cand,
                           dlite_qstats* qs, const dlite_taps* taps, dlite_stream_t stream) {
  RUN(check_round_args(h, B, hidden, anchor, temperature, pos, cand, qs));
  cudaStream_t s = (cudaStream_t)stream;
  RUN(run_backbone(h, B, hidden, anchor, taps, s));
  if (h->gated)  // the head's vectors (r) go to the hs tap
    return run_gated_head(h, B, anchor, temperature, seed, pos, cand, qs, taps ? taps->hs : nullptr, s);
  RUN(run_seq_head(h, B, taps ? taps->hs : nullptr, s));
  RUN(run_lm_head(h, B, temperature, seed, pos, cand, qs, s));
  return DLITE_OK;
}

int dlite_draft_round(dlite_handle* h, int B, const void* hidden, const int32_t* anchor,
                      float temperature, uint64_t seed, const int64_t* pos, int32_t* cand,
                      dlite_qstats* qs, dlite_stream_t stream) {
  return dlite_draft_round_taps(h, B, hidden, anchor, temperature, seed, pos, cand, qs, nullptr,
                                stream);
}

int dlite_backbone(dlite_handle* h, int B, const void* hidden, const int32_t* anchor, float* b,
                   dlite_stream_t stream) {
  if (!h || !hidden || !anchor || !b || B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  dlite_taps taps = {nullptr, nullptr, b, nullptr};
  return run_backbone(h, B, hidden, anchor, &taps, (cudaStream_t)stream);
}

int dlite_seq_head(dlite_handle* h, int B, const float* b, float* hs, dlite_stream_t stream) {
  if (!h || !b || !hs || B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  if (h->gated) return DLITE_ERR_UNSUPPORTED_SHAPE;  // the gated head runs inside dlite_draft_round
  cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)B * h->cfg.K * h->cfg.D;
  CK(launch_split(b, n, h->bp, h->b, s));
  return run_seq_head(h, B, hs, s);
}

int dlite_lm_head(dlite_handle* h, int B, const float* hs, float temperature, uint64_t seed,
                  const int64_t* pos, int32_t* cand, dlite_qstats* qs, dlite_stream_t stream) {
  if (!h || !hs || !cand || B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  if (h->gated) return DLITE_ERR_UNSUPPORTED_SHAPE;  // the gated head runs inside dlite_draft_round
  if (!(temperature >= 0.f) || isinf(temperature)) return DLITE_ERR_INVALID_ARG;
  if (temperature > 0.f && (!pos || !qs)) return DLITE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)B * h->cfg.K * h->cfg.D;
  CK(launch_split(hs, n, h->hp, h->hs, s));
  return run_lm_head(h, B, temperature, seed, pos, cand, qs, s);
}

// Where verification recomputes q(v) = exp(w_v . x_i / T - lse_i): the tied E and
// the head outputs h_i (D wide), or, for the gated head, W_o and r_i (R wide).
void set_q_source(dlite_handle* h, VerifyArgs* v, const float* vec) {
  if (h->gated) {
    v->D = h->cfg.R;
    v->hs = vec ? vec : h->g_r;
    if (h->f32)
      v->Ef = h->Wo32;
    else
      v->Eb = h->Wo[0];
    return;
  }
  v->D = h->cfg.D;
  v->hs = vec ? vec : h->hs;
  if (h->f32)
    v->Ef = (const float*)h->E_src;
  else
    v->Eb = h->E[0];
}

int dlite_verify(dlite_handle* h, int B, const int32_t* cand, const int32_t* tgt, int32_t* accepted,
                 int32_t* commits, int32_t* n_commit, int32_t* next_anchor, dlite_stream_t stream) {
  if (!h || !cand || !tgt || !accepted || !commits || !n_commit || !next_anchor)
    return DLITE_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  VerifyArgs v;
  v.B = B;
  v.K = h->cfg.K;
  v.V = h->cfg.V;
  v.cand = cand;
  v.tgt = tgt;
  v.accepted = accepted;
  v.commits = commits;
  v.n_commit = n_commit;
  v.next_anchor = next_anchor;
  v.status = h->status;
  CK(launch_verify_greedy(v, (cudaStream_t)stream));
  mark(h, "verify_greedy");
  return DLITE_OK;
}

int dlite_verify_sample(dlite_handle* h, int B, const int32_t* cand, const dlite_qstats* qs,
                        const float* hs, const float* probs, float temperature, uint64_t seed,
                        const int64_t* pos, int32_t* accepted, int32_t* commits, int32_t* n_commit,
                        int32_t* next_anchor, dlite_stream_t stream) {
  if (!h || !cand || !qs || !probs || !pos || !accepted || !commits || !n_commit || !next_anchor)
    return DLITE_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || isinf(temperature)) return DLITE_ERR_INVALID_ARG;
  VerifyArgs v;
  v.B = B;
  v.K = h->cfg.K;
  v.V = h->cfg.V;
  v.D = h->cfg.D;
  v.cand = cand;
  v.qs = qs;
  v.probs = probs;
  set_q_source(h, &v, hs);
  v.resid = h->resid;
  v.counters = h->counters;
  v.T = (double)temperature;
  seed_key(seed, &v.k0, &v.k1);
  v.pos = pos;
  v.accepted = accepted;
  v.commits = commits;
  v.n_commit = n_commit;
  v.next_anchor = next_anchor;
  v.status = h->status;
  CK(launch_verify_sample(v, (cudaStream_t)stream));
  mark(h, "verify_sample");
  return DLITE_OK;
}

int dlite_verify_ex(dlite_handle* h, const dlite_verify_args* a, dlite_stream_t stream) {
  if (!h || !a) return DLITE_ERR_INVALID_ARG;
  const dlite_config& c = h->cfg;
  if (a->B < 1 || a->B > c.B_max || a->n_verify < 0 || a->n_verify > c.K) return DLITE_ERR_INVALID_ARG;
  if (!a->candidates || !a->accepted || !a->commits || !a->n_commit || !a->next_anchor)
    return DLITE_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  VerifyArgs v;
  v.B = a->B;
  v.K = c.K;
  v.V = c.V;
  v.D = c.D;
  v.kv = a->n_verify;
  v.cand = a->candidates;
  v.accepted = a->accepted;
  v.commits = a->commits;
  v.n_commit = a->n_commit;
  v.next_anchor = a->next_anchor;
  v.status = h->status;
  switch (a->mode) {
    case DLITE_VERIFY_GREEDY:
      if (!a->target_tokens) return DLITE_ERR_INVALID_ARG;
      v.tgt = a->target_tokens;
      CK(launch_verify_greedy(v, s));
      mark(h, "verify_greedy");
      return DLITE_OK;
    case DLITE_VERIFY_SAMPLE:
      if (!a->qstats || !a->target_probs || !a->pos) return DLITE_ERR_INVALID_ARG;
      if (!(a->temperature > 0.f) || isinf(a->temperature)) return DLITE_ERR_INVALID_ARG;
      v.qs = a->qstats;
      v.probs = a->target_probs;
      set_q_source(h, &v, a->hs);
      v.resid = h->resid;
      v.counters = h->counters;
      v.T = (double)a->temperature;
      seed_key(a->seed, &v.k0, &v.k1);
      v.pos = a->pos;
      CK(launch_verify_sample(v, s));
      mark(h, "verify_sample");
      return DLITE_OK;
    case DLITE_VERIFY_MATCH:
      if (!a->target_probs || !a->pos) return DLITE_ERR_INVALID_ARG;
      v.probs = a->target_probs;
      seed_key(a->seed, &v.k0, &v.k1);
      v.pos = a->pos;
      v.tsamp = h->tsamp;
      CK(launch_match_sample(v, s));
      mark(h, "match_sample");
      v.tgt = h->tsamp;  // then greedy verification against the target's samples
      CK(launch_verify_greedy(v, s));
      mark(h, "verify_match");
      return DLITE_OK;
    default:
      return DLITE_ERR_INVALID_ARG;
  }
}

int dlite_shift_group(dlite_handle* h, int B, const int32_t* commits, const int32_t* n_commit,
                      int32_t* group, dlite_stream_t stream) {
  if (!h || !commits || !n_commit || !group || B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  CK(launch_shift_group(B, group_of(&h->cfg), h->cfg.K + 1, commits, n_commit, group, (cudaStream_t)stream));
  return DLITE_OK;
}

int dlite_advance(dlite_handle* h, int B, const int32_t* n_commit, int64_t* pos,
                  dlite_stream_t stream) {
  if (!h || !n_commit || !pos || B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  CK(launch_advance(B, n_commit, pos, (cudaStream_t)stream));
  return DLITE_OK;
}

int dlite_round_host(dlite_handle* h, int B, const void* hidden_host, const int32_t* anchor_host,
                     const int64_t* pos_host, const int32_t* tgt_host, const float* probs_host,
                     float temperature, uint64_t seed, int32_t* accepted_host, int32_t* commits_host,
                     int32_t* n_commit_host, int32_t* next_anchor_host, dlite_stream_t stream) {
  if (!h || !hidden_host || !anchor_host || !accepted_host || !commits_host || !n_commit_host ||
      !next_anchor_host)
    return DLITE_ERR_INVALID_ARG;
  if (B < 1 || B > h->cfg.B_max) return DLITE_ERR_INVALID_ARG;
  const bool sampling = temperature > 0.f;
  if (sampling ? (!probs_host || !pos_host) : !tgt_host) return DLITE_ERR_INVALID_ARG;
  const dlite_config& c = h->cfg;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t hb = (size_t)B * c.m * c.D * (h->f32 ? 4 : 2);
  // the target rows (155 MB of probabilities at B = 32, V = 151936) are only
  // read by the verification: they cross on the handle's copy stream while the
  // draft runs, after whatever `stream` had queued (an earlier verification
  // may still read the staging buffer)
  // Pinned, device-mapped probabilities are not copied at all: the
  // verification reads the entries and rows it uses in place (over the
  // CPU-GPU link), a few percent of the tensor.
  const float* probs_dev = h->d_probs;
  if (sampling) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, probs_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer)
      probs_dev = (const float*)pa.devicePointer;
    else
      cudaGetLastError();  // not a CUDA allocation: copied below
  }
  CK(cudaEventRecord(h->ev_in, s));
  CK(cudaStreamWaitEvent(h->cstream, h->ev_in, 0));
  if (sampling && probs_dev == h->d_probs)
    CK(cudaMemcpyAsync(h->d_probs, probs_host, (size_t)B * (c.K + 1) * c.V * 4,
                       cudaMemcpyHostToDevice, h->cstream));
  else if (!sampling)
    CK(cudaMemcpyAsync(h->d_tgt, tgt_host, (size_t)B * (c.K + 1) * 4, cudaMemcpyHostToDevice, h->cstream));
  CK(cudaEventRecord(h->ev_cp, h->cstream));
  CK(cudaMemcpyAsync(h->d_hidden, hidden_host, hb, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(h->d_anchor, anchor_host, (size_t)B * group_of(&c) * 4, cudaMemcpyHostToDevice, s));
  if (pos_host) CK(cudaMemcpyAsync(h->d_pos, pos_host, (size_t)B * 8, cudaMemcpyHostToDevice, s));
  RUN(dlite_draft_round(h, B, h->d_hidden, h->d_anchor, temperature, seed,
                        pos_host ? h->d_pos : nullptr, h->d_cand, h->d_qs, stream));
  CK(cudaStreamWaitEvent(s, h->ev_cp, 0));
  if (sampling)
    RUN(dlite_verify_sample(h, B, h->d_cand, h->d_qs, nullptr, probs_dev, temperature, seed,
                            h->d_pos, h->d_acc, h->d_commits, h->d_ncommit, h->d_next, stream));
  else
    RUN(dlite_verify(h, B, h->d_cand, h->d_tgt, h->d_acc, h->d_commits, h->d_ncommit, h->d_next,
                     stream));
  CK(cudaMemcpyAsync(accepted_host, h->d_acc, (size_t)B * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(commits_host, h->d_commits, (size_t)B * (c.K + 1) * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(n_commit_host, h->d_ncommit, (size_t)B * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(next_anchor_host, h->d_next, (size_t)B * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  return DLITE_OK;
}

int dlite_device_status(dlite_handle* h, int clear, int* status_out, dlite_stream_t stream) {
  if (!h || !status_out) return DLITE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  CK(cudaMemcpyAsync(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost, s));
  if (clear) CK(cudaMemsetAsync(h->status, 0, sizeof(int), s));
  CK(cudaStreamSynchronize(s));
  *status_out = v;
  if (v & DLITE_DEV_TIMEOUT) return DLITE_ERR_DEVICE_TIMEOUT;
  if (v & DLITE_DEV_BOUNDS) return DLITE_ERR_BOUNDS;
  return DLITE_OK;
}

int dlite_stage_times(dlite_handle* h, int B, const void* hidden, const int32_t* anchor,
                      float temperature, uint64_t seed, const int64_t* pos,
                      const int32_t* target_tokens, const float* target_probs, int32_t* cand,
                      dlite_qstats* qs, int32_t* accepted, int32_t* commits, int32_t* n_commit,
                      int32_t* next_anchor, float* times_ms, const char** names, int cap,
                      dlite_stream_t stream) {
  RUN(check_round_args(h, B, hidden, anchor, temperature, pos, cand, qs));
  if (!times_ms || cap < 1) return DLITE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  h->prof_stream = s;
  h->prof_n = 0;
  CK(cudaEventRecord(h->prof_ev[0], s));
  int rc = dlite_draft_round(h, B, hidden, anchor, temperature, seed, pos, cand, qs, stream);
  if (!rc && temperature > 0.f && target_probs)
    rc = dlite_verify_sample(h, B, cand, qs, nullptr, target_probs, temperature, seed, pos,
                             accepted, commits, n_commit, next_anchor, stream);
  else if (!rc && temperature == 0.f && target_tokens)
    rc = dlite_verify(h, B, cand, target_tokens, accepted, commits, n_commit, next_anchor, stream);
  const int n = h->prof_n;
  h->prof_n = -1;
  if (rc) return rc;
  CK(cudaStreamSynchronize(s));
  for (int i = 0; i < n && i < cap; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, h->prof_ev[i], h->prof_ev[i + 1]));
    times_ms[i] = ms;
    if (names) names[i] = h->prof_name[i];
  }
  return n;
}

int dlite_selftest_gemm(int rows, int outs, int K, int xplanes, int wplanes, const void* X0,
                        const void* X1, int x_rows, const void* W0, const void* W1, float* part,
                        int* status, const int* plan_override, dlite_stream_t stream) {
  if (rows < 1 || outs < 8 || outs % 8 || K < 64 || K % 64 || xplanes < 1 || xplanes > 2 ||
      wplanes < 1 || wplanes > 2 || !X0 || !W0 || !part || x_rows < rows || x_rows % 128)
    return DLITE_ERR_INVALID_ARG;
  if ((xplanes == 2 && !X1) || (wplanes == 2 && !W1)) return DLITE_ERR_INVALID_ARG;
  if (xplanes == 1 && wplanes == 2) return DLITE_ERR_INVALID_ARG;  // plane products x0w0 (+x1w0) (+x0w1)
  const int wrows = (outs + 63) / 64 * 64;
  if (!plan_override && tc::use_pair_engine(rows, xplanes, wplanes)) {  // the round's route
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DLITE_ERR_CUDA;
    const tc::PairPlan pp = tc::pair_plan(rows, outs, K, sms);
    if (pp.ok && pp.S <= 16) {  // `part` holds 16 planes
      CUtensorMap mx, mw;
      if (!tc::make_map(&mx, X0, x_rows, K, 128) || !tc::make_map_tiled(&mw, W0, wrows, K, 128))
        return DLITE_ERR_CUDA;
      tc::PairParams prm;
      prm.rows = rows;
      prm.outs = outs;
      prm.part = part;
      prm.status = status;
      CK(tc::launch_pair(pp, &mx, &mw, prm, (cudaStream_t)stream));
      return pp.S;
    }
  }
  tc::Plan pl = tc::plan(rows, outs, K, xplanes, wplanes, false);
  if (!pl.ok) return DLITE_ERR_UNSUPPORTED_SHAPE;
  if (plan_override) {  // {N, S, stages}; 0 keeps the planner's choice
    if (plan_override[0]) pl.N = plan_override[0];
    if (plan_override[1]) {
      pl.S = plan_override[1];
      pl.kb_per_split = (pl.kblocks + pl.S - 1) / pl.S;
      pl.S = (pl.kblocks + pl.kb_per_split - 1) / pl.kb_per_split;
    }
    pl.stage_bytes = (uint32_t)wplanes * pl.N * 128 + (uint32_t)pl.n_mt * xplanes * tc::a_slot_bytes(tc::x_box_rows(rows));
    pl.tail_pad = tc::x_box_rows(rows) < 128 ? (uint32_t)tc::kTailPad : 0u;
    int stmax = (int)((tc::kSmemBudget - 2048 - pl.tail_pad) / pl.stage_bytes);
    pl.stages = plan_override[2] ? plan_override[2] : (stmax > 8 ? 8 : stmax);
    int cols = 32;
    while (cols < pl.N * pl.n_mt) cols <<= 1;
    pl.tmem_cols = cols;
    if (pl.N < 64 || pl.N > 256 || pl.N % 64 || pl.N > (outs + 63) / 64 * 64 || pl.N * pl.n_mt > 512 ||
        pl.stages < 2 ||
        pl.stages > stmax || pl.S > 16)
      return DLITE_ERR_INVALID_ARG;
  }
  CUtensorMap mx0, mx1, mw0, mw1;
  const int xb = tc::x_box_rows(rows);
  if (!tc::make_map(&mx0, X0, x_rows, K, xb) || !tc::make_map_tiled(&mw0, W0, wrows, K, pl.N))
    return DLITE_ERR_CUDA;
  if (xplanes == 2 && !tc::make_map(&mx1, X1, x_rows, K, xb)) return DLITE_ERR_CUDA;
  if (wplanes == 2 && !tc::make_map_tiled(&mw1, W1, wrows, K, pl.N)) return DLITE_ERR_CUDA;
  tc::TcParams prm;
  prm.rows = rows;
  prm.outs = outs;
  prm.K = K;
  prm.xplanes = xplanes;
  prm.wplanes = wplanes;
  prm.x_box = xb;
  prm.part = part;
  prm.status = status;
  CUtensorMap mo;
  if (!tc::make_out_map(&mo, part, pl.S, rows, outs)) return DLITE_ERR_CUDA;
  CK(tc::launch(pl, &mx0, xplanes == 2 ? &mx1 : nullptr, &mw0, wplanes == 2 ? &mw1 : nullptr, prm,
                (cudaStream_t)stream, &mo));
  return pl.S;
}

int dlite_counters(dlite_handle* h, int reset, int64_t* out, dlite_stream_t stream) {
  if (!h || !out) return DLITE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaMemcpyAsync(out, h->counters, 5 * sizeof(int64_t), cudaMemcpyDeviceToHost, s));
  if (reset) CK(cudaMemsetAsync(h->counters, 0, 8 * sizeof(int64_t), s));
  CK(cudaStreamSynchronize(s));
  return DLITE_OK;
}

int dlite_history_reset(dlite_handle* h, dlite_stream_t stream) {
  if (!h || !h->H) return DLITE_ERR_INVALID_ARG;
  HistFillArgs f;
  f.k = h->hk_ring;
  f.v = h->hv_ring;
  f.cursor = h->hcursor;
  f.L = h->cfg.L_D;
  f.Bm = h->cfg.B_max;
  f.n_kv = h->cfg.n_kv;
  f.H = h->H;
  f.Hx = h->hHx;
  f.rows = h->hrows;
  f.d_h = h->cfg.d_h;
  CK(launch_hist_fill(f, (cudaStream_t)stream));
  return DLITE_OK;
}

int dlite_history_read(dlite_handle* h, int layer, int request, int which, void* dst, int32_t* cursor,
                       dlite_stream_t stream) {
  if (!h || !h->H || !dst || layer < 0 || layer >= h->cfg.L_D || request < 0 || request >= h->cfg.B_max ||
      (which != 0 && which != 1))
    return DLITE_ERR_INVALID_ARG;
  const dlite_config& c = h->cfg;
  const size_t row = (size_t)c.d_h * sizeof(bf16);
  const bf16* src = (which ? h->hv_ring : h->hk_ring) + (size_t)layer * h->hrows * c.d_h +
                    (size_t)request * c.n_kv * h->hHx * c.d_h;
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaMemcpy2DAsync(dst, h->H * row, src, h->hHx * row, h->H * row, c.n_kv, cudaMemcpyDeviceToDevice, s));
  if (cursor) {
    CK(cudaMemcpyAsync(cursor, h->hcursor + request, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
  }
  return DLITE_OK;
}

int dlite_selftest_wait(dlite_handle* h, uint64_t limit_ns, int32_t* result, dlite_stream_t stream) {
  if (!h || !result || limit_ns < 1 || limit_ns > 1000000000ull) return DLITE_ERR_INVALID_ARG;
  CK(launch_wait_probe(limit_ns, h->status, result, (cudaStream_t)stream));
  return DLITE_OK;
}

int dlite_launch_count(dlite_handle* h, int B, float temperature) {
  if (!h || B < 1) return -1;
  (void)temperature;
  // stage + per layer {qkv, ctx-kv, attention, o, resnorm, gate/up (+ swiglu on the pair
  // engine; the one-CTA engine fuses it), down, resnorm} + head {ce, chain, P, out}
  // + lm {head, merge} + verify
  const int L = B * (group_of(&h->cfg) + h->cfg.K);
  const bool fused = !tc::use_pair_engine(L, h->xp, h->np);
  const int per_layer = (fused ? 8 : 9) - (fuse_ctx(h, B) ? 1 : 0);  // one product for [y; z] when fused
  // history-KV control: + {history attention, combine} per layer + the cursor advance
  const int hist = h->H ? 2 * h->cfg.L_D + 1 : 0;
  if (h->gated)  // head: {W_h u product, sum} + K x {state (+ r), lm, merge} + final (+ the warm-up's state)
    return 1 + per_layer * h->cfg.L_D + hist + 2 + (gated_fused(h, B) ? 3 : 4) * h->cfg.K + 1 +
           (h->cfg.head_warmup ? 1 : 0);
  // head {ce, chain, P + residual} (+ out when no single-split plan fits the P product)
  const int head = B * h->cfg.K <= 64 && tc::plan(B * h->cfg.K, h->cfg.D, h->Rp, 2, h->np, false, true).ok &&
                   h->cfg.D % 16 == 0 ? 3 : 4;
  return 1 + per_layer * h->cfg.L_D + hist + head + 2 + 1;
}

}  // extern "C"
