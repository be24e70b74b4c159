// tcgen05 GEMM engine: plan, tensor maps and launch.
#pragma once

#include <cuda.h>

#include <vector>

#include "internal.h"

namespace dlite {
namespace tc {

constexpr int kEpiGroups = 2;                    // epilogue warp groups (each 4 warps)
constexpr int kThreads = 64 + 128 * kEpiGroups;  // TMA warp, MMA warp, epilogue warps
// the one-CTA engine: four epilogue groups (its epilogue is on the critical path)
constexpr int kGemmEpiGroups = 4;
constexpr int kGemmThreads = 64 + 128 * kGemmEpiGroups;
constexpr size_t kSmemBudget = 226 * 1024;  // dynamic shared memory per CTA (all of it)
constexpr size_t kTailPad = 16 * 1024;      // overhang room for a 128-row operand read of a short slot

struct Plan {
  bool ok = false;
  int N = 0;             // weight rows (output features) per CTA slab
  int S = 1;             // K splits
  int kb_per_split = 0;  // 64-wide k blocks per split
  int kblocks = 0;
  int n_mt = 1;          // 128-row M-tiles per CTA
  int groups = 1;        // row groups (grid.z)
  int stages = 2;
  uint32_t stage_bytes = 0;
  int tmem_cols = 32;
  uint32_t tail_pad = 0;  // behind the last stage when the activation slots hold < 128 rows
};

struct TcParams {
  int rows = 0, outs = 0, K = 0;
  int n_mt = 1, xplanes = 1, wplanes = 1, N = 0, kb_per_split = 0, kblocks = 0, stages = 0;
  uint32_t stage_bytes = 0, tmem_cols = 32;
  int x_box = 128;         // rows of each activation tile load (<= 128, multiple of 8)
  int mode = 0;            // 0: fp32 partials [split][rows][outs]; 1: LM-head records;
                           // 2: SwiGLU of gate / up columns interleaved in blocks of 32 (one split);
                           // 3: out32 = res + product as fp32 and as two bf16 planes act[0..1] (one split)
  float* part = nullptr;
  bf16* act[2] = {nullptr, nullptr};  // mode 2: a = silu(gate) * up, [rows, outs / 2] bf16 planes
  int act_planes = 1;
  LmRec* rec = nullptr;    // [slabs * kGemmEpiGroups][rows]
  float inv_T = 0.f;
  uint32_t k0 = 0, k1 = 0;
  const int64_t* pos = nullptr;
  int K_draft = 1;
  int* status = nullptr;
  int tma_out = 0;         // mode 0: partials leave through bulk tensor stores (the out map)
  const float* res = nullptr;  // mode 3: [rows, outs] addend
  float* out32 = nullptr;      // mode 3: [rows, outs] result
  float* tap32 = nullptr;      // mode 3: optional copy of the result
  // mode 0: a CTA whose rows all lie at or past skip_row0 (> 0) and whose
  // columns all lie before skip_cols does nothing (a product over stacked
  // operands whose lower rows need only the upper columns)
  int skip_row0 = 0, skip_cols = 0;
};

// Tensor map of a bf16 row-major [rows, K] matrix, box = 64 (k) x box_rows.
bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows);
// Tensor map of a bf16 weight in the tiled layout (rows a multiple of 64), box = one
// k block of box_rows (a multiple of 64) rows.
bool make_map_tiled(CUtensorMap* m, const void* base, int rows, int K, int box_rows);
// Tensor map of fp32 split-K partials part[S][rows][outs] for 32-row x 32-column
// bulk stores (128-byte swizzle): rows and columns past the extents are not written.
bool make_out_map(CUtensorMap* m, const void* base, int S, int rows, int outs);
// lm or one_split: no k splits (the LM head; products whose epilogue needs the full sums)
// skip_row0 / skip_cols: the tiles TcParams::skip_row0 / skip_cols describe do no work
Plan plan(int rows, int outs, int K, int xplanes, int wplanes, bool lm, bool one_split = false, int skip_row0 = 0,
          int skip_cols = 0);
// Rows of the activation tile loads: the valid rows (rounded to 8) when they fit one tile.
inline int x_box_rows(int rows) { return rows >= 128 ? 128 : ((rows + 7) / 8) * 8; }
// Shared-memory slot of one activation tile: the loaded rows, rounded to a 1 KB swizzle atom group.
__host__ __device__ inline uint32_t a_slot_bytes(int x_box) { return (uint32_t)((x_box * 128 + 1023) / 1024 * 1024); }
size_t smem_bytes(const Plan& pl);
// Every feasible plan of a one-CTA-engine product (for timing-based selection).
std::vector<Plan> plan_candidates(int rows, int outs, int K, int xplanes, int wplanes, bool one_split);

// Persistent LM-head kernel (rows <= 256): one CTA per SM walking the
// vocabulary slabs with double-buffered TMEM accumulators (sampling epilogue
// overlapped with the E stream); rows 129..256 use CTA pairs, one 128-row tile
// of h each, on the same slabs. Records are [n_units][rows].
struct LmPlan {
  bool ok = false;
  bool paired = false;
  bool rep = false;  // rows <= 32 copied into all four TMEM lane quadrants (short k: the epilogue paces a slab)
  int N = 0, x_box0 = 0, x_box1 = 0, kblocks = 0, stages = 0, n_slabs = 0, n_units = 0, grid = 0,
      groups = 0;
  uint32_t stage_bytes = 0;
  size_t tail_pad = 0;
};
struct LmParams {
  int rows = 0, outs = 0;
  int n_slabs = 0, kblocks = 0, stages = 0, x_box0 = 0, x_box1 = 0, paired = 0, rep = 0;
  uint32_t stage_bytes = 0;
  LmRec* rec = nullptr;
  float inv_T = 0.f;  // 0 = greedy
  uint32_t k0 = 0, k1 = 0;
  const int64_t* pos = nullptr;
  int K_draft = 1;
  int* status = nullptr;
};
// Pair GEMM (2-SM MMA, persistent stream-K; rows 129..4096, bf16 operands):
// grid = 2 x G CTAs in clusters of two; W maps with 128-row boxes, X maps with
// 128-row boxes; partials laid out as pair_splits() describes.
struct PairPlan {
  bool ok = false;
  int kblocks = 0, slabs = 0, groups = 0, stages = 0, G = 0, S = 1;
  long long U = 0;
};
struct PairParams {
  int rows = 0, outs = 0;
  int kblocks = 0, slabs = 0, stages = 0, G = 1;
  long long U = 1;
  float* part = nullptr;
  int* status = nullptr;
};
bool use_pair_engine(int rows, int xplanes, int wplanes);
PairPlan pair_plan(int rows, int outs, int K, int num_sms);
Splits pair_splits(const PairPlan& pl);
size_t pair_smem_bytes(const PairPlan& pl);
cudaError_t launch_pair(const PairPlan& pl, const CUtensorMap* x, const CUtensorMap* w, PairParams prm,
                        cudaStream_t s);

LmPlan lm_plan_persistent(int rows, int outs, int K, int num_sms);
size_t lm_smem_bytes(const LmPlan& pl);
cudaError_t launch_lm_persistent(const LmPlan& pl, const CUtensorMap* x0, const CUtensorMap* x1,
                                 const CUtensorMap* w, LmParams prm, cudaStream_t s);
// out: the partials' map (make_out_map) for mode 0, or null (16-byte stores from registers)
cudaError_t launch(const Plan& pl, const CUtensorMap* x0, const CUtensorMap* x1, const CUtensorMap* w0,
                   const CUtensorMap* w1, TcParams prm, cudaStream_t s, const CUtensorMap* out = nullptr);

}  // namespace tc
}  // namespace dlite
