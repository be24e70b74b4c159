/*
 * dlite.h — C ABI of the DLite draft-and-verify round on one GB300 GPU.
 *
 * The method (DLite: history-free speculative decoding) drafts K tokens from
 * the target model's current pivot features alone — m selected target-layer
 * hidden states at the last processed position plus the anchor token — with
 * no draft-side history KV, then verifies them against the target.
 * Sources, cited by page / section / equation:
 *   [P1] "DLite 完全拆解:面向智能体的无历史投机解码" (pinghaoyang.com.cn)
 *   [P2] "DLite: History-free Speculative Decoding for Agentic AI" summary (yomxxx.com)
 *
 * Conventions for every call below
 *   - Array arguments are DEVICE pointers owned by the caller, unless the
 *     name ends in _host. They must stay valid until the stream reaches the
 *     call. Layouts are dense, row-major, in the shapes given.
 *   - Calls are stream-ordered and asynchronous: they enqueue kernels on
 *     `stream` and return; they never allocate device memory and never
 *     synchronise (except dlite_create, dlite_destroy, dlite_device_status
 *     and dlite_round_host, which say so).
 *   - Return value: DLITE_OK (0) or a negative DLITE_ERR_* code. Arguments are
 *     validated on the host before anything is launched; on an error nothing
 *     is enqueued. Device-side problems (an out-of-range token id, a bounded
 *     wait that ran out) set bits in the handle's sticky device status word,
 *     read with dlite_device_status; kernels never trap.
 *   - A handle may be used from one stream at a time; calls on one handle
 *     share its workspace, so calls that overlap on the GPU race.
 */
#ifndef DLITE_H
#define DLITE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dlite_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

enum dlite_dtype { DLITE_F32 = 0, DLITE_BF16 = 1 };

enum dlite_status {
    DLITE_OK = 0,
    DLITE_ERR_INVALID_ARG = -1,       /* null pointer, B out of [1, B_max], bad enum */
    DLITE_ERR_UNSUPPORTED_SHAPE = -2, /* config outside what the kernels handle */
    DLITE_ERR_CUDA = -3,              /* a CUDA runtime call failed (launch, copy, ...) */
    DLITE_ERR_DEVICE_TIMEOUT = -4,    /* device status: a bounded wait ran out */
    DLITE_ERR_BOUNDS = -5,            /* device status: an id was out of range (clamped) */
    DLITE_ERR_OOM = -6                /* dlite_create could not allocate */
};

/* Device status word bits (dlite_device_status). */
#define DLITE_DEV_TIMEOUT 1
#define DLITE_DEV_BOUNDS 2

/* Drafter shape. Positions: block = anchor + K placeholders ([P1] §"草稿块长与
 * 验证块长不是一个参数": block_size 8 = 1 anchor + 7 drafts). */
typedef struct {
    int B_max;        /* largest batch any call will pass */
    int D;            /* hidden width; multiple of 64 */
    int m;            /* selected target layers (context slots); m + K + max(1, anchor_group) <= 32 */
    int K;            /* draft positions, 1..31 */
    int L_D;          /* backbone layers, 1..DLITE_MAX_LAYERS */
    int n_q, n_kv, d_h; /* attention heads; n_q % n_kv == 0; d_h in {64, 128} */
    int F;            /* SwiGLU inner width; multiple of 64 */
    int R;            /* sequential-head rank; multiple of 32, <= 512 */
    int V;            /* vocabulary (tied embedding / LM head); multiple of 8, <= 262144 */
    int dtype;        /* DLITE_F32 or DLITE_BF16: type of all weights and of `hidden` */
    float rms_eps;    /* RMSNorm epsilon (1e-6) */
    float rope_theta; /* RoPE base (1e6) */
    int anchor_group; /* G: local token group ending at the anchor ([P1] §"局部位置编码切断草稿端的
                       * 全局位置增长": a fixed-length local group whose start is the origin);
                       * 0 or 1 = the anchor alone; m + K + G <= 32, G <= 8. The group rows sit at
                       * local positions 0..G-1, the placeholders at G..G+K-1, and the `anchor`
                       * argument of the draft calls is then [B, G] int32 (oldest first, the anchor
                       * last) */
    int head_type;    /* DLITE_HEAD_RNN (0): the low-rank RNN head with one tied D->V projection;
                       * DLITE_HEAD_GATED (1): the official gated token-feedback head (weights in
                       * dlite_weights.gated; R a multiple of 64) */
    int history;      /* H: history-KV control of the history-cost comparison. 0 (the method):
                       * history-free, no draft KV. H > 0: the conventional drafter the method is
                       * measured against ([P1] §"本轮临时 K/V 仍然需要计算", eq. M_draftKV; [P2]
                       * §"实验：三类负载，逐项看数字", the sliding-window ablation): every backbone
                       * layer keeps a ring of the last H local key /
                       * value rows of each request slot (bf16, 2 L_D H n_kv d_h values per slot,
                       * allocated by dlite_create and filled with the synthetic history that
                       * dlite_history_reset describes); each backbone pass attends over the H
                       * ring rows beside the block, then writes its G + K local rows at slots
                       * (cursor + j) mod H and advances the slot's cursor by G + K. A 512-row
                       * ring is the sliding-window variant. Requires DLITE_BF16,
                       * G + K <= H <= 2^20 and (n_q / n_kv) (G + K) <= 128 */
    int act_planes;   /* precision of the backbone activations of a DLITE_BF16 drafter:
                       * 0 or 1 = bf16 (the fast form: z, y, q, k, v, o and the SwiGLU output
                       * are stored as bf16); 2 = fp32-class, each stored as two bf16 planes
                       * hi + lo (about 16 significant bits) and multiplied as two products, so
                       * that with bf16 weights and fp32 accumulation the round follows float64
                       * arithmetic on the same weights to ~1e-5 (about twice the tensor work
                       * and activation traffic of the backbone products; not with history > 0).
                       * DLITE_F32 drafters always keep fp32-class activations. */
    int head_warmup;  /* DLITE_HEAD_GATED with anchor_group >= 2 only: 1 = warm the head's state up
                       * on the token before the anchor ([P1] §"官方顺序头具体算了什么": when the
                       * configuration allows, one token before the anchor gives a fixed-length
                       * warm-up): s_0 is one state update from the zero state on E_R of the
                       * group's second-to-last token, with no output; 0 = s_0 = 0 */
} dlite_config;

enum dlite_head_type { DLITE_HEAD_RNN = 0, DLITE_HEAD_GATED = 1 };

#define DLITE_MAX_LAYERS 8

/* Weights of one backbone layer, nn.Linear layout W[out, in], element type
 * cfg.dtype. Shapes: g_attn, g_ffn [D]; Wq [n_q*d_h, D]; Wk, Wv [n_kv*d_h, D];
 * Wo [D, n_q*d_h]; Wg, Wu [F, D]; Wd [D, F]. */
typedef struct {
    const void *g_attn, *Wq, *Wk, *Wv, *Wo, *g_ffn, *Wg, *Wu, *Wd;
} dlite_layer_weights;

/* All drafter weights (device pointers, element type cfg.dtype):
 *   e_depth [m, D]   depth embedding ([P1] §"History-Free 到底省掉了什么", eq. z_t)
 *   g_stage [D]      RMSNorm gain after the depth embedding is added
 *   e_ph [D]         placeholder embedding ([P1] §"锚点是已经确定...")
 *   E [V, D]         tied token embedding / LM head
 *   g_final [D]      final RMSNorm gain of the backbone
 *   Q [R, 2D]        sequential head, acting on [b_i ; h_{i-1}]
 *   P [D, R]         sequential head output map: h_i = b_i + P tanh(Q [b_i; h_{i-1}]) */
typedef struct {
    const void *e_depth, *g_stage, *e_ph, *E, *g_final, *Q, *P;
    dlite_layer_weights layer[DLITE_MAX_LAYERS];
    /* the gated token-feedback head ([P1] §"官方顺序头具体算了什么"), head_type 1 only:
     *   E_R [V, R] token embedding of the head;  W_s [2R, 2R], b_s [2R] acting on
     *   [s_{i-1}; v_i] (outputs g first, then c);  W_h [R, R + D], b_h [R] acting on
     *   [s_i; u_i];  W_o [V, R] vocabulary projection. Q and P are then unused. */
    struct {
        const void *E_R, *W_s, *b_s, *W_h, *b_h, *W_o;
    } gated;
} dlite_weights;

/* Draft statistics of one draft slot for sampling verification: the logit of
 * the drawn token and log-sum-exp of logits / T, so q(d) = exp(logit/T - lse). */
typedef struct {
    float logit;
    float lse;
} dlite_qstats;

typedef struct dlite_handle dlite_handle;

/* Create a drafter on the current CUDA device. Copies and repacks the weights
 * into handle-owned device memory (caller buffers may be freed afterwards),
 * precomputes the sequential head's R x R matrix Q_h P, and allocates the
 * workspace for batches up to B_max. Synchronises the device.
 * Errors: INVALID_ARG (null), UNSUPPORTED_SHAPE, OOM, CUDA. */
int dlite_create(const dlite_config *cfg, const dlite_weights *w, dlite_handle **out);

/* Free everything the handle owns. Synchronises the device. NULL is a no-op. */
void dlite_destroy(dlite_handle *h);

/* One history-free draft ([P1] §"从目标隐藏状态到并行草稿表示", Fig. 3;
 * [P2] §设计).
 *   hidden [B, m, D] (cfg.dtype)  pivot features: the current hidden states of
 *                                 the m selected target layers (no KV, no history)
 *   anchor [B] int32              the token already chosen but not yet run
 *                                 ([B, G] with anchor_group G > 1: the local group, anchor last)
 *                                 through the target ([P1] §"锚点...")
 *   temperature                   0 = greedy argmax; > 0 = an exact draw from
 *                                 q_i = softmax(l_i / T) in two levels: Gumbel-max over
 *                                 chunks of 16 ids on their log-mass L_k (noise: word
 *                                 k & 3 of Philox(k >> 2, position, b, 1)), then the
 *                                 inverse CDF inside the chosen chunk k at word 0 of
 *                                 Philox(k, position, b, 8)
 *   seed, pos [B] int64           RNG key and per-request position offset; draft
 *                                 slot i (1..K) uses position pos[b] + i
 *                                 (ignored when temperature == 0; pos may be NULL then)
 *   candidates [B, K] int32       out: d_1..d_K
 *   qstats [B, K]                 out: draft statistics (may be NULL when T == 0)
 * Local rows: anchor at local position 0, placeholders at 1..K (with a group:
 * group tokens at 0..G-1, placeholders at G..G+K-1); the context
 * slots are key/value-only rows at position 0. Out-of-range anchors are
 * clamped to 0 and flag DLITE_DEV_BOUNDS. */
int dlite_draft_round(dlite_handle *h, int B, const void *hidden, const int32_t *anchor,
                      float temperature, uint64_t seed, const int64_t *pos,
                      int32_t *candidates, dlite_qstats *qstats, dlite_stream_t stream);

/* Optional intermediate outputs of a draft (device pointers, float32; any may
 * be NULL): z [B, m, D] staged context features; x [L_D, B, G+K, D] residual
 * stream after each layer; b [B, K, D] backbone outputs; hs [B, K, D]
 * sequential-head outputs (gated head: its vectors r_i, [B, K, R]). */
typedef struct {
    float *z, *x, *b, *hs;
} dlite_taps;

/* dlite_draft_round plus taps (for checking hidden representations). */
int dlite_draft_round_taps(dlite_handle *h, int B, const void *hidden, const int32_t *anchor,
                           float temperature, uint64_t seed, const int64_t *pos,
                           int32_t *candidates, dlite_qstats *qstats, const dlite_taps *taps,
                           dlite_stream_t stream);

/* Stage entry points (the same kernels as dlite_draft_round, split at the
 * stage boundaries, for stage-by-stage checks).
 *   dlite_backbone:   hidden, anchor -> b [B, K, D] float32 (staging + L_D layers + final norm)
 *   dlite_seq_head:   b [B, K, D] float32 -> hs [B, K, D] float32 (sequential head)
 *   dlite_lm_head:    hs [B, K, D] float32 -> candidates, qstats (vocabulary
 *                     projection with the fused argmax / two-level draw + LSE) */
int dlite_backbone(dlite_handle *h, int B, const void *hidden, const int32_t *anchor, float *b,
                   dlite_stream_t stream);
int dlite_seq_head(dlite_handle *h, int B, const float *b, float *hs, dlite_stream_t stream);
int dlite_lm_head(dlite_handle *h, int B, const float *hs, float temperature, uint64_t seed,
                  const int64_t *pos, int32_t *candidates, dlite_qstats *qstats,
                  dlite_stream_t stream);

/* Greedy verification ([P1] §"一次因果前向评估整条候选", §"贪心模式与随机模式").
 *   candidates [B, K], target_tokens [B, K+1] int32: target_tokens[b, j] is the
 *   target's argmax at input index j of [a, d_1..d_K] (its choice for position j+1).
 * Outputs: accepted [B] = A (leading matches, 0..K); commits [B, K+1] =
 * d_1..d_A then target_tokens[b, A], entries past A set to -1;
 * n_commit [B] = A + 1; next_anchor [B] = target_tokens[b, A].
 * next_anchor may alias the anchor buffer of the draft that produced the
 * candidates (it is written after the draft has read it). */
int dlite_verify(dlite_handle *h, int B, const int32_t *candidates, const int32_t *target_tokens,
                 int32_t *accepted, int32_t *commits, int32_t *n_commit, int32_t *next_anchor,
                 dlite_stream_t stream);

/* Speculative-sampling verification ([P1] §"贪心模式与随机模式要分别说明",
 * eqs. alpha(d) = min(1, p(d)/q(d)) and p_res = [p - q]_+ / sum).
 *   candidates [B, K], qstats [B, K]     from the draft (temperature T > 0)
 *   hs [B, K, D] float32 or NULL         sequential-head outputs the candidates were
 *                                        drawn from (NULL: the handle's copy from its
 *                                        most recent dlite_draft_round)
 *   target_probs [B, K+1, V] float32     p_j: target distribution at input index j
 * d_i is accepted iff u_i * q_i(d_i) < p_{i-1}(d_i), u_i = Philox(seed, request b,
 * position pos[b]+i). At the first rejection the replacement is drawn from the
 * residual by proposal-rejection (v ~ p, kept w.p. max(0, 1 - q(v)/p(v)), 32
 * proposals, then inverse CDF over [p - q]_+); with no rejection the bonus token
 * is drawn from p_K. Decisions are taken in float64. Outputs as dlite_verify. */
int dlite_verify_sample(dlite_handle *h, int B, const int32_t *candidates,
                        const dlite_qstats *qstats, const float *hs, const float *target_probs,
                        float temperature, uint64_t seed, const int64_t *pos, int32_t *accepted,
                        int32_t *commits, int32_t *n_commit, int32_t *next_anchor,
                        dlite_stream_t stream);

/* Verification with a window and a choice of rule ([P1] §"草稿块长与验证块长不是
 * 一个参数": the verification window counts the anchor and may be shorter than
 * the drafted block, which is then truncated; §"贪心模式与随机模式要分别说明":
 * the official `match` mode).
 *   mode      DLITE_VERIFY_GREEDY: as dlite_verify (target_tokens)
 *             DLITE_VERIFY_SAMPLE: as dlite_verify_sample (qstats, hs, target_probs,
 *                                  temperature, seed, pos)
 *             DLITE_VERIFY_MATCH:  the candidates (the draft's greedy choices) against
 *                                  the target's own samples t_j ~ p_j: t_j = inverse CDF of
 *                                  target_probs[b, j] at u = Philox(seed, request b, position
 *                                  pos[b]+j+1, tag 5); A = leading run of d_{j+1} == t_j,
 *                                  commits d_1..d_A then t_A (target_probs, seed, pos)
 *   n_verify  candidates handed to verification, 0..K (K: all); the rest are dropped:
 *             A <= n_verify and the token after the verified prefix comes from index
 *             A (sampling: the bonus from p_{n_verify} at position pos[b]+n_verify+1)
 * Outputs as dlite_verify (commits [B, K+1], entries past A set to -1). Fields a mode
 * does not use may be NULL / 0. Match mode keeps its samples in handle workspace;
 * everything is stream-ordered and allocation-free (graph-capturable).
 * Errors: INVALID_ARG for a NULL the mode needs, B outside [1, B_max], n_verify
 * outside [0, K] or an unknown mode. */
enum dlite_verify_mode { DLITE_VERIFY_GREEDY = 0, DLITE_VERIFY_SAMPLE = 1, DLITE_VERIFY_MATCH = 2 };
typedef struct {
    int mode;                       /* dlite_verify_mode */
    int B;
    int n_verify;
    const int32_t *candidates;      /* [B, K] */
    const int32_t *target_tokens;   /* [B, K+1], GREEDY */
    const dlite_qstats *qstats;     /* [B, K], SAMPLE */
    const float *hs;                /* [B, K, D] or NULL, SAMPLE */
    const float *target_probs;      /* [B, K+1, V], SAMPLE and MATCH */
    float temperature;              /* SAMPLE */
    uint64_t seed;                  /* SAMPLE and MATCH */
    const int64_t *pos;             /* [B], SAMPLE and MATCH */
    int32_t *accepted, *commits, *n_commit, *next_anchor;
} dlite_verify_args;
int dlite_verify_ex(dlite_handle *h, const dlite_verify_args *args, dlite_stream_t stream);

/* Allocation-free sampling verification (no counterpart on the method's pages;
 * a library convenience). Same computation and outputs as dlite_verify_sample,
 * without a handle and without allocating: for callers that cannot allocate
 * device memory where they verify (allocator-less embedders, arena-owned
 * memory, hot loops that forbid cudaMalloc because it synchronises).
 *   K, V, D          draft positions, vocabulary (multiple of 8, <= 262144), width (multiple of 4)
 *   hs [B, K, D]     float32 head states the candidates were drawn from
 *   E [V, D]         float32 row-major LM-head weights (used for q(v) = exp(E_v . h / T - lse))
 *   other arguments  as dlite_verify_sample.
 * Scratch: the exact-fallback residual row lives in a static device array of
 * 2^20 fixed-point entries (8 MiB) that every GPU loading the library holds
 * until exit; B * V above 2^20 is rejected with DLITE_ERR_UNSUPPORTED_SHAPE.
 * The first call on a device looks up that array's device address (no
 * allocation); make that first call before any stream capture. The address
 * is cached per device for the life of the process: after cudaDeviceReset on
 * a device this call must not be used there again. All calls share the array,
 * which keeps the last call's contents (each call rewrites what it reads), so
 * calls that overlap on the GPU race.
 * E, hs and target_probs must be 16-byte aligned (INVALID_ARG otherwise).
 * Without a handle there is no device status word: a candidate id outside
 * [0, V) is not reported (it is scored as id 0 and committed unchanged), so
 * callers pass candidates from a draft of the same vocabulary. */
int dlite_verify_sample_static(int B, int K, int V, int D, const int32_t *candidates,
                               const dlite_qstats *qstats, const float *hs, const float *E,
                               const float *target_probs, float temperature, uint64_t seed,
                               const int64_t *pos, int32_t *accepted, int32_t *commits,
                               int32_t *n_commit, int32_t *next_anchor, dlite_stream_t stream);

/* History-KV control (cfg.history = H > 0). dlite_history_reset refills every
 * ring with the synthetic history and sets every cursor to 0 (dlite_create has
 * done so): element (slot t, head g, column d) of layer l, request slot b, keys
 * (which = 0) or values (which = 1) is bf16((u0 + u1 + u2 + u3 - 2) sqrt(3)),
 * every step in fp32, u_i the four uniforms ((x >> 9) + 1/2) 2^-23 of
 * Philox4x32-10(counter = (t d_h + d, (2 l + which) n_kv + g, b, 6),
 * key = (0x00000001, 0x48495354)): mean 0, variance 1.
 * dlite_history_read copies one ring, [n_kv][H][d_h] bf16 (slot-major per
 * head), to the device buffer dst on `stream` and, when cursor is non-null,
 * the slot's cursor to host memory (synchronising the stream).
 * Errors: INVALID_ARG (no history, layer / request / which out of range, null dst), CUDA. */
int dlite_history_reset(dlite_handle *h, dlite_stream_t stream);
int dlite_history_read(dlite_handle *h, int layer, int request, int which, void *dst, int32_t *cursor,
                       dlite_stream_t stream);

/* Round bookkeeping for a local token group (anchor_group G): group [B, G] becomes the
 * last G tokens of (group ++ commits[b, 0..n_commit[b]-1]), i.e. the G most recent
 * tokens ending at the new anchor. commits [B, K+1] and n_commit [B] as written by the
 * verification calls; with G = 1 this is the next anchor. In place, stream-ordered. */
int dlite_shift_group(dlite_handle *h, int B, const int32_t *commits, const int32_t *n_commit,
                      int32_t *group, dlite_stream_t stream);

/* Round bookkeeping: pos[b] += n_commit[b] (the RNG positions follow the
 * committed tokens; [P1] §"一轮执行后..." — each round advances A+1). */
int dlite_advance(dlite_handle *h, int B, const int32_t *n_commit, int64_t *pos,
                  dlite_stream_t stream);

/* One whole round from HOST buffers: copies hidden_host [B, m, D] (cfg.dtype),
 * anchor_host [B, G], pos_host [B] and either target_tokens_host [B, K+1]
 * (temperature == 0) or target_probs_host [B, K+1, V] (temperature > 0) to the
 * device, runs draft + verify, copies accepted/commits/n_commit/next_anchor
 * back into the *_host outputs, and synchronises `stream`. Host buffers should
 * be pinned for asynchronous copies. Uses handle-owned device staging buffers;
 * the target rows cross on a handle-owned copy stream while the draft runs on
 * `stream` (the verification waits for them). Target probabilities in pinned,
 * device-mapped host memory (cudaHostAlloc / pinned tensors on a unified-address
 * system) are not copied: the verification reads the entries and rows it uses
 * in place, so only those cross the CPU-GPU link. */
int dlite_round_host(dlite_handle *h, int B, const void *hidden_host, const int32_t *anchor_host,
                     const int64_t *pos_host, const int32_t *target_tokens_host,
                     const float *target_probs_host, float temperature, uint64_t seed,
                     int32_t *accepted_host, int32_t *commits_host, int32_t *n_commit_host,
                     int32_t *next_anchor_host, dlite_stream_t stream);

/* Synthetic target tokens for timing whole rounds with a realistic acceptance.
 * This library holds the drafter and the verification rule, not the target
 * model; this call stands in for the target's greedy choices in the
 * acceptance workloads (it is not a step of the method). The acceptance model
 * is the per-position conditional acceptance c_i whose products give the
 * prefix survival P(A >= k) = prod c_i ([P1] §"分布重叠怎样影响平均推进量"):
 *   target_tokens[b, j], j < K: = candidates[b, j] with probability c_j, else a
 *                               uniform id different from it;
 *   target_tokens[b, K]:        a uniform id (the bonus position).
 * Draws: the words (w0, w1, w2, w3) of Philox4x32-10(counter = (0, pos[b] + j + 1
 * (low 32 bits), b, 7), key = (seed & 0xffffffff, seed >> 32)); agreement iff
 * ((w0 >> 9) + 1/2) 2^-23 < c_j; a disagreeing id is (d + 1 + floor(w1 (V-1) / 2^32))
 * mod V, the bonus id floor(w1 V / 2^32).
 *   accept_c [n_tables, B, K] float32  c per table, request and index; the call uses
 *                                      table (*round_counter mod n_tables) and then
 *                                      increments *round_counter (device int32; NULL:
 *                                      table 0, nothing incremented)
 *   candidates [B, K], pos [B] int64, target_tokens [B, K+1] int32 (out), device pointers.
 * Out-of-range candidates are read as id 0. One single-CTA launch, stream-ordered,
 * allocation-free. Errors: INVALID_ARG (NULL, B < 1, K outside 1..31, V < 2,
 * n_tables < 1), CUDA. */
int dlite_synthetic_target(int B, int K, int V, const int32_t *candidates, const float *accept_c,
                           int n_tables, int32_t *round_counter, uint64_t seed, const int64_t *pos,
                           int32_t *target_tokens, dlite_stream_t stream);

/* Failure-detection probe of the bounded device waits (no fault is involved).
 * Enqueues one kernel that waits on an mbarrier no thread arrives at, through
 * the same bounded-wait helpers the tensor-core kernels use, with the limit
 * limit_ns (1 ns .. 1 s) in place of their 2 s; each wait gives up, sets
 * DLITE_DEV_TIMEOUT in the handle's status word and returns. Then one kernel
 * makes the engines' entry check of that word. result [3] device int32 (out):
 * [0] = 1 if the warp-wide wait gave up, [1] = 1 if the single-thread wait gave
 * up, [2] = 1 if the second kernel saw the flag and would skip its work.
 * Afterwards dlite_device_status returns DLITE_ERR_DEVICE_TIMEOUT (and clears
 * the flag if asked). Errors: INVALID_ARG, CUDA. */
int dlite_selftest_wait(dlite_handle *h, uint64_t limit_ns, int32_t *result, dlite_stream_t stream);

/* Read (and with clear != 0, reset) the sticky device status word.
 * Synchronises `stream`. *status_out gets DLITE_DEV_* bits. Returns
 * DLITE_ERR_DEVICE_TIMEOUT or DLITE_ERR_BOUNDS when those bits are set. */
int dlite_device_status(dlite_handle *h, int clear, int *status_out, dlite_stream_t stream);

/* Static description of a status code. */
const char *dlite_status_string(int status);

/* Name and description of the CUDA runtime error behind the most recent
 * DLITE_ERR_CUDA returned on the calling host thread ("no error" if none).
 * The string is static; no GPU work is done. */
const char *dlite_last_cuda_error(void);

/* Profiling: run one draft (and, when target_tokens / target_probs is given,
 * its greedy / sampling verification) eagerly on `stream`, recording a CUDA
 * event after every kernel launch; synchronises `stream`. Writes the elapsed
 * milliseconds of launch i into times_ms[i] and a static kernel name into
 * names[i] (names may be NULL), for up to `cap` launches. Returns the number
 * of launches (> 0) or a negative DLITE_ERR_*. Arguments as dlite_draft_round
 * and dlite_verify / dlite_verify_sample. */
int dlite_stage_times(dlite_handle *h, int B, const void *hidden, const int32_t *anchor,
                      float temperature, uint64_t seed, const int64_t *pos,
                      const int32_t *target_tokens, const float *target_probs, int32_t *candidates,
                      dlite_qstats *qstats, int32_t *accepted, int32_t *commits, int32_t *n_commit,
                      int32_t *next_anchor, float *times_ms, const char **names, int cap,
                      dlite_stream_t stream);

/* Diagnostic: one tensor-core product through the same engine the round uses,
 * part[z][r][o] = sum over k-split z of X[r, :] . W[o, :], with X given as 1 or
 * 2 bf16 planes [x_rows, K] (x_rows a multiple of 128, >= rows) and W as 1 or 2
 * bf16 planes of [outs, K] in the library's tiled weight layout: rows padded with
 * zeros to a multiple of 64, stored as 64 x 64 tiles, tile (i, j) = rows 64i.., columns
 * 64j.., tiles in row-tile-major order, each tile row-major (two W planes need two
 * X planes); K a multiple of 64, outs a multiple of 8. `part` must
 * hold 16 * rows * outs floats; the sum over the returned number of splits
 * (> 0) is the product. `status` is a device int receiving DLITE_DEV_* bits.
 * plan_override: NULL selects what the round uses (one bf16 plane on each side
 * and more than 512 rows: the CTA-pair engine with 2-SM MMAs; otherwise the
 * one-CTA engine with the planner's tiling); a host int[3] {slab width N,
 * k splits, pipeline stages} (0 = planner's choice) forces the one-CTA engine
 * with that tiling, for sweeps.
 * Returns the split count or a negative DLITE_ERR_*. */
int dlite_selftest_gemm(int rows, int outs, int K, int xplanes, int wplanes, const void *X0,
                        const void *X1, int x_rows, const void *W0, const void *W1, float *part,
                        int *status, const int *plan_override, dlite_stream_t stream);

/* Counters since creation or the last reset, copied to host memory out[5]:
 * [0] residual draws, [1] proposals evaluated, [2] residual draws that needed
 * the exact inverse-CDF fallback, [3] bonus draws (sampling verification);
 * [4] LM-head rows whose 4 finalists were within 0.02 (score units) of each
 * other. Synchronises `stream`; reset != 0 zeroes them. */
int dlite_counters(dlite_handle *h, int reset, int64_t *out, dlite_stream_t stream);

/* Number of kernels the last draft+verify path enqueues for batch B
 * (greedy when temperature == 0), for launch accounting. */
int dlite_launch_count(dlite_handle *h, int B, float temperature);

#ifdef __cplusplus
}
#endif

#endif /* DLITE_H */
