"""Plain CPU oracle for the DLite draft-and-verify round (numpy, float64).

TEST INFRASTRUCTURE ONLY. This module is the slow, obviously-correct statement
of what the round computes. Only tests/, the smoke check in __graft_entry__ and
the bench's CPU-baseline / reference leg may import it; the product path never
does, and it shares no code with the CUDA library.

Sources (web pages on the method; cited by page, section and equation):
  [P1] "DLite 完全拆解:面向智能体的无历史投机解码" (pinghaoyang.com.cn, 2026-10-19)
  [P2] "DLite: History-free Speculative Decoding for Agentic AI" paper summary
       (yomxxx.com, 2026-10-20)
  [P3] "DFlash block diffusion speculative decoding" (charlestar.github.io)

Every function works on ONE request (the method is per-request independent);
batching is a loop in draft_round / verify_* callers.

Two precision modes:
  mirror=False  every value in float64 ("pure").
  mirror=True   float64 arithmetic, but values are rounded to bfloat16 at the
                points where the bf16 GPU path stores bf16 activations (listed
                in `BF16_POINTS`). Weights are taken as given (already bf16).

Readings where the pages are silent (each is restated beside the code):
  * RMSNorm everywhere, eps from the config (1e-6), applied after adding the
    depth embedding, before attention, before the FFN and at the end.
  * Context slots are key/value-only rows: each layer projects the staged z
    with that layer's W_k, W_v; they get no query, no RoPE (local position 0)
    and no residual update.
  * Anchor at local position 0, placeholder i at local position i; RoPE is
    rotate-half with base theta from the config.
  * One shared placeholder embedding e_ph; the anchor row is the tied E row.
  * Sequential head, low-rank RNN form: h_0 = 0,
        h_i = b_i + P tanh(Q^T [b_i; h_{i-1}]),  i = 1..K,
    followed by ONE vocabulary projection l_i = E h_i.
  * Argmax ties go to the lowest token id.
  * Sampling draws d_i from q_i = softmax(l_i / T) in two levels (sample_logits):
    Gumbel-max over chunks of 16 ids on their log-mass, then the inverse CDF
    inside the chosen chunk, all noise from Philox.
"""
import numpy as np

from . import philox as _ph

BF16_POINTS = ("z", "y_attn", "q", "k", "v", "o", "y_ffn", "a")


# ---------------------------------------------------------------- precision

def bf16_round(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64.

    fp64 -> fp32 (round to nearest even), then fp32 -> bf16 on the bit
    pattern: add 0x7FFF plus the lowest kept bit, clear the low 16 bits.
    """
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _r(x, mirror):
    return bf16_round(x) if mirror else x


def f64(a):
    """Any array-like (numpy, or a CPU torch tensor via numpy()) as float64."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().float().numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- building blocks

def rmsnorm(x, g, eps):
    """RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps)."""
    x = f64(x)
    return f64(g) * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope_rotate_half(x, positions, theta):
    """Rotary embedding, rotate-half form, on x[..., rows, heads, d_h].

    Pair (j, j + d_h/2) is rotated by angle pos * theta^(-2j/d_h).
    [P1] §"局部位置编码切断草稿端的全局位置增长": the drafter uses local
    coordinates only (anchor at 0, placeholders 1, 2, 3, ...).
    """
    x = f64(x)
    d = x.shape[-1]
    half = d // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]   # [rows, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def block_attention(q, k, v, n_q, n_kv):
    """Non-causal attention over the whole local block.

    q: [Tq, n_q, d_h]; k, v: [Tk, n_kv, d_h]. Query head h reads key/value head
    floor(h * n_kv / n_q). Scores q.k / sqrt(d_h), softmax over ALL keys (no
    mask). [P1] §"锚点是已经确定、尚待目标前向处理的输入": the backbone runs
    non-causal attention inside the short block so every placeholder is
    computed at once.
    """
    q, k, v = f64(q), f64(k), f64(v)
    d_h = q.shape[-1]
    group = n_q // n_kv
    out = np.empty_like(q)
    for h in range(n_q):
        g = h // group
        s = q[:, h, :] @ k[:, g, :].T / np.sqrt(d_h)          # [Tq, Tk]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out.reshape(q.shape[0], n_q * d_h)


# ---------------------------------------------------------------- history-KV control

def history_values(H, n_kv, d_h, layer, request, which):
    """Synthetic history rows of the control drafter, [H, n_kv, d_h], bf16 values.

    Element (slot t, head g, column d) of K (which = 0) or V (which = 1) of a
    layer and request: with the four uniforms u0..u3 of Philox(counter =
    (t d_h + d, (2 layer + which) n_kv + g, request, TAG_HIST), key = HIST_SEED),
    bf16(float32((u0 + u1 + u2 + u3 - 2) * sqrt(3))) -- mean 0, variance 1, a
    stand-in for the N(0, 1) history of the control workload; every step is
    computed in float32 so that the GPU forms the same bits.
    """
    t = np.arange(H, dtype=np.int64)[:, None, None]
    g = np.arange(n_kv, dtype=np.int64)[None, :, None]
    d = np.arange(d_h, dtype=np.int64)[None, None, :]
    k0, k1 = _ph.seed_key(_ph.HIST_SEED)
    w = _ph.philox4x32_10(t * d_h + d, (2 * layer + which) * n_kv + g, request, _ph.TAG_HIST, k0, k1)
    u = [_ph.uniform_open(x).astype(np.float32) for x in w]
    acc = ((u[0] + u[1]) + u[2]) + u[3]
    val = (acc - np.float32(2.0)) * np.float32(1.7320508075688772)
    return bf16_round(val.astype(np.float64))


class HistoryCache:
    """The control drafter's per-layer draft KV of one request: a ring of the
    last H local K/V rows ([P1] §"本轮临时 K/V 仍然需要计算": a conventional
    drafter keeps its own KV and it grows with the history; here a window of
    H rows), initially the synthetic history_values. Each round attends over
    the H cached rows beside the block, then writes its G + K local rows at
    slots (cursor + j) mod H and advances the cursor."""

    def __init__(self, cfg, H, request):
        self.H = H
        self.cursor = 0
        self.k = [history_values(H, cfg.n_kv, cfg.d_h, l, request, 0) for l in range(cfg.L_D)]
        self.v = [history_values(H, cfg.n_kv, cfg.d_h, l, request, 1) for l in range(cfg.L_D)]

    def layer(self, l):
        return self.k[l], self.v[l]

    def append(self, local):
        """local: per layer (k_loc, v_loc) [G+K, n_kv, d_h] of the finished round."""
        n = local[0][0].shape[0]
        slots = (self.cursor + np.arange(n)) % self.H
        for l, (k_loc, v_loc) in enumerate(local):
            self.k[l][slots] = k_loc
            self.v[l][slots] = v_loc
        self.cursor = (self.cursor + n) % self.H


def silu(x):
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------- the drafter

def anchor_group(anchor, cfg):
    """The request's local token group: G token ids ending at the anchor."""
    g = [int(t) for t in np.atleast_1d(np.asarray(anchor))]
    if len(g) != cfg.G:
        raise ValueError("the anchor group holds G = %d tokens" % cfg.G)
    return g


def stage(hidden, anchor, W, cfg, mirror=False):
    """Depth-embedding staging and the local rows of one request.

    z_j = RMSNorm(h_j + e_depth_j) * g_stage for the m selected target layers
    ([P1] §"History-Free 到底省掉了什么", eq. z_t = h_t + e_depth, "官方实现还
    会对相加后的特征做归一化"). Local rows: x_0 = E[anchor] (tied embedding),
    x_i = e_ph for the K placeholders ([P1] §"锚点是已经确定...").
    With a local token group of G tokens ending at the anchor ([P1]
    §"局部位置编码切断草稿端的全局位置增长": build_block_position_ids takes a
    fixed-length local group, its start the origin) the first G rows are the
    group's embeddings and the K placeholders follow.
    Returns z [m, D] and the fp32-class residual stream x [G+K, D].
    """
    h = f64(hidden)                                          # [m, D]
    z = _r(rmsnorm(h + f64(W["e_depth"]), W["g_stage"], cfg.eps), mirror)
    D, K, G = cfg.D, cfg.K, cfg.G
    group = anchor_group(anchor, cfg)
    x = np.empty((G + K, D))
    for i, t in enumerate(group):
        x[i] = f64(W["E"][t])
    x[G:] = f64(W["e_ph"])[None, :]
    return z, x


def backbone_layer(x, z, Wl, cfg, mirror=False, hist=None, local_out=None):
    """One pre-norm block over [m context slots | anchor group | K placeholders].

    Queries exist only for the anchor and placeholders; keys/values for the
    context slots and the local rows ([P1] §"本轮临时 K/V 仍然需要计算").
    Context slots are K/V-only rows projected from z with no extra norm and
    sit at local position 0, where RoPE is the identity; the group rows sit at
    0..G-1 (its start is the origin) and placeholder i at G-1+i.
    """
    K1 = cfg.G + cfg.K
    n_q, n_kv, d_h = cfg.n_q, cfg.n_kv, cfg.d_h
    y = _r(rmsnorm(x, Wl["g_attn"], cfg.eps), mirror)
    pos = np.arange(K1)
    q = y @ f64(Wl["Wq"]).T
    k_loc = y @ f64(Wl["Wk"]).T
    v_loc = y @ f64(Wl["Wv"]).T
    q = _r(rope_rotate_half(q.reshape(K1, n_q, d_h), pos, cfg.theta), mirror)
    k_loc = _r(rope_rotate_half(k_loc.reshape(K1, n_kv, d_h), pos, cfg.theta), mirror)
    v_loc = _r(v_loc.reshape(K1, n_kv, d_h), mirror)
    k_ctx = _r((z @ f64(Wl["Wk"]).T).reshape(-1, n_kv, d_h), mirror)
    v_ctx = _r((z @ f64(Wl["Wv"]).T).reshape(-1, n_kv, d_h), mirror)
    k_all = np.concatenate([k_ctx, k_loc], axis=0)
    v_all = np.concatenate([v_ctx, v_loc], axis=0)
    if hist is not None:   # the control's draft KV: H more keys / values beside the block
        k_all = np.concatenate([hist[0], k_all], axis=0)
        v_all = np.concatenate([hist[1], v_all], axis=0)
    if local_out is not None:
        local_out.append((k_loc, v_loc))
    o = _r(block_attention(q, k_all, v_all, n_q, n_kv), mirror)
    x = x + o @ f64(Wl["Wo"]).T
    y2 = _r(rmsnorm(x, Wl["g_ffn"], cfg.eps), mirror)
    a = _r(silu(y2 @ f64(Wl["Wg"]).T) * (y2 @ f64(Wl["Wu"]).T), mirror)
    return x + a @ f64(Wl["Wd"]).T


def backbone(hidden, anchor, W, cfg, mirror=False, taps=None, history=None, local_out=None):
    """Parallel backbone: b_i = RMSNorm(x_i) * g_final for placeholders i=1..K.

    [P1] §"主干并行输出的是表示,还不是有因果联系的完整候选": the backbone
    emits one vector per draft position, u_1..u_K, all at once.
    """
    z, x = stage(hidden, anchor, W, cfg, mirror)
    if taps is not None:
        taps["z"] = z
        taps["x"] = []
    for l, Wl in enumerate(W["layers"]):
        x = backbone_layer(x, z, Wl, cfg, mirror, history.layer(l) if history is not None else None, local_out)
        if taps is not None:
            taps["x"].append(x.copy())
    return rmsnorm(x[cfg.G:], W["g_final"], cfg.eps)


def sequential_head(b, Q, P):
    """Low-rank RNN head, direct form, state reset at the start of the block.

    h_0 = 0;  h_i = b_i + P tanh(Q^T [b_i ; h_{i-1}]).  Q is stored as the
    [R, 2D] matrix that maps [b; h] to R values, P as [D, R].
    [P2] §设计 (sequential head): a low-rank RNN integrates in-block
    dependencies in hidden space; [P1] §"官方顺序头具体算了什么": the state is
    initialised at the start of each block.
    """
    b = f64(b)
    Q, P = f64(Q), f64(P)
    h_prev = np.zeros(b.shape[1])
    out = np.empty_like(b)
    for i in range(b.shape[0]):
        t = np.tanh(Q @ np.concatenate([b[i], h_prev]))
        out[i] = b[i] + P @ t
        h_prev = out[i]
    return out


CHUNK = 16   # vocabulary ids per chunk of the two-level draw


def sample_logits(ell_i, temperature, seed, position, request):
    """The draft's choice from one row of logits l over V ids; returns (d, gap, lse).

    T = 0: d = argmax l (lowest id on ties); gap = the top-2 logit gap.
    T > 0: an exact draw from q = softmax(l / T) ([P1] §"官方顺序头具体算了什么":
    q_i from the temperature-scaled softmax of the logits, d_i drawn from it),
    in two levels:
      1. chunks of CHUNK consecutive ids, chunk k = ids [16k, 16k + 16) within V,
         with log-mass L_k = log sum_{v in k} exp(l_v / T); Gumbel-max over the
         chunks: k* = argmax_k L_k + g_k (lowest k on ties), with
         g_k = -log(-log u_k), u_k from word k & 3 of Philox(k >> 2, position,
         request, TAG_GUMBEL); so P(k* = k) = exp(L_k) / sum_j exp(L_j);
      2. inside chunk k*: the inverse CDF of exp(l_v / T - L_k*) at u' from word
         0 of Philox(k*, position, request, TAG_PICK).
    P(d = v) = exp(l_v / T) / sum_w exp(l_w / T). gap = the smaller of the top-2
    gap of the chunk scores and the distance of u' from the nearest CDF step
    of the chosen chunk (how close the draw was to going another way).
    lse = log sum_v exp(l_v / T).
    """
    ell_i = f64(ell_i)
    if temperature == 0.0:
        d = int(np.argmax(ell_i))
        return d, float(_top2_gap(ell_i[None, :])[0]), float("nan")
    V = ell_i.shape[0]
    z = ell_i / temperature
    m = float(z.max())
    lse = m + float(np.log(np.exp(z - m).sum()))
    n_chunks = (V + CHUNK - 1) // CHUNK
    L = np.array([np.log(np.exp(z[k * CHUNK:(k + 1) * CHUNK] - m).sum()) + m for k in range(n_chunks)])
    score = L + _ph.gumbel_row(seed, position, request, n_chunks)
    k = int(np.argmax(score))
    gap = float(_top2_gap(score[None, :])[0]) if n_chunks > 1 else float("inf")
    u = float(_ph.draw(seed, k, position, request, _ph.TAG_PICK, 0))
    zc = z[k * CHUNK:(k + 1) * CHUNK]
    w = np.exp(zc - zc.max())
    j = inverse_cdf(w, u)
    c = np.cumsum(w) / w.sum()
    edges = [c[j]] + ([c[j - 1]] if j > 0 else [])
    gap = min(gap, min(abs(u - e) for e in edges))
    return k * CHUNK + j, gap, lse


def _pick(ell_i, temperature, seed, position, request):
    return sample_logits(ell_i, temperature, seed, position, request)


def gated_state_step(s_prev, token, W):
    """One state update of the gated head on the previous token's embedding:
    [g, c] = W_s [s_prev; E_R(token)] + b_s;  f = sigmoid(g);
    s = f * s_prev + (1 - f) * tanh(c)  ([P1] §"官方顺序头具体算了什么", eq. block)."""
    E_R, W_s, b_s = f64(W["E_R"]), f64(W["W_s"]), f64(W["b_s"])
    R = E_R.shape[1]
    gc = W_s @ np.concatenate([s_prev, E_R[int(token)]]) + b_s
    f = 1.0 / (1.0 + np.exp(-gc[:R]))
    return f * s_prev + (1.0 - f) * np.tanh(gc[R:])


def gated_head(b, anchor_token, W, temperature=0.0, seed=0, pos=0, request=0, warm_token=None):
    """The official gated token-feedback head, direct form ([P1] §"官方顺序头具体
    算了什么", eq. block), one request:
        v_i = E_R(d_{i-1}), d_0 = the anchor;
        [g_i, c_i] = W_s [s_{i-1}; v_i] + b_s;   f_i = sigmoid(g_i);
        s_i = f_i * s_{i-1} + (1 - f_i) * tanh(c_i),  s_0 = 0 (the state starts
              with the block);
        r_i = W_h [s_i; u_i] + b_h;   l_i = W_o r_i,
    and d_i is drawn from l_i like the main head's candidates (argmax, or
    the two-level draw of sample_logits at position pos + i) before step i + 1 reads it.
    g is the first R outputs of W_s, c the last R; W_h acts on [s; u].
    Warm-up (the same passage: when the configuration allows, the one token
    before the anchor warms the state up for a fixed length): with warm_token,
    s_0 is one state update from the zero state on E_R(warm_token), with no
    output; step 1 then reads s_0 and the anchor as before.
    Returns dict(cand, logit_d, lse, gap, r [K, R], logits [K, V]).
    """
    u = f64(b)
    K = u.shape[0]
    E_R, W_s, b_s = f64(W["E_R"]), f64(W["W_s"]), f64(W["b_s"])
    W_h, b_h, W_o = f64(W["W_h"]), f64(W["b_h"]), f64(W["W_o"])
    R = E_R.shape[1]
    temperature = float(np.float32(temperature))
    s_prev = np.zeros(R)
    if warm_token is not None:
        s_prev = gated_state_step(s_prev, warm_token, W)
    d_prev = int(anchor_token)
    cand, logit_d, lse, gap = [], [], [], []
    rs, ells = np.empty((K, R)), []
    for i in range(K):
        gc = W_s @ np.concatenate([s_prev, E_R[d_prev]]) + b_s
        f = 1.0 / (1.0 + np.exp(-gc[:R]))
        s_i = f * s_prev + (1.0 - f) * np.tanh(gc[R:])
        r = W_h @ np.concatenate([s_i, u[i]]) + b_h
        ell = W_o @ r
        d, gp, l = _pick(ell, temperature, seed, pos + i + 1, request)
        cand.append(d)
        logit_d.append(float(ell[d]))
        lse.append(l)
        gap.append(gp)
        rs[i] = r
        ells.append(ell)
        s_prev, d_prev = s_i, d
    return dict(cand=np.array(cand, dtype=np.int64), logit_d=np.array(logit_d), lse=np.array(lse),
                gap=np.array(gap), r=rs, logits=np.stack(ells))


def lm_logits(h, E, chunk=16384):
    """The single vocabulary projection l = E h (tied E [V, D]), chunked over V.

    [P2] §设计: the vocabulary projection is done once, after the block's
    dependencies are integrated; [P1] §"避免的是昂贵的中间词表投影".
    """
    h = f64(h)
    V = E.shape[0]
    out = np.empty((h.shape[0], V))
    for s in range(0, V, chunk):
        out[:, s:s + chunk] = h @ f64(E[s:s + chunk]).T
    return out


def _top2_gap(s):
    part = np.partition(s, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def draft_request(hidden, anchor, W, cfg, temperature=0.0, seed=0, pos=0, request=0,
                  mirror=False, taps=None, history=None):
    """One request's draft: candidates d_1..d_K plus what verification needs.

    Greedy (T = 0): d_i = argmax_v l_iv (lowest id on ties).
    Sampling (T > 0): d_i is the two-level draw of sample_logits at position
    pos + i, an exact draw from q_i = softmax(l_i / T) ([P1] §"从 logits 经过
    温度缩放和 softmax,得到草稿分布 q_i").
    Returns dict(cand, logit_d, lse, gap, b, h).
    """
    temperature = float(np.float32(temperature))   # a float32 quantity, as in the C ABI
    local = [] if history is not None else None
    b = backbone(hidden, anchor, W, cfg, mirror, taps, history, local)
    if history is not None:   # the round's local rows join the draft KV afterwards
        history.append(local)
    if getattr(cfg, "head", "rnn") == "gated":   # token feedback: vocabulary projection inside each step
        group = anchor_group(anchor, cfg)
        warm = group[-2] if getattr(cfg, "warmup", 0) else None   # the token before the anchor
        r = gated_head(b, group[-1], W, temperature, seed, pos, request, warm_token=warm)
        if taps is not None:
            taps["b"] = b
            taps["h"] = r["r"]
            taps["logits"] = r["logits"]
        return dict(cand=r["cand"], logit_d=r["logit_d"], lse=r["lse"], gap=r["gap"], b=b, h=r["r"])
    h = sequential_head(b, W["Q"], W["P"])
    ell = lm_logits(h, W["E"])
    K = cfg.K
    if temperature == 0.0:
        cand = np.argmax(ell, axis=1)
        gap = _top2_gap(ell)
        logit_d = ell[np.arange(K), cand]
        lse = np.full(K, np.nan)
    else:
        picks = [sample_logits(ell[i], temperature, seed, pos + i + 1, request) for i in range(K)]
        cand = np.array([p[0] for p in picks])
        gap = np.array([p[1] for p in picks])
        logit_d = ell[np.arange(K), cand]
        lse = np.array([p[2] for p in picks])
    if taps is not None:
        taps["b"] = b
        taps["h"] = h
        taps["logits"] = ell
    return dict(cand=cand.astype(np.int64), logit_d=logit_d, lse=lse, gap=gap, b=b, h=h)


# ---------------------------------------------------------------- verification

def _n_verify(K, n_verify):
    """Candidates handed to verification: all K by default, else the first
    n_verify; the rest are dropped ([P1] §"草稿块长与验证块长不是一个参数":
    a verification window of n_verify + 1 tokens including the anchor truncates
    verification, not drafting)."""
    kv = K if n_verify is None else int(n_verify)
    if not 0 <= kv <= K:
        raise ValueError("n_verify must lie in [0, K]")
    return kv


def verify_greedy(cand, target_tokens, n_verify=None):
    """Longest accepted prefix, greedy mode.

    target_tokens[j] is the target's argmax at input index j of [a, d_1..d_K],
    i.e. its choice for position j+1. Draft d_i passes iff d_i equals
    target_tokens[i-1]; A is the length of the leading run of passes (the
    cumulative product of the pass flags: "pass, pass, fail, pass" gives A = 2).
    The round commits d_1..d_A then target_tokens[A] (correction, or the bonus
    token when A = K); that token is the next anchor.
    [P1] §"一次因果前向评估整条候选", §"贪心模式与随机模式要分别说明",
    §"一轮执行后..." steps 4-5.
    With n_verify = w < K only d_1..d_w are verified (A <= w) and the token
    committed after them is target_tokens[A].
    """
    cand = [int(c) for c in cand]
    K = _n_verify(len(cand), n_verify)
    A = 0
    while A < K and cand[A] == int(target_tokens[A]):
        A += 1
    tok = int(target_tokens[A])
    return dict(A=A, commits=cand[:A] + [tok], n_commit=A + 1, next_anchor=tok)


def next_group(group, commits):
    """The next round's local token group: the G most recent tokens, i.e. the
    last G of the current group followed by the committed tokens (the last
    committed token is the new anchor; [P1] §"一轮执行后..." step 5)."""
    seq = [int(t) for t in np.atleast_1d(group)] + [int(c) for c in commits]
    return seq[-len(np.atleast_1d(group)):]


def inverse_cdf(w, u):
    """Smallest index v with sum_{w<=v} w > u * sum(w), prefix sums in float64."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    return int(np.searchsorted(c, u * c[-1], side="right"))


N_PROPOSALS = 32


def verify_sample(cand, logit_d, lse, h, E, p, temperature, seed, pos, request, n_verify=None):
    """Speculative rejection sampling with residual resampling, one request.

    For i = 1..K: q_i(d_i) = exp(l_{i,d_i}/T - lse_i); with
    u_i = Philox(0, pos + i, request, TAG_ACCEPT) word 0, d_i is accepted iff
    u_i * q_i(d_i) < p_{i-1}(d_i), i.e. with probability min(1, p/q)
    ([P1] §"贪心模式与随机模式要分别说明", eq. alpha(d) = min(1, p(d)/q(d))).
    A = index of the first rejection (K if none).
    A < K: draw from p_res = [p_A - q_{A+1}]_+ / sum ([P1] eq. p_res) by
      proposal-rejection: propose v ~ p_A by inverse CDF with
      u = Philox(j, pos+A+1, request, TAG_RESID) word 0 and keep it iff
      word 1 * p(v) < p(v) - q(v); this keeps v with probability
      max(0, 1 - q(v)/p(v)), so kept draws follow p_res exactly. After
      N_PROPOSALS misses, inverse CDF over [p - q]_+ itself with
      u = Philox(N_PROPOSALS, ...) word 0 (over p if that mass is 0).
    A = K: the bonus token is drawn from p_K by inverse CDF with
      u = Philox(0, pos+K+1, request, TAG_BONUS) word 0.
    q(v) for arbitrary v is recomputed from the head state: exp(E_v.h/T - lse).
    With n_verify = w < K the round runs as if K were w (only d_1..d_w are
    tested; the bonus comes from p_w at position pos + w + 1).
    """
    T = float(np.float32(temperature))   # a float32 quantity, as in the C ABI
    cand = [int(c) for c in cand]
    K = _n_verify(len(cand), n_verify)
    p = f64(p)
    A = K
    for i in range(1, K + 1):
        d = cand[i - 1]
        q_d = np.exp(float(logit_d[i - 1]) / T - float(lse[i - 1]))
        u = float(_ph.draw(seed, 0, pos + i, request, _ph.TAG_ACCEPT, 0))
        if not (u * q_d < p[i - 1, d]):
            A = i - 1
            break
    resampled = "bonus"
    if A == K:
        u = float(_ph.draw(seed, 0, pos + K + 1, request, _ph.TAG_BONUS, 0))
        tok = inverse_cdf(p[K], u)
    else:
        row = p[A]
        hrow = f64(h[A])
        lse_a = float(lse[A])
        tok = None
        for j in range(N_PROPOSALS):
            u1 = float(_ph.draw(seed, j, pos + A + 1, request, _ph.TAG_RESID, 0))
            u2 = float(_ph.draw(seed, j, pos + A + 1, request, _ph.TAG_RESID, 1))
            v = inverse_cdf(row, u1)
            q_v = np.exp(float(f64(E[v]) @ hrow) / T - lse_a)
            if u2 * row[v] < row[v] - q_v:
                tok = v
                resampled = "proposal"
                break
        if tok is None:
            q_all = np.exp(lm_logits(hrow[None, :], E)[0] / T - lse_a)
            r = np.maximum(row - q_all, 0.0)
            u3 = float(_ph.draw(seed, N_PROPOSALS, pos + A + 1, request, _ph.TAG_RESID, 0))
            tok = inverse_cdf(r if r.sum() > 0 else row, u3)
            resampled = "fallback"
    return dict(A=A, commits=cand[:A] + [tok], n_commit=A + 1, next_anchor=tok, how=resampled)


def match_target_token(p_row, seed, pos, request, j):
    """The target's own sample at input index j (its choice for position j + 1):
    inverse CDF over p_j with u = Philox(0, pos + j + 1, request, TAG_MATCH) word 0."""
    u = float(_ph.draw(seed, 0, pos + j + 1, request, _ph.TAG_MATCH, 0))
    return inverse_cdf(p_row, u)


def verify_match(cand, p, seed, pos, request, n_verify=None):
    """Match verification, one request ([P1] §"贪心模式与随机模式要分别说明",
    the official `match` mode): the candidates are the draft's greedy choices,
    the target samples every position from its own distribution p_j (rows given
    at the target's temperature), A is the leading run of positions where the
    candidate equals the target's sample, and the round commits d_1..d_A then
    the target's sample at index A (at the first mismatch, or after the last
    verified candidate). Unlike rejection sampling this is no p/q rule: for a
    fixed candidate d the chance of a match at index j is p_j(d).
    """
    cand = [int(c) for c in cand]
    K = _n_verify(len(cand), n_verify)
    p = f64(p)
    t = [match_target_token(p[j], seed, pos, request, j) for j in range(K + 1)]
    A = 0
    while A < K and cand[A] == t[A]:
        A += 1
    tok = t[A]
    return dict(A=A, commits=cand[:A] + [tok], n_commit=A + 1, next_anchor=tok, targets=t)


# ---------------------------------------------------------------- synthetic target

def synthetic_target_tokens(cand, c, seed, pos, request, V):
    """Target choices [K+1] of one request that stand in for the target model
    in the acceptance workloads.

    The acceptance model is the per-position conditional acceptance c_i of
    [P1] §"分布重叠怎样影响平均推进量" and of the DFlash page's prefix-survival
    formula P(A >= k) = prod_{i<=k} c_i: the target's choice at input index j
    (its choice for position j + 1) equals the candidate d_{j+1} with
    probability c_j, independently per position, and is otherwise a uniform
    id different from it; the choice at index K (the bonus position) is a
    uniform id.
    Draws: the words (w0, w1, w2, w3) of Philox(counter = (0, pos + j + 1,
    request, TAG_TARGET), key = seed). Agreement iff uniform_open(w0) < c_j
    (c_j a float32 value; both sides exact in float64). A disagreeing choice
    is (d_{j+1} + 1 + floor(w1 (V - 1) / 2^32)) mod V; the bonus choice is
    floor(w1 V / 2^32). Integer arithmetic throughout, so both sides agree
    bit for bit.
    """
    cand = [int(x) for x in cand]
    K = len(cand)
    c = np.asarray(c, dtype=np.float32).astype(np.float64)
    out = []
    for j in range(K + 1):
        w = _ph.words(seed, 0, pos + j + 1, request, _ph.TAG_TARGET)
        if j == K:
            out.append((int(w[1]) * V) >> 32)
            break
        if float(_ph.uniform_open(w[0])) < c[j]:
            out.append(cand[j])
        else:
            out.append((cand[j] + 1 + ((int(w[1]) * (V - 1)) >> 32)) % V)
    return out


# ---------------------------------------------------------------- batch drivers

def draft_round(hidden, anchor, W, cfg, temperature=0.0, seed=0, pos=None, mirror=False,
                requests=None):
    """Draft for each request b in `requests` (default: all rows of `hidden`)."""
    B = len(anchor)
    pos = np.zeros(B, dtype=np.int64) if pos is None else np.asarray(pos)
    reqs = range(B) if requests is None else requests
    return {b: draft_request(hidden[b], anchor[b], W, cfg, temperature, seed, int(pos[b]), b, mirror)
            for b in reqs}


# ---------------------------------------------------------------- cost model

def draft_kv_bytes(L_D, H, n_kv, d_h, bytes_per_elem):
    """History draft-KV size M = 2 L_D H n_kv d_h b ([P1] §"本轮临时 K/V 仍然需要计算")."""
    return 2 * L_D * H * n_kv * d_h * bytes_per_elem
