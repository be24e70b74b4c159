"""Round-level cost model and roofline arithmetic used by the bench.

Time model of one speculative round ([P1] "DLite 完全拆解", §"先拆开一次投机
轮次的时间"): a round costs T_D + T_V + T_S and commits tau = E[A + 1] tokens
on average, so T_token ~ (T_D + T_V + T_S) / tau and the speed-up over plain
autoregressive decoding is S ~ T_AR * tau / (T_D + T_V + T_S).
Workflow-level Amdahl form ([P1] §"哪些请求更可能受益"):
S_workflow = 1 / ((1 - f) + f / S_D).
"""


def time_per_token(t_draft, t_verify, t_state, tau):
    return (t_draft + t_verify + t_state) / tau


def speedup(t_ar, tau, t_round):
    """S ~ T_AR * tau / T_round with T_round = T_D + T_V + T_S."""
    return t_ar * tau / t_round


def relative_rate(s_a, s_b):
    """Rate of method a relative to method b, both quoted as speed-ups over the same baseline."""
    return s_a / s_b


def time_saved(rate):
    """Fraction of decode time saved when running `rate` times faster: 1 - 1/rate."""
    return 1.0 - 1.0 / rate


def workflow_speedup(f, s_d):
    return 1.0 / ((1.0 - f) + f / s_d)


def expected_advance(p_ge):
    """E[A+1] = 1 + sum_{j=1..K} Pr(A >= j) ([P1] §"分布重叠怎样影响平均推进量")."""
    return 1.0 + sum(p_ge)


def prefix_survival(c):
    """P(A >= k) = prod_{i<=k} c_i for per-position conditional acceptance c_i."""
    out, acc = [], 1.0
    for ci in c:
        acc *= ci
        out.append(acc)
    return out


# ---------------------------------------------------------------- byte / flop accounting

def round_bytes(cfg, B):
    """Algorithmic HBM bytes of one draft+verify round over B requests.

    Every weight read once (weight element size from cfg.dtype), the pivot
    hidden states read once, plus the small per-round I/O (anchors, candidates,
    commits). Target probabilities for sampling verification are counted by
    the caller (they are an input of verification, read only where needed).
    """
    wb = 4 if cfg.dtype == "f32" else 2
    D, F, R, V = cfg.D, cfg.F, cfg.R, cfg.V
    qkv = (cfg.n_q + 2 * cfg.n_kv) * cfg.d_h * D
    layer = qkv + D * cfg.n_q * cfg.d_h + 3 * D * F
    weights = cfg.L_D * layer + 2 * D * R + D * R + V * D
    small = (cfg.m * D + cfg.L_D * 2 * D + 3 * D) * wb
    hidden = B * cfg.m * D * wb
    io = B * (4 + 4 * cfg.K * 2 + 4 * (cfg.K + 1) + 16)
    return weights * wb + small + hidden + io + history_bytes(cfg, B)


def history_bytes(cfg, B):
    """History-KV control: per layer every ring read once (bf16 keys and values)
    and the round's G + K rows written into it; 0 for the history-free drafter."""
    H = getattr(cfg, "history", 0)
    if not H:
        return 0
    K1 = getattr(cfg, "G", 1) + cfg.K
    return cfg.L_D * B * cfg.n_kv * cfg.d_h * 2 * 2 * (H + K1)


def hist_attn_bytes(cfg, B):
    """One launch of the history attention (one layer): the ring and the block's
    keys / values read once, the block's queries read once (bf16)."""
    K1 = getattr(cfg, "G", 1) + cfg.K
    Tk = cfg.m + K1
    QR = cfg.n_q // cfg.n_kv * K1
    return B * cfg.n_kv * cfg.d_h * 2 * (2 * (cfg.history + Tk) + QR)


def round_flops(cfg, B):
    """2 * rows * in * out over the round's GEMMs plus attention and the RNN chain."""
    D, F, R, V, K, m = cfg.D, cfg.F, cfg.R, cfg.V, cfg.K, cfg.m
    qd, kvd = cfg.n_q * cfg.d_h, cfg.n_kv * cfg.d_h
    loc = B * (K + 1)
    ctx = B * m
    per_layer = 2 * loc * D * (qd + 2 * kvd) + 2 * ctx * D * 2 * kvd \
        + 2 * loc * qd * D + 2 * loc * D * 2 * F + 2 * loc * F * D
    attn = 2 * 2 * loc * cfg.n_q * (m + K + 1) * cfg.d_h
    head = 2 * B * K * D * 2 * R + 2 * B * K * R * R + 2 * B * K * R * D
    lm = 2 * B * K * D * V
    hist = 2 * 2 * B * cfg.n_q * (getattr(cfg, "G", 1) + K) * getattr(cfg, "history", 0) * cfg.d_h
    return cfg.L_D * (per_layer + attn + hist) + head + lm


def lm_head_bytes(cfg, B):
    wb = 4 if cfg.dtype == "f32" else 2
    return cfg.V * cfg.D * wb + B * cfg.K * cfg.D * 4


def lm_head_flops(cfg, B):
    return 2 * B * cfg.K * cfg.D * cfg.V


def gated_lm_bytes(cfg, B):
    """One step's vocabulary projection of the gated head: W_o [V, R] once, r [B, R] (bf16)."""
    wb = 4 if cfg.dtype == "f32" else 2
    return cfg.V * cfg.R * wb + B * cfg.R * 2


def gated_lm_flops(cfg, B):
    return 2 * B * cfg.R * cfg.V


def roofline_floor_s(nbytes, flops, hbm_gbs, tflops):
    return max(nbytes / (hbm_gbs * 1e9), flops / (tflops * 1e12))
