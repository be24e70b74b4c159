"""Seeded synthetic workloads for the DLite round (shapes, weights, inputs).

This module draws random numbers and nothing else: it holds none of the
method's arithmetic. Both the CUDA path (through the tests and the bench) and
the CPU oracle (through the tests) take their inputs from here.

Shapes follow the drafters the method is evaluated with: Qwen3-4B- and
Qwen3-8B-shaped drafters with K = 7 draft positions, 12-14 selected target
layers, a 3-layer backbone and a low-rank sequential head (rank 320 / 512),
plus a tiny fp32 configuration for exhaustive checks.
"""
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class DraftConfig:
    name: str
    D: int          # hidden width (drafter = target width)
    m: int          # selected target layers (context slots)
    K: int          # draft positions (block = anchor + K placeholders)
    L_D: int        # backbone layers
    n_q: int        # query heads
    n_kv: int       # key/value heads
    d_h: int        # head width
    F: int          # SwiGLU inner width
    R: int          # sequential-head rank
    V: int          # vocabulary
    dtype: str      # "f32" or "bf16" (weights, hidden inputs)
    eps: float = 1e-6
    theta: float = 1e6
    G: int = 1      # local token group ending at the anchor (local positions 0..G-1)
    head: str = "rnn"   # "rnn": low-rank RNN head + tied D->V projection; "gated": token-feedback head
    history: int = 0    # H > 0: history-KV control (a ring of the last H draft K/V rows per layer)
    act_planes: int = 1  # bf16 drafters: 1 = bf16 activations; 2 = fp32-class (two bf16 planes)
    warmup: int = 0     # gated head: warm the state up on the token before the anchor (needs G >= 2)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def n_params(self):
        D, F, R, V = self.D, self.F, self.R, self.V
        qkv = (self.n_q + 2 * self.n_kv) * self.d_h * D
        per_layer = qkv + D * self.n_q * self.d_h + 3 * D * F + 2 * D
        return (self.L_D * per_layer + self.m * D + 3 * D + V * D + 2 * D * R + D * R)


TINY = DraftConfig("tiny-fp32", D=256, m=4, K=4, L_D=1, n_q=4, n_kv=2, d_h=64, F=768,
                   R=32, V=2048, dtype="f32")
QWEN3_4B = DraftConfig("qwen3-4b-shape", D=2560, m=12, K=7, L_D=3, n_q=32, n_kv=8, d_h=128,
                       F=9728, R=320, V=151936, dtype="bf16")
QWEN3_8B = DraftConfig("qwen3-8b-shape", D=4096, m=14, K=7, L_D=3, n_q=32, n_kv=8, d_h=128,
                       F=12288, R=512, V=151936, dtype="bf16")


@dataclass(frozen=True)
class Workload:
    """A named workload: drafter shape, batch, verification mode, seeds."""
    name: str
    cfg: DraftConfig
    B: int
    temperature: float
    index: int                 # seeds are 1234/1235/1236 + 100 * index
    accept_c: float = 0.0      # greedy: per-position agreement probability
    scaled_hidden: bool = True
    accept_classes: bool = False   # greedy: two request classes, c ~ Beta(6, 4) / Beta(18, 2)

    @property
    def weight_seed(self):
        return 1234 + 100 * self.index

    @property
    def input_seed(self):
        return 1235 + 100 * self.index

    @property
    def rng_seed(self):
        return 1236 + 100 * self.index


WORKLOADS = {
    "tiny": Workload("tiny-fp32-b4-greedy", TINY, B=4, temperature=0.0, index=0,
                     accept_c=0.8, scaled_hidden=False),
    "qwen3-4b-b1": Workload("qwen3-4b-shape-b1-greedy", QWEN3_4B, B=1, temperature=0.0,
                            index=1, accept_c=0.85),
    "qwen3-8b-b32": Workload("qwen3-8b-shape-b32-sample-t0.7", QWEN3_8B, B=32,
                             temperature=0.7, index=2),
    "qwen3-8b-sweep": Workload("qwen3-8b-shape-sweep", QWEN3_8B, B=64, temperature=0.0,
                               index=3, accept_classes=True),
    "qwen3-8b-history": Workload("qwen3-8b-shape-b8-history-control", QWEN3_8B, B=8,
                                 temperature=0.0, index=4, accept_classes=True),
}

SWEEP_BATCHES = (1, 2, 4, 8, 16, 32, 64)


def shrink(cfg, **kw):
    """A smaller drafter of the same family (used for fast parity cases)."""
    return replace(cfg, **kw)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


WEIGHT_STD = 0.02


def make_weights(cfg, seed, device="cpu", gain_jitter=False):
    """All matrices and embeddings ~ N(0, 0.02^2); RMSNorm gains 1.0.

    gain_jitter=True draws the gains from U[0.5, 1.5] instead (used to prove
    the gains are applied). Matrices are stored nn.Linear-style, W[out, in].
    Q is the [R, 2D] matrix acting on [b; h]; P is [D, R].
    """
    g = _gen(seed, device)
    dt = cfg.torch_dtype
    D, F, R, V = cfg.D, cfg.F, cfg.R, cfg.V
    qd, kvd = cfg.n_q * cfg.d_h, cfg.n_kv * cfg.d_h

    def mat(*shape):
        return (torch.randn(*shape, generator=g, device=device) * WEIGHT_STD).to(dt)

    def gain():
        if gain_jitter:
            return (0.5 + torch.rand(D, generator=g, device=device)).to(dt)
        return torch.ones(D, device=device, dtype=dt)

    W = {
        "e_depth": mat(cfg.m, D),
        "g_stage": gain(),
        "e_ph": mat(D),
        "E": mat(V, D),
        "layers": [],
    }
    for _ in range(cfg.L_D):
        W["layers"].append({
            "g_attn": gain(),
            "Wq": mat(qd, D), "Wk": mat(kvd, D), "Wv": mat(kvd, D), "Wo": mat(D, qd),
            "g_ffn": gain(),
            "Wg": mat(F, D), "Wu": mat(F, D), "Wd": mat(D, F),
        })
    W["g_final"] = gain()
    W["Q"] = mat(R, 2 * D)
    W["P"] = mat(D, R)
    if cfg.head == "gated":   # the token-feedback head: E_R [V, R], W_s [2R, 2R], W_h [R, R + D], W_o [V, R]
        W["E_R"] = mat(V, R)
        W["W_s"] = mat(2 * R, 2 * R)
        W["b_s"] = mat(2 * R)
        W["W_h"] = mat(R, R + D)
        W["b_h"] = mat(R)
        W["W_o"] = mat(V, R)
    return W


def weights_to(W, device):
    out = {k: v.to(device) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: v.to(device) for k, v in l.items()} for l in W["layers"]]
    return out


def make_round_inputs(wl, B=None, round_index=0, device="cpu", cfg=None):
    """Pivot hidden states [B, m, D], anchors [B] (int32), RNG positions [B] (int64).

    hidden: N(0,1), scaled per selected layer by s_j ~ U[0.5, 4] (the scales are
    fixed per workload seed) when wl.scaled_hidden; anchors uniform in [0, V).
    """
    cfg = cfg or wl.cfg
    B = wl.B if B is None else B
    gs = _gen(wl.input_seed, "cpu")
    scales = 0.5 + 3.5 * torch.rand(cfg.m, generator=gs)
    g = _gen(wl.input_seed * 1000003 + round_index, device)
    hidden = torch.randn(B, cfg.m, cfg.D, generator=g, device=device)
    if wl.scaled_hidden:
        hidden = hidden * scales.to(device)[None, :, None]
    anchor = torch.randint(0, cfg.V, (B,), generator=g, device=device, dtype=torch.int64)
    pos = torch.randint(0, 1 << 20, (B,), generator=g, device=device, dtype=torch.int64)
    return hidden.to(cfg.torch_dtype), anchor.to(torch.int32), pos


def make_target_tokens(ref_cand, accept_p, V, seed, device="cpu"):
    """Synthetic target choices [B, K+1] for greedy verification.

    Position j < K agrees with ref_cand[:, j] with probability accept_p[:, j]
    (scalar or [B, K]), otherwise it is a uniform id different from it; the
    bonus position K is a uniform id.
    """
    ref = torch.as_tensor(ref_cand, device=device).to(torch.int64)
    B, K = ref.shape
    g = _gen(seed, device)
    p = torch.as_tensor(accept_p, dtype=torch.float64, device=device)
    p = p.expand(B, K) if p.dim() else p.new_full((B, K), float(p))
    agree = torch.rand(B, K, generator=g, device=device, dtype=torch.float64) < p
    other = (ref + 1 + torch.randint(0, V - 1, (B, K), generator=g, device=device)) % V
    tgt = torch.empty(B, K + 1, dtype=torch.int64, device=device)
    tgt[:, :K] = torch.where(agree, ref, other)
    tgt[:, K] = torch.randint(0, V, (B,), generator=g, device=device)
    return tgt.to(torch.int32)


def make_beta_accept(B, K, seed, device="cpu", n_tables=None):
    """Per-position agreement probabilities for the two-class sweep.

    Even requests: c ~ Beta(6, 4) (agentic-like); odd: c ~ Beta(18, 2)
    (structured-output-like); drawn iid per (table, request, position). With
    n_tables the result is [n_tables, B, K] (one table per round, cycled by the
    synthetic target's round counter), else [B, K]. float64.
    """
    rng = np.random.default_rng(int(seed))
    n = 1 if n_tables is None else int(n_tables)
    a = np.array([6.0 if b % 2 == 0 else 18.0 for b in range(B)])[None, :, None] * np.ones((n, 1, K))
    bb = np.array([4.0 if b % 2 == 0 else 2.0 for b in range(B)])[None, :, None] * np.ones((n, 1, K))
    c = torch.from_numpy(rng.beta(a, bb)).to(device)
    return c if n_tables is not None else c[0]


def make_const_accept(B, K, c, n_tables=1, device="cpu"):
    """A constant agreement probability c for every (table, request, position): [n_tables, B, K]."""
    return torch.full((n_tables, B, K), float(c), dtype=torch.float64, device=device)


def make_target_probs(B, K, V, seed, device="cpu", support=64, logit_std=3.0, tail=1e-3,
                      force=None):
    """Target distributions p [B, K+1, V] (float32, rows sum to 1).

    Each row: a support of `support` ids drawn uniformly without replacement,
    softmax of N(0, logit_std^2) logits on it scaled by (1 - tail), and the
    mass `tail` spread evenly over the other V - support ids. `force` [B, K]
    optionally puts ids into the support of rows 0..K-1 (statistical tests).
    """
    g = _gen(seed, device)
    rows = B * (K + 1)
    keys = torch.rand(rows, V, generator=g, device=device)
    if force is not None:
        f = torch.as_tensor(force, device=device).to(torch.int64)
        idx = torch.arange(B, device=device)[:, None] * (K + 1) + torch.arange(K, device=device)[None, :]
        keys[idx.reshape(-1), f.reshape(-1)] = 2.0
    sup = keys.topk(support, dim=1).indices
    logits = torch.randn(rows, support, generator=g, device=device) * logit_std
    p = torch.full((rows, V), tail / (V - support), device=device, dtype=torch.float64)
    p.scatter_(1, sup, (1.0 - tail) * torch.softmax(logits.double(), dim=1))
    p = p / p.sum(dim=1, keepdim=True)
    return p.to(torch.float32).reshape(B, K + 1, V)
