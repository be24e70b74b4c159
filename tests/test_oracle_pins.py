"""Pins of the CPU oracle against facts fixed outside itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, an off-by-one index) fails at least one:
published known-answer vectors, closed forms, library routines on special
cases, brute force on tiny inputs, and distributional identities checked by
Monte Carlo.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import dlite_oracle as O
from oracle import philox as ph
from history_free_speculative_gb300 import workload as wk
from history_free_speculative_gb300 import reporter as rp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.strip() for l in f if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------- RNG

def test_philox_known_answers():
    for line in _golden_lines("philox4x32_10_kat.txt"):
        lhs, rhs = line.split("->")
        c0, c1, c2, c3, k0, k1 = (int(t, 16) for t in lhs.split())
        want = [int(t, 16) for t in rhs.split()]
        got = ph.philox4x32_10(c0, c1, c2, c3, k0, k1)
        assert [int(g) for g in got] == want


def test_uniform_open_interval_and_exact_in_fp32():
    x = np.array([0, 1, 511, 512, 0x7FFFFFFF, 0xFFFFFFFF], dtype=np.uint64)
    u = ph.uniform_open(x)
    assert u[0] == 0.5 * 2.0 ** -23 and u[-1] == 1.0 - 0.5 * 2.0 ** -23
    assert np.all((u > 0) & (u < 1))
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_gumbel_max_matches_softmax():
    """Gumbel-max over l/T draws from softmax(l/T): chi-square over 8 ids."""
    rng = np.random.default_rng(0)
    V, T, N = 8, 0.7, 30000
    ell = rng.normal(0, 1.0, V)
    counts = np.zeros(V)
    for n in range(N):
        s = ell / T + ph.gumbel_row(77, n, 3, V)
        counts[np.argmax(s)] += 1
    p = np.exp(ell / T - ell.max() / T)
    p /= p.sum()
    chi2 = ((counts - N * p) ** 2 / (N * p)).sum()
    assert chi2 < 30.0          # 7 dof; P(chi2 > 30) ~ 1e-4


def test_two_level_draw_matches_softmax():
    """The draft's sampling draw (chunk Gumbel-max on the chunks' log-mass, then
    the inverse CDF inside the chosen chunk) follows softmax(l / T): chi-square
    over 40 ids (chunks of 16, 16 and a partial 8)."""
    rng = np.random.default_rng(1)
    V, T, N = 40, 0.7, 40000
    ell = rng.normal(0, 1.0, V)
    counts = np.zeros(V)
    for n in range(N):
        counts[O.sample_logits(ell, T, 77, n, 3)[0]] += 1
    p = np.exp(ell / T - ell.max() / T)
    p /= p.sum()
    chi2 = ((counts - N * p) ** 2 / (N * p)).sum()
    assert chi2 < 92.0          # 39 dof: mean 39, sd 8.8; P(chi2 > 92) < 1e-6


def test_two_level_draw_single_chunk_is_the_inverse_cdf():
    """With V <= 16 there is one chunk: the draw is the inverse CDF of
    softmax(l / T) at word 0 of Philox(0, position, request, TAG_PICK)."""
    rng = np.random.default_rng(2)
    ell = rng.normal(0, 1.0, 12)
    q = np.exp(ell / 0.7 - ell.max() / 0.7)
    q /= q.sum()
    for pos in range(200):
        u = float(ph.draw(5, 0, pos, 4, ph.TAG_PICK, 0))
        want = int(np.searchsorted(np.cumsum(q), u, side="right"))
        assert O.sample_logits(ell, 0.7, 5, pos, 4)[0] == want


def test_two_level_draw_follows_the_chunk_mass():
    """All mass in chunk 2 (ids 32..47): every draw lands there, with the
    within-chunk frequencies of softmax; T = 0 is the plain argmax."""
    rng = np.random.default_rng(3)
    ell = np.full(64, -1e3)
    ell[32:48] = rng.normal(0, 1.0, 16)
    counts = np.zeros(64)
    N = 8000
    for n in range(N):
        counts[O.sample_logits(ell, 0.7, 9, n, 0)[0]] += 1
    assert counts[:32].sum() == 0 and counts[48:].sum() == 0
    p = np.exp(ell[32:48] / 0.7 - ell[32:48].max() / 0.7)
    p /= p.sum()
    chi2 = ((counts[32:48] - N * p) ** 2 / (N * p)).sum()
    assert chi2 < 60.0          # 15 dof
    assert O.sample_logits(ell, 0.0, 9, 0, 0)[0] == 32 + int(np.argmax(ell[32:48]))


def test_draws_are_keyed_by_seed_request_position_tag():
    base = ph.draw(5, 0, 10, 2, ph.TAG_ACCEPT, 0)
    for args in [(6, 0, 10, 2, ph.TAG_ACCEPT), (5, 1, 10, 2, ph.TAG_ACCEPT),
                 (5, 0, 11, 2, ph.TAG_ACCEPT), (5, 0, 10, 3, ph.TAG_ACCEPT),
                 (5, 0, 10, 2, ph.TAG_RESID)]:
        assert ph.draw(*args, 0) != base
    assert ph.draw(5, 0, 10, 2, ph.TAG_ACCEPT, 0) == base


# ---------------------------------------------------------------- precision helper

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 1, 10000), rng.normal(0, 1e-3, 1000), rng.normal(0, 1e4, 1000)])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_round(x32), want)


# ---------------------------------------------------------------- building blocks

def test_rmsnorm_closed_form():
    y = O.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [3 / r, 8 / r], rtol=0, atol=1e-15)
    x = np.random.default_rng(2).normal(0, 5, (6, 64))
    y = O.rmsnorm(x, np.full(64, 1.5), 0.0)
    assert np.allclose(np.sqrt((y ** 2).mean(axis=1)), 1.5, atol=1e-12)


def test_rope_is_complex_rotation_and_identity_at_zero():
    rng = np.random.default_rng(3)
    d, theta = 16, 1e6
    x = rng.normal(size=(5, 2, d))
    pos = np.arange(5)
    y = O.rope_rotate_half(x, pos, theta)
    assert np.array_equal(y[0], x[0])                      # position 0 = identity
    # independent statement: (x_j + i x_{j+d/2}) * exp(i * pos * theta^(-2j/d))
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = theta ** (-2.0 * np.arange(half) / d)
    w = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    assert np.allclose(y[..., :half], w.real, atol=1e-12)
    assert np.allclose(y[..., half:], w.imag, atol=1e-12)


def test_attention_matches_sdpa_library():
    rng = np.random.default_rng(4)
    n_q, n_kv, d = 8, 2, 32
    q = rng.normal(size=(5, n_q, d))
    k = rng.normal(size=(9, n_kv, d))
    v = rng.normal(size=(9, n_kv, d))
    got = O.block_attention(q, k, v, n_q, n_kv)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).repeat_interleave(n_q // n_kv, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).repeat_interleave(n_q // n_kv, dim=1).permute(1, 0, 2)[None]
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)
    want = want[0].permute(1, 0, 2).reshape(5, n_q * d).numpy()
    assert np.allclose(got, want, atol=1e-12)


def test_attention_zero_query_is_mean_of_values():
    rng = np.random.default_rng(5)
    v = rng.normal(size=(7, 1, 4))
    o = O.block_attention(np.zeros((3, 2, 4)), rng.normal(size=(7, 1, 4)), v, 2, 1)
    assert np.allclose(o.reshape(3, 2, 4), v.mean(axis=0)[None], atol=1e-14)


# ---------------------------------------------------------------- drafter structure

def _tiny(**kw):
    return wk.shrink(wk.TINY, **kw)


def _weights(cfg, seed=11, jitter=False):
    W = wk.make_weights(cfg, seed, gain_jitter=jitter)
    return W


def test_layer_is_residual():
    cfg = _tiny()
    W = _weights(cfg)
    Wl = dict(W["layers"][0])
    Wl["Wo"] = torch.zeros_like(Wl["Wo"])
    Wl["Wd"] = torch.zeros_like(Wl["Wd"])
    rng = np.random.default_rng(6)
    x = rng.normal(size=(cfg.K + 1, cfg.D))
    z = rng.normal(size=(cfg.m, cfg.D))
    assert np.array_equal(O.backbone_layer(x, z, Wl, cfg), x)


def test_context_slots_are_an_unordered_set():
    """Sequence-dim context slots all sit at local position 0: permuting
    (hidden_j, e_depth_j) pairs together cannot change the draft."""
    cfg = _tiny()
    W = _weights(cfg)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    perm = torch.tensor([2, 0, 3, 1])
    b0 = O.backbone(hidden[0], anchor[0], W, cfg)
    W2 = dict(W)
    W2["e_depth"] = W["e_depth"][perm]
    b1 = O.backbone(hidden[0][perm], anchor[0], W2, cfg)
    assert np.allclose(b0, b1, atol=1e-12)
    # ... while moving one slot's feature to another depth does change it
    hid3 = hidden[0].clone()
    hid3[[0, 1]] = hid3[[1, 0]]
    b3 = O.backbone(hid3, anchor[0], W, cfg)
    assert np.abs(b3 - b0).max() > 1e-3


def test_block_attention_is_non_causal():
    """The anchor row (position 0) sees the placeholders: changing e_ph moves it."""
    cfg = _tiny()
    W = _weights(cfg)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    z, x = O.stage(hidden[0], anchor[0], W, cfg)
    x_a = O.backbone_layer(x, z, W["layers"][0], cfg)
    W2 = dict(W)
    W2["e_ph"] = W["e_ph"] * 3.0
    z2, x2 = O.stage(hidden[0], anchor[0], W2, cfg)
    x_b = O.backbone_layer(x2, z2, W["layers"][0], cfg)
    assert np.array_equal(x[0], x2[0])
    assert np.abs(x_a[0] - x_b[0]).max() > 1e-4


def test_gains_are_applied():
    cfg = _tiny()
    Wj = _weights(cfg, jitter=True)
    W1 = _weights(cfg, jitter=False)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    b_j = O.backbone(hidden[0], anchor[0], Wj, cfg)
    b_1 = O.backbone(hidden[0], anchor[0], W1, cfg)
    g = O.f64(Wj["g_final"])
    # b / g_final is the plain normalised stream: unit RMS up to the eps term
    assert np.allclose(np.sqrt(((b_j / g) ** 2).mean(axis=1)), 1.0, atol=1e-3)
    assert np.abs(b_j - b_1).max() > 0.05


def test_staging_closed_form():
    cfg = _tiny()
    W = _weights(cfg, jitter=True)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    z, x = O.stage(hidden[0], anchor[0], W, cfg)
    s = O.f64(hidden[0]) + O.f64(W["e_depth"])
    j = 2
    want = O.f64(W["g_stage"]) * s[j] / math.sqrt(float(np.dot(s[j], s[j])) / cfg.D + cfg.eps)
    assert np.allclose(z[j], want, atol=1e-12)
    assert np.array_equal(x[0], O.f64(W["E"][int(anchor[0])]))
    assert all(np.array_equal(x[i], O.f64(W["e_ph"])) for i in range(1, cfg.K + 1))


# ---------------------------------------------------------------- local token group

def test_group_staging_layout():
    """G tokens ending at the anchor fill the first G local rows (tied E rows),
    the K placeholders follow; G = 1 with a list equals the scalar anchor."""
    cfg = _tiny(G=3)
    W = _weights(cfg)
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    group = [5, 17, 3]
    z, x = O.stage(hidden[0], group, W, cfg)
    assert x.shape == (cfg.G + cfg.K, cfg.D)
    for i, t in enumerate(group):
        assert np.array_equal(x[i], O.f64(W["E"][t]))
    assert all(np.array_equal(x[i], O.f64(W["e_ph"])) for i in range(cfg.G, cfg.G + cfg.K))
    c1 = _tiny()
    W1 = _weights(c1)
    assert np.array_equal(O.backbone(hidden[0], [7], W1, c1), O.backbone(hidden[0], 7, W1, c1))
    with pytest.raises(ValueError):
        O.stage(hidden[0], [1, 2], W, cfg)


def test_group_positions_follow_the_group():
    """Local rows that enter with identical inputs differ only by their RoPE
    positions. With every group token's embedding equal to e_ph, a G = 2 block
    of K = 3 placeholders and a G = 1 block of K = 4 placeholders hold the same
    5 identical rows at positions 0..4, so the last three outputs agree; a
    slip in the positions (placeholders restarting at 1, say) breaks this."""
    c2, c1 = _tiny(G=2, K=3), _tiny(G=1, K=4)
    W = _weights(c2)
    W = dict(W)
    E = W["E"].clone()
    E[[11, 12]] = W["e_ph"]
    W["E"] = E
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    b2 = O.backbone(hidden[0], [11, 12], W, c2)
    b1 = O.backbone(hidden[0], 11, W, c1)
    assert np.allclose(b2, b1[1:], rtol=0, atol=1e-12)
    assert not np.allclose(b1[0], b1[1], atol=1e-6)        # positions do matter


def test_group_zero_blocks_closed_form_and_dependence():
    """With zero output projections (Wo = Wd = 0) the residual stream keeps its
    staged rows, so every placeholder's b is RMSNorm(e_ph) g_final whatever the
    group; with the real weights the group's first token changes the outputs."""
    cfg = _tiny(G=2)
    W = _weights(cfg, jitter=True)
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    Wz = dict(W)
    Wz["layers"] = [dict(l, Wo=np.zeros_like(l["Wo"]), Wd=np.zeros_like(l["Wd"])) for l in W["layers"]]
    e = O.f64(W["e_ph"])
    want = O.f64(W["g_final"]) * e / math.sqrt(float(e @ e) / cfg.D + cfg.eps)
    for group in ([1, 2], [300, 9]):
        b = O.backbone(hidden[0], group, Wz, cfg)
        assert np.allclose(b, want[None, :], atol=1e-12)
    assert not np.allclose(O.backbone(hidden[0], [1, 2], W, cfg), O.backbone(hidden[0], [3, 2], W, cfg))


def test_next_group_is_the_most_recent_tokens():
    """G = 1: the next group is the verification's next anchor; generally the
    last G tokens of the group followed by the commits (brute force)."""
    rng = np.random.default_rng(41)
    for _ in range(200):
        G = int(rng.integers(1, 6))
        group = [int(t) for t in rng.integers(0, 100, G)]
        n = int(rng.integers(1, 9))
        commits = [int(t) for t in rng.integers(100, 200, n)]
        ng = O.next_group(group, commits)
        assert len(ng) == G and ng[-1] == commits[-1]
        full = group + commits
        assert ng == full[len(full) - G:]
    r = O.verify_greedy([1, 2, 3], [1, 2, 9, 4])
    assert O.next_group([5], r["commits"]) == [r["next_anchor"]]


# ---------------------------------------------------------------- gated token-feedback head

def _gated_setup(seed=5, V=64, R=16, D=32, K=5):
    rng = np.random.default_rng(seed)
    W = {"E_R": rng.normal(0, 0.5, (V, R)), "W_s": rng.normal(0, 0.3, (2 * R, 2 * R)),
         "b_s": rng.normal(0, 0.3, 2 * R), "W_h": rng.normal(0, 0.3, (R, R + D)),
         "b_h": rng.normal(0, 0.3, R), "W_o": rng.normal(0, 0.5, (V, R))}
    u = rng.normal(0, 1.0, (K, D))
    return W, u, R


def test_gated_head_saturated_gate_ignores_feedback():
    """f = sigmoid(g) -> 1 (large gate bias): the state stays at s_0 = 0, so
    r_i = W_h[:, R:] u_i + b_h and l_i = W_o r_i whatever the tokens fed back."""
    W, u, R = _gated_setup()
    W["b_s"] = W["b_s"].copy()
    W["b_s"][:R] = 60.0
    want_r = u @ W["W_h"][:, R:].T + W["b_h"]
    for anchor in (0, 17, 63):
        out = O.gated_head(u, anchor, W)
        assert np.allclose(out["r"], want_r, atol=1e-12)
        assert np.allclose(out["logits"], want_r @ W["W_o"].T, atol=1e-12)
        assert list(out["cand"]) == list(np.argmax(want_r @ W["W_o"].T, axis=1))


def test_gated_head_open_gate_reads_the_previous_token():
    """f -> 0 and no state-to-candidate weights: s_i = tanh(W_s[R:, R:] E_R[d_{i-1}]
    + b_s[R:]), so each step depends on the previous token only (d_0 = anchor);
    swapping the g / c halves, feeding d_i instead of d_{i-1} or the [s; u]
    order of W_h would all break this."""
    W, u, R = _gated_setup(6)
    W["b_s"] = W["b_s"].copy()
    W["b_s"][:R] = -60.0
    W["W_s"] = W["W_s"].copy()
    W["W_s"][R:, :R] = 0.0
    anchor = 9
    out = O.gated_head(u, anchor, W)
    prev = anchor
    for i in range(u.shape[0]):
        s_i = np.tanh(W["W_s"][R:, R:] @ W["E_R"][prev] + W["b_s"][R:])
        r = W["W_h"][:, :R] @ s_i + W["W_h"][:, R:] @ u[i] + W["b_h"]
        assert np.allclose(out["r"][i], r, atol=1e-12)
        prev = int(out["cand"][i])
        assert prev == int(np.argmax(W["W_o"] @ r))
    other = O.gated_head(u, 10, W)
    assert not np.allclose(other["r"][0], out["r"][0])   # the anchor is fed back


def test_gated_head_warmup_saturated_gate_is_a_no_op():
    """Warm-up on the token before the anchor ([P1] §"官方顺序头具体算了什么"): with
    f -> 1 the warm-up step keeps the zero state (s_0 = 1 * 0 + 0 * tanh c), so
    the head's outputs equal those without warm-up, whatever the token."""
    W, u, R = _gated_setup(8)
    W["b_s"] = W["b_s"].copy()
    W["b_s"][:R] = 60.0
    base = O.gated_head(u, 5, W)
    for w in (0, 31, 63):
        out = O.gated_head(u, 5, W, warm_token=w)
        assert np.array_equal(out["r"], base["r"]) and list(out["cand"]) == list(base["cand"])


def test_gated_head_warmup_open_gate_closed_form():
    """With f -> 0 the warm-up state is s_0 = tanh(W_s^c [0; E_R(w)] + b_s^c) (c the
    last R outputs of W_s); step 1 then updates from s_0 on the anchor's
    embedding: s_1 = tanh(W_s^c [s_0; E_R(a)] + b_s^c), r_1 = W_h [s_1; u_1] + b_h.
    A warm-up that read the anchor, skipped the zero start, or fed its state to
    r (an output for the warm-up token) fails this."""
    W, u, R = _gated_setup(9)
    W["b_s"] = W["b_s"].copy()
    W["b_s"][:R] = -60.0
    a, w = 12, 40
    s0 = np.tanh(W["W_s"][R:, R:] @ W["E_R"][w] + W["b_s"][R:])
    s1 = np.tanh(W["W_s"][R:, :R] @ s0 + W["W_s"][R:, R:] @ W["E_R"][a] + W["b_s"][R:])
    r1 = W["W_h"][:, :R] @ s1 + W["W_h"][:, R:] @ u[0] + W["b_h"]
    out = O.gated_head(u, a, W, warm_token=w)
    assert np.allclose(out["r"][0], r1, atol=1e-12)
    assert out["r"].shape[0] == u.shape[0]                       # K outputs, none for the warm-up
    assert not np.allclose(O.gated_head(u, a, W, warm_token=w + 1)["r"][0], r1)   # the token matters


def test_draft_warmup_takes_the_token_before_the_anchor():
    """In a drafted round the warm-up token is the group's second-to-last token."""
    cfg = _tiny(G=3, head="gated", warmup=1, R=64)
    W = _weights(cfg, seed=13)
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1, cfg=cfg)
    group = [7, 21, 9]
    r = O.draft_request(hidden[0], group, W, cfg)
    b = O.backbone(hidden[0], group, W, cfg)
    want = O.gated_head(b, 9, W, warm_token=21)
    assert list(r["cand"]) == list(want["cand"]) and np.allclose(r["h"], want["r"], atol=1e-12)


def test_gated_head_sampling_follows_softmax():
    """T > 0: the first candidate is a draw from softmax(l_1 / T) (chi-square
    over positions), and lse is the log-sum-exp of l_1 / T."""
    W, u, R = _gated_setup(7, V=8)
    T, N = 0.8, 12000
    ell = O.gated_head(u, 3, W)["logits"][0]
    p = np.exp(ell / np.float32(T) - (ell / np.float32(T)).max())
    p /= p.sum()
    counts = np.zeros(8)
    for n in range(N):
        out = O.gated_head(u[:1], 3, W, temperature=T, seed=2, pos=10 * n, request=1)
        counts[out["cand"][0]] += 1
    chi2 = ((counts - N * p) ** 2 / (N * p)).sum()
    assert chi2 < 30.0                                    # 7 dof
    want = float(torch.logsumexp(torch.tensor(ell / float(np.float32(T))), 0))
    assert abs(out["lse"][0] - want) < 1e-9


# ---------------------------------------------------------------- history-KV control

def test_history_values_statistics_and_keying():
    """Synthetic history: bf16 values with mean 0, variance 1 (a sum of four
    uniforms), different for every (layer, request, K/V) key."""
    a = O.history_values(512, 2, 64, 0, 0, 0)
    assert np.array_equal(a, O.bf16_round(a))
    assert abs(a.mean()) < 0.02 and abs(a.var() - 1.0) < 0.03
    assert abs(a.max()) <= 2 * math.sqrt(3.0) + 1e-6
    others = [O.history_values(512, 2, 64, 1, 0, 0), O.history_values(512, 2, 64, 0, 1, 0),
              O.history_values(512, 2, 64, 0, 0, 1)]
    for b in others:
        assert np.corrcoef(a.ravel(), b.ravel())[0, 1] < 0.05


def test_history_is_an_unordered_set_of_extra_keys():
    """The history rows are plain extra keys / values (no position): permuting
    the ring's slots changes nothing, while the history does change the round;
    and a zero-key history with constant values c mixes c in with weight
    H / (H + sum_j exp(s_j)) per query."""
    cfg = _tiny(L_D=1)
    W = _weights(cfg)
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    H = 40
    h1 = O.HistoryCache(cfg, H, 0)
    h2 = O.HistoryCache(cfg, H, 0)
    perm = np.random.default_rng(3).permutation(H)
    h2.k[0], h2.v[0] = h2.k[0][perm], h2.v[0][perm]
    b1 = O.backbone(hidden[0], 5, W, cfg, history=h1)
    b2 = O.backbone(hidden[0], 5, W, cfg, history=h2)
    assert np.allclose(b1, b2, atol=1e-12)
    assert not np.allclose(b1, O.backbone(hidden[0], 5, W, cfg), atol=1e-6)
    rng = np.random.default_rng(4)
    n_q, n_kv, d_h, T = 4, 2, 8, 6
    q, k, v = rng.normal(size=(3, n_q, d_h)), rng.normal(size=(T, n_kv, d_h)), rng.normal(size=(T, n_kv, d_h))
    c = rng.normal(size=(n_kv, d_h))
    kh = np.zeros((H, n_kv, d_h))
    vh = np.broadcast_to(c, (H, n_kv, d_h))
    got = O.block_attention(q, np.concatenate([kh, k]), np.concatenate([vh, v]), n_q, n_kv).reshape(3, n_q, d_h)
    base = O.block_attention(q, k, v, n_q, n_kv).reshape(3, n_q, d_h)
    for h in range(n_q):
        g = h // (n_q // n_kv)
        Z = np.exp(q[:, h] @ k[:, g].T / math.sqrt(d_h)).sum(axis=1)
        want = (base[:, h] * Z[:, None] + H * c[g][None, :]) / (Z + H)[:, None]
        assert np.allclose(got[:, h], want, atol=1e-12)


def test_history_ring_holds_the_last_rounds():
    """After each round the ring holds that round's local K/V rows at slots
    (cursor + j) mod H; older rows survive until overwritten."""
    cfg = _tiny(L_D=2)
    W = _weights(cfg)
    hidden, _, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    H, K1 = 12, cfg.K + 1
    hc = O.HistoryCache(cfg, H, 2)
    init_k1 = hc.k[1].copy()
    seen = []
    for rnd in range(4):
        local = []
        O.backbone(hidden[0], rnd + 1, W, cfg, history=hc, local_out=local)
        before = hc.cursor
        hc.append(local)
        seen.append((before, local))
    for rnd, (cur, local) in enumerate(seen):
        for j in range(K1):
            slot = (cur + j) % H
            newer = any(((slot - c2) % H) < K1 for c2, _ in seen[rnd + 1:])
            if not newer:
                assert np.array_equal(hc.k[1][slot], local[1][0][j])
                assert np.array_equal(hc.v[0][slot], local[0][1][j])
    untouched = set(range(H)) - {(c + j) % H for c, _ in seen for j in range(K1)}
    for slot in untouched:
        assert np.array_equal(hc.k[1][slot], init_k1[slot])
    assert hc.cursor == (4 * K1) % H


# ---------------------------------------------------------------- sequential head

def test_head_with_zero_P_is_identity():
    rng = np.random.default_rng(7)
    b = rng.normal(size=(5, 16))
    assert np.array_equal(O.sequential_head(b, rng.normal(size=(4, 32)), np.zeros((16, 4))), b)


def test_head_first_step_closed_form():
    """h_0 = 0 and the [b; h] order: h_1 = b_1 + P tanh(Q[:, :D] b_1)."""
    rng = np.random.default_rng(8)
    D, R = 16, 4
    b = rng.normal(size=(1, D))
    Q = rng.normal(size=(R, 2 * D)) * 0.3
    P = rng.normal(size=(D, R))
    h = O.sequential_head(b, Q, P)
    assert np.allclose(h[0], b[0] + P @ np.tanh(Q[:, :D] @ b[0]), atol=1e-14)


def test_head_low_rank_recurrence_identity():
    """Feeding back h_{i-1} = b_{i-1} + P t_{i-1} gives the R x R recurrence
    t_i = tanh(Q_b b_i + Q_h b_{i-1} + (Q_h P) t_{i-1}); the two forms agree."""
    rng = np.random.default_rng(9)
    D, R, K = 24, 6, 7
    b = rng.normal(size=(K, D))
    Q = rng.normal(size=(R, 2 * D)) * 0.2
    P = rng.normal(size=(D, R)) * 0.5
    Qb, Qh = Q[:, :D], Q[:, D:]
    M = Qh @ P
    t_prev = np.zeros(R)
    e_prev = np.zeros(R)
    want = np.empty_like(b)
    for i in range(K):
        t = np.tanh(Qb @ b[i] + e_prev + M @ t_prev)
        want[i] = b[i] + P @ t
        t_prev, e_prev = t, Qh @ b[i]
    assert np.allclose(O.sequential_head(b, Q, P), want, atol=1e-12)


# ---------------------------------------------------------------- LM head

def test_greedy_ties_go_to_lowest_id():
    cfg = _tiny(V=8, D=4, K=1)
    h = np.array([[1.0, 0.0, 0.0, 0.0]])
    E = np.zeros((8, 4))
    E[[2, 5, 6], 0] = 1.0
    ell = O.lm_logits(h, E)
    assert int(np.argmax(ell[0])) == 2


def test_lse_matches_library():
    from scipy.special import logsumexp
    cfg = _tiny()
    W = _weights(cfg)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    r = O.draft_request(hidden[0], anchor[0], W, cfg, temperature=0.7, seed=3, pos=5, request=0)
    ell = O.lm_logits(r["h"], W["E"])
    assert np.allclose(r["lse"], logsumexp(ell / 0.7, axis=1), atol=1e-12)
    assert np.allclose(r["logit_d"], ell[np.arange(cfg.K), r["cand"]], atol=0)


# ---------------------------------------------------------------- verification

def test_pages_prefix_example():
    for line in _golden_lines("pages_examples.txt"):
        if line.startswith("prefix_flags"):
            flags = [int(t) for t in line.split("->")[0].split()[1:]]
            want = int(line.split("->")[1].split()[1])
            cand = [7, 8, 9, 10]
            tgt = [c if f else c + 1 for c, f in zip(cand, flags)] + [99]
            r = O.verify_greedy(cand, tgt)
            assert r["A"] == want and r["n_commit"] == want + 1
            assert r["commits"] == cand[:want] + [tgt[want]] and r["next_anchor"] == tgt[want]
        if line.startswith("next_index"):
            A = int(line.split()[2])
            idx = int(line.split("->")[1])
            cand = [1, 2, 3, 4]
            tgt = [1, 2, 3, 4, 5]
            tgt[A] = 0 if A < 4 else tgt[A]
            r = O.verify_greedy(cand, tgt)
            assert r["A"] == A == idx


def test_greedy_prefix_brute_force_exhaustive():
    """All candidate/target pairs for V = 3, K = 3 against the cumprod rule."""
    import itertools
    V, K = 3, 3
    for cand in itertools.product(range(V), repeat=K):
        for tgt in itertools.product(range(V), repeat=K + 1):
            r = O.verify_greedy(cand, tgt)
            passes = np.array([cand[i] == tgt[i] for i in range(K)], dtype=np.int64)
            A = int(np.cumprod(passes).sum())
            assert r["A"] == A and 0 <= A <= K
            assert r["commits"] == list(cand[:A]) + [tgt[A]]


def _q_setup(V, ell):
    """E = I, h = l, so that E h = l exactly (D = V)."""
    E = np.eye(V)
    return E, np.asarray(ell, dtype=np.float64)


@pytest.mark.parametrize("case", ["disjoint", "overlapping"])
def test_speculative_sampling_preserves_target(case):
    """Committed token ~ p and first-position acceptance ~ sum_v min(p, q)."""
    rng = np.random.default_rng(12 if case == "disjoint" else 13)
    V, T, N = 6, 0.7, 12000
    ell = rng.normal(0, 1.0, V)
    E, h = _q_setup(V, ell)
    q = np.exp(ell / T - ell.max() / T)
    q /= q.sum()
    if case == "disjoint":
        p = rng.dirichlet(np.ones(V) * 0.5)
    else:                                  # p close to q: rejections rare, fallback exercised
        p = 0.93 * q + 0.07 * rng.dirichlet(np.ones(V))
    lse = float(np.log(np.exp(ell / T).sum()))
    counts = np.zeros(V)
    accepted = 0
    hows = {}
    for n in range(N):
        d = O.sample_logits(ell, T, 21, n + 1, 0)[0]
        pp = np.stack([p, np.full(V, 1.0 / V)])          # K = 1: row 0 verifies, row 1 bonus
        r = O.verify_sample([d], [ell[d]], [lse], h[None, :], E, pp, T, 21, n, 0)
        if r["A"] == 1:
            accepted += 1
            counts[d] += 1
        else:
            counts[r["commits"][0]] += 1
        hows[r["how"]] = hows.get(r["how"], 0) + 1
    beta = np.minimum(p, q).sum()
    assert abs(accepted / N - beta) < 5 * math.sqrt(beta * (1 - beta) / N)
    # chi-square with every bin's expected count >= 5: the rarest ids pooled, smallest first
    order = np.argsort(p)
    n_pool = int(np.searchsorted(np.cumsum(N * p[order]), 5.0)) + 1
    pool, rest = order[:n_pool], order[n_pool:]
    obs = np.append(counts[rest], counts[pool].sum())
    exp_ = np.append(N * p[rest], N * p[pool].sum())
    chi2 = ((obs - exp_) ** 2 / exp_).sum()
    assert chi2 < 35.0                                    # <= 5 dof; P(chi2 > 35) ~ 1e-6
    if case == "overlapping":
        assert hows.get("fallback", 0) > 0


def test_prefix_survival_is_product_of_conditionals():
    """P(A >= k) = prod c_i, and E[A+1] = 1 + sum_k P(A >= k)."""
    rng = np.random.default_rng(14)
    K, N, V = 5, 40000, 50
    c = np.array([0.9, 0.8, 0.85, 0.6, 0.95])
    cand = rng.integers(0, V, size=(N, K))
    agree = rng.random((N, K)) < c
    tgt = np.where(agree, cand, (cand + 1 + rng.integers(0, V - 1, size=(N, K))) % V)
    tgt = np.concatenate([tgt, rng.integers(0, V, size=(N, 1))], axis=1)
    A = np.array([O.verify_greedy(cand[n], tgt[n])["A"] for n in range(N)])
    want = np.cumprod(c)
    for k in range(1, K + 1):
        est = (A >= k).mean()
        assert abs(est - want[k - 1]) < 5 * math.sqrt(want[k - 1] * (1 - want[k - 1]) / N)
    assert abs((A + 1).mean() - rp.expected_advance(rp.prefix_survival(c))) < 0.03


# ---------------------------------------------------------------- verification window, match mode

def test_verification_window_is_the_shorter_round():
    """n_verify = w gives exactly the round of a drafter with K = w on the first
    w candidates and target rows 0..w (greedy and sampling, including the
    Philox positions of the bonus draw), and n_verify = K changes nothing."""
    rng = np.random.default_rng(31)
    V, K, T = 6, 4, 0.7
    E = np.eye(V)
    for trial in range(60):
        cand = [int(c) for c in rng.integers(0, 3, size=K)]
        tgt = [int(t) for t in rng.integers(0, 3, size=K + 1)]
        ell = rng.normal(0, 1.0, (K, V))
        lse = [float(np.log(np.exp(e / T).sum())) for e in ell]
        logit_d = [float(ell[i, cand[i]]) for i in range(K)]
        p = rng.dirichlet(np.ones(V), size=K + 1)
        assert O.verify_greedy(cand, tgt, n_verify=K) == O.verify_greedy(cand, tgt)
        full = O.verify_sample(cand, logit_d, lse, ell, E, p, T, 5, 100 + trial, 3)
        assert O.verify_sample(cand, logit_d, lse, ell, E, p, T, 5, 100 + trial, 3, n_verify=K) == full
        for w in range(K + 1):
            g = O.verify_greedy(cand, tgt, n_verify=w)
            assert g == O.verify_greedy(cand[:w], tgt[:w + 1])
            assert g["A"] <= w
            r = O.verify_sample(cand, logit_d, lse, ell, E, p, T, 5, 100 + trial, 3, n_verify=w)
            assert r == O.verify_sample(cand[:w], logit_d[:w], lse[:w], ell[:w + 1], E, p[:w + 1], T, 5,
                                        100 + trial, 3)
    with pytest.raises(ValueError):
        O.verify_greedy([1, 2], [1, 2, 3], n_verify=3)


def test_match_with_deterministic_target_is_greedy():
    """One-hot target rows: every sample is the row's id, so match verification
    reduces to greedy verification against those ids (every window)."""
    rng = np.random.default_rng(32)
    V, K = 5, 4
    for trial in range(50):
        tgt = [int(t) for t in rng.integers(0, V, size=K + 1)]
        cand = [t if rng.random() < 0.7 else int(rng.integers(0, V)) for t in tgt[:K]]
        p = np.zeros((K + 1, V))
        p[np.arange(K + 1), tgt] = 1.0
        for w in range(K + 1):
            r = O.verify_match(cand, p, 9, trial, 1, n_verify=w)
            g = O.verify_greedy(cand, tgt, n_verify=w)
            assert r["targets"] == tgt[:w + 1]
            assert {k: r[k] for k in g} == g


def test_match_statistics():
    """P(A >= k) = prod_{j<k} p_j(d_{j+1}) (independent target samples), and at a
    mismatch the committed token follows p_A restricted to ids other than the
    candidate: p_A(v) / (1 - p_A(d)), v != d. Monte Carlo over positions."""
    rng = np.random.default_rng(33)
    V, K, N = 4, 3, 20000
    p = rng.dirichlet(np.ones(V) * 2.0, size=K + 1)
    cand = [int(np.argmax(p[j])) for j in range(K)]      # a greedy draft that guessed the argmax
    A = np.zeros(N, dtype=np.int64)
    first = np.zeros(V)
    for n in range(N):
        r = O.verify_match(cand, p, 44, 10 * n, 2)
        A[n] = r["A"]
        if r["A"] == 0:
            first[r["commits"][0]] += 1
    pm = np.array([p[j, cand[j]] for j in range(K)])
    want = np.cumprod(pm)
    for k in range(1, K + 1):
        est = (A >= k).mean()
        assert abs(est - want[k - 1]) < 5 * math.sqrt(want[k - 1] * (1 - want[k - 1]) / N)
    n0 = first.sum()
    cond = p[0].copy()
    cond[cand[0]] = 0.0
    cond /= cond.sum()
    assert first[cand[0]] == 0
    m = cond > 0
    chi2 = ((first[m] - n0 * cond[m]) ** 2 / (n0 * cond[m])).sum()
    assert chi2 < 25.0                                    # V - 2 dof


def test_match_uses_its_own_stream():
    """The target samples come from tag TAG_MATCH at position pos + j + 1 and
    differ from the bonus stream of sampling verification."""
    V = 64
    p = np.full((2, V), 1.0 / V)
    t = O.verify_match([0], p, 123, 40, 5)["targets"]
    for j in range(2):
        u = float(ph.draw(123, 0, 40 + j + 1, 5, ph.TAG_MATCH, 0))
        assert t[j] == min(int(u * V), V - 1)            # uniform row: floor(u V)
    assert ph.TAG_MATCH not in (ph.TAG_GUMBEL, ph.TAG_ACCEPT, ph.TAG_RESID, ph.TAG_BONUS)


# ---------------------------------------------------------------- cost-model arithmetic

def test_pages_time_model_examples():
    for line in _golden_lines("pages_examples.txt"):
        t = line.split()
        if t[0] == "speedup":
            assert rp.speedup(float(t[2]), float(t[4]), float(t[6])) == pytest.approx(float(t[-1]))
        if t[0] == "relative":
            assert rp.relative_rate(float(t[1]), float(t[2])) == pytest.approx(float(t[-1]), abs=0.005)
        if t[0] == "time_saved":
            assert rp.time_saved(float(t[1])) == pytest.approx(float(t[-1]), abs=0.005)
        if t[0] == "workflow":
            assert rp.workflow_speedup(float(t[2]), float(t[4])) == pytest.approx(float(t[-1]))


def test_draft_kv_formula_and_history_control_sizes():
    # 2 * L_D * H * n_kv * d_h * b with the 8B-shaped drafter, bf16
    assert O.draft_kv_bytes(3, 8192, 8, 128, 2) == 100663296
    assert O.draft_kv_bytes(3, 118000, 8, 128, 2) == 1449984000


def test_mirror_differs_from_pure_by_bf16_scale():
    cfg = _tiny()
    W = _weights(cfg)
    hidden, anchor, _ = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=1)
    b0 = O.backbone(hidden[0], anchor[0], W, cfg, mirror=False)
    b1 = O.backbone(hidden[0], anchor[0], W, cfg, mirror=True)
    rel = np.linalg.norm(b1 - b0) / np.linalg.norm(b0)
    assert 1e-5 < rel < 2e-2


def test_ffn_gate_goes_through_silu_up_is_linear():
    """silu(y W_g^T) * (y W_u^T): the FFN increment is linear in W_u and W_d but not in W_g,
    so a swapped gate / up matrix or a missing nonlinearity changes which scaling is linear."""
    cfg = _tiny()
    W = _weights(cfg, seed=23)
    rng = np.random.default_rng(24)
    x = rng.normal(size=(cfg.K + 1, cfg.D))
    z = rng.normal(size=(cfg.m, cfg.D))
    base = dict(W["layers"][0])
    base["Wo"] = torch.zeros_like(base["Wo"])          # attention contributes nothing
    delta = O.backbone_layer(x, z, base, cfg) - x
    for name, linear in (("Wu", True), ("Wd", True), ("Wg", False)):
        Wl = dict(base)
        Wl[name] = base[name] * 2.0          # exact in binary floating point
        d2 = O.backbone_layer(x, z, Wl, cfg) - x
        close = np.allclose(d2, 2.0 * delta, rtol=1e-9, atol=1e-12)
        assert close == linear, name


# ---------------------------------------------------------------- attention wiring of a layer

def _wiring_setup(G=1, seed=31):
    # jittered gains: the staged z is then far from unit RMS, so a context row
    # taken through the pre-attention norm differs from z itself
    cfg = _tiny(G=G)
    W = _weights(cfg, seed=seed, jitter=True)
    rng = np.random.default_rng(seed + 1)
    x = rng.normal(size=(cfg.G + cfg.K, cfg.D))
    hidden = torch.from_numpy(rng.normal(size=(cfg.m, cfg.D)))
    z, _ = O.stage(hidden, [0] * cfg.G if G > 1 else 0, W, cfg)
    return cfg, W, x, z


def test_layer_with_zero_queries_averages_the_value_rows():
    """W_q = 0 makes every score zero, so each query head returns the plain mean
    of its KV group's value rows over all m + G + K keys: the context rows
    projected from the staged z as it is, the local rows from the normed
    y = RMSNorm(x) g_attn, neither rotated. With W_d = 0 the layer output is
    then x + mean W_o^T in closed form ([P1] §"本轮临时 K/V 仍然需要计算":
    context and local rows both give keys / values)."""
    cfg, W, x, z = _wiring_setup()
    Wl = dict(W["layers"][0])
    Wl["Wq"] = torch.zeros_like(Wl["Wq"])
    Wl["Wd"] = torch.zeros_like(Wl["Wd"])
    g = O.f64(Wl["g_attn"])
    y = g * x / np.sqrt((x * x).mean(axis=1, keepdims=True) + cfg.eps)
    Wv = O.f64(Wl["Wv"])
    rows = np.concatenate([z, y]) @ Wv.T                       # [m + K1, n_kv d_h]
    mean = rows.mean(axis=0).reshape(cfg.n_kv, cfg.d_h)
    group = cfg.n_q // cfg.n_kv
    o = np.concatenate([mean[h // group] for h in range(cfg.n_q)])
    want = x + (o @ O.f64(Wl["Wo"]).T)[None, :]
    got = O.backbone_layer(x, z, Wl, cfg)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2])
def test_layer_attention_inputs_follow_the_local_positions(G, monkeypatch):
    """What a layer hands to the attention, against an independent statement in
    complex form: local row i (position i: the group at 0..G-1, placeholders
    after it) gives q_i = rot_i(W_q y_i) and k_i = rot_i(W_k y_i), where rot_p
    multiplies the pair (j, j + d_h/2), read as one complex number, by
    exp(i p theta^(-2j/d_h)); context row j gives k = W_k z_j with no rotation
    (position 0) and no norm; values are never rotated. The score matrix
    q k^T / sqrt(d_h) and the values are compared ([P1]
    §"局部位置编码切断草稿端的全局位置增长")."""
    cfg, W, x, z = _wiring_setup(G=G, seed=37 + G)
    Wl = W["layers"][0]
    seen = {}
    real = O.block_attention

    def spy(q, k, v, n_q, n_kv):
        seen.update(q=np.array(q), k=np.array(k), v=np.array(v))
        return real(q, k, v, n_q, n_kv)

    monkeypatch.setattr(O, "block_attention", spy)
    O.backbone_layer(x, z, Wl, cfg)
    K1, d = cfg.G + cfg.K, cfg.d_h
    g = O.f64(Wl["g_attn"])
    y = g * x / np.sqrt((x * x).mean(axis=1, keepdims=True) + cfg.eps)

    def rot(rows, pos):   # rows [T, heads, d]
        half = d // 2
        c = rows[..., :half] + 1j * rows[..., half:]
        w = np.exp(1j * np.outer(pos, cfg.theta ** (-2.0 * np.arange(half) / d)))[:, None, :]
        c = c * w
        return np.concatenate([c.real, c.imag], axis=-1)

    pos = np.arange(K1, dtype=np.float64)
    q = rot((y @ O.f64(Wl["Wq"]).T).reshape(K1, cfg.n_q, d), pos)
    k_loc = rot((y @ O.f64(Wl["Wk"]).T).reshape(K1, cfg.n_kv, d), pos)
    k_ctx = (z @ O.f64(Wl["Wk"]).T).reshape(cfg.m, cfg.n_kv, d)
    v = (np.concatenate([z, y]) @ O.f64(Wl["Wv"]).T).reshape(cfg.m + K1, cfg.n_kv, d)
    k = np.concatenate([k_ctx, k_loc])
    group = cfg.n_q // cfg.n_kv
    for h in range(cfg.n_q):
        want = q[:, h] @ k[:, h // group].T / math.sqrt(d)
        got = seen["q"][:, h] @ seen["k"][:, h // group].T / math.sqrt(d)
        assert np.allclose(got, want, rtol=0, atol=1e-10), h
    assert np.allclose(seen["v"], v, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- synthetic target of the acceptance workloads

def test_synthetic_target_extremes():
    """c = 1: the target agrees everywhere (A = K); c = 0: it never agrees and
    every disagreeing id differs from the candidate (A = 0)."""
    rng = np.random.default_rng(51)
    V, K = 37, 6
    for r in range(300):
        cand = [int(t) for t in rng.integers(0, V, K)]
        t1 = O.synthetic_target_tokens(cand, np.ones(K), 9, r, 2, V)
        assert t1[:K] == cand and 0 <= t1[K] < V
        t0 = O.synthetic_target_tokens(cand, np.zeros(K), 9, r, 2, V)
        assert all(a != b and 0 <= a < V for a, b in zip(t0[:K], cand))
        assert O.verify_greedy(cand, t1)["A"] == K and O.verify_greedy(cand, t0)["A"] == 0


def test_synthetic_target_other_ids_are_uniform():
    """A disagreeing choice is uniform over the V - 1 other ids and the bonus
    choice uniform over all V (chi-square)."""
    V, K, N = 5, 3, 6000
    other = np.zeros(V)
    bonus = np.zeros(V)
    for r in range(N):
        t = O.synthetic_target_tokens([2] * K, np.zeros(K), 17, 10 * r, 1, V)
        for x in t[:K]:
            other[x] += 1
        bonus[t[K]] += 1
    assert other[2] == 0
    e = K * N / (V - 1)
    chi_o = (((other - e) ** 2) / e)[[0, 1, 3, 4]].sum()
    chi_b = (((bonus - N / V) ** 2) / (N / V)).sum()
    assert chi_o < 25.0 and chi_b < 25.0        # 3 and 4 dof; P(> 25) < 1e-4


def test_synthetic_target_prefix_survival():
    """Greedy verification against the synthetic target: P(A >= k) = prod c_i
    (DFlash page, prefix survival; [P1] §"分布重叠怎样影响平均推进量"), within
    5 sigma binomial bands, and E[A + 1] = 1 + sum_k P(A >= k)."""
    c = np.array([0.9, 0.8, 0.7, 0.95, 0.6], dtype=np.float32)
    K, V, N = len(c), 1000, 20000
    cand = [3, 1, 4, 1, 5]
    A = np.array([O.verify_greedy(cand, O.synthetic_target_tokens(cand, c, 23, 8 * n, n % 7, V))["A"]
                  for n in range(N)])
    surv = np.cumprod(c.astype(np.float64))
    for k in range(1, K + 1):
        p = surv[k - 1]
        assert abs((A >= k).mean() - p) < 5 * math.sqrt(p * (1 - p) / N), k
    assert abs((A + 1).mean() - rp.expected_advance(surv)) < 5 * (A + 1).std() / math.sqrt(N)


def test_synthetic_target_is_keyed():
    """Different seeds, positions and requests give different draws; the same
    key gives the same tokens."""
    cand = list(range(10, 17))
    c = np.full(7, 0.5)
    base = O.synthetic_target_tokens(cand, c, 5, 100, 3, 151936)
    assert base == O.synthetic_target_tokens(cand, c, 5, 100, 3, 151936)
    for kw in ({"seed": 6}, {"pos": 101}, {"request": 4}):
        args = dict(seed=5, pos=100, request=3)
        args.update(kw)
        assert O.synthetic_target_tokens(cand, c, args["seed"], args["pos"], args["request"], 151936) != base
