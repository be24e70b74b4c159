"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances (from the method's stated agreement bar):
  * token ids, A and commits: bit-exact;
  * hidden representations: relative L2 error <= 2e-2 per tensor against the
    pure fp64 oracle (bf16 weights, fp32 accumulate);
  * candidates: >= 99.9% identical, and every mismatch only where the
    oracle's top-2 gap (logits, or perturbed scores when sampling) is < 1e-3.
"""
import numpy as np
import pytest
import torch

from history_free_speculative_gb300 import binding
from history_free_speculative_gb300 import workload as wk
from oracle import dlite_oracle as O
from oracle import philox as ph
from parity import HIDDEN_REL_TOL, check_candidates, check_candidates_bf16, check_fed_back_candidates, f64_weights, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _drafter(cfg, W, B_max):
    return binding.Drafter(cfg, wk.weights_to(W, DEV), B_max=B_max)


@pytest.fixture(scope="module")
def tiny():
    wl = wk.WORKLOADS["tiny"]
    W = wk.make_weights(wl.cfg, wl.weight_seed, gain_jitter=True)
    dr = _drafter(wl.cfg, W, B_max=16)
    yield wl, W, dr
    dr.close()


# ---------------------------------------------------------------- tiny fp32 round, greedy

def test_tiny_round_hidden_and_candidates(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 16
    cands, ocands, gaps = [], [], []
    for rnd in range(3):
        hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=rnd)
        out = dr.new_outputs(B, DEV)
        taps = {"z": torch.empty(B, cfg.m, cfg.D, device=DEV),
                "x": torch.empty(cfg.L_D, B, cfg.K + 1, cfg.D, device=DEV),
                "b": torch.empty(B, cfg.K, cfg.D, device=DEV),
                "hs": torch.empty(B, cfg.K, cfg.D, device=DEV)}
        dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, 0, pos.to(DEV), out["cand"],
                       out["qstats"], taps=taps)
        torch.cuda.synchronize()
        for b in range(B):
            t = {}
            r = O.draft_request(hidden[b], int(anchor[b]), W, cfg, taps=t)
            assert rel_err(taps["z"][b].cpu(), t["z"]) < 1e-5
            for l in range(cfg.L_D):
                assert rel_err(taps["x"][l, b].cpu(), t["x"][l]) < 1e-4
            assert rel_err(taps["b"][b].cpu(), t["b"]) < 1e-4
            assert rel_err(taps["hs"][b].cpu(), t["h"]) < 1e-4
            cands.append(out["cand"][b].cpu().numpy())
            ocands.append(r["cand"])
            gaps.append(r["gap"])
    check_candidates(np.stack(cands), np.stack(ocands), np.stack(gaps))


def test_tiny_round_verify_commits(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 16
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=7)
    ref = O.draft_round(hidden, anchor.numpy(), W, cfg)
    ocand = np.stack([ref[b]["cand"] for b in range(B)])
    tgt = wk.make_target_tokens(ocand, wl.accept_c, cfg.V, wl.rng_seed)
    out = dr.new_outputs(B, DEV)
    dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, 0, pos.to(DEV), out["cand"], out["qstats"])
    dr.verify(out["cand"], tgt.to(DEV), out["accepted"], out["commits"], out["n_commit"],
              out["next_anchor"])
    torch.cuda.synchronize()
    assert np.array_equal(out["cand"].cpu().numpy(), ocand)
    for b in range(B):
        ov = O.verify_greedy(ocand[b], tgt[b].numpy())
        assert int(out["accepted"][b]) == ov["A"]
        assert int(out["n_commit"][b]) == ov["n_commit"]
        assert out["commits"][b, :ov["n_commit"]].tolist() == ov["commits"]
        assert int(out["next_anchor"][b]) == ov["next_anchor"]


def test_tiny_round_sampling(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B, T, seed = 16, 0.7, 4242
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=3)
    out = dr.new_outputs(B, DEV)
    dr.draft_round(hidden.to(DEV), anchor.to(DEV), T, seed, pos.to(DEV), out["cand"], out["qstats"])
    torch.cuda.synchronize()
    qs = out["qstats"].cpu().numpy()
    cands, ocands, gaps = [], [], []
    for b in range(B):
        r = O.draft_request(hidden[b], int(anchor[b]), W, cfg, temperature=T, seed=seed,
                            pos=int(pos[b]), request=b)
        cands.append(out["cand"][b].cpu().numpy())
        ocands.append(r["cand"])
        gaps.append(r["gap"])
        same = out["cand"][b].cpu().numpy() == r["cand"]
        assert np.allclose(qs[b, same, 0], r["logit_d"][same], rtol=1e-4, atol=1e-4)
        assert np.allclose(qs[b, :, 1], r["lse"], rtol=1e-5, atol=1e-4)
    check_candidates(np.stack(cands), np.stack(ocands), np.stack(gaps))


@pytest.fixture(scope="module")
def midvocab():
    # bf16 drafter whose vocabulary spans several slabs per CTA with a ragged
    # last slab (100000 is not a multiple of 128 or 256)
    cfg = wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=1, n_q=4, n_kv=2, R=64, V=100000, m=2)
    W = wk.make_weights(cfg, 77)
    dr = _drafter(cfg, W, B_max=40)
    yield cfg, W, dr
    dr.close()


@pytest.mark.parametrize("B", [3, 20, 40])   # 21 rows (one M-tile), 140 (two), 280 (one-slab kernel)
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_lm_head_identical_inputs_multislab(midvocab, B, T):
    cfg, W, dr = midvocab
    hs = _rand_hs(cfg, B, 6 + B)
    pos = torch.arange(B, dtype=torch.int64) * 977 + 5
    cand = torch.empty(B, cfg.K, dtype=torch.int32, device=DEV)
    qs = torch.empty(B, cfg.K, 2, device=DEV)
    dr.lm_head(hs.to(DEV), T, 123, pos.to(DEV), cand, qs)
    torch.cuda.synchronize()
    E = O.f64(W["E"])
    ell = O.lm_logits(hs.reshape(-1, cfg.D).numpy().astype(np.float64), E).reshape(B, cfg.K, -1)
    Tq = float(np.float32(T))
    picks = [[O.sample_logits(ell[b, i], Tq, 123, int(pos[b]) + i + 1, b) for i in range(cfg.K)] for b in range(B)]
    oc = np.array([[p[0] for p in row] for row in picks])
    gap = np.array([[p[1] for p in row] for row in picks])
    c = cand.cpu().numpy()
    check_candidates(c, oc, gap)
    q = qs.cpu().numpy()
    # the reported logit is the exact re-score of the chosen id
    chosen = np.take_along_axis(ell, c[..., None].astype(np.int64), 2)[..., 0]
    assert np.allclose(q[..., 0], chosen, rtol=1e-5, atol=1e-4)
    if T > 0:
        lse = np.log(np.exp(ell / Tq - (ell / Tq).max(axis=2, keepdims=True)).sum(axis=2)) + \
            (ell / Tq).max(axis=2)
        assert np.allclose(q[..., 1], lse, rtol=0, atol=2e-3)


# ---------------------------------------------------------------- stage checks on identical inputs

def _rand_hs(cfg, B, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, cfg.K, cfg.D, generator=g) * scale


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_lm_head_identical_inputs_tiny(tiny, T):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 16
    hs = _rand_hs(cfg, B, 5)
    pos = torch.arange(B, dtype=torch.int64) * 100
    cand = torch.empty(B, cfg.K, dtype=torch.int32, device=DEV)
    qs = torch.empty(B, cfg.K, 2, device=DEV)
    dr.lm_head(hs.to(DEV), T, 99, pos.to(DEV), cand, qs)
    torch.cuda.synchronize()
    E = O.f64(W["E"])
    ell = O.lm_logits(hs.reshape(-1, cfg.D).numpy(), E).reshape(B, cfg.K, -1)
    Tq = float(np.float32(T))
    picks = [[O.sample_logits(ell[b, i], Tq, 99, int(pos[b]) + i + 1, b) for i in range(cfg.K)] for b in range(B)]
    oc = np.array([[p[0] for p in row] for row in picks])
    gap = np.array([[p[1] for p in row] for row in picks])
    check_candidates(cand.cpu().numpy(), oc, gap, gap_tol=1e-4)


def test_seq_head_identical_inputs_tiny(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 16
    b = _rand_hs(cfg, B, 6)
    hs = torch.empty(B, cfg.K, cfg.D, device=DEV)
    dr.seq_head(b.to(DEV), hs)
    torch.cuda.synchronize()
    for r in range(B):
        want = O.sequential_head(b[r].numpy(), W["Q"], W["P"])
        assert rel_err(hs[r].cpu(), want) < 1e-5


# ---------------------------------------------------------------- verify (K5)

@pytest.fixture(scope="module")
def small_v():
    """A tiny-vocabulary drafter for exhaustive verify checks (V = 8, K = 3)."""
    cfg = wk.shrink(wk.TINY, V=8, K=3, D=64, F=128, R=32, n_q=2, n_kv=1, m=2)
    W = wk.make_weights(cfg, 7)
    dr = _drafter(cfg, W, B_max=4096)
    yield cfg, W, dr
    dr.close()


def test_verify_greedy_exhaustive(small_v):
    """All candidate / target pairs over 3 ids with K = 3, against brute force."""
    import itertools
    cfg, W, dr = small_v
    cands = np.array(list(itertools.product(range(3), repeat=3)), dtype=np.int32)
    tgts = np.array(list(itertools.product(range(3), repeat=4)), dtype=np.int32)
    C = np.repeat(cands, len(tgts), axis=0)
    Tt = np.tile(tgts, (len(cands), 1))
    B = len(C)
    out = dr.new_outputs(B, DEV)
    dr.verify(torch.from_numpy(C).to(DEV), torch.from_numpy(Tt).to(DEV), out["accepted"],
              out["commits"], out["n_commit"], out["next_anchor"])
    torch.cuda.synchronize()
    acc = out["accepted"].cpu().numpy()
    com = out["commits"].cpu().numpy()
    for i in range(B):
        passes = (C[i] == Tt[i, :3]).astype(np.int64)
        A = int(np.cumprod(passes).sum())
        assert acc[i] == A
        assert list(com[i, :A + 1]) == list(C[i, :A]) + [Tt[i, A]]
        assert all(com[i, A + 1:] == -1)
    assert np.array_equal(out["n_commit"].cpu().numpy(), acc + 1)


def _sample_inputs(cfg, W, B, seed, overlap):
    """Candidates drawn from q, q statistics and target rows (oracle-computed)."""
    rng = np.random.default_rng(seed)
    hs = rng.normal(0, 1.0, (B, cfg.K, cfg.D))
    E = O.f64(W["E"])
    ell = O.lm_logits(hs.reshape(-1, cfg.D), E).reshape(B, cfg.K, cfg.V)
    T = float(np.float32(0.7))
    lse = np.log(np.exp(ell / T).sum(axis=2))
    cand = np.empty((B, cfg.K), dtype=np.int64)
    pos = rng.integers(0, 1 << 20, B)
    for b in range(B):
        for i in range(cfg.K):
            cand[b, i] = np.argmax(ell[b, i] / T + ph.gumbel_row(1, pos[b] + i + 1, b, cfg.V))
    q = np.exp(ell / T - lse[..., None])
    p = np.empty((B, cfg.K + 1, cfg.V))
    for b in range(B):
        for j in range(cfg.K + 1):
            d = rng.dirichlet(np.ones(cfg.V) * 0.7)
            p[b, j] = (overlap * q[b, min(j, cfg.K - 1)] + (1 - overlap) * d) if overlap else d
    p = (p / p.sum(axis=2, keepdims=True)).astype(np.float32)
    logit_d = np.take_along_axis(ell, cand[..., None], 2)[..., 0]
    return hs.astype(np.float32), cand, logit_d.astype(np.float32), lse.astype(np.float32), p, pos


@pytest.mark.parametrize("overlap", [0.0, 0.97])
def test_verify_sample_identical_inputs(small_v, overlap):
    """Accept/reject, residual proposals and the inverse-CDF fallback: bit-exact."""
    cfg, W, dr = small_v
    B, T, seed = 2048, 0.7, 1
    hs, cand, logit_d, lse, p, pos = _sample_inputs(cfg, W, B, 31 + int(overlap * 100), overlap)
    qs = np.stack([logit_d, lse], axis=-1)
    out = dr.new_outputs(B, DEV)
    dr.verify_sample(torch.from_numpy(cand.astype(np.int32)).to(DEV), torch.from_numpy(qs).to(DEV),
                     torch.from_numpy(hs).to(DEV), torch.from_numpy(p).to(DEV), T, seed,
                     torch.from_numpy(pos).to(DEV), out["accepted"], out["commits"],
                     out["n_commit"], out["next_anchor"])
    torch.cuda.synchronize()
    acc = out["accepted"].cpu().numpy()
    com = out["commits"].cpu().numpy()
    hows = {}
    for b in range(B):
        r = O.verify_sample(cand[b], logit_d[b], lse[b], hs[b], W["E"], p[b], T, seed, int(pos[b]), b)
        hows[r["how"]] = hows.get(r["how"], 0) + 1
        assert acc[b] == r["A"], (b, acc[b], r)
        assert list(com[b, :r["n_commit"]]) == r["commits"], (b, com[b], r)
    assert np.array_equal(out["next_anchor"].cpu().numpy(), com[np.arange(B), acc])
    if overlap:
        assert hows.get("fallback", 0) > 0, hows


def test_verify_sample_preserves_target_distribution(small_v):
    """GPU speculative sampling: the committed first token follows p (chi-square)."""
    cfg, W, dr = small_v
    V, N, T = cfg.V, 4096, 0.7
    rng = np.random.default_rng(3)
    h1 = rng.normal(0, 1.0, cfg.D)
    E = O.f64(W["E"])
    ell = E @ h1
    Tq = float(np.float32(T))
    q = np.exp(ell / Tq - ell.max() / Tq)
    q /= q.sum()
    lse = float(np.log(np.exp(ell / Tq).sum()))
    p0 = rng.dirichlet(np.ones(V))
    pos = np.arange(N, dtype=np.int64) * 16
    cand = np.zeros((N, cfg.K), dtype=np.int64)
    for n in range(N):
        cand[n, 0] = np.argmax(ell / Tq + ph.gumbel_row(5, pos[n] + 1, n, V))
    hs = np.tile(h1, (N, cfg.K, 1)).astype(np.float32)
    p = np.tile(p0, (N, cfg.K + 1, 1)).astype(np.float32)
    qs = np.zeros((N, cfg.K, 2), dtype=np.float32)
    qs[:, :, 0] = ell[cand].astype(np.float32)
    qs[:, :, 1] = lse
    out = dr.new_outputs(N, DEV)
    dr.verify_sample(torch.from_numpy(cand.astype(np.int32)).to(DEV), torch.from_numpy(qs).to(DEV),
                     torch.from_numpy(hs).to(DEV), torch.from_numpy(p).to(DEV), T, 5,
                     torch.from_numpy(pos).to(DEV), out["accepted"], out["commits"],
                     out["n_commit"], out["next_anchor"])
    torch.cuda.synchronize()
    first = out["commits"][:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    pp = p0.astype(np.float32).astype(np.float64)
    pp /= pp.sum()
    chi2 = ((counts - N * pp) ** 2 / (N * pp)).sum()
    assert chi2 < 40.0, (chi2, counts, N * pp)     # 7 dof
    beta = np.minimum(pp, q).sum()
    acc1 = (out["accepted"].cpu().numpy() >= 1).mean()
    assert abs(acc1 - beta) < 5 * np.sqrt(beta * (1 - beta) / N)


# ---------------------------------------------------------------- verification window and match mode

def _t(x, dtype=None):
    x = np.asarray(x)
    return torch.from_numpy(x.astype(dtype) if dtype else x).to(DEV)


@pytest.mark.parametrize("n_verify", [0, 1, 2, 3])
def test_verify_window_identical_inputs(small_v, n_verify):
    """dlite_verify_ex with a verification window: greedy and sampling bit-exact
    against the oracle's truncated rounds (n_verify = K is the full round)."""
    cfg, W, dr = small_v
    B, T, seed = 1024, 0.7, 3
    rng = np.random.default_rng(50 + n_verify)
    C = rng.integers(0, 3, size=(B, cfg.K)).astype(np.int32)
    Tt = rng.integers(0, 3, size=(B, cfg.K + 1)).astype(np.int32)
    out = dr.new_outputs(B, DEV)
    dr.verify_ex(binding.VERIFY_GREEDY, _t(C), out["accepted"], out["commits"], out["n_commit"],
                 out["next_anchor"], n_verify=n_verify, target_tokens=_t(Tt))
    torch.cuda.synchronize()
    acc, com = out["accepted"].cpu().numpy(), out["commits"].cpu().numpy()
    for b in range(B):
        r = O.verify_greedy(C[b], Tt[b], n_verify=n_verify)
        assert acc[b] == r["A"] and list(com[b, :r["n_commit"]]) == r["commits"]
        assert all(com[b, r["n_commit"]:] == -1)
    hs, cand, logit_d, lse, p, pos = _sample_inputs(cfg, W, B, 60 + n_verify, 0.6)
    qs = np.stack([logit_d, lse], axis=-1)
    out = dr.new_outputs(B, DEV)
    dr.verify_ex(binding.VERIFY_SAMPLE, _t(cand, np.int32), out["accepted"], out["commits"], out["n_commit"],
                 out["next_anchor"], n_verify=n_verify, qstats=_t(qs), hs=_t(hs), probs=_t(p),
                 temperature=T, seed=seed, pos=_t(pos))
    torch.cuda.synchronize()
    acc, com = out["accepted"].cpu().numpy(), out["commits"].cpu().numpy()
    for b in range(B):
        r = O.verify_sample(cand[b], logit_d[b], lse[b], hs[b], W["E"], p[b], T, seed, int(pos[b]), b,
                            n_verify=n_verify)
        assert acc[b] == r["A"] <= n_verify, (b, acc[b], r)
        assert list(com[b, :r["n_commit"]]) == r["commits"], (b, com[b], r)
    assert np.array_equal(out["next_anchor"].cpu().numpy(), com[np.arange(B), acc])


def _match_inputs(cfg, B, seed, agree):
    """Target rows p_j and greedy candidates that equal the row's mode w.p. agree."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(cfg.V) * 0.3, size=(B, cfg.K + 1)).astype(np.float32)
    mode = np.argmax(p[:, :cfg.K], axis=2)
    rand = rng.integers(0, cfg.V, size=(B, cfg.K))
    cand = np.where(rng.random((B, cfg.K)) < agree, mode, rand).astype(np.int32)
    pos = rng.integers(0, 1 << 20, B)
    return cand, p, pos


@pytest.mark.parametrize("n_verify", [None, 1, 0])
def test_verify_match_identical_inputs(small_v, n_verify):
    """Match verification (the target's own samples, Philox tag 5): A, commits and
    the next anchor bit-exact against the oracle, for several windows."""
    cfg, W, dr = small_v
    B, seed = 2048, 11
    cand, p, pos = _match_inputs(cfg, B, 70, 0.8)
    out = dr.new_outputs(B, DEV)
    dr.verify_ex(binding.VERIFY_MATCH, _t(cand), out["accepted"], out["commits"], out["n_commit"],
                 out["next_anchor"], n_verify=n_verify, probs=_t(p), seed=seed, pos=_t(pos))
    torch.cuda.synchronize()
    acc, com = out["accepted"].cpu().numpy(), out["commits"].cpu().numpy()
    hist = np.zeros(cfg.K + 1, dtype=np.int64)
    for b in range(B):
        r = O.verify_match(cand[b], p[b], seed, int(pos[b]), b, n_verify=n_verify)
        hist[r["A"]] += 1
        assert acc[b] == r["A"], (b, acc[b], r)
        assert list(com[b, :r["n_commit"]]) == r["commits"], (b, com[b], r)
    assert np.array_equal(out["n_commit"].cpu().numpy(), acc + 1)
    kv = cfg.K if n_verify is None else n_verify
    assert hist[kv] > 0 and (kv == 0 or hist[0] > 0)        # both ends of the range occur


@pytest.mark.parametrize("B", [1, 8, 16, 40])   # clusters of 8, 4, 2 and 1 CTAs per sampled row
def test_verify_match_large_vocabulary(midvocab, B):
    """Match verification over a 100k vocabulary (multi-segment inverse CDF in
    every CTA of the cluster, for each cluster size), against the oracle."""
    cfg, W, dr = midvocab
    seed = 5
    cand, p, pos = _match_inputs(cfg, B, 71, 0.9)
    out = dr.new_outputs(B, DEV)
    dr.verify_ex(binding.VERIFY_MATCH, _t(cand), out["accepted"], out["commits"], out["n_commit"],
                 out["next_anchor"], probs=_t(p), seed=seed, pos=_t(pos))
    torch.cuda.synchronize()
    acc, com = out["accepted"].cpu().numpy(), out["commits"].cpu().numpy()
    for b in range(B):
        r = O.verify_match(cand[b], p[b], seed, int(pos[b]), b)
        assert acc[b] == r["A"] and list(com[b, :r["n_commit"]]) == r["commits"], (b, r)


def test_verify_ex_rejects_bad_arguments(small_v):
    cfg, W, dr = small_v
    cand = torch.zeros(4, cfg.K, dtype=torch.int32, device=DEV)
    out = dr.new_outputs(4, DEV)
    for kw in (dict(n_verify=cfg.K + 1, target_tokens=cand), dict(n_verify=-1, target_tokens=cand),
               dict(target_tokens=None)):
        with pytest.raises(RuntimeError):
            dr.verify_ex(binding.VERIFY_GREEDY, cand, out["accepted"], out["commits"], out["n_commit"],
                         out["next_anchor"], **kw)
    with pytest.raises(RuntimeError):
        dr.verify_ex(7, cand, out["accepted"], out["commits"], out["n_commit"], out["next_anchor"])


# ---------------------------------------------------------------- local token group

@pytest.mark.parametrize("name,G", [("tiny", 2), ("bf16", 3)])
def test_group_round_parity(name, G):
    """A local token group of G tokens: staging, attention over G + K local rows
    at positions 0..G+K-1 and the placeholder outputs, against the oracle."""
    if name == "tiny":
        cfg = wk.shrink(wk.TINY, G=G)
        W = wk.make_weights(cfg, 21, gain_jitter=True)
        tol = 1e-4
    else:
        cfg = wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=2, n_q=4, n_kv=2, R=64, V=4096, m=6, G=G)
        W = wk.make_weights(cfg, 22)
        tol = HIDDEN_REL_TOL
    wl = wk.WORKLOADS["tiny"]
    B = 12
    dr = _drafter(cfg, W, B_max=B)
    try:
        hidden, _, pos = wk.make_round_inputs(wl, B=B, cfg=cfg)
        rng = np.random.default_rng(G)
        groups = torch.from_numpy(rng.integers(0, cfg.V, size=(B, G)).astype(np.int32))
        out = dr.new_outputs(B, DEV)
        taps = {"z": torch.empty(B, cfg.m, cfg.D, device=DEV),
                "x": torch.empty(cfg.L_D, B, G + cfg.K, cfg.D, device=DEV),
                "b": torch.empty(B, cfg.K, cfg.D, device=DEV),
                "hs": torch.empty(B, cfg.K, cfg.D, device=DEV)}
        dr.draft_round(hidden.to(DEV), groups.to(DEV), 0.0, 0, pos.to(DEV), out["cand"], out["qstats"], taps=taps)
        torch.cuda.synchronize()
        cands, ocands, gaps, hmir = [], [], [], []
        for b in range(B):
            t = {}
            r = O.draft_request(hidden[b], groups[b].numpy(), W, cfg, taps=t, mirror=(cfg.dtype == "bf16"))
            for l in range(cfg.L_D):
                assert rel_err(taps["x"][l, b].cpu(), t["x"][l]) < tol
            assert rel_err(taps["b"][b].cpu(), t["b"]) < tol
            cands.append(out["cand"][b].cpu().numpy())
            ocands.append(r["cand"])
            gaps.append(r["gap"])
            hmir.append(t["h"])
        if cfg.dtype == "bf16":   # a flip must be the own head state's exact choice at a bridgeable gap
            check_candidates_bf16(np.stack(cands), np.stack(ocands), np.stack(gaps), O.f64(W["E"]),
                                  taps["hs"].cpu().numpy(), hmir, lambda n, i, ell: int(np.argmax(ell)))
        else:
            check_candidates(np.stack(cands), np.stack(ocands), np.stack(gaps))
    finally:
        dr.close()


def test_shift_group_matches_oracle(small_v):
    """dlite_shift_group against the oracle's next_group (G = 1 in this drafter:
    the next anchor), and a G = 4 drafter over random commit lengths."""
    for G in (1, 4):
        cfg = wk.shrink(wk.TINY, V=8, K=3, D=64, F=128, R=32, n_q=2, n_kv=1, m=2, G=G)
        dr = _drafter(cfg, wk.make_weights(cfg, 7), B_max=64)
        try:
            rng = np.random.default_rng(90 + G)
            B = 64
            group = rng.integers(0, 8, size=(B, G)).astype(np.int32)
            n = rng.integers(1, cfg.K + 2, size=B).astype(np.int32)
            commits = np.where(np.arange(cfg.K + 1)[None, :] < n[:, None],
                               rng.integers(0, 8, size=(B, cfg.K + 1)), -1).astype(np.int32)
            g = _t(group)
            dr.shift_group(_t(commits), _t(n), g)
            torch.cuda.synchronize()
            got = g.cpu().numpy()
            for b in range(B):
                assert list(got[b]) == O.next_group(group[b], commits[b, :n[b]])
        finally:
            dr.close()


# ---------------------------------------------------------------- gated token-feedback head

@pytest.mark.parametrize("name", ["tiny", "bf16", "bf16-r512-b32"])
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_gated_head_round_parity(name, T):
    """The official gated head: per-step vectors r_i and candidates (greedy and
    sampled, token fed back each step) against the oracle. With one weight plane
    the step's r runs in the state kernel's launch when all its clusters (R / 32
    CTAs, 4 requests each) are resident at once: R = 128 with 12 requests takes
    that form; R = 512 with 32 requests (eight 16-CTA clusters) the two launches
    on devices that hold fewer clusters at once."""
    B = 12
    if name == "tiny":
        cfg = wk.shrink(wk.TINY, R=64, head="gated")
        W = wk.make_weights(cfg, 31, gain_jitter=True)
        tol = 1e-4
    elif name == "bf16":
        cfg = wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=2, n_q=4, n_kv=2, R=128, V=4096, m=6, head="gated")
        W = wk.make_weights(cfg, 32)
        tol = HIDDEN_REL_TOL
    else:
        cfg = wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=1, n_q=4, n_kv=2, R=512, V=4096, m=6, head="gated")
        W = wk.make_weights(cfg, 33)
        tol = HIDDEN_REL_TOL
        B = 32
    wl = wk.WORKLOADS["tiny"]
    seed = 77
    dr = _drafter(cfg, W, B_max=B)
    try:
        hidden, anchor, pos = wk.make_round_inputs(wl, B=B, cfg=cfg)
        anchor = anchor % cfg.V
        out = dr.new_outputs(B, DEV)
        taps = {"z": torch.empty(B, cfg.m, cfg.D, device=DEV),
                "x": torch.empty(cfg.L_D, B, cfg.K + 1, cfg.D, device=DEV),
                "b": torch.empty(B, cfg.K, cfg.D, device=DEV),
                "hs": torch.empty(B, cfg.K, cfg.R, device=DEV)}
        dr.draft_round(hidden.to(DEV), anchor.to(DEV), T, seed, pos.to(DEV), out["cand"], out["qstats"],
                       taps=taps)
        torch.cuda.synchronize()
        cand = out["cand"].cpu().numpy()
        qs = out["qstats"].cpu().numpy()
        cands, ocands, gaps, hmir = [], [], [], []
        for b in range(B):
            r = O.draft_request(hidden[b], int(anchor[b]), W, cfg, temperature=T, seed=seed, pos=int(pos[b]),
                                request=b, mirror=(cfg.dtype == "bf16"))
            if np.array_equal(cand[b], r["cand"]):   # same tokens fed back: the vectors agree
                assert rel_err(taps["hs"][b].cpu(), r["h"]) < tol
                if T > 0:
                    assert np.allclose(qs[b, :, 1], r["lse"], rtol=1e-5, atol=1e-3)
            else:                                    # a near-tie flipped a token: earlier steps still agree
                k = int(np.argmax(cand[b] != r["cand"]))
                assert rel_err(taps["hs"][b, :k + 1].cpu(), r["h"][:k + 1]) < tol
            cands.append(cand[b])
            ocands.append(r["cand"])
            gaps.append(r["gap"])
            hmir.append(r["h"])
        Tq = float(np.float32(T))
        own = lambda n, i, ell: O.sample_logits(ell, Tq if T > 0 else 0.0, seed, int(pos[n]) + i + 1, n)[0]
        check_fed_back_candidates(np.stack(cands), np.stack(ocands), np.stack(gaps), O.f64(W["W_o"]),
                                  taps["hs"].cpu().numpy(), hmir, own, T=Tq, bf16=cfg.dtype == "bf16")
    finally:
        dr.close()


@pytest.mark.parametrize("name", ["tiny", "bf16"])
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_gated_head_warmup_round_parity(name, T):
    """The gated head with its state warmed up on the token before the anchor
    (local group of 3 tokens): head vectors and candidates against the oracle;
    and the warm-up changes the head's first vector (it is not a no-op)."""
    G = 3
    if name == "tiny":
        cfg = wk.shrink(wk.TINY, R=64, head="gated", G=G, warmup=1)
        W = wk.make_weights(cfg, 35, gain_jitter=True)
        tol = 1e-4
    else:
        cfg = wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=2, n_q=4, n_kv=2, R=128, V=4096, m=6, head="gated", G=G,
                        warmup=1)
        W = wk.make_weights(cfg, 36)
        tol = HIDDEN_REL_TOL
    # a state that matters: larger token embeddings and state weights (powers of two: exact in bf16)
    W = dict(W, E_R=W["E_R"] * 64, W_s=W["W_s"] * 16)
    B, seed = 12, 79
    dr = _drafter(cfg, W, B_max=B)
    try:
        hidden, _, pos = wk.make_round_inputs(wk.WORKLOADS["tiny"], B=B, cfg=cfg)
        group = torch.randint(0, cfg.V, (B, G), generator=torch.Generator().manual_seed(5), dtype=torch.int32)
        out = dr.new_outputs(B, DEV)
        rv = torch.empty(B, cfg.K, cfg.R, device=DEV)
        dr.draft_round(hidden.to(DEV), group.to(DEV), T, seed, pos.to(DEV), out["cand"], out["qstats"],
                       taps={"z": None, "x": None, "b": None, "hs": rv})
        torch.cuda.synchronize()
        cand, rvec = out["cand"].cpu().numpy(), rv.cpu().numpy()
        cands, ocands, gaps, hmir = [], [], [], []
        for b in range(B):
            r = O.draft_request(hidden[b], group[b].tolist(), W, cfg, temperature=T, seed=seed, pos=int(pos[b]),
                                request=b, mirror=(cfg.dtype == "bf16"))
            k = cfg.K if np.array_equal(cand[b], r["cand"]) else int(np.argmax(cand[b] != r["cand"])) + 1
            assert rel_err(rvec[b, :k], r["h"][:k]) < tol, b
            cold = O.gated_head(O.backbone(hidden[b], group[b].tolist(), W, cfg, mirror=(cfg.dtype == "bf16")),
                                int(group[b, -1]), W, T, seed, int(pos[b]), b)
            e_warm, e_cold = rel_err(rvec[b, :1], r["h"][:1]), rel_err(rvec[b, :1], cold["r"][:1])
            assert e_warm < e_cold / 4, (b, e_warm, e_cold)   # the GPU's s_0 is the warmed-up one
            cands.append(cand[b])
            ocands.append(r["cand"])
            gaps.append(r["gap"])
            hmir.append(r["h"])
        Tq = float(np.float32(T))
        own = lambda n, i, ell: O.sample_logits(ell, Tq if T > 0 else 0.0, seed, int(pos[n]) + i + 1, n)[0]
        check_fed_back_candidates(np.stack(cands), np.stack(ocands), np.stack(gaps), O.f64(W["W_o"]), rvec, hmir,
                                  own, T=Tq, bf16=cfg.dtype == "bf16")
    finally:
        dr.close()


def test_gated_head_sampling_verification():
    """Sampling verification with the gated head: q(v) from W_o and the head's
    r vectors kept by the handle; bit-exact against the oracle on identical inputs."""
    cfg = wk.shrink(wk.TINY, R=64, V=512, head="gated")
    W = wk.make_weights(cfg, 33)
    B, T, seed = 64, 0.7, 5
    dr = _drafter(cfg, W, B_max=B)
    try:
        wl = wk.WORKLOADS["tiny"]
        hidden, anchor, pos = wk.make_round_inputs(wl, B=B, cfg=cfg)
        anchor = anchor % cfg.V
        out = dr.new_outputs(B, DEV)
        rvec = torch.empty(B, cfg.K, cfg.R, device=DEV)
        taps = {"z": None, "x": None, "b": None, "hs": rvec}
        dr.draft_round(hidden.to(DEV), anchor.to(DEV), T, seed, pos.to(DEV), out["cand"], out["qstats"], taps=taps)
        p = wk.make_target_probs(B, cfg.K, cfg.V, 9, device=DEV)
        dr.verify_sample(out["cand"], out["qstats"], None, p, T, seed, pos.to(DEV), out["accepted"],
                         out["commits"], out["n_commit"], out["next_anchor"])
        torch.cuda.synchronize()
        cand, qs, rv = out["cand"].cpu().numpy(), out["qstats"].cpu().numpy(), rvec.cpu().numpy()
        acc, com, pn = out["accepted"].cpu().numpy(), out["commits"].cpu().numpy(), p.cpu().numpy()
        for b in range(B):
            o = O.verify_sample(cand[b], qs[b, :, 0], qs[b, :, 1], rv[b], W["W_o"], pn[b], T, seed, int(pos[b]), b)
            assert acc[b] == o["A"] and list(com[b, :o["n_commit"]]) == o["commits"], (b, o)
    finally:
        dr.close()


# ---------------------------------------------------------------- invariants and robustness

def test_history_free_and_deterministic(tiny):
    """Same (hidden, anchor, key) -> bit-identical draft, whatever ran before."""
    wl, W, dr = tiny
    B = 16
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=11)
    args = (hidden.to(DEV), anchor.to(DEV))
    o1 = dr.new_outputs(B, DEV)
    dr.draft_round(*args, 0.7, 5, pos.to(DEV), o1["cand"], o1["qstats"])
    for k in range(5):        # unrelated rounds in between
        h2, a2, p2 = wk.make_round_inputs(wl, B=B, round_index=100 + k)
        o = dr.new_outputs(B, DEV)
        dr.draft_round(h2.to(DEV), a2.to(DEV), 0.7, 9, p2.to(DEV), o["cand"], o["qstats"])
    o2 = dr.new_outputs(B, DEV)
    dr.draft_round(*args, 0.7, 5, pos.to(DEV), o2["cand"], o2["qstats"])
    torch.cuda.synchronize()
    assert torch.equal(o1["cand"], o2["cand"])
    assert torch.equal(o1["qstats"], o2["qstats"])


def test_out_of_range_anchor_flags_status(tiny):
    wl, W, dr = tiny
    B = 2
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=1)
    anchor[1] = wl.cfg.V + 5
    out = dr.new_outputs(B, DEV)
    dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, 0, pos.to(DEV), out["cand"], out["qstats"])
    rc, st = dr.device_status(clear=True)
    assert st & 2 and rc == -5
    rc, st = dr.device_status(clear=True)
    assert rc == 0 and st == 0


def test_graph_capture_matches_eager(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 8
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=2)
    hd, ad, pd = hidden.to(DEV), anchor.to(DEV), pos.to(DEV)
    tgt = wk.make_target_tokens(np.zeros((B, cfg.K), dtype=np.int64), 0.0, cfg.V, 3).to(DEV)
    eager = dr.new_outputs(B, DEV)
    dr.draft_round(hd, ad, 0.0, 0, pd, eager["cand"], eager["qstats"])
    dr.verify(eager["cand"], tgt, eager["accepted"], eager["commits"], eager["n_commit"],
              eager["next_anchor"])
    g_out = dr.new_outputs(B, DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            dr.draft_round(hd, ad, 0.0, 0, pd, g_out["cand"], g_out["qstats"], stream=s)
            dr.verify(g_out["cand"], tgt, g_out["accepted"], g_out["commits"], g_out["n_commit"],
                      g_out["next_anchor"], stream=s)
    graph.replay()
    torch.cuda.synchronize()
    for k in ("cand", "accepted", "commits", "n_commit", "next_anchor"):
        assert torch.equal(eager[k], g_out[k]), k


def test_round_host_matches_device_path(tiny):
    wl, W, dr = tiny
    cfg = wl.cfg
    B = 4
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=4)
    tgt = wk.make_target_tokens(np.zeros((B, cfg.K), dtype=np.int64), 0.0, cfg.V, 3)
    dev = dr.new_outputs(B, DEV)
    dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, 0, pos.to(DEV), dev["cand"], dev["qstats"])
    dr.verify(dev["cand"], tgt.to(DEV), dev["accepted"], dev["commits"], dev["n_commit"],
              dev["next_anchor"])
    host = {k: v.cpu().pin_memory() for k, v in dr.new_outputs(B, "cpu").items()}
    dr.round_host(hidden.pin_memory(), anchor.pin_memory(), pos.pin_memory(), tgt.pin_memory(),
                  None, 0.0, 0, host)
    for k in ("accepted", "commits", "n_commit", "next_anchor"):
        assert torch.equal(dev[k].cpu(), host[k]), k


def test_round_host_sampling_matches_device_path(tiny):
    """Sampling through the host-buffer call: target probabilities in pinned
    (device-mapped, read in place) and in pageable (copied) host memory both
    give the device path's accepted lengths and commits."""
    wl, W, dr = tiny
    cfg = wl.cfg
    B, T, seed = 4, 0.7, 99
    hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=5)
    probs = wk.make_target_probs(B, cfg.K, cfg.V, 5)
    dev = dr.new_outputs(B, DEV)
    dr.draft_round(hidden.to(DEV), anchor.to(DEV), T, seed, pos.to(DEV), dev["cand"], dev["qstats"])
    dr.verify_sample(dev["cand"], dev["qstats"], None, probs.to(DEV), T, seed, pos.to(DEV), dev["accepted"],
                     dev["commits"], dev["n_commit"], dev["next_anchor"])
    for pinned in (True, False):
        host = {k: v.cpu().pin_memory() for k, v in dr.new_outputs(B, "cpu").items()}
        p_h = probs.pin_memory() if pinned else probs.clone()
        dr.round_host(hidden.pin_memory(), anchor.pin_memory(), pos.pin_memory(), None, p_h, T, seed, host)
        for k in ("accepted", "commits", "n_commit", "next_anchor"):
            assert torch.equal(dev[k].cpu(), host[k]), (pinned, k)


# ---------------------------------------------------------------- full-size shapes, sampled

@pytest.mark.parametrize("name", ["qwen3-4b-b1", "qwen3-8b-b32"])
def test_full_size_round_sampled_requests(name):
    """Full-size drafter in the bench's launch configuration; the oracle checks
    two sampled requests end to end (pure for hidden states, mirror for tokens;
    a differing token must be the exact choice of the drafter's own head state
    at a gap within reach of the head-state difference)."""
    wl = wk.WORKLOADS[name]
    cfg = wl.cfg
    B = wl.B
    W = wk.make_weights(cfg, wl.weight_seed, device=DEV)
    dr = binding.Drafter(cfg, W, B_max=B)
    hidden, anchor, pos = wk.make_round_inputs(wl, device=DEV)
    out = dr.new_outputs(B, DEV)
    taps = {"b": torch.empty(B, cfg.K, cfg.D, device=DEV),
            "hs": torch.empty(B, cfg.K, cfg.D, device=DEV)}
    T = wl.temperature
    dr.draft_round(hidden, anchor, T, wl.rng_seed, pos, out["cand"], out["qstats"], taps=taps)
    torch.cuda.synchronize()
    rc, st = dr.device_status()
    assert rc == 0
    Wc = f64_weights(wk.weights_to(W, "cpu"))
    del W
    dr_cand = out["cand"].cpu().numpy()
    sample = [0, B - 1] if B > 1 else [0]
    cands, ocands, gaps, hgpu, hmir = [], [], [], [], []
    for b in sample:
        pure = O.draft_request(hidden[b].cpu(), int(anchor[b]), Wc, cfg, temperature=T,
                               seed=wl.rng_seed, pos=int(pos[b]), request=b, mirror=False)
        tm = {}
        mir = O.draft_request(hidden[b].cpu(), int(anchor[b]), Wc, cfg, temperature=T,
                              seed=wl.rng_seed, pos=int(pos[b]), request=b, mirror=True, taps=tm)
        assert rel_err(taps["b"][b].cpu(), pure["b"]) < HIDDEN_REL_TOL
        assert rel_err(taps["hs"][b].cpu(), pure["h"]) < HIDDEN_REL_TOL
        cands.append(dr_cand[b])
        ocands.append(mir["cand"])
        gaps.append(mir["gap"])
        hgpu.append(taps["hs"][b].cpu().numpy())
        hmir.append(tm["h"])
    # bf16 activations: a differing candidate must be the exact choice of the
    # drafter's own head state, at a gap the head-state difference can bridge
    Tq = float(np.float32(T))
    own = lambda n, i, ell: O.sample_logits(ell, Tq if T > 0 else 0.0, wl.rng_seed,
                                            int(pos[sample[n]]) + i + 1, sample[n])[0]
    check_candidates_bf16(np.stack(cands), np.stack(ocands), np.stack(gaps), Wc["E"], hgpu, hmir, own, T=Tq)
    dr.close()


# ---------------------------------------------------------------- history-KV control

def _history_cfg(name, H):
    if name == "d128":   # 4 query heads per key/value head, as in the 8B shape: 32 query rows per head
        return wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=2, n_q=8, n_kv=2, R=64, V=4096, m=6, history=H)
    if name == "d128wide":   # 8 query heads x 9 local rows = 72 query rows per head: one key split per tile
        return wk.shrink(wk.QWEN3_8B, D=512, F=1024, L_D=1, n_q=16, n_kv=2, K=8, R=64, V=4096, m=6, history=H)
    return wk.shrink(wk.TINY, dtype="bf16", history=H)   # d_h = 64, 2 heads per group


@pytest.mark.parametrize("name", ["d128", "d64"])
def test_history_fill_matches_oracle(name):
    """The synthetic history in every ring, bit for bit, and the cursors at 0."""
    H = 80
    cfg = _history_cfg(name, H)
    dr = _drafter(cfg, wk.make_weights(cfg, 41), B_max=3)
    try:
        for l in range(cfg.L_D):
            for b in range(3):
                for which in (0, 1):
                    ring, cur = dr.history_read(l, b, which)
                    got = ring.float().cpu().numpy().transpose(1, 0, 2)
                    ref = O.history_values(H, cfg.n_kv, cfg.d_h, l, b, which)
                    assert np.array_equal(got, ref), (l, b, which)
                    assert cur == 0
    finally:
        dr.close()


@pytest.mark.parametrize("name,H", [("d128", 300), ("d128", 64), ("d64", 200), ("d64", 12), ("d128wide", 150)])
def test_history_round_parity(name, H):
    """Three rounds of the history-KV control (the 12-row ring wraps): hidden rows and candidates against
    the oracle drafter attending over its own ring (bf16 activations: a differing
    candidate must be the exact choice of the drafter's own head state at a
    near-tie that the head-state difference explains), then each ring after the
    append (slots no round has written bit-exact, the written rows within the
    hidden tolerance: the appended rows are the drafter's own) and the cursors."""
    cfg = _history_cfg(name, H)
    W = wk.make_weights(cfg, 42)
    wl = wk.WORKLOADS["tiny"]
    B = 4
    dr = _drafter(cfg, W, B_max=B)
    K1 = cfg.G + cfg.K
    E64 = O.f64(W["E"])
    try:
        hist = [O.HistoryCache(cfg, H, b) for b in range(B)]
        written = np.zeros((B, H), dtype=bool)
        for rnd in range(3):
            hidden, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=rnd, cfg=cfg)
            anchor = anchor % cfg.V
            out = dr.new_outputs(B, DEV)
            taps = {"z": torch.empty(B, cfg.m, cfg.D, device=DEV),
                    "x": torch.empty(cfg.L_D, B, K1, cfg.D, device=DEV),
                    "b": torch.empty(B, cfg.K, cfg.D, device=DEV),
                    "hs": torch.empty(B, cfg.K, cfg.D, device=DEV)}
            dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, 0, pos.to(DEV), out["cand"], out["qstats"],
                           taps=taps)
            torch.cuda.synchronize()
            cursor0 = [hc.cursor for hc in hist]
            cands, ocands, gaps, hmir = [], [], [], []
            for b in range(B):
                t = {}
                r = O.draft_request(hidden[b], int(anchor[b]), W, cfg, taps=t, mirror=True, history=hist[b])
                for l in range(cfg.L_D):
                    assert rel_err(taps["x"][l, b].cpu(), t["x"][l]) < HIDDEN_REL_TOL, (rnd, b, l)
                assert rel_err(taps["b"][b].cpu(), t["b"]) < HIDDEN_REL_TOL
                cands.append(out["cand"][b].cpu().numpy())
                ocands.append(r["cand"])
                gaps.append(r["gap"])
                hmir.append(t["h"])
            check_candidates_bf16(np.stack(cands), np.stack(ocands), np.stack(gaps), E64,
                                  taps["hs"].cpu().numpy(), hmir, lambda n, i, ell: int(np.argmax(ell)))
            for b in range(B):
                written[b, (cursor0[b] + np.arange(K1)) % H] = True   # rows of this and earlier rounds
                slots, keep = written[b], ~written[b]
                for l in range(cfg.L_D):
                    for which, ref in ((0, hist[b].k[l]), (1, hist[b].v[l])):
                        ring, cur = dr.history_read(l, b, which)
                        got = ring.float().cpu().numpy().transpose(1, 0, 2)
                        assert np.array_equal(got[keep], ref[keep]), (rnd, b, l, which)
                        assert rel_err(got[slots], ref[slots]) < HIDDEN_REL_TOL, (rnd, b, l, which)
                        assert cur == hist[b].cursor == (cursor0[b] + K1) % H
    finally:
        dr.close()


def test_history_calls_need_a_ring(tiny):
    """A drafter built with history = 0 keeps no ring: the history calls refuse it."""
    wl, W, dr = tiny
    with pytest.raises(binding.DliteError):
        dr.history_reset()


def test_full_size_history_round_sampled_requests():
    """The 8B-shape history-KV control at B = 8 with an 8192-row ring, in the
    bench's launch configuration: two sampled requests against the oracle
    drafter attending over its own ring (pure for hidden states, mirror for
    tokens; a differing token must be the exact choice of the drafter's own
    head state at a gap within reach of the head-state difference), and their
    rings after the append."""
    H = 8192
    wl = wk.WORKLOADS["qwen3-8b-history"]
    cfg = wk.shrink(wl.cfg, history=H)
    B = wl.B
    K1 = cfg.G + cfg.K
    W = wk.make_weights(cfg, wl.weight_seed, device=DEV)
    dr = binding.Drafter(cfg, W, B_max=B)
    hidden, anchor, pos = wk.make_round_inputs(wl, device=DEV)
    out = dr.new_outputs(B, DEV)
    taps = {"b": torch.empty(B, cfg.K, cfg.D, device=DEV), "hs": torch.empty(B, cfg.K, cfg.D, device=DEV)}
    dr.draft_round(hidden, anchor, 0.0, wl.rng_seed, pos, out["cand"], out["qstats"], taps=taps)
    torch.cuda.synchronize()
    rc, st = dr.device_status()
    assert rc == 0 and st == 0
    Wc = f64_weights(wk.weights_to(W, "cpu"))
    del W
    cands, ocands, gaps, hgpu, hmir = [], [], [], [], []
    for b in (1, B - 1):
        hp = O.HistoryCache(cfg, H, b)
        hm = O.HistoryCache(cfg, H, b)
        pure = O.draft_request(hidden[b].cpu(), int(anchor[b]), Wc, cfg, mirror=False, history=hp)
        tm = {}
        mir = O.draft_request(hidden[b].cpu(), int(anchor[b]), Wc, cfg, mirror=True, history=hm, taps=tm)
        assert rel_err(taps["b"][b].cpu(), pure["b"]) < HIDDEN_REL_TOL
        cands.append(out["cand"][b].cpu().numpy())
        ocands.append(mir["cand"])
        gaps.append(mir["gap"])
        hgpu.append(taps["hs"][b].cpu().numpy())
        hmir.append(tm["h"])
        for l in range(cfg.L_D):
            ring, cur = dr.history_read(l, b, 0)
            got = ring.float().cpu().numpy().transpose(1, 0, 2)
            assert cur == K1 and hm.cursor == K1
            assert np.array_equal(got[K1:], hm.k[l][K1:])
            assert rel_err(got[:K1], hm.k[l][:K1]) < HIDDEN_REL_TOL
    # bf16 activations: a differing candidate must be the exact choice of the
    # drafter's own head state, at a gap the head-state difference can bridge
    check_candidates_bf16(np.stack(cands), np.stack(ocands), np.stack(gaps), Wc["E"], hgpu, hmir,
                          lambda n, i, ell: int(np.argmax(ell)))
    dr.close()


def test_history_ring_memory_matches_draft_kv_formula():
    """The control's device memory grows by the draft-KV formula 2 L_D H n_kv d_h b
    per request slot (DLite 完全拆解, §"本轮临时 K/V 仍然需要计算", eq. M_draftKV).
    Two ring sizes: the difference of what their handles hold equals the
    formula's difference up to the rounding of the two ring allocations (2 MiB
    each), so the rest of the control's workspace (block rows behind each ring,
    staged queries, chunk partials) does not grow with H; and the larger ring's
    handle holds at least the formula more than the history-free handle."""
    H1, H2, Bm = 32768, 65536, 4
    cfg0, cfg1, cfg2 = (_history_cfg("d128", H) for H in (0, H1, H2))
    W = wk.make_weights(cfg2, 43)
    Wd = wk.weights_to(W, DEV)
    held = []
    drs = []
    try:
        for cfg in (cfg0, cfg1, cfg2):
            torch.cuda.synchronize()
            f0 = torch.cuda.mem_get_info()[0]
            drs.append(binding.Drafter(cfg, Wd, B_max=Bm))
            torch.cuda.synchronize()
            held.append(f0 - torch.cuda.mem_get_info()[0])
        formula = lambda H: 2 * cfg2.L_D * H * cfg2.n_kv * cfg2.d_h * 2 * Bm
        step = held[2] - held[1]
        assert abs(step - (formula(H2) - formula(H1))) <= (4 << 20), (step, formula(H2) - formula(H1))
        assert held[2] - held[0] >= formula(H2), (held, formula(H2))
    finally:
        for d in drs:
            d.close()
