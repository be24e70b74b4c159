"""Shared comparison helpers for the GPU-vs-oracle parity tests."""
import numpy as np

HIDDEN_REL_TOL = 2e-2      # hidden representations, relative L2 error
CAND_MATCH_MIN = 0.999     # fraction of identical candidate tokens
CAND_GAP_TOL = 1e-3        # a mismatch is allowed only where the oracle's top-2 gap is below this


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def check_candidates(cand, ocand, ogap, gap_tol=CAND_GAP_TOL, min_match=CAND_MATCH_MIN):
    cand = np.asarray(cand)
    ocand = np.asarray(ocand)
    ogap = np.asarray(ogap)
    bad = cand != ocand
    frac = 1.0 - bad.mean()
    assert np.all(ogap[bad] < gap_tol), (
        f"candidate mismatch outside the tie band: gaps {ogap[bad]}, "
        f"gpu {cand[bad]}, oracle {ocand[bad]}")
    # >= 99.9% identical; on samples under 1000 tokens one tie-band mismatch is allowed
    allowed = max(1, int((1.0 - min_match) * cand.size))
    assert bad.sum() <= allowed, f"only {frac:.4%} identical ({bad.sum()} of {cand.size})"
    return int(bad.sum()), frac


def f64_weights(W):
    """fp64 numpy copy of a weight dict (speeds up repeated oracle calls)."""
    from oracle.dlite_oracle import f64
    out = {k: f64(v) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: f64(v) for k, v in l.items()} for l in W["layers"]]
    return out


def check_candidates_bf16(cand, ocand, ogap, E, h_gpu, h_mir, own_choice, T=0.0, max_frac=0.02):
    """Candidates of a drafter with bf16 backbone activations against the mirror oracle.

    Both round the activations to bf16 at the same points, but once an input of
    one rounding differs in its last fp32 bits (another accumulation order) the
    two sides' rounding decisions decorrelate: the head states differ by a
    bf16-noise amount and a near-tie can go either way. Each mismatch must
    (1) be the exact choice of the drafter's own head state, own_choice(n, i,
    E h_gpu[n, i]) in float64, and (2) sit where the mirror's gap is within
    reach of the head-state difference: a logit shift of at most
    s = max_v |E (h_gpu - h_mir)| moves a greedy top-2 gap by at most 2 s, a
    chunk-score gap of the two-level draw by at most 2 s / T and a CDF step
    inside a chunk by at most exp(2 s / T) - 1. At most max_frac of the
    candidates may differ (one on samples under 1 / max_frac).
    """
    cand, ocand, ogap = np.asarray(cand), np.asarray(ocand), np.asarray(ogap)
    E = np.asarray(E, dtype=np.float64)
    bad = np.argwhere(cand != ocand)
    for n, i in bad:
        hg = np.asarray(h_gpu[n][i], dtype=np.float64)
        assert own_choice(n, i, E @ hg) == cand[n, i], ("not the exact choice of its own head state", n, i)
        s = float(np.abs(E @ (hg - np.asarray(h_mir[n][i], dtype=np.float64))).max())
        reach = 2.0 * s if T == 0 else float(np.expm1(2.0 * s / T))
        assert ogap[n, i] < reach, ("a gap the head-state difference cannot bridge", n, i, ogap[n, i], reach)
    allowed = max(1, int(max_frac * cand.size))
    assert len(bad) <= allowed, f"{len(bad)} of {cand.size} candidates differ"
    return len(bad)


def check_fed_back_candidates(cand, ocand, ogap, E, h_gpu, h_mir, own_choice, T=0.0, bf16=True):
    """Candidates of a head that feeds each step's token into the next step (the
    gated head): after a request's first differing token the two sides draft from
    different prefixes, so the positions past it are not compared; the first
    difference itself is checked like any other (check_candidates_bf16 for bf16
    activations, the tie band otherwise)."""
    cand, ocand = np.array(cand), np.asarray(ocand)
    for n in range(cand.shape[0]):
        bad = np.nonzero(cand[n] != ocand[n])[0]
        if len(bad):
            cand[n, bad[0] + 1:] = ocand[n, bad[0] + 1:]
    if bf16:
        return check_candidates_bf16(cand, ocand, ogap, E, h_gpu, h_mir, own_choice, T)
    return check_candidates(cand, ocand, ogap)
