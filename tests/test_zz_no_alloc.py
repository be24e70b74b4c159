"""The allocation-free sampling verification against the handle-based entry point.

dlite_verify_sample_static serves callers that cannot allocate device memory
where they verify; it keeps its fallback scratch in a static device array
shared by all calls. This file is collected last on purpose, so that a run
stopping at the first failure has already run every other test. It checks
two calls in a row (the second must not see the first one's scratch).
"""
import numpy as np
import pytest
import torch

from history_free_speculative_gb300 import binding
from history_free_speculative_gb300 import workload as wk
from oracle import dlite_oracle as O
from oracle import philox as ph

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(cfg, W, B, seed, overlap):
    rng = np.random.default_rng(seed)
    hs = rng.normal(0, 1.0, (B, cfg.K, cfg.D))
    ell = O.lm_logits(hs.reshape(-1, cfg.D), O.f64(W["E"])).reshape(B, cfg.K, cfg.V)
    T = float(np.float32(0.7))
    lse = np.log(np.exp(ell / T).sum(axis=2))
    pos = rng.integers(0, 1 << 20, B)
    cand = np.empty((B, cfg.K), dtype=np.int64)
    for b in range(B):
        for i in range(cfg.K):
            cand[b, i] = np.argmax(ell[b, i] / T + ph.gumbel_row(9, pos[b] + i + 1, b, cfg.V))
    q = np.exp(ell / T - lse[..., None])
    p = np.empty((B, cfg.K + 1, cfg.V))
    for b in range(B):
        for j in range(cfg.K + 1):
            p[b, j] = overlap * q[b, min(j, cfg.K - 1)] + (1 - overlap) * rng.dirichlet(np.ones(cfg.V))
    p = (p / p.sum(axis=2, keepdims=True)).astype(np.float32)
    logit_d = np.take_along_axis(ell, cand[..., None], 2)[..., 0]
    qs = np.stack([logit_d, lse], axis=-1).astype(np.float32)
    t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.astype(dt))).to(DEV)
    return dict(cand=t(cand, np.int32), qs=t(qs), hs=t(hs, np.float32), p=t(p), pos=t(pos, np.int64))


def test_static_scratch_verify_matches_handle_path():
    # fp32 drafter so the handle's verification reads the same fp32 row-major E
    cfg = wk.shrink(wk.TINY, V=64, K=3, D=64, F=128, R=32, n_q=2, n_kv=1, m=2)
    W = wk.make_weights(cfg, 19)
    B = 512
    dr = binding.Drafter(cfg, wk.weights_to(W, DEV), B_max=B)
    E = W["E"].to(DEV).float().contiguous()
    try:
        dr.counters(reset=True)
        for call, (seed, overlap) in enumerate([(101, 0.97), (202, 0.9)]):
            x = _inputs(cfg, W, B, seed, overlap)
            ref = dr.new_outputs(B, DEV)
            dr.verify_sample(x["cand"], x["qs"], x["hs"], x["p"], 0.7, seed, x["pos"], ref["accepted"],
                             ref["commits"], ref["n_commit"], ref["next_anchor"])
            got = dr.new_outputs(B, DEV)
            binding.verify_sample_static(x["cand"], x["qs"], x["hs"], E, x["p"], 0.7, seed, x["pos"],
                                         got["accepted"], got["commits"], got["n_commit"],
                                         got["next_anchor"])
            torch.cuda.synchronize()
            for k in ("accepted", "commits", "n_commit", "next_anchor"):
                assert torch.equal(ref[k], got[k]), (call, k)
        # the scratch-backed exact fallback really ran
        assert dr.counters()["fallback"] > 0
    finally:
        dr.close()


def test_static_scratch_rejects_oversize():
    B, K, V, D = 16, 3, 131072, 64   # B * V = 2^21 > the 2^20-entry scratch
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=DEV)
    with pytest.raises(binding.DliteError) as e:
        binding.verify_sample_static(z(B, K, dt=torch.int32), z(B, K, 2), z(B, K, D), z(V, D),
                                     z(B, K + 1, V), 0.7, 1, z(B, dt=torch.int64),
                                     z(B, dt=torch.int32), z(B, K + 1, dt=torch.int32),
                                     z(B, dt=torch.int32), z(B, dt=torch.int32))
    assert e.value.code == -2
