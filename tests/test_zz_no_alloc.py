"""The allocation-free sampling verification against the handle-based entry point
and against the oracle.

dlite_verify_sample_static serves callers that cannot allocate device memory
where they verify; it keeps its fallback scratch in a static device array
shared by all calls. This file is collected last on purpose, so that a run
stopping at the first failure has already run every other test.

Two calls in a row with different batch sizes and vocabularies: the second
call's residual rows sit at other offsets of the shared array than the first
call's, so a row it failed to rewrite would be read with the first call's
contents and change its draws. Each call is compared with the handle path and
with the oracle's sampling verification request by request, and the oracle
shows that the exact fallback (the only reader of the scratch) ran.
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
T = 0.7


def _inputs(cfg, W, B, seed, overlap):
    rng = np.random.default_rng(seed)
    hs = rng.normal(0, 1.0, (B, cfg.K, cfg.D)).astype(np.float32)
    ell = O.lm_logits(hs.reshape(-1, cfg.D), O.f64(W["E"])).reshape(B, cfg.K, cfg.V)
    Tq = float(np.float32(T))
    lse = np.log(np.exp(ell / Tq).sum(axis=2))
    pos = rng.integers(0, 1 << 20, B)
    cand = np.empty((B, cfg.K), dtype=np.int64)
    for b in range(B):
        for i in range(cfg.K):
            cand[b, i] = np.argmax(ell[b, i] / Tq + ph.gumbel_row(9, pos[b] + i + 1, b, cfg.V))
    q = np.exp(ell / Tq - lse[..., None])
    p = np.empty((B, cfg.K + 1, cfg.V))
    for b in range(B):
        for j in range(cfg.K + 1):
            p[b, j] = overlap * q[b, min(j, cfg.K - 1)] + (1 - overlap) * rng.dirichlet(np.ones(cfg.V))
    p = (p / p.sum(axis=2, keepdims=True)).astype(np.float32)
    logit_d = np.take_along_axis(ell, cand[..., None], 2)[..., 0].astype(np.float32)
    lse = lse.astype(np.float32)
    return dict(cand=cand, logit_d=logit_d, lse=lse, hs=hs, p=p, pos=pos)


def _dev(a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a if dt is None else a.astype(dt))).to(DEV)


@pytest.mark.parametrize("order", ["small_first", "large_first"])
def test_static_scratch_verify_matches_handle_path_and_oracle(order):
    # fp32 drafters, so the handle's verification reads the same fp32 row-major E
    calls = [(64, 512, 101), (256, 96, 202)]
    if order == "large_first":
        calls = calls[::-1]
    for call, (V, B, seed) in enumerate(calls):
        cfg = wk.shrink(wk.TINY, V=V, K=3, D=64, F=128, R=32, n_q=2, n_kv=1, m=2)
        W = wk.make_weights(cfg, 19 + V)
        x = _inputs(cfg, W, B, seed, 0.97)
        qs = np.stack([x["logit_d"], x["lse"]], axis=-1)
        cand, qsd, hs, p, pos = (_dev(x["cand"], np.int32), _dev(qs), _dev(x["hs"]), _dev(x["p"]),
                                 _dev(x["pos"], np.int64))
        dr = binding.Drafter(cfg, wk.weights_to(W, DEV), B_max=B)
        try:
            ref = dr.new_outputs(B, DEV)
            dr.verify_sample(cand, qsd, hs, p, T, seed, pos, ref["accepted"], ref["commits"], ref["n_commit"],
                             ref["next_anchor"])
            got = dr.new_outputs(B, DEV)
            E = W["E"].to(DEV).float().contiguous()
            binding.verify_sample_static(cand, qsd, hs, E, p, T, seed, pos, got["accepted"], got["commits"],
                                         got["n_commit"], got["next_anchor"])
            torch.cuda.synchronize()
            for k in ("accepted", "commits", "n_commit", "next_anchor"):
                assert torch.equal(ref[k], got[k]), (call, k)
        finally:
            dr.close()
        acc = got["accepted"].cpu().numpy()
        com = got["commits"].cpu().numpy()
        hows = {}
        for b in range(B):
            r = O.verify_sample(x["cand"][b], x["logit_d"][b], x["lse"][b], x["hs"][b], W["E"], x["p"][b], T, seed,
                                int(x["pos"][b]), b)
            hows[r["how"]] = hows.get(r["how"], 0) + 1
            assert acc[b] == r["A"], (call, b, acc[b], r)
            assert list(com[b, :r["n_commit"]]) == r["commits"], (call, b, com[b], r)
        assert hows.get("fallback", 0) > 0, (call, hows)   # the scratch-backed exact draw ran


def test_static_scratch_rejects_oversize_and_bad_arguments():
    B, K, V, D = 16, 3, 131072, 64   # B * V = 2^21 > the 2^20-entry scratch
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=DEV)
    args = lambda E: (z(B, K, dt=torch.int32), z(B, K, 2), z(B, K, D), E, z(B, K + 1, V), 0.7, 1,
                      z(B, dt=torch.int64), z(B, dt=torch.int32), z(B, K + 1, dt=torch.int32),
                      z(B, dt=torch.int32), z(B, dt=torch.int32))
    with pytest.raises(binding.DliteError) as e:
        binding.verify_sample_static(*args(z(V, D)))
    assert e.value.code == -2
    with pytest.raises(ValueError):   # bf16 LM-head weights are not what this call reads
        binding.verify_sample_static(*args(z(V, D, dt=torch.bfloat16)))
