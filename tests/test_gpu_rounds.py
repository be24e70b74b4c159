"""GPU: round bookkeeping, the synthetic target of the acceptance workloads and
the bounded device waits, through the C ABI against the CPU oracle.

  * dlite_synthetic_target: bit-exact against the oracle's statement of the
    acceptance model (table selection by the device round counter included);
  * chained rounds replayed from one captured graph (draft, synthetic target,
    greedy verification, position advance): target tokens, A, commits and the
    positions pos + sum n_commit bit-exact against the oracle on the GPU's own
    candidates, and the candidates within the tie band of the oracle's draft;
  * the bounded waits: a wait nobody answers gives up after its limit, flags
    DLITE_ERR_DEVICE_TIMEOUT, a following kernel sees the flag, and the
    context stays usable.
"""
import numpy as np
import pytest
import torch

from history_free_speculative_gb300 import binding
from history_free_speculative_gb300 import workload as wk
from oracle import dlite_oracle as O
from parity import check_candidates

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_synthetic_target_matches_oracle():
    B, K, V, NT, seed = 64, 7, 151936, 3, 77
    c = wk.make_beta_accept(B, K, 5, n_tables=NT).to(torch.float32)   # [NT, B, K]
    rng = np.random.default_rng(8)
    ctr = torch.zeros(1, dtype=torch.int32, device=DEV)
    tgt = torch.empty(B, K + 1, dtype=torch.int32, device=DEV)
    for call in range(4):
        cand = rng.integers(0, V, (B, K))
        pos = rng.integers(0, 1 << 30, B)
        binding.synthetic_target(torch.from_numpy(cand.astype(np.int32)).to(DEV), c.to(DEV), seed,
                                 torch.from_numpy(pos).to(DEV), tgt, V, round_counter=ctr)
        torch.cuda.synchronize()
        got = tgt.cpu().numpy()
        for b in range(B):
            want = O.synthetic_target_tokens(cand[b], c[call % NT, b].numpy(), seed, int(pos[b]), b, V)
            assert list(got[b]) == want, (call, b)
    assert int(ctr.item()) == 4


def test_synthetic_target_rejects_bad_arguments():
    z = torch.zeros(2, 3, dtype=torch.int32, device=DEV)
    c = torch.zeros(1, 2, 3, dtype=torch.float32, device=DEV)
    pos = torch.zeros(2, dtype=torch.int64, device=DEV)
    out = torch.empty(2, 4, dtype=torch.int32, device=DEV)
    with pytest.raises(binding.DliteError) as e:
        binding.synthetic_target(z, c, 1, pos, out, 1)   # V < 2
    assert e.value.code == -1


def test_chained_graph_rounds_advance_positions():
    """Four rounds from one captured graph: the anchor is the previous round's
    next anchor (written in place), pos += n_commit on the device."""
    wl = wk.WORKLOADS["tiny"]
    cfg = wl.cfg
    B, R = wl.B, 4
    W = wk.make_weights(cfg, wl.weight_seed)
    dr = binding.Drafter(cfg, wk.weights_to(W, DEV), B_max=B)
    try:
        hidden, anchor, pos = wk.make_round_inputs(wl, round_index=3)
        hd, ad, pd = hidden.to(DEV), anchor.to(DEV), pos.to(DEV)
        c = torch.full((1, B, cfg.K), 0.8, dtype=torch.float32, device=DEV)
        ctr = torch.zeros(1, dtype=torch.int32, device=DEV)
        tgt = torch.empty(B, cfg.K + 1, dtype=torch.int32, device=DEV)
        out = dr.new_outputs(B, DEV)
        s = torch.cuda.Stream(device=DEV)

        def enqueue():
            dr.draft_round(hd, ad, 0.0, wl.rng_seed, pd, out["cand"], out["qstats"], stream=s)
            binding.synthetic_target(out["cand"], c, wl.rng_seed, pd, tgt, cfg.V, round_counter=ctr, stream=s)
            dr.verify(out["cand"], tgt, out["accepted"], out["commits"], out["n_commit"], ad, stream=s)
            dr.advance(out["n_commit"], pd, stream=s)

        a0, p0 = ad.clone(), pd.clone()
        with torch.cuda.stream(s):   # eager round (sets kernel attributes), then undo its effects
            enqueue()
        s.synchronize()
        ad.copy_(a0)
        pd.copy_(p0)
        ctr.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                enqueue()
        s.synchronize()
        o_anchor = anchor.numpy().astype(np.int64)
        o_pos = pos.numpy().astype(np.int64)
        total_commit = 0
        for r in range(R):
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
            cand = out["cand"].cpu().numpy()
            ref = O.draft_round(hidden, o_anchor, W, cfg)
            check_candidates(cand, np.stack([ref[b]["cand"] for b in range(B)]),
                             np.stack([ref[b]["gap"] for b in range(B)]))
            got_t = tgt.cpu().numpy()
            acc = out["accepted"].cpu().numpy()
            com = out["commits"].cpu().numpy()
            for b in range(B):
                t = O.synthetic_target_tokens(cand[b], np.full(cfg.K, 0.8, dtype=np.float32), wl.rng_seed,
                                              int(o_pos[b]), b, cfg.V)
                assert list(got_t[b]) == t, (r, b)
                v = O.verify_greedy(cand[b], t)
                assert acc[b] == v["A"] and list(com[b, :v["n_commit"]]) == v["commits"], (r, b)
                o_anchor[b] = v["next_anchor"]
                o_pos[b] += v["n_commit"]
                total_commit += v["n_commit"]
            assert np.array_equal(ad.cpu().numpy(), o_anchor), r
            assert np.array_equal(pd.cpu().numpy(), o_pos), r
        assert int(ctr.item()) == R
        assert total_commit > R * B     # some candidates were accepted (c = 0.8)
        rc, st = dr.device_status()
        assert rc == 0 and st == 0
    finally:
        dr.close()


def test_bounded_wait_gives_up_and_flags_timeout():
    """A wait nobody answers returns after its ~1 ms limit with the timeout bit
    set; a following kernel sees the bit (the engines then skip their work);
    the status reads DLITE_ERR_DEVICE_TIMEOUT once and the context stays usable."""
    wl = wk.WORKLOADS["tiny"]
    cfg = wl.cfg
    W = wk.make_weights(cfg, wl.weight_seed)
    dr = binding.Drafter(cfg, wk.weights_to(W, DEV), B_max=wl.B)
    try:
        res = torch.zeros(3, dtype=torch.int32, device=DEV)
        import time
        t0 = time.perf_counter()
        dr.selftest_wait(1_000_000, res)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert res.tolist() == [1, 1, 1]
        assert dt < 5.0, dt
        rc, st = dr.device_status(clear=True)
        assert rc == -4 and st & 1
        rc, st = dr.device_status(clear=False)
        assert rc == 0 and st == 0
        # a normal round after the probe runs and matches the oracle
        hidden, anchor, pos = wk.make_round_inputs(wl)
        out = dr.new_outputs(wl.B, DEV)
        dr.draft_round(hidden.to(DEV), anchor.to(DEV), 0.0, wl.rng_seed, pos.to(DEV), out["cand"], out["qstats"])
        torch.cuda.synchronize()
        ref = O.draft_round(hidden, anchor.numpy(), W, cfg)
        check_candidates(out["cand"].cpu().numpy(), np.stack([ref[b]["cand"] for b in range(wl.B)]),
                         np.stack([ref[b]["gap"] for b in range(wl.B)]))
        assert dr.device_status()[0] == 0
        with pytest.raises(binding.DliteError):
            dr.selftest_wait(0, res)
    finally:
        dr.close()
