"""Byte and FLOP accounting of the bench (CPU): the draft-memory figures of the
history-cost workload and the per-launch bytes of the history attention.

The draft KV of the control drafter is 2 L_D H n_kv d_h values per request
(DLite 完全拆解, §"本轮临时 K/V 仍然需要计算", eq. M_draftKV ≈ 2 L_D H n_kv d_h b; bf16):
at the 8B shape (L_D 3, 8 KV heads of 128) 100.7 MB at H = 8192, 503.3 MB at
H = 40960 and 1.450 GB at H = 118000, per request.
"""
import dataclasses

import pytest

from history_free_speculative_gb300 import reporter as rp
from history_free_speculative_gb300 import workload as wk

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("H,mb", [(8192, 100.7), (40960, 503.3), (118000, 1450.0)])
def test_draft_kv_bytes_per_request(H, mb):
    cfg = dataclasses.replace(wk.QWEN3_8B, history=H)
    per_request = 2 * cfg.L_D * H * cfg.n_kv * cfg.d_h * 2
    assert per_request / 1e6 == pytest.approx(mb, rel=2e-3)
    # the round reads every ring once and writes the round's G + K rows into it
    K1 = cfg.G + cfg.K
    assert rp.history_bytes(cfg, 1) == per_request + 2 * cfg.L_D * K1 * cfg.n_kv * cfg.d_h * 2


def test_history_free_round_has_no_history_bytes():
    cfg = wk.QWEN3_8B
    assert rp.history_bytes(cfg, 32) == 0
    with_h = dataclasses.replace(cfg, history=512)
    assert rp.round_bytes(with_h, 8) - rp.round_bytes(cfg, 8) == rp.history_bytes(with_h, 8)
    assert rp.round_flops(with_h, 8) > rp.round_flops(cfg, 8)


def test_hist_attn_bytes_one_layer():
    cfg = dataclasses.replace(wk.QWEN3_8B, history=40960)
    B = 8
    K1 = cfg.G + cfg.K
    Tk = cfg.m + K1
    rows = cfg.n_q // cfg.n_kv * K1
    ring_and_block = B * cfg.n_kv * (cfg.history + Tk) * cfg.d_h * 2 * 2   # keys and values, bf16
    queries = B * cfg.n_kv * rows * cfg.d_h * 2
    assert rp.hist_attn_bytes(cfg, B) == ring_and_block + queries
    # three launches per round read the whole draft KV of the 8 requests once
    assert 3 * rp.hist_attn_bytes(cfg, B) == pytest.approx(rp.history_bytes(cfg, B), rel=2e-3)


def test_gated_projection_bytes():
    cfg = dataclasses.replace(wk.QWEN3_8B, head="gated")
    assert rp.gated_lm_bytes(cfg, 32) == cfg.V * cfg.R * 2 + 32 * cfg.R * 2
    assert rp.gated_lm_flops(cfg, 32) == 2 * 32 * cfg.R * cfg.V
