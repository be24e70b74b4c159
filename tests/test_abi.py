"""The C ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

import pytest

from history_free_speculative_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dlite_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def so():
    path = build.build()
    return ctypes.CDLL(path)


def test_every_declared_symbol_is_exported(so):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(so, n), n


def test_binding_covers_declared_symbols():
    assert sorted(binding.EXPORTED) == _declared()


def test_missing_library_fails_loudly():
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError):
            binding.load("/nonexistent/libdlite.so")
    finally:
        binding._lib = saved


def test_host_side_validation_needs_no_gpu(so):
    """Argument errors are returned before any CUDA call is made."""
    lib = binding.load()
    h = ctypes.c_void_p()
    assert lib.dlite_create(None, None, ctypes.byref(h)) == -1
    bad = binding.Config(B_max=1, D=100, m=4, K=4, L_D=1, n_q=4, n_kv=2, d_h=64, F=768, R=32,
                         V=2048, dtype=0, rms_eps=1e-6, rope_theta=1e6)
    w = binding.Weights()
    for n in ("e_depth", "g_stage", "e_ph", "E", "g_final", "Q", "P"):
        setattr(w, n, 1)
    assert lib.dlite_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == -2
    bad.D = 256
    bad.m = 30   # m + K + 1 > 32: block does not fit one warp of keys
    assert lib.dlite_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == -2
    assert lib.dlite_draft_round(None, 1, None, None, 0.0, 0, None, None, None, None) == -1
    assert lib.dlite_verify(None, 1, None, None, None, None, None, None, None) == -1
    assert lib.dlite_status_string(-2) == b"unsupported shape"
    lib.dlite_destroy(None)


@pytest.mark.parametrize("field,value,code", [
    ("history", -1, -1),            # negative history: invalid
    ("history", 2, -2),             # a ring shorter than the round's G + K rows
    ("history", (1 << 20) + 1, -2),  # past the synthetic history's counter range
    ("anchor_group", 9, -2),        # local token group longer than 8
    ("head_type", 2, -1),           # no such head
    ("R", 96, -2),                  # gated head: R must be a multiple of 64 (with head_type 1 below)
    ("act_planes", 3, -1),          # activation planes: 1 (bf16) or 2 (fp32-class)
    ("act_planes", -1, -1),
])
def test_config_checks_need_no_gpu(so, field, value, code):
    """The history, group and head fields of dlite_config are checked before any CUDA call."""
    lib = binding.load()
    h = ctypes.c_void_p()
    cfg = binding.Config(B_max=1, D=256, m=4, K=4, L_D=1, n_q=4, n_kv=2, d_h=64, F=768, R=64,
                         V=2048, dtype=1, rms_eps=1e-6, rope_theta=1e6, anchor_group=1, head_type=0,
                         history=0)
    setattr(cfg, field, value)
    if field == "R":
        cfg.head_type = 1
    w = binding.Weights()
    for n in ("e_depth", "g_stage", "e_ph", "E", "g_final", "Q", "P"):
        setattr(w, n, 1)
    for n in binding.GATED_FIELDS:
        setattr(w.gated, n, 1)
    assert lib.dlite_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == code


def test_history_needs_bf16_and_few_query_rows(so):
    lib = binding.load()
    h = ctypes.c_void_p()
    w = binding.Weights()
    for n in ("e_depth", "g_stage", "e_ph", "E", "g_final", "Q", "P"):
        setattr(w, n, 1)
    cfg = binding.Config(B_max=1, D=256, m=4, K=4, L_D=1, n_q=4, n_kv=2, d_h=64, F=768, R=64,
                         V=2048, dtype=0, rms_eps=1e-6, rope_theta=1e6, history=64)
    assert lib.dlite_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2   # fp32 drafter
    cfg.dtype = 1
    cfg.n_q, cfg.n_kv, cfg.K = 32, 1, 7   # 32 heads x 8 rows = 256 query rows per KV head
    assert lib.dlite_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    cfg.n_q, cfg.n_kv, cfg.K, cfg.act_planes = 4, 2, 4, 2   # the history kernels keep bf16 activations
    assert lib.dlite_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    assert lib.dlite_history_reset(None, None) == -1
    assert lib.dlite_history_read(None, 0, 0, 0, None, None, None) == -1
