"""Thin ctypes binding of libdlite.so (argument marshalling only).

Every step of the round runs in the CUDA library; this module only turns
torch tensors into device pointers and checks return codes. It fails loudly
when the library is missing: there is no fallback path.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdlite.so")

DLITE_F32, DLITE_BF16 = 0, 1
MAX_LAYERS = 8

STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "CUDA runtime error",
    -4: "device wait timed out", -5: "id out of range on the device", -6: "device allocation failed",
}


class DliteError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B_max", "D", "m", "K", "L_D", "n_q", "n_kv", "d_h", "F", "R", "V", "dtype")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("anchor_group", ctypes.c_int),
                ("head_type", ctypes.c_int), ("history", ctypes.c_int), ("act_planes", ctypes.c_int),
                ("head_warmup", ctypes.c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("g_attn", "Wq", "Wk", "Wv", "Wo", "g_ffn", "Wg", "Wu", "Wd")]


GATED_FIELDS = ("E_R", "W_s", "b_s", "W_h", "b_h", "W_o")


class GatedWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in GATED_FIELDS]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("e_depth", "g_stage", "e_ph", "E", "g_final", "Q", "P")] + \
               [("layer", LayerWeights * MAX_LAYERS), ("gated", GatedWeights)]


VERIFY_GREEDY, VERIFY_SAMPLE, VERIFY_MATCH = 0, 1, 2


class VerifyArgs(ctypes.Structure):
    """dlite_verify_args (include/dlite.h)."""
    _fields_ = [("mode", ctypes.c_int), ("B", ctypes.c_int), ("n_verify", ctypes.c_int),
                ("candidates", ctypes.c_void_p), ("target_tokens", ctypes.c_void_p),
                ("qstats", ctypes.c_void_p), ("hs", ctypes.c_void_p), ("target_probs", ctypes.c_void_p),
                ("temperature", ctypes.c_float), ("seed", ctypes.c_uint64), ("pos", ctypes.c_void_p),
                ("accepted", ctypes.c_void_p), ("commits", ctypes.c_void_p), ("n_commit", ctypes.c_void_p),
                ("next_anchor", ctypes.c_void_p)]


class Taps(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("z", "x", "b", "hs")]


_lib = None

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_U64 = ctypes.c_uint64
_SIGS = {
    "dlite_create": (_I, [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(_P)]),
    "dlite_destroy": (None, [_P]),
    "dlite_draft_round": (_I, [_P, _I, _P, _P, _F, _U64, _P, _P, _P, _P]),
    "dlite_draft_round_taps": (_I, [_P, _I, _P, _P, _F, _U64, _P, _P, _P, ctypes.POINTER(Taps), _P]),
    "dlite_backbone": (_I, [_P, _I, _P, _P, _P, _P]),
    "dlite_seq_head": (_I, [_P, _I, _P, _P, _P]),
    "dlite_lm_head": (_I, [_P, _I, _P, _F, _U64, _P, _P, _P, _P]),
    "dlite_verify": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "dlite_verify_sample": (_I, [_P, _I, _P, _P, _P, _P, _F, _U64, _P, _P, _P, _P, _P, _P]),
    "dlite_verify_ex": (_I, [_P, ctypes.POINTER(VerifyArgs), _P]),
    "dlite_advance": (_I, [_P, _I, _P, _P, _P]),
    "dlite_shift_group": (_I, [_P, _I, _P, _P, _P, _P]),
    "dlite_history_reset": (_I, [_P, _P]),
    "dlite_history_read": (_I, [_P, _I, _I, _I, _P, ctypes.POINTER(ctypes.c_int32), _P]),
    "dlite_verify_sample_static": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _F, _U64, _P, _P, _P,
                                        _P, _P, _P]),
    "dlite_round_host": (_I, [_P, _I, _P, _P, _P, _P, _P, _F, _U64, _P, _P, _P, _P, _P]),
    "dlite_synthetic_target": (_I, [_I, _I, _I, _P, _P, _I, _P, _U64, _P, _P, _P]),
    "dlite_selftest_wait": (_I, [_P, _U64, _P, _P]),
    "dlite_device_status": (_I, [_P, _I, ctypes.POINTER(_I), _P]),
    "dlite_status_string": (ctypes.c_char_p, [_I]),
    "dlite_last_cuda_error": (ctypes.c_char_p, []),
    "dlite_launch_count": (_I, [_P, _I, _F]),
    "dlite_counters": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int64), _P]),
    "dlite_selftest_gemm": (_I, [_I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P,
                                 ctypes.POINTER(ctypes.c_int), _P]),
    "dlite_stage_times": (_I, [_P, _I, _P, _P, _F, _U64, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, ctypes.POINTER(ctypes.c_char_p), _I, _P]),
}

EXPORTED = tuple(_SIGS)


def load(path=None):
    """Load libdlite.so (built by history_free_speculative_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libdlite.so not built ({path}); run `python -m "
                           "history_free_speculative_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("contiguous host tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, what):
    if code != 0:
        if code == -3 and _lib is not None:   # DLITE_ERR_CUDA: name the runtime error
            what = f"{what} [{_lib.dlite_last_cuda_error().decode()}]"
        raise DliteError(code, what)


def selftest_gemm(X, W, rows=None, stream=None, plan=None, part=None, outs=None):
    """Tensor-core product X[:rows] @ W^T through the round's GEMM engine.

    X, W: lists of 1 or 2 bf16 device planes ([x_rows, K] with x_rows a multiple
    of 128; W in the tiled weight layout, rows padded to 64). Returns
    (fp32 [rows, outs] device tensor, status).
    """
    lib = load()
    rows = X[0].shape[0] if rows is None else rows
    wrows, K = W[0].shape
    outs = wrows if outs is None else outs
    if part is None:
        part = torch.zeros(16 * rows * outs, dtype=torch.float32, device=X[0].device)
    st = torch.zeros(1, dtype=torch.int32, device=X[0].device)
    ov = (ctypes.c_int * 3)(*plan) if plan is not None else None
    S = lib.dlite_selftest_gemm(rows, outs, K, len(X), len(W), _ptr(X[0]),
                                _ptr(X[1]) if len(X) > 1 else None, X[0].shape[0], _ptr(W[0]),
                                _ptr(W[1]) if len(W) > 1 else None, _ptr(part), _ptr(st), ov,
                                _stream(stream))
    if S < 0:
        raise DliteError(S, "dlite_selftest_gemm")
    return part[:S * rows * outs].view(S, rows, outs).sum(0), st


def verify_sample_static(cand, qstats, hs, E, probs, temperature, seed, pos, accepted, commits,
                         n_commit, next_anchor, stream=None):
    """Allocation-free sampling verification (no handle; E float32 row-major [V, D])."""
    lib = load()
    B, K = cand.shape
    V, D = E.shape
    want = ((cand, torch.int32, (B, K)), (qstats, torch.float32, (B, K, 2)), (hs, torch.float32, (B, K, D)),
            (E, torch.float32, (V, D)), (probs, torch.float32, (B, K + 1, V)), (pos, torch.int64, (B,)),
            (accepted, torch.int32, (B,)), (commits, torch.int32, (B, K + 1)), (n_commit, torch.int32, (B,)),
            (next_anchor, torch.int32, (B,)))
    for t, dt, shape in want:
        if t.dtype != dt or tuple(t.shape) != shape:
            raise ValueError(f"verify_sample_static: expected {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
    _check(lib.dlite_verify_sample_static(B, K, V, D, _ptr(cand), _ptr(qstats), _ptr(hs), _ptr(E),
                                          _ptr(probs), temperature, seed, _ptr(pos), _ptr(accepted),
                                          _ptr(commits), _ptr(n_commit), _ptr(next_anchor),
                                          _stream(stream)), "dlite_verify_sample_static")


def synthetic_target(cand, accept_c, seed, pos, target_tokens, V, round_counter=None, stream=None):
    """Synthetic target tokens [B, K+1] (dlite_synthetic_target): accept_c is
    [n_tables, B, K] float32 on the device, round_counter a device int32 (or None)."""
    lib = load()
    B, K = cand.shape
    if accept_c.dtype != torch.float32 or accept_c.dim() != 3 or tuple(accept_c.shape[1:]) != (B, K):
        raise ValueError("accept_c must be float32 [n_tables, B, K]")
    if cand.dtype != torch.int32 or pos.dtype != torch.int64 or target_tokens.dtype != torch.int32:
        raise ValueError("candidates / target_tokens int32, pos int64 expected")
    if tuple(target_tokens.shape) != (B, K + 1) or tuple(pos.shape) != (B,):
        raise ValueError("target_tokens [B, K+1] and pos [B] expected")
    if round_counter is not None and round_counter.dtype != torch.int32:
        raise ValueError("round_counter must be a device int32")
    _check(lib.dlite_synthetic_target(B, K, V, _ptr(cand), _ptr(accept_c), accept_c.shape[0],
                                      _ptr(round_counter), seed, _ptr(pos), _ptr(target_tokens),
                                      _stream(stream)), "dlite_synthetic_target")


def config_struct(cfg, B_max):
    return Config(B_max=B_max, D=cfg.D, m=cfg.m, K=cfg.K, L_D=cfg.L_D, n_q=cfg.n_q,
                  n_kv=cfg.n_kv, d_h=cfg.d_h, F=cfg.F, R=cfg.R, V=cfg.V,
                  dtype=DLITE_F32 if cfg.dtype == "f32" else DLITE_BF16,
                  rms_eps=cfg.eps, rope_theta=cfg.theta, anchor_group=getattr(cfg, "G", 1),
                  head_type=1 if getattr(cfg, "head", "rnn") == "gated" else 0,
                  history=getattr(cfg, "history", 0), act_planes=getattr(cfg, "act_planes", 1),
                  head_warmup=getattr(cfg, "warmup", 0))


class Drafter:
    """A drafter handle on the current CUDA device.

    W is the weight dict of workload.make_weights (tensors on the device, in
    the config's dtype). The library copies and repacks them at creation.
    """

    def __init__(self, cfg, W, B_max):
        self.lib = load()
        self.cfg = cfg
        self.B_max = B_max
        c = config_struct(cfg, B_max)
        w = Weights()
        for n in ("e_depth", "g_stage", "e_ph", "E", "g_final", "Q", "P"):
            setattr(w, n, _ptr(W[n]).value)
        for i, L in enumerate(W["layers"]):
            for n in ("g_attn", "Wq", "Wk", "Wv", "Wo", "g_ffn", "Wg", "Wu", "Wd"):
                setattr(w.layer[i], n, _ptr(L[n]).value)
        if getattr(cfg, "head", "rnn") == "gated":
            for n in GATED_FIELDS:
                setattr(w.gated, n, _ptr(W[n]).value)
        h = ctypes.c_void_p()
        _check(self.lib.dlite_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)), "dlite_create")
        self.h = h

    def close(self):
        if self.h:
            self.lib.dlite_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- outputs helpers
    def new_outputs(self, B, device="cuda"):
        K = self.cfg.K
        return dict(
            cand=torch.empty(B, K, dtype=torch.int32, device=device),
            qstats=torch.empty(B, K, 2, dtype=torch.float32, device=device),
            accepted=torch.empty(B, dtype=torch.int32, device=device),
            commits=torch.empty(B, K + 1, dtype=torch.int32, device=device),
            n_commit=torch.empty(B, dtype=torch.int32, device=device),
            next_anchor=torch.empty(B, dtype=torch.int32, device=device),
        )

    # ---- calls
    def draft_round(self, hidden, anchor, temperature, seed, pos, cand, qstats, stream=None,
                    taps=None):
        B = hidden.shape[0]
        if taps is None:
            rc = self.lib.dlite_draft_round(self.h, B, _ptr(hidden), _ptr(anchor), temperature,
                                            seed, _ptr(pos), _ptr(cand), _ptr(qstats), _stream(stream))
        else:
            t = Taps(*(None if taps.get(k) is None else taps[k].data_ptr() for k in ("z", "x", "b", "hs")))
            rc = self.lib.dlite_draft_round_taps(self.h, B, _ptr(hidden), _ptr(anchor), temperature,
                                                 seed, _ptr(pos), _ptr(cand), _ptr(qstats),
                                                 ctypes.byref(t), _stream(stream))
        _check(rc, "dlite_draft_round")

    def backbone(self, hidden, anchor, b, stream=None):
        _check(self.lib.dlite_backbone(self.h, hidden.shape[0], _ptr(hidden), _ptr(anchor), _ptr(b),
                                       _stream(stream)), "dlite_backbone")

    def seq_head(self, b, hs, stream=None):
        _check(self.lib.dlite_seq_head(self.h, b.shape[0], _ptr(b), _ptr(hs), _stream(stream)),
               "dlite_seq_head")

    def lm_head(self, hs, temperature, seed, pos, cand, qstats, stream=None):
        _check(self.lib.dlite_lm_head(self.h, hs.shape[0], _ptr(hs), temperature, seed, _ptr(pos),
                                      _ptr(cand), _ptr(qstats), _stream(stream)), "dlite_lm_head")

    def verify(self, cand, target_tokens, accepted, commits, n_commit, next_anchor, stream=None):
        _check(self.lib.dlite_verify(self.h, cand.shape[0], _ptr(cand), _ptr(target_tokens),
                                     _ptr(accepted), _ptr(commits), _ptr(n_commit),
                                     _ptr(next_anchor), _stream(stream)), "dlite_verify")

    def verify_sample(self, cand, qstats, hs, probs, temperature, seed, pos, accepted, commits,
                      n_commit, next_anchor, stream=None):
        _check(self.lib.dlite_verify_sample(self.h, cand.shape[0], _ptr(cand), _ptr(qstats),
                                            _ptr(hs), _ptr(probs), temperature, seed, _ptr(pos),
                                            _ptr(accepted), _ptr(commits), _ptr(n_commit),
                                            _ptr(next_anchor), _stream(stream)),
               "dlite_verify_sample")

    def verify_ex(self, mode, cand, accepted, commits, n_commit, next_anchor, n_verify=None,
                  target_tokens=None, qstats=None, hs=None, probs=None, temperature=0.0, seed=0, pos=None,
                  stream=None):
        """dlite_verify_ex: greedy / sampling / match verification over the first
        n_verify candidates (default all K)."""
        a = VerifyArgs(mode=mode, B=cand.shape[0], n_verify=cand.shape[1] if n_verify is None else n_verify,
                       candidates=_ptr(cand), target_tokens=_ptr(target_tokens), qstats=_ptr(qstats),
                       hs=_ptr(hs), target_probs=_ptr(probs), temperature=temperature, seed=seed,
                       pos=_ptr(pos), accepted=_ptr(accepted), commits=_ptr(commits),
                       n_commit=_ptr(n_commit), next_anchor=_ptr(next_anchor))
        _check(self.lib.dlite_verify_ex(self.h, ctypes.byref(a), _stream(stream)), "dlite_verify_ex")

    def history_reset(self, stream=None):
        """Refill every draft-KV ring with the synthetic history; cursors to 0."""
        _check(self.lib.dlite_history_reset(self.h, _stream(stream)), "dlite_history_reset")

    def history_read(self, layer, request, which, stream=None):
        """One ring of the history-KV control: ([n_kv, H, d_h] bf16 on the device, cursor)."""
        c = self.cfg
        dst = torch.empty(c.n_kv, c.history, c.d_h, dtype=torch.bfloat16, device="cuda")
        cur = ctypes.c_int32(0)
        _check(self.lib.dlite_history_read(self.h, layer, request, which, _ptr(dst), ctypes.byref(cur),
                                           _stream(stream)), "dlite_history_read")
        return dst, int(cur.value)

    def shift_group(self, commits, n_commit, group, stream=None):
        _check(self.lib.dlite_shift_group(self.h, n_commit.shape[0], _ptr(commits), _ptr(n_commit), _ptr(group),
                                          _stream(stream)), "dlite_shift_group")

    def advance(self, n_commit, pos, stream=None):
        _check(self.lib.dlite_advance(self.h, n_commit.shape[0], _ptr(n_commit), _ptr(pos),
                                      _stream(stream)), "dlite_advance")

    def round_host(self, hidden_h, anchor_h, pos_h, tgt_h, probs_h, temperature, seed, out_h,
                   stream=None):
        _check(self.lib.dlite_round_host(self.h, hidden_h.shape[0], _hptr(hidden_h), _hptr(anchor_h),
                                         _hptr(pos_h), _hptr(tgt_h), _hptr(probs_h), temperature,
                                         seed, _hptr(out_h["accepted"]), _hptr(out_h["commits"]),
                                         _hptr(out_h["n_commit"]), _hptr(out_h["next_anchor"]),
                                         _stream(stream)), "dlite_round_host")

    def device_status(self, clear=True, stream=None):
        v = ctypes.c_int(0)
        rc = self.lib.dlite_device_status(self.h, 1 if clear else 0, ctypes.byref(v), _stream(stream))
        return rc, v.value

    def stage_times(self, hidden, anchor, temperature, seed, pos, out, target_tokens=None,
                    target_probs=None, stream=None, cap=128):
        """Per-launch CUDA-event times (ms) of one eager draft (+ verify): [(name, ms)]."""
        times = (ctypes.c_float * cap)()
        names = (ctypes.c_char_p * cap)()
        n = self.lib.dlite_stage_times(
            self.h, hidden.shape[0], _ptr(hidden), _ptr(anchor), temperature, seed, _ptr(pos),
            _ptr(target_tokens), _ptr(target_probs), _ptr(out["cand"]), _ptr(out["qstats"]),
            _ptr(out["accepted"]), _ptr(out["commits"]), _ptr(out["n_commit"]),
            _ptr(out["next_anchor"]), times, names, cap, _stream(stream))
        if n < 0:
            raise DliteError(n, "dlite_stage_times")
        return [(names[i].decode(), times[i]) for i in range(min(n, cap))]

    def selftest_wait(self, limit_ns, result, stream=None):
        """Bounded-wait probe (dlite_selftest_wait): result is a device int32 [3]."""
        _check(self.lib.dlite_selftest_wait(self.h, int(limit_ns), _ptr(result), _stream(stream)),
               "dlite_selftest_wait")

    def counters(self, reset=False, stream=None):
        """Sampling-verify counters: residual draws, proposals, fallbacks, bonus draws."""
        out = (ctypes.c_int64 * 5)()
        _check(self.lib.dlite_counters(self.h, 1 if reset else 0, out, _stream(stream)), "dlite_counters")
        return dict(residual=out[0], proposals=out[1], fallback=out[2], bonus=out[3],
                    lm_close_calls=out[4])

    def launch_count(self, B, temperature):
        return self.lib.dlite_launch_count(self.h, B, temperature)
