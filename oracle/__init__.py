"""Python access to the CPU oracle (plain C, fp64 accumulation).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports this
package and this package never imports the CUDA library.

`build()` compiles oracle.c with gcc into oracle/_build/liboracle.so.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    hdr = os.path.join(_HERE, "oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Dims(C.Structure):
    _fields_ = [("V", C.c_int), ("d", C.c_int), ("slots", C.c_int), ("K", C.c_int),
                ("r", C.c_int), ("H", C.c_int), ("ln_eps", C.c_double),
                ("beam_width", C.c_int), ("beam_topm", C.c_int)]


class Weights(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_float)) for n in (
        "w_cand", "w_ctx", "w_fuse", "ln_gamma", "ln_beta", "w_pair", "w1", "b1", "w2", "b2", "w_io")]


class Inter(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_double)) for n in ("b", "g", "z", "s", "o", "in_")]


_PD = C.POINTER(C.c_double)
_PF = C.POINTER(C.c_float)
_PI = C.POINTER(C.c_int32)
_PU = C.POINTER(C.c_uint16)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_topk_row.argtypes = [_PU, C.c_int, C.c_int, _PI, _PF]
            L.orc_ln0.argtypes = [_PD, C.c_int, C.c_double, _PD]
            L.orc_gelu.argtypes = [C.c_double]
            L.orc_gelu.restype = C.c_double
            L.orc_context.argtypes = [C.POINTER(Dims), C.POINTER(Weights), _PU, _PD]
            L.orc_candidate.argtypes = [C.POINTER(Dims), C.POINTER(Weights), _PU, _PD, _PD, _PD]
            L.orc_pair_state.argtypes = [C.POINTER(Dims), C.POINTER(Weights), _PU, _PU, _PD]
            L.orc_transition.argtypes = [C.POINTER(Dims), C.POINTER(Weights), _PD, _PD, _PD,
                                         C.c_double, C.c_double]
            L.orc_transition.restype = C.c_double
            L.orc_cosine_vectors.argtypes = [C.POINTER(Dims), C.POINTER(Weights), _PU, _PU, _PD, _PD]
            L.orc_cosine_transition.argtypes = [C.c_int, C.c_double, _PD, _PD, C.c_double]
            L.orc_cosine_transition.restype = C.c_double
            L.orc_walk.argtypes = [_PD, C.c_int, C.c_int, _PI, _PD]
            L.orc_viterbi.argtypes = [_PD, C.c_int, C.c_int, _PI, _PD]
            L.orc_viterbi_f32.argtypes = [_PF, C.c_int, C.c_int, _PI, _PF]
            L.orc_beam.argtypes = [_PD, C.c_int, C.c_int, C.c_int, C.c_int, _PI, _PD]
            L.orc_topk_features.argtypes = [_PU, C.c_int, C.c_int, _PD]
            L.orc_verify_stochastic.argtypes = [_PU, C.c_int64, C.c_int, C.c_int, _PI, _PF, C.c_float, _PI, _PI,
                                                _PD]
            L.orc_beam_f32.argtypes = [_PF, C.c_int, C.c_int, C.c_int, C.c_int, _PI, _PF]
            L.orc_verify.argtypes = [_PI, _PI, C.c_int]
            L.orc_verify.restype = C.c_int
            L.orc_expected_yield.argtypes = [_PD, C.c_int, _PD]
            L.orc_expected_yield.restype = C.c_double
            L.orc_param_count.argtypes = [C.c_int, C.c_int, C.c_int]
            L.orc_param_count.restype = C.c_longlong
            L.orc_correct_request.argtypes = [
                C.POINTER(Dims), C.POINTER(Weights), C.c_int, C.c_double, C.c_int,
                _PU, C.c_int64, _PU, _PU, _PI,
                _PI, _PF, _PD, _PI, _PI, _PD, _PI, C.POINTER(Inter)]
            L.orc_correct_request.restype = C.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ctype))


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


class Model:
    """Holds fp32 weights (kept alive) and the dims struct for the C calls."""

    def __init__(self, weights: dict[str, np.ndarray], V: int, d: int, slots: int = 16,
                 K: int = 16, r: int = 128, H: int = 256, ln_eps: float = 1e-5, beam_width: int = 2,
                 beam_topm: int = 0):
        self.w = {k: np.ascontiguousarray(v, dtype=np.float32) for k, v in weights.items()}
        self.dims = Dims(V, d, slots, K, r, H, ln_eps, beam_width, beam_topm)
        self.cw = Weights(*[_p(self.w.get(f[0]), C.c_float) for f in Weights._fields_])

    @property
    def B(self):
        return self.dims.slots - 1


# ------------------------------------------------------------------ steps
def topk_row(row_bits: np.ndarray, K: int):
    row = _u16(row_bits)
    ids = np.empty(K, np.int32)
    vals = np.empty(K, np.float32)
    lib().orc_topk_row(_p(row, C.c_uint16), row.shape[0], K, _p(ids, C.c_int32), _p(vals, C.c_float))
    return ids, vals


def ln0(x: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().orc_ln0(_p(x, C.c_double), x.shape[0], eps, _p(y, C.c_double))
    return y


def gelu(x: float) -> float:
    return lib().orc_gelu(float(x))


def context(m: Model, h_bits):
    h = _u16(h_bits)
    g = np.empty(m.dims.r, np.float64)
    lib().orc_context(C.byref(m.dims), C.byref(m.cw), _p(h, C.c_uint16), _p(g, C.c_double))
    return g


def candidate(m: Model, e_bits, g):
    e = _u16(e_bits)
    g = np.ascontiguousarray(g, dtype=np.float64)
    b = np.empty(m.dims.r, np.float64)
    z = np.empty(m.dims.r, np.float64)
    lib().orc_candidate(C.byref(m.dims), C.byref(m.cw), _p(e, C.c_uint16), _p(g, C.c_double),
                        _p(b, C.c_double), _p(z, C.c_double))
    return b, z


def pair_state(m: Model, hp_bits, hq_bits):
    hp, hq = _u16(hp_bits), _u16(hq_bits)
    s = np.empty(m.dims.r, np.float64)
    lib().orc_pair_state(C.byref(m.dims), C.byref(m.cw), _p(hp, C.c_uint16), _p(hq, C.c_uint16),
                         _p(s, C.c_double))
    return s


def transition(m: Model, s, z_a, z_b, l_a: float, l_b: float) -> float:
    s, z_a, z_b = (np.ascontiguousarray(v, dtype=np.float64) for v in (s, z_a, z_b))
    return lib().orc_transition(C.byref(m.dims), C.byref(m.cw), _p(s, C.c_double),
                                _p(z_a, C.c_double), _p(z_b, C.c_double), float(l_a), float(l_b))


def cosine_vectors(m: Model, e_bits, h_bits):
    e, h = _u16(e_bits), _u16(h_bits)
    o = np.empty(m.dims.r, np.float64)
    i = np.empty(m.dims.r, np.float64)
    lib().orc_cosine_vectors(C.byref(m.dims), C.byref(m.cw), _p(e, C.c_uint16), _p(h, C.c_uint16),
                             _p(o, C.c_double), _p(i, C.c_double))
    return o, i


def cosine_transition(sigma: float, o_a, in_b, l_b: float) -> float:
    o_a, in_b = (np.ascontiguousarray(v, dtype=np.float64) for v in (o_a, in_b))
    return lib().orc_cosine_transition(o_a.shape[0], float(sigma), _p(o_a, C.c_double),
                                       _p(in_b, C.c_double), float(l_b))


def walk(scores: np.ndarray):
    """scores [B-1, K, K] -> (choice [B], margin [B-1])."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    P, K, _ = s.shape
    choice = np.empty(P + 1, np.int32)
    margin = np.empty(P, np.float64)
    lib().orc_walk(_p(s, C.c_double), P + 1, K, _p(choice, C.c_int32), _p(margin, C.c_double))
    return choice, margin


def viterbi(scores: np.ndarray):
    """scores [B-1, K, K] -> (choice [B], margin [B-1]) of the highest-scoring path."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    P, K, _ = s.shape
    choice = np.empty(P + 1, np.int32)
    margin = np.empty(P, np.float64)
    lib().orc_viterbi(_p(s, C.c_double), P + 1, K, _p(choice, C.c_int32), _p(margin, C.c_double))
    return choice, margin


def viterbi_f32(scores: np.ndarray):
    """The highest-scoring path with single-precision totals (scores given as float32)."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    P, K, _ = s.shape
    choice = np.empty(P + 1, np.int32)
    margin = np.empty(P, np.float32)
    lib().orc_viterbi_f32(_p(s, C.c_float), P + 1, K, _p(choice, C.c_int32), _p(margin, C.c_float))
    return choice, margin


def beam(scores: np.ndarray, width: int, topm: int = 0):
    """scores [B-1, K, K] -> (choice [B], margin [B-1]) of the beam walk."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    P, K, _ = s.shape
    choice = np.empty(P + 1, np.int32)
    margin = np.empty(P, np.float64)
    lib().orc_beam(_p(s, C.c_double), P + 1, K, width, topm, _p(choice, C.c_int32), _p(margin, C.c_double))
    return choice, margin


def beam_f32(scores: np.ndarray, width: int, topm: int = 0):
    """The beam walk with float totals (scores given as float32)."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    P, K, _ = s.shape
    choice = np.empty(P + 1, np.int32)
    margin = np.empty(P, np.float32)
    lib().orc_beam_f32(_p(s, C.c_float), P + 1, K, width, topm, _p(choice, C.c_int32), _p(margin, C.c_float))
    return choice, margin


def select_path(scores: np.ndarray, path_rule: int = 0, width: int = 2, topm: int = 0):
    """path_rule 0: greedy walk, 1: highest-scoring path, 2: beam walk."""
    if path_rule == 1:
        return viterbi(scores)
    if path_rule == 2:
        return beam(scores, width, topm)
    return walk(scores)


def topk_features(row_bits, K: int, V: int | None = None):
    """row [stride] u16 (bf16 bits; the first V columns are the vocabulary) ->
    features [K, 5] = (log p, p, l_0 - l_k, k / K, k == 0)."""
    r = _u16(row_bits)
    feat = np.empty((K, 5), np.float64)
    lib().orc_topk_features(_p(r, C.c_uint16), V or r.shape[-1], K, _p(feat, C.c_double))
    return feat


def verify_stochastic(target_logits, tokens, u_acc, u_draw: float, V: int | None = None):
    """target_logits [B+1, stride] u16 (bf16 bits; the first V columns are the
    vocabulary), tokens [B], u_acc [B] -> (accept_len, next_token, q_acc [B])."""
    tl = _u16(target_logits)
    tk = np.ascontiguousarray(tokens, dtype=np.int32)
    ua = np.ascontiguousarray(u_acc, dtype=np.float32)
    B = tk.shape[0]
    al = np.zeros(1, np.int32)
    nt = np.zeros(1, np.int32)
    q = np.empty(B, np.float64)
    lib().orc_verify_stochastic(_p(tl, C.c_uint16), tl.shape[-1], V or tl.shape[-1], B, _p(tk, C.c_int32),
                                _p(ua, C.c_float), float(u_draw), _p(al, C.c_int32), _p(nt, C.c_int32),
                                _p(q, C.c_double))
    return int(al[0]), int(nt[0]), q


def verify(tokens, target) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    g = np.ascontiguousarray(target, dtype=np.int32)
    return lib().orc_verify(_p(t, C.c_int32), _p(g, C.c_int32), t.shape[0])


def expected_yield(cond):
    c = np.ascontiguousarray(cond, dtype=np.float64)
    surv = np.empty_like(c)
    ey = lib().orc_expected_yield(_p(c, C.c_double), c.shape[0], _p(surv, C.c_double))
    return ey, surv


def param_count(d: int, r: int = 128, H: int = 256) -> int:
    return int(lib().orc_param_count(d, r, H))


# ------------------------------------------------------------------ whole path
def correct_request(m: Model, logits_req, hidden_req, E, target=None, variant: int = 0,
                    sigma: float = 1.0, intermediates: bool = False, path_rule: int = 0):
    """One request.  logits_req [slots, stride] u16, hidden_req [slots, d] u16, E [V, d] u16."""
    dm = m.dims
    B, K, r = dm.slots - 1, dm.K, dm.r
    lg = _u16(logits_req)
    hd = _u16(hidden_req)
    E = _u16(E)
    tg = None if target is None else np.ascontiguousarray(target, dtype=np.int32)
    out = {
        "topk_ids": np.empty((B, K), np.int32),
        "topk_val": np.empty((B, K), np.float32),
        "scores": np.empty((B - 1, K, K), np.float64),
        "choice": np.empty(B, np.int32),
        "tokens": np.empty(B, np.int32),
        "margin": np.empty(B - 1, np.float64),
        "accept_len": np.zeros(1, np.int32),
    }
    inter = None
    if intermediates:
        if variant == 0:
            out["b"] = np.empty((B, K, r)); out["z"] = np.empty((B, K, r))
            out["g"] = np.empty((B, r)); out["s"] = np.empty((B - 1, r))
            inter = Inter(_p(out["b"], C.c_double), _p(out["g"], C.c_double), _p(out["z"], C.c_double),
                          _p(out["s"], C.c_double), None, None)
        else:
            out["o"] = np.empty((B, K, r)); out["in"] = np.empty((B, K, r))
            inter = Inter(None, None, None, None, _p(out["o"], C.c_double), _p(out["in"], C.c_double))
    rc = lib().orc_correct_request(
        C.byref(dm), C.byref(m.cw), variant, sigma, path_rule, _p(lg, C.c_uint16), lg.shape[-1],
        _p(hd, C.c_uint16), _p(E, C.c_uint16), _p(tg, C.c_int32),
        _p(out["topk_ids"], C.c_int32), _p(out["topk_val"], C.c_float), _p(out["scores"], C.c_double),
        _p(out["choice"], C.c_int32), _p(out["tokens"], C.c_int32), _p(out["margin"], C.c_double),
        _p(out["accept_len"], C.c_int32) if tg is not None else None,
        C.byref(inter) if inter is not None else None)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    out["accept_len"] = int(out["accept_len"][0]) if tg is not None else None
    return out


def correct_batch(m: Model, logits, hidden, E, targets=None, variant: int = 0, sigma: float = 1.0,
                  requests=None, threads: int | None = None, path_rule: int = 0):
    """Run `correct_request` over requests (all, or the listed indices) on a thread pool."""
    N = logits.shape[0]
    req = list(range(N)) if requests is None else list(requests)
    E = _u16(E)
    threads = threads or min(len(req), os.cpu_count() or 1)

    def one(n):
        return correct_request(m, logits[n], hidden[n], E, None if targets is None else targets[n],
                               variant, sigma, path_rule=path_rule)

    if threads <= 1:
        res = [one(n) for n in req]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            res = list(ex.map(one, req))
    keys = ("topk_ids", "topk_val", "scores", "choice", "tokens", "margin")
    out = {k: np.stack([r[k] for r in res]) for k in keys}
    out["accept_len"] = None if targets is None else np.array([r["accept_len"] for r in res], np.int32)
    out["requests"] = np.array(req)
    return out
