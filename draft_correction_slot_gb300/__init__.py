"""GB300 (sm_103a) draft-correction library: thin Python binding of include/dcoco.h.

Every function here only marshals arguments (tensor data pointers, sizes,
the current CUDA stream) into the C ABI of libdcoco.so; every step of the
correction path runs in the library's CUDA kernels.  There is no CPU path:
importing the binding without the built library raises.

Build the library first:  python draft_correction_slot_gb300/build.py
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdcoco.so")

DCOCO_OK = 0
DCOCO_EINVAL = -1
DCOCO_EUNSUPPORTED = -2
DCOCO_EBATCH = -3
DCOCO_ECUDA = -4
DCOCO_ENOMEM = -5
DCOCO_EDEVICE = -6


class DcocoError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {dcoco_status_string(status)} ({status})")
        self.status = status


class dcoco_config(C.Structure):
    _fields_ = [("vocab", C.c_int), ("hidden", C.c_int), ("slots", C.c_int), ("topk", C.c_int),
                ("rank", C.c_int), ("mlp_hidden", C.c_int), ("max_batch", C.c_int),
                ("variant", C.c_int), ("sigma", C.c_float), ("ln_eps", C.c_float),
                ("host_staging", C.c_int), ("path_rule", C.c_int), ("beam_width", C.c_int),
                ("beam_topm", C.c_int)]


WEIGHT_NAMES = ("w_cand", "w_ctx", "w_fuse", "ln_gamma", "ln_beta", "w_pair", "w1", "b1", "w2",
                "b2", "w_io")


class dcoco_weight_ptrs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_NAMES] + [("on_device", C.c_int)]


class dcoco_inputs(C.Structure):
    _fields_ = [("logits", C.c_void_p), ("logits_slot_stride", C.c_int64), ("hidden", C.c_void_p),
                ("cand_embed", C.c_void_p), ("target_tokens", C.c_void_p)]


class dcoco_outputs(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("choice", C.c_void_p), ("scores", C.c_void_p),
                ("accept_len", C.c_void_p), ("topk_ids", C.c_void_p), ("topk_val", C.c_void_p),
                ("margin", C.c_void_p), ("cand_feat", C.c_void_p)]


EXPORTED = ("dcoco_version", "dcoco_status_string", "dcoco_create", "dcoco_weights_create",
            "dcoco_correct", "dcoco_correct_host", "dcoco_topk", "dcoco_get_device_status",
            "dcoco_selftest_wait_timeout",
            "dcoco_weights_destroy", "dcoco_destroy", "dcoco_kernel_launches",
            "dcoco_stage_timing", "dcoco_stage_read", "dcoco_stage_name", "dcoco_topk_noalloc",
            "dcoco_topk_noalloc_plan", "dcoco_verify_stochastic", "dcoco_host_range_covers")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python draft_correction_slot_gb300/build.py` (there is no CPU fallback)")
    L = C.CDLL(LIB_PATH)
    L.dcoco_version.restype = C.c_int
    L.dcoco_status_string.argtypes = [C.c_int]
    L.dcoco_status_string.restype = C.c_char_p
    L.dcoco_create.argtypes = [C.POINTER(dcoco_config), C.POINTER(C.c_void_p)]
    L.dcoco_weights_create.argtypes = [C.c_void_p, C.POINTER(dcoco_weight_ptrs), C.c_void_p,
                                       C.POINTER(C.c_void_p)]
    for f in (L.dcoco_correct, L.dcoco_correct_host):
        f.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.POINTER(dcoco_inputs),
                      C.POINTER(dcoco_outputs), C.c_void_p]
    L.dcoco_verify_stochastic.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.dcoco_topk.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                             C.c_void_p]
    L.dcoco_topk_noalloc.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int64,
                                     C.c_void_p, C.c_void_p, C.c_void_p]
    L.dcoco_topk_noalloc_plan.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int),
                                          C.POINTER(C.c_int)]
    L.dcoco_host_range_covers.argtypes = [C.c_uint64, C.c_uint64, C.c_uint64, C.c_uint64]
    L.dcoco_get_device_status.argtypes = [C.c_void_p]
    L.dcoco_selftest_wait_timeout.argtypes = [C.c_void_p, C.c_longlong, C.c_void_p]
    L.dcoco_weights_destroy.argtypes = [C.c_void_p]
    L.dcoco_weights_destroy.restype = None
    L.dcoco_destroy.argtypes = [C.c_void_p]
    L.dcoco_destroy.restype = None
    L.dcoco_kernel_launches.argtypes = [C.c_void_p]
    L.dcoco_kernel_launches.restype = C.c_longlong
    L.dcoco_stage_timing.argtypes = [C.c_void_p, C.c_int]
    L.dcoco_stage_read.argtypes = [C.c_void_p, C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_int),
                                   C.POINTER(C.c_int)]
    L.dcoco_stage_name.argtypes = [C.c_void_p, C.c_int]
    L.dcoco_stage_name.restype = C.c_char_p
    return L


_lib = _load()


def lib():
    return _lib


def _check(rc: int, what: str):
    if rc != DCOCO_OK:
        raise DcocoError(rc, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ------------------------------------------------------------------ C ABI, same names
def dcoco_version() -> int:
    return _lib.dcoco_version()


def dcoco_status_string(status: int) -> str:
    return _lib.dcoco_status_string(status).decode()


def dcoco_create(vocab: int, hidden: int, slots: int = 16, topk: int = 16, max_batch: int = 32,
                 variant: int = 0, sigma: float = 1.0, ln_eps: float = 1e-5, rank: int = 128,
                 mlp_hidden: int = 256, host_staging: bool = False, path_rule: int = 0,
                 beam_width: int = 2, beam_topm: int = 0) -> C.c_void_p:
    """path_rule 0: prefix-first greedy walk; 1: highest-scoring path; 2: beam walk
    (beam_width partial paths, beam_topm successors each, 0 = all)."""
    cfg = dcoco_config(vocab, hidden, slots, topk, rank, mlp_hidden, max_batch, variant, sigma, ln_eps,
                       int(host_staging), int(path_rule), int(beam_width), int(beam_topm))
    h = C.c_void_p()
    _check(_lib.dcoco_create(C.byref(cfg), C.byref(h)), "dcoco_create")
    return h


def dcoco_weights_create(handle, weights: dict, stream=None) -> C.c_void_p:
    """weights: name -> fp32 tensor (all on the GPU, or all on the CPU)."""
    keep = {}
    on_dev = None
    for n in WEIGHT_NAMES:
        t = weights.get(n)
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            t = torch.as_tensor(t)
        t = t.detach().to(torch.float32).contiguous()
        dev = t.is_cuda
        if on_dev is None:
            on_dev = dev
        elif on_dev != dev:
            raise ValueError("weights must all be on the GPU or all on the CPU")
        keep[n] = t
    ptrs = dcoco_weight_ptrs(*[_ptr(keep.get(n)) for n in WEIGHT_NAMES], int(bool(on_dev)))
    w = C.c_void_p()
    _check(_lib.dcoco_weights_create(handle, C.byref(ptrs), _stream(stream) if on_dev else None,
                                     C.byref(w)), "dcoco_weights_create")
    return w


def _io(logits, hidden, cand_embed, target_tokens, logits_slot_stride, outs):
    stride = logits_slot_stride if logits_slot_stride is not None else logits.shape[-1]
    ins = dcoco_inputs(_ptr(logits), int(stride), _ptr(hidden), _ptr(cand_embed), _ptr(target_tokens))
    o = dcoco_outputs(*[_ptr(outs.get(k)) for k in ("tokens", "choice", "scores", "accept_len",
                                                    "topk_ids", "topk_val", "margin", "cand_feat")])
    return ins, o


def dcoco_correct(handle, weights, batch: int, logits, hidden, cand_embed, target_tokens=None, *,
                  tokens, choice=None, scores=None, accept_len=None, topk_ids=None, topk_val=None,
                  margin=None, cand_feat=None, logits_slot_stride: int | None = None, stream=None) -> None:
    """Device buffers in, device buffers out (see include/dcoco.h for layouts)."""
    ins, o = _io(logits, hidden, cand_embed, target_tokens, logits_slot_stride,
                 dict(tokens=tokens, choice=choice, scores=scores, accept_len=accept_len,
                      topk_ids=topk_ids, topk_val=topk_val, margin=margin, cand_feat=cand_feat))
    _check(_lib.dcoco_correct(handle, weights, batch, C.byref(ins), C.byref(o), _stream(stream)),
           "dcoco_correct")


def dcoco_correct_host(handle, weights, batch: int, logits, hidden, cand_embed, target_tokens=None,
                       *, tokens, choice=None, scores=None, accept_len=None, topk_ids=None,
                       topk_val=None, margin=None, logits_slot_stride: int | None = None,
                       stream=None) -> None:
    """Host (ideally pinned) logits/hidden/targets/outputs; cand_embed stays on the device."""
    ins, o = _io(logits, hidden, cand_embed, target_tokens, logits_slot_stride,
                 dict(tokens=tokens, choice=choice, scores=scores, accept_len=accept_len,
                      topk_ids=topk_ids, topk_val=topk_val, margin=margin))
    _check(_lib.dcoco_correct_host(handle, weights, batch, C.byref(ins), C.byref(o), _stream(stream)),
           "dcoco_correct_host")


def dcoco_topk(handle, batch: int, logits, topk_ids, topk_val, logits_slot_stride: int | None = None,
               stream=None) -> None:
    stride = logits_slot_stride if logits_slot_stride is not None else logits.shape[-1]
    _check(_lib.dcoco_topk(handle, batch, _ptr(logits), int(stride), _ptr(topk_ids), _ptr(topk_val),
                           _stream(stream)), "dcoco_topk")


def dcoco_verify_stochastic(handle, batch: int, target_logits, tokens, u_accept, u_draw, accept_len,
                            next_token, q_accept=None, target_stride: int | None = None, stream=None) -> None:
    """Stochastic verification (temperature 1) of the proposal `tokens` against
    target_logits [batch, B+1, stride] (bf16), with caller-drawn uniforms."""
    stride = target_stride if target_stride is not None else target_logits.shape[-1]
    _check(_lib.dcoco_verify_stochastic(handle, batch, _ptr(target_logits), int(stride), _ptr(tokens),
                                        _ptr(u_accept), _ptr(u_draw), _ptr(accept_len), _ptr(next_token),
                                        _ptr(q_accept) if q_accept is not None else None, _stream(stream)),
           "dcoco_verify_stochastic")


def dcoco_topk_noalloc(batch: int, slots: int, vocab: int, topk: int, logits, topk_ids, topk_val,
                       logits_slot_stride: int | None = None, stream=None) -> None:
    """Step 1 without a handle and without any device allocation (for callers
    that cannot allocate); same results as dcoco_topk."""
    stride = logits_slot_stride if logits_slot_stride is not None else logits.shape[-1]
    _check(_lib.dcoco_topk_noalloc(batch, slots, vocab, topk, _ptr(logits), int(stride), _ptr(topk_ids),
                                   _ptr(topk_val), _stream(stream)), "dcoco_topk_noalloc")


def dcoco_topk_noalloc_plan(batch: int, slots: int, vocab: int, topk: int) -> tuple[int, int]:
    """-> (segments per row dcoco_topk_noalloc would use, segments dcoco_topk would use)."""
    seg, planned = C.c_int(), C.c_int()
    _check(_lib.dcoco_topk_noalloc_plan(batch, slots, vocab, topk, C.byref(seg), C.byref(planned)),
           "dcoco_topk_noalloc_plan")
    return seg.value, planned.value


def dcoco_host_range_covers(range_start: int, range_size: int, ptr: int, nbytes: int) -> bool:
    """Whether [ptr, ptr + nbytes) lies inside the range (the host entry's in-place test)."""
    return bool(_lib.dcoco_host_range_covers(range_start, range_size, ptr, nbytes))


def dcoco_get_device_status(handle) -> int:
    return _lib.dcoco_get_device_status(handle)


def dcoco_selftest_wait_timeout(handle, limit_ns: int, stream: int = 0) -> None:
    """One block waits on an mbarrier nothing completes, with the kernels' own
    bounded wait (limit_ns); the handle's device status then reads DCOCO_EDEVICE."""
    _check(_lib.dcoco_selftest_wait_timeout(handle, int(limit_ns), C.c_void_p(stream)),
           "dcoco_selftest_wait_timeout")


def dcoco_weights_destroy(weights) -> None:
    _lib.dcoco_weights_destroy(weights)


def dcoco_destroy(handle) -> None:
    _lib.dcoco_destroy(handle)


def dcoco_kernel_launches(handle) -> int:
    return int(_lib.dcoco_kernel_launches(handle))


def dcoco_stage_timing(handle, enable: bool) -> None:
    _check(_lib.dcoco_stage_timing(handle, int(bool(enable))), "dcoco_stage_timing")


def dcoco_stage_read(handle) -> tuple[dict, int]:
    """-> ({stage name: summed ms}, number of calls summed)."""
    ms = (C.c_float * 8)()
    calls, ns = C.c_int(), C.c_int()
    _check(_lib.dcoco_stage_read(handle, 8, ms, C.byref(calls), C.byref(ns)), "dcoco_stage_read")
    return {dcoco_stage_name(handle, s): float(ms[s]) for s in range(ns.value)}, calls.value


def dcoco_stage_name(handle, s: int) -> str | None:
    r = _lib.dcoco_stage_name(handle, s)
    return None if r is None else r.decode()


# ------------------------------------------------------------------ convenience wrapper
class Corrector:
    """Owns a handle + packed weights; allocates output tensors per call."""

    def __init__(self, weights: dict, vocab: int, hidden: int, slots: int = 16, topk: int = 16,
                 max_batch: int = 32, variant: int = 0, sigma: float = 1.0, ln_eps: float = 1e-5,
                 host_staging: bool = False, path_rule: int = 0, beam_width: int = 2, beam_topm: int = 0):
        self.vocab, self.hidden, self.slots, self.topk = vocab, hidden, slots, topk
        self.B = slots - 1
        self.max_batch = max_batch
        self.path_rule = path_rule
        self.handle = dcoco_create(vocab, hidden, slots, topk, max_batch, variant, sigma, ln_eps,
                                   host_staging=host_staging, path_rule=path_rule, beam_width=beam_width,
                                   beam_topm=beam_topm)
        try:
            self.weights = dcoco_weights_create(self.handle, weights)
        except Exception:
            dcoco_destroy(self.handle)
            raise

    def close(self):
        if getattr(self, "weights", None) is not None:
            dcoco_weights_destroy(self.weights)
            self.weights = None
        if getattr(self, "handle", None) is not None:
            dcoco_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, N: int, device="cuda", full: bool = True, features: bool = False):
        B, K = self.B, self.topk
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        out = {"tokens": torch.empty(N, B, **i32), "accept_len": torch.empty(N, **i32)}
        if full:
            out.update(choice=torch.empty(N, B, **i32), scores=torch.empty(N, B - 1, K, K, **f32),
                       topk_ids=torch.empty(N, B, K, **i32), topk_val=torch.empty(N, B, K, **f32),
                       margin=torch.empty(N, B - 1, **f32))
        if features:
            out["cand_feat"] = torch.empty(N, B, K, 5, **f32)
        return out

    def correct(self, logits, hidden, cand_embed, target_tokens=None, out=None, full=True,
                logits_slot_stride=None, stream=None):
        N = logits.shape[0]
        out = out if out is not None else self.alloc_outputs(N, logits.device, full)
        kw = {k: v for k, v in out.items() if k != "accept_len"}
        dcoco_correct(self.handle, self.weights, N, logits, hidden, cand_embed, target_tokens,
                      accept_len=out.get("accept_len") if target_tokens is not None else None,
                      logits_slot_stride=logits_slot_stride, stream=stream, **kw)
        return out

    def verify_stochastic(self, target_logits, tokens, u_accept, u_draw, target_stride=None, stream=None):
        """-> dict(accept_len [N], next_token [N], q_accept [N, B]) on the tokens' device."""
        N = tokens.shape[0]
        dev = tokens.device
        out = {"accept_len": torch.empty(N, dtype=torch.int32, device=dev),
               "next_token": torch.empty(N, dtype=torch.int32, device=dev),
               "q_accept": torch.empty(N, self.B, dtype=torch.float32, device=dev)}
        dcoco_verify_stochastic(self.handle, N, target_logits, tokens, u_accept, u_draw, out["accept_len"],
                                out["next_token"], out["q_accept"], target_stride, stream)
        return out

    def status(self) -> int:
        return dcoco_get_device_status(self.handle)
