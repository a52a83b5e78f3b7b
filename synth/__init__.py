"""Seeded synthetic inputs for the draft-correction path.

This module only draws random numbers and packs them into arrays.  It holds
none of the correction method's arithmetic, so both the CPU oracle tests and
the CUDA library tests can use it.  Every draw is from a NumPy PCG64 generator
seeded by the caller.

Recipe (shapes follow a Qwen3-8B-sized DFlash drafter, as the DCOCO page
"Contextual Correction of Parallel Drafts for Speculative Decoding" describes
in its method section: 16 block positions = 1 anchor + 15 draft slots, top-16
candidates, a frozen V x d embedding table, r = 128, a 386 -> 256 -> 1 MLP):

* logits: bf16( 2 * N(0,1) + boost ), with `planted` distinct token ids per
  slot (uniform without replacement) receiving boost ~ U(lo, hi); computed in
  fp32 and rounded to bf16 (round-to-nearest-even).  Shape [N, slots, stride].
* hidden states: bf16 N(0,1), shape [N, slots, d].
* embedding table: bf16 N(0, 0.02^2), shape [V, d].
* weights: fp32 Xavier-uniform (gain 1) for every matrix; b1 = b2 = 0,
  gamma = 1, beta = 0.  `perturb=True` also draws b1, b2, gamma-1, beta from
  N(0, 0.1^2) so those terms are exercised.  `zero_out=True` zeroes the
  MLP's output layer (w2 = 0, b2 = 0), the initialisation the DCOCO page
  describes, under which the learned correction term vanishes.
* target tokens: with probability 0.6 uniform over the slot's top-16
  candidate ids (which the caller supplies), else uniform over [0, V).
"""
from __future__ import annotations

import os

import numpy as np

__all__ = [
    "bf16_bits", "bf16_to_f32", "make_logits", "make_hidden", "make_embedding",
    "make_weights", "make_cosine_weights", "draw_targets", "CONFIGS",
]

# Named workloads (sizes only).  Entries: N requests, slots (incl. anchor),
# V vocabulary, d hidden width, K candidates, planted ids per slot, boost range.
CONFIGS = {
    "tiny": dict(N=1, slots=16, V=151936, d=4096, K=16, planted=32, boost=(4.0, 12.0)),
    "qwen3_8b_c32": dict(N=32, slots=16, V=151936, d=4096, K=16, planted=32, boost=(4.0, 12.0)),
    "cosine_c16": dict(N=16, slots=16, V=151936, d=4096, K=16, planted=32, boost=(4.0, 12.0)),
    "wide_k32_d5120": dict(N=32, slots=16, V=151936, d=5120, K=32, planted=8, boost=(8.0, 16.0)),
    "tier_low": dict(slots=16, V=151936, d=4096, K=16, planted=64, boost=(2.0, 6.0)),
    "tier_mid": dict(slots=16, V=151936, d=4096, K=16, planted=64, boost=(4.0, 12.0)),
    "tier_high": dict(slots=16, V=151936, d=4096, K=16, planted=64, boost=(8.0, 16.0)),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_logits(rng: np.random.Generator, N: int, slots: int, V: int, planted: int,
                boost: tuple[float, float], stride: int | None = None) -> np.ndarray:
    """bf16 logits [N, slots, stride]; columns >= V (row padding) are -inf."""
    stride = V if stride is None else stride
    assert stride >= V
    base = rng.standard_normal((N, slots, V), dtype=np.float32) * np.float32(2.0)
    if planted > 0:
        for n in range(N):
            for s in range(slots):
                ids = rng.choice(V, size=min(planted, V), replace=False)
                base[n, s, ids] += rng.uniform(boost[0], boost[1], size=ids.shape[0]).astype(np.float32)
    out = np.full((N, slots, stride), 0xFF80, dtype=np.uint16)
    out[:, :, :V] = bf16_bits(base)
    return out


def make_hidden(rng: np.random.Generator, N: int, slots: int, d: int) -> np.ndarray:
    return bf16_bits(rng.standard_normal((N, slots, d), dtype=np.float32))


def make_embedding(rng: np.random.Generator, V: int, d: int, std: float = 0.02,
                   rows_per_draw: int = 8192, threads: int | None = None) -> np.ndarray:
    """bf16 N(0, std^2) table [V, d].  Row blocks are drawn from child generators
    (seeded from `rng`) on a thread pool, so the result depends only on `rng`."""
    from concurrent.futures import ThreadPoolExecutor
    out = np.empty((V, d), dtype=np.uint16)
    starts = list(range(0, V, rows_per_draw))
    children = np.random.SeedSequence(int(rng.integers(0, 2**63))).spawn(len(starts))

    def fill(k):
        r0 = starts[k]
        r1 = min(V, r0 + rows_per_draw)
        g = np.random.Generator(np.random.PCG64(children[k]))
        out[r0:r1] = bf16_bits(g.standard_normal((r1 - r0, d), dtype=np.float32) * np.float32(std))

    with ThreadPoolExecutor(max_workers=threads or min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(len(starts))))
    return out


def _xavier(rng: np.random.Generator, fan_out: int, fan_in: int) -> np.ndarray:
    a = np.sqrt(6.0 / (fan_in + fan_out))
    return rng.uniform(-a, a, size=(fan_out, fan_in)).astype(np.float32)


def make_weights(rng: np.random.Generator, d: int, r: int = 128, H: int = 256,
                 zero_out: bool = False, perturb: bool = False) -> dict[str, np.ndarray]:
    """Corrector weights, PyTorch Linear layout [out, in], fp32."""
    w = {
        "w_cand": _xavier(rng, r, d),
        "w_ctx": _xavier(rng, r, d),
        "w_fuse": _xavier(rng, r, 2 * r),
        "ln_gamma": np.ones(r, dtype=np.float32),
        "ln_beta": np.zeros(r, dtype=np.float32),
        "w_pair": _xavier(rng, r, 2 * d),
        "w1": _xavier(rng, H, 3 * r + 2),
        "b1": np.zeros(H, dtype=np.float32),
        "w2": _xavier(rng, 1, H).reshape(H),
        "b2": np.zeros(1, dtype=np.float32),
    }
    if perturb:
        w["b1"] = (rng.standard_normal(H) * 0.1).astype(np.float32)
        w["b2"] = (rng.standard_normal(1) * 0.1).astype(np.float32)
        w["ln_gamma"] = (1.0 + rng.standard_normal(r) * 0.1).astype(np.float32)
        w["ln_beta"] = (rng.standard_normal(r) * 0.1).astype(np.float32)
    if zero_out:
        w["w2"] = np.zeros(H, dtype=np.float32)
        w["b2"] = np.zeros(1, dtype=np.float32)
    return w


def make_cosine_weights(rng: np.random.Generator, d: int, r: int = 128) -> dict[str, np.ndarray]:
    """The in/out projection of the cosine variant: W_io [2r, 2d], no bias."""
    return {"w_io": _xavier(rng, 2 * r, 2 * d)}


def draw_targets(rng: np.random.Generator, top16_ids: np.ndarray, V: int, p_hit: float = 0.6) -> np.ndarray:
    """Target tokens [N, B]: w.p. p_hit a uniform pick from the slot's top-16 ids, else uniform in [0, V)."""
    N, B, K16 = top16_ids.shape
    hit = rng.random((N, B)) < p_hit
    pick = rng.integers(0, K16, size=(N, B))
    uni = rng.integers(0, V, size=(N, B))
    from_top = np.take_along_axis(top16_ids, pick[..., None], axis=2)[..., 0]
    return np.where(hit, from_top, uni).astype(np.int32)
