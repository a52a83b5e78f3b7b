"""Seeded problems shared by the GPU parity tests: synthetic inputs (synth),
the CPU oracle's answer, the CUDA library's answer, and the comparison rules.

Comparison rules (fixed before any kernel ran; `compare_path` holds the
rules of the highest-scoring-path selection):
  * top-K ids and values, chosen tokens and accept_len: bit-exact;
  * scores: max |GPU - oracle| <= SCORE_TOL = 2e-3 (fp32 vs fp64);
  * the walk: a choice may differ from the oracle only where the oracle's
    best and second-best successor scores are within SCORE_TOL (a near tie),
    and the GPU's pick must then be within SCORE_TOL of the best.  After such
    a divergence the oracle is re-walked from the GPU's prefix, tokens are
    checked against the GPU's choices, and accept_len against the oracle's
    verify of the GPU's tokens.  Divergences are counted and reported.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

SCORE_TOL = 2e-3

_E_CACHE: dict = {}


def embedding(seed: int, V: int, d: int) -> np.ndarray:
    """The embedding table of a problem depends only on (seed, V, d); cached."""
    key = (seed, V, d)
    if key not in _E_CACHE:
        if len(_E_CACHE) >= 2:
            _E_CACHE.pop(next(iter(_E_CACHE)))
        _E_CACHE[key] = synth.make_embedding(np.random.default_rng([seed, V, d, 0xE]), V, d)
    return _E_CACHE[key]


class Problem:
    def __init__(self, seed: int, N: int, V: int, d: int, K: int = 16, slots: int = 16,
                 planted: int = 32, boost=(4.0, 12.0), stride: int | None = None, variant: int = 0,
                 sigma: float = 1.0, zero_out: bool = False, perturb: bool = False,
                 targets: bool = True, path_rule: int = 0, beam_width: int = 2, beam_topm: int = 0):
        rng = np.random.default_rng(seed)
        self.N, self.V, self.d, self.K, self.slots, self.B = N, V, d, K, slots, slots - 1
        self.variant, self.sigma, self.path_rule = variant, sigma, path_rule
        self.beam_width, self.beam_topm = beam_width, beam_topm
        self.stride = stride if stride is not None else ((V + 7) // 8) * 8
        self.logits = synth.make_logits(rng, N, slots, V, planted, boost, stride=self.stride)
        self.hidden = synth.make_hidden(rng, N, slots, d)
        self.E = embedding(seed, V, d)
        if variant == 0:
            self.w = synth.make_weights(rng, d, zero_out=zero_out, perturb=perturb)
        else:
            self.w = synth.make_cosine_weights(rng, d)
        self.model = oracle.Model(self.w, V=V, d=d, slots=slots, K=K, beam_width=beam_width, beam_topm=beam_topm)
        self.rng = rng
        self.targets = None
        if targets:
            top16 = self.oracle_top16()
            self.targets = synth.draw_targets(rng, top16, V)

    def oracle_top16(self, requests=None):
        req = range(self.N) if requests is None else requests
        k16 = min(16, self.V)
        return np.stack([np.stack([oracle.topk_row(self.logits[n, i + 1, :self.V], k16)[0]
                                   for i in range(self.B)]) for n in req])

    def oracle(self, requests=None):
        return oracle.correct_batch(self.model, self.logits, self.hidden, self.E, self.targets,
                                    variant=self.variant, sigma=self.sigma, requests=requests,
                                    path_rule=self.path_rule)


def bf16_tensor(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def make_corrector(prob: Problem, max_batch: int | None = None):
    import torch
    import draft_correction_slot_gb300 as dc
    return dc.Corrector({k: torch.from_numpy(v) for k, v in prob.w.items()}, prob.V, prob.d,
                        prob.slots, prob.K, max_batch=max_batch or prob.N, variant=prob.variant,
                        sigma=prob.sigma, path_rule=prob.path_rule, beam_width=prob.beam_width,
                        beam_topm=prob.beam_topm)


def run_gpu(prob: Problem, max_batch: int | None = None, corr=None, E_dev=None):
    import torch
    import draft_correction_slot_gb300 as dc
    own = corr is None
    if own:
        corr = make_corrector(prob, max_batch)
    E_dev = E_dev if E_dev is not None else bf16_tensor(prob.E)
    tg = None if prob.targets is None else torch.from_numpy(prob.targets).cuda()
    out = corr.correct(bf16_tensor(prob.logits), bf16_tensor(prob.hidden), E_dev, tg,
                       logits_slot_stride=prob.stride)
    torch.cuda.synchronize()
    status = corr.status()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    if own:
        corr.close()
    assert status == dc.DCOCO_OK, f"device status {status}"
    return res


def compare(prob: Problem, gpu: dict, ref: dict, tol: float = SCORE_TOL) -> dict:
    """Apply the comparison rules; returns stats (max score error, divergences)."""
    req = ref["requests"]
    g = {k: v[req] for k, v in gpu.items()}
    np.testing.assert_array_equal(g["topk_ids"], ref["topk_ids"], err_msg="top-K ids")
    np.testing.assert_array_equal(g["topk_val"], ref["topk_val"], err_msg="top-K values")
    err = float(np.abs(g["scores"].astype(np.float64) - ref["scores"]).max()) if ref["scores"].size else 0.0
    assert err <= tol, f"max |score error| {err:.3e} > {tol}"
    diverged = 0
    for j, n in enumerate(req):
        gc = g["choice"][j]
        sc = ref["scores"][j]
        assert gc[0] == 0
        for p in range(prob.B - 1):
            row = sc[p, gc[p]]
            best = int(np.flatnonzero(row == row.max())[0])
            if gc[p + 1] != best:
                second = np.max(np.delete(row, best))
                assert row[best] - second < tol and row[gc[p + 1]] >= row[best] - tol, (
                    f"request {n} slot {p + 2}: GPU picked {gc[p + 1]}, oracle {best}, "
                    f"margin {row[best] - second:.3e}")
                diverged += 1
            np.testing.assert_allclose(g["margin"][j, p], row[best] - np.max(np.delete(row, best)),
                                       atol=2 * tol)
        toks = ref["topk_ids"][j][np.arange(prob.B), gc]
        np.testing.assert_array_equal(g["tokens"][j], toks, err_msg=f"tokens of request {n}")
        if prob.targets is not None:
            assert g["accept_len"][j] == oracle.verify(toks, prob.targets[n])
            if diverged == 0:
                assert g["accept_len"][j] == ref["accept_len"][j]
    if diverged == 0:
        np.testing.assert_array_equal(g["tokens"], ref["tokens"])
    return {"max_score_err": err, "diverged": diverged}


def path_total(sc: np.ndarray, path) -> float:
    return float(sum(sc[p, path[p], path[p + 1]] for p in range(sc.shape[0])))


def compare_path(prob: Problem, gpu: dict, ref: dict, tol: float = SCORE_TOL) -> dict:
    """Rules for the highest-scoring path (path_rule 1) and the beam walk
    (path_rule 2; there the optimum bound does not apply, the beam being no
    exact optimizer):
      * top-K ids and values bit-exact, scores within tol (as `compare`);
      * on the GPU's own scores the oracle's dynamic program with the kernel's
        single-precision totals (the same order of additions and the same tie
        rule) must give the GPU's path and margins exactly;
      * on the oracle's scores the GPU's path must score within 2 (B-1) tol of
        the oracle's optimum (each of the B-1 terms moves by at most tol);
        paths that differ are counted as divergences;
      * tokens are the chosen candidates' ids and accept_len the verify of
        those tokens (and the oracle's own when no request diverged)."""
    req = ref["requests"]
    g = {k: v[req] for k, v in gpu.items()}
    np.testing.assert_array_equal(g["topk_ids"], ref["topk_ids"], err_msg="top-K ids")
    np.testing.assert_array_equal(g["topk_val"], ref["topk_val"], err_msg="top-K values")
    err = float(np.abs(g["scores"].astype(np.float64) - ref["scores"]).max()) if ref["scores"].size else 0.0
    assert err <= tol, f"max |score error| {err:.3e} > {tol}"
    diverged = 0
    for j, n in enumerate(req):
        gc = g["choice"][j]
        if prob.path_rule == 1:
            own_choice, own_margin = oracle.viterbi_f32(g["scores"][j])
        else:
            own_choice, own_margin = oracle.beam_f32(g["scores"][j], prob.beam_width, prob.beam_topm)
        np.testing.assert_array_equal(gc, own_choice, err_msg=f"request {n}: path on the GPU's scores")
        np.testing.assert_array_equal(g["margin"][j], own_margin, err_msg=f"request {n}: margins")
        sc = ref["scores"][j]
        if prob.path_rule == 1:
            best = path_total(sc, ref["choice"][j])
            mine = path_total(sc, gc)
            assert mine >= best - 2 * (prob.B - 1) * tol, (
                f"request {n}: GPU path total {mine:.6f} vs optimum {best:.6f}")
        if not np.array_equal(gc, ref["choice"][j]):
            diverged += 1
        toks = ref["topk_ids"][j][np.arange(prob.B), gc]
        np.testing.assert_array_equal(g["tokens"][j], toks, err_msg=f"tokens of request {n}")
        if prob.targets is not None:
            assert g["accept_len"][j] == oracle.verify(toks, prob.targets[n])
    if diverged == 0:
        np.testing.assert_array_equal(g["tokens"], ref["tokens"])
        if prob.targets is not None:
            np.testing.assert_array_equal(g["accept_len"][:len(req)], ref["accept_len"])
    return {"max_score_err": err, "diverged": diverged}
