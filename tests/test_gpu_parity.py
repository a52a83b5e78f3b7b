"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs.  Rules in tests/problem.py: ids, tokens and
accept_len bit-exact; scores within 2e-3; walk divergences only at oracle
near-ties (counted)."""
import copy

import numpy as np
import pytest

import oracle
import synth
from problem import make_corrector, compare_path, Problem, bf16_tensor, compare, run_gpu

pytestmark = pytest.mark.gpu

V_QWEN, D_QWEN = 151936, 4096


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


def report(name, stats):
    print(f"[parity] {name}: max|dS|={stats['max_score_err']:.2e} near-tie divergences={stats['diverged']}")


# ------------------------------------------------------------------ top-K edge cases
def _adversarial_rows(rng, V, stride):
    rows = []
    f = lambda a: synth.bf16_bits(np.asarray(a, np.float32))  # noqa: E731
    rows.append(np.full(V, f([1.5])[0], np.uint16))                        # all equal
    r = np.full(V, f([-np.inf])[0], np.uint16)                             # mostly -inf
    r[rng.choice(V, 5, replace=False)] = f(rng.standard_normal(5))
    rows.append(r)
    rows.append(np.full(V, f([-np.inf])[0], np.uint16))                    # all -inf
    r = f(np.round(rng.standard_normal(V)))                                # few levels, many ties
    rows.append(r)
    r = np.zeros(V, np.uint16); r[rng.choice(V, V // 2, replace=False)] = 0x8000  # -0 / +0 mix
    rows.append(r)
    r = f(rng.standard_normal(V) - 10); r[-(V % 8 or 8):] = f([50.0])[0]   # maxima in the tail
    rows.append(r)
    r = f(-np.abs(rng.standard_normal(V)) - 1)                             # all negative
    rows.append(r)
    r = f(rng.standard_normal(V)); r[::2048 * 8] = f([30.0])[0]            # chunk boundaries
    r[2048 * 8 - 1::2048 * 8] = f([29.0])[0]
    rows.append(r)
    r = f(np.full(V, 2.0)); r[rng.choice(V, 3, replace=False)] = f([3.0])[0]  # K-th value tied
    rows.append(r)
    out = np.full((len(rows), stride), 0xFF80, np.uint16)
    for i, r in enumerate(rows):
        out[i, :V] = r
    return out


@pytest.mark.parametrize("V,K", [(151936, 16), (151933, 32), (4099, 8), (40, 16), (20000, 32)])
def test_topk_adversarial(torch_cuda, V, K):
    torch = torch_cuda
    import draft_correction_slot_gb300 as dc
    rng = np.random.default_rng(V + K)
    stride = ((V + 7) // 8) * 8
    rows = _adversarial_rows(rng, V, stride)
    slots = rows.shape[0] + 1
    logits = np.full((1, slots, stride), 0xFF80, np.uint16)
    logits[0, 1:] = rows
    h = dc.dcoco_create(V, 64, slots, K, max_batch=1)
    try:
        ids = torch.empty(1, slots - 1, K, dtype=torch.int32, device="cuda")
        vals = torch.empty(1, slots - 1, K, dtype=torch.float32, device="cuda")
        for _ in range(2):  # twice: the row counters must reset themselves
            dc.dcoco_topk(h, 1, bf16_tensor(logits), ids, vals, logits_slot_stride=stride)
            torch.cuda.synchronize()
            gi, gv = ids.cpu().numpy()[0], vals.cpu().numpy()[0]
            for i in range(slots - 1):
                ri, rv = oracle.topk_row(logits[0, i + 1, :V], K)
                np.testing.assert_array_equal(gi[i], ri, err_msg=f"row {i} ids")
                np.testing.assert_array_equal(gv[i].view(np.uint32), rv.view(np.uint32),
                                              err_msg=f"row {i} values (bitwise, +0 canonical)")
    finally:
        dc.dcoco_destroy(h)


def test_topk_random_many_rows(torch_cuda):
    prob = Problem(1, N=8, V=V_QWEN, d=64, targets=False)
    import draft_correction_slot_gb300 as dc
    torch = torch_cuda
    h = dc.dcoco_create(V_QWEN, 64, 16, 16, max_batch=8)
    ids = torch.empty(8, 15, 16, dtype=torch.int32, device="cuda")
    vals = torch.empty(8, 15, 16, dtype=torch.float32, device="cuda")
    dc.dcoco_topk(h, 8, bf16_tensor(prob.logits), ids, vals)
    torch.cuda.synchronize()
    dc.dcoco_destroy(h)
    ref = prob.oracle_top16()
    np.testing.assert_array_equal(ids.cpu().numpy(), ref)


# ------------------------------------------------------------------ whole path
def test_tiny_single_request(torch_cuda):
    """One request, Qwen3-8B shapes: V=151,936, d=4096, K=16, 16 slots."""
    prob = Problem(0, N=1, V=V_QWEN, d=D_QWEN)
    report("tiny", compare(prob, run_gpu(prob), prob.oracle()))


def test_tiny_zero_output_layer(torch_cuda):
    """Output layer zeroed: scores equal l_{p+1}(b) exactly and the walk returns the draft argmax."""
    prob = Problem(0, N=1, V=V_QWEN, d=D_QWEN, zero_out=True)
    g = run_gpu(prob)
    report("zero-output", compare(prob, g, prob.oracle()))
    vals = g["topk_val"][0]
    for p in range(prob.B - 1):
        np.testing.assert_array_equal(g["scores"][0, p], np.broadcast_to(vals[p + 1], (16, 16)))
    np.testing.assert_array_equal(g["choice"], 0)
    np.testing.assert_array_equal(g["tokens"][0], g["topk_ids"][0, :, 0])


def test_ragged_small_shapes(torch_cuda):
    """Ragged vocabulary (V % 8 != 0, padded stride) and a small hidden width."""
    prob = Problem(3, N=3, V=4099, d=256, stride=4112, perturb=True)
    report("ragged", compare(prob, run_gpu(prob, max_batch=5), prob.oracle()))


@pytest.mark.parametrize("K", [8, 32])
def test_other_candidate_counts(torch_cuda, K):
    prob = Problem(4 + K, N=2, V=20011, d=512, K=K, planted=8, boost=(8.0, 16.0))
    report(f"K={K}", compare(prob, run_gpu(prob), prob.oracle()))


def test_wide_k32_d5120(torch_cuda):
    """K=32, d=5120, low-entropy logits (8 planted ids, U(8,16)): 14 x 32^2 transitions."""
    prob = Problem(5, N=2, V=V_QWEN, d=5120, K=32, planted=8, boost=(8.0, 16.0))
    report("wide", compare(prob, run_gpu(prob), prob.oracle()))


def test_back_to_back_handles(torch_cuda):
    """Two handles in turn, the second after the first is closed: its buffers
    may take the first one's addresses, and every kernel must read this
    call's results, not lines cached from the earlier handle's calls (the
    kernels launched early read the previous kernel's outputs through L2)."""
    first = Problem(36, N=2, V=20011, d=512, K=32, planted=8, boost=(8.0, 16.0))
    report("handle-1", compare(first, run_gpu(first), first.oracle()))
    second = Problem(5, N=2, V=V_QWEN, d=5120, K=32, planted=8, boost=(8.0, 16.0))
    report("handle-2", compare(second, run_gpu(second), second.oracle()))


def test_bounded_wait_expires_into_device_status(torch_cuda):
    """The kernels' bounded wait, on an mbarrier nothing completes, gives up
    after its limit: the status word reads DCOCO_EDEVICE once, is cleared by
    the read, and the context keeps working (a parity run on the same handle)."""
    import torch
    import draft_correction_slot_gb300 as dc
    prob = Problem(21, N=1, V=4099, d=128)
    corr = dc.Corrector({k: torch.from_numpy(v) for k, v in prob.w.items()}, prob.V, prob.d, prob.slots,
                        prob.K, max_batch=1)
    try:
        assert corr.status() == dc.DCOCO_OK
        dc.dcoco_selftest_wait_timeout(corr.handle, 2_000_000, torch.cuda.current_stream().cuda_stream)
        assert corr.status() == dc.DCOCO_EDEVICE
        assert corr.status() == dc.DCOCO_OK
        report("after-timeout", compare(prob, run_gpu(prob, corr=corr), prob.oracle()))
        with pytest.raises(dc.DcocoError):
            dc.dcoco_selftest_wait_timeout(corr.handle, 10, 0)  # below the 1 us floor
    finally:
        corr.close()


def test_cosine_variant(torch_cuda):
    prob = Problem(6, N=2, V=V_QWEN, d=D_QWEN, variant=1, sigma=1.0)
    report("cosine", compare(prob, run_gpu(prob), prob.oracle()))


def test_cosine_variant_sigma8(torch_cuda):
    prob = Problem(7, N=2, V=5003, d=128, variant=1, sigma=8.0)
    report("cosine-sigma8", compare(prob, run_gpu(prob), prob.oracle()))


def test_short_block(torch_cuda):
    """slots = 3 (B = 2 draft slots, one pair) and slots = 32 (B = 31)."""
    for slots in (3, 32):
        prob = Problem(8 + slots, N=2, V=3001, d=128, slots=slots)
        report(f"slots={slots}", compare(prob, run_gpu(prob), prob.oracle()))


def test_determinism_and_batch_invariance(torch_cuda):
    """Within one handle: the same call twice gives the same bits, and a
    request's results do not depend on the batch it came in.  A handle whose
    max_batch selects another projection split count (here 4 and 32 requests:
    eight and four splits) sums the projection in another order: its
    discrete outputs are the same and its scores agree to fp32 rounding."""
    prob = Problem(9, N=4, V=V_QWEN, d=D_QWEN, targets=True)
    corr = make_corrector(prob, max_batch=32)
    try:
        a = run_gpu(prob, corr=corr)
        a2 = run_gpu(prob, corr=corr)
        for k in a:
            np.testing.assert_array_equal(a[k], a2[k], err_msg=f"{k} not deterministic")
        one = copy.copy(prob)
        one.N = 1
        one.logits, one.hidden, one.targets = prob.logits[2:3], prob.hidden[2:3], prob.targets[2:3]
        c = run_gpu(one, corr=corr)
        for k in c:
            np.testing.assert_array_equal(c[k][0], a[k][2], err_msg=f"{k} depends on the batch")
    finally:
        corr.close()
    b = run_gpu(prob)  # a handle for 4 requests: eight splits instead of four
    for k in ("tokens", "choice", "accept_len", "topk_ids", "topk_val"):
        if k in a:
            np.testing.assert_array_equal(a[k], b[k], err_msg=f"{k} differs between split counts")
    np.testing.assert_allclose(a["scores"], b["scores"], rtol=0, atol=1e-4)


@pytest.mark.parametrize("tier,boost", [("low", (2.0, 6.0)), ("mid", (4.0, 12.0)), ("high", (8.0, 16.0))])
def test_entropy_tiers(torch_cuda, tier, boost):
    """Serving-sweep tiers: 64 planted ids per slot; accept_len is oracle-checked."""
    prob = Problem(20, N=4, V=V_QWEN, d=D_QWEN, planted=64, boost=boost)
    ref = prob.oracle()
    stats = compare(prob, run_gpu(prob), ref)
    report(f"tier-{tier}", stats)
    print(f"[tier] {tier}: mean accept_len = {ref['accept_len'].mean():.3f}")


@pytest.mark.slow
def test_full_size_batch32_sampled(torch_cuda):
    """Batch 32 at Qwen3-8B shapes, the launch the benchmark times; the oracle
    checks sampled requests."""
    prob = Problem(1, N=32, V=V_QWEN, d=D_QWEN, targets=False)
    sample = [0, 13, 31]
    top16 = prob.oracle_top16()
    prob.targets = synth.draw_targets(prob.rng, top16, prob.V)
    g = run_gpu(prob)
    report("batch32", compare(prob, g, prob.oracle(requests=sample)))
    # top-K of every request is cheap to check in full
    np.testing.assert_array_equal(g["topk_ids"], top16)


@pytest.mark.slow
def test_full_size_cosine_batch16_sampled(torch_cuda):
    """The cosine variant at its own batch of 16 (Qwen3-8B shapes, the
    launch the benchmark times): every request's top-K in full, the oracle
    on sampled requests."""
    prob = Problem(41, N=16, V=V_QWEN, d=D_QWEN, variant=1, sigma=1.0, targets=False)
    top16 = prob.oracle_top16()
    prob.targets = synth.draw_targets(prob.rng, top16, prob.V)
    g = run_gpu(prob)
    np.testing.assert_array_equal(g["topk_ids"], top16)
    report("cosine batch16", compare(prob, g, prob.oracle(requests=[0, 7, 15])))


@pytest.mark.slow
def test_full_size_wide_k32_d5120_batch32_sampled(torch_cuda):
    """d = 5120, K = 32, 8 planted tokens per slot with boost U(8,16), at the
    batch of 32 the benchmark times: 60 candidate tiles of the projection
    (66 four-CTA clusters with the draft-slot tiles, more than one wave) and
    1920 pair scores.  Every request's top-K in full (the first 16 of the
    oracle's top 32 for the targets), the oracle on sampled requests."""
    prob = Problem(42, N=32, V=V_QWEN, d=5120, K=32, planted=8, boost=(8.0, 16.0), targets=False)
    top32 = np.stack([np.stack([oracle.topk_row(prob.logits[n, i + 1, :prob.V], 32)[0] for i in range(prob.B)])
                      for n in range(prob.N)])
    prob.targets = synth.draw_targets(prob.rng, top32[..., :16], prob.V)
    g = run_gpu(prob)
    np.testing.assert_array_equal(g["topk_ids"], top32)
    report("wide batch32", compare(prob, g, prob.oracle(requests=[0, 31])))


def test_host_entry_matches_device_entry(torch_cuda):
    torch = torch_cuda
    import draft_correction_slot_gb300 as dc
    prob = Problem(11, N=3, V=4099, d=256, stride=4104)
    dev = run_gpu(prob)
    corr = dc.Corrector({k: torch.from_numpy(v) for k, v in prob.w.items()}, prob.V, prob.d,
                        max_batch=3, host_staging=True)
    E = bf16_tensor(prob.E)
    # pinned logits are read in place; pageable ones go through the staging copy
    for pinned in (True, False):
        lg = torch.from_numpy(prob.logits.view(np.int16).copy())
        lg = lg.pin_memory() if pinned else lg
        hd = torch.from_numpy(prob.hidden.view(np.int16)).pin_memory()
        tg = torch.from_numpy(prob.targets).pin_memory()
        out = {k: torch.empty_like(torch.from_numpy(dev[k])).pin_memory()
               for k in ("tokens", "accept_len", "scores", "topk_ids")}
        dc.dcoco_correct_host(corr.handle, corr.weights, 3, lg, hd, E, tg, logits_slot_stride=prob.stride,
                              **out)
        for k, v in out.items():
            np.testing.assert_array_equal(v.numpy(), dev[k], err_msg=f"{k} (pinned={pinned})")
    corr.close()


def test_argument_errors(torch_cuda):
    torch = torch_cuda
    import draft_correction_slot_gb300 as dc
    prob = Problem(12, N=2, V=4099, d=256, stride=4104)
    corr = dc.Corrector({k: torch.from_numpy(v) for k, v in prob.w.items()}, prob.V, prob.d, max_batch=2)
    lg, hd, E = bf16_tensor(prob.logits), bf16_tensor(prob.hidden), bf16_tensor(prob.E)
    tok = torch.empty(3, 15, dtype=torch.int32, device="cuda")
    with pytest.raises(dc.DcocoError) as e:       # batch above max_batch
        dc.dcoco_correct(corr.handle, corr.weights, 3, lg, hd, E, tokens=tok, logits_slot_stride=4104)
    assert e.value.status == dc.DCOCO_EBATCH
    with pytest.raises(dc.DcocoError) as e:       # stride not a multiple of 8
        dc.dcoco_correct(corr.handle, corr.weights, 1, lg, hd, E, tokens=tok, logits_slot_stride=4100)
    assert e.value.status == dc.DCOCO_EINVAL
    with pytest.raises(dc.DcocoError) as e:       # misaligned logits pointer
        dc.dcoco_correct(corr.handle, corr.weights, 1, lg.view(-1)[1:], hd, E, tokens=tok,
                         logits_slot_stride=4104)
    assert e.value.status == dc.DCOCO_EINVAL
    with pytest.raises(dc.DcocoError) as e:       # targets without accept_len
        dc.dcoco_correct(corr.handle, corr.weights, 1, lg, hd, E, torch.zeros(2, 15, dtype=torch.int32,
                         device="cuda"), tokens=tok, logits_slot_stride=4104)
    assert e.value.status == dc.DCOCO_EINVAL
    dc.dcoco_correct(corr.handle, corr.weights, 0, lg, hd, E, tokens=tok)  # batch 0: no-op
    assert corr.status() == dc.DCOCO_OK
    corr.close()


# ------------------------------------------------------------------ highest-scoring path
def test_viterbi_tiny_single_request(torch_cuda):
    """Path rule 1 (LiLiCorr App. E Eq. (12)) at Qwen3-8B shapes, one request."""
    prob = Problem(20, N=1, V=V_QWEN, d=D_QWEN, path_rule=1)
    report("viterbi tiny", compare_path(prob, run_gpu(prob), prob.oracle()))


def test_viterbi_zero_output_layer(torch_cuda):
    """Delta = 0: the highest-scoring path is the per-slot draft argmax."""
    prob = Problem(21, N=2, V=20011, d=512, zero_out=True, path_rule=1)
    g = run_gpu(prob)
    report("viterbi zero-output", compare_path(prob, g, prob.oracle()))
    np.testing.assert_array_equal(g["choice"], 0)


@pytest.mark.parametrize("K", [8, 16, 32])
def test_viterbi_batch(torch_cuda, K):
    prob = Problem(22 + K, N=4, V=20011, d=512, K=K, perturb=True, path_rule=1)
    report(f"viterbi K={K}", compare_path(prob, run_gpu(prob), prob.oracle()))


def test_viterbi_cosine_variant(torch_cuda):
    """The cosine variant selects its path in the stand-alone step-5 launch."""
    prob = Problem(23, N=3, V=20011, d=512, variant=1, path_rule=1)
    report("viterbi cosine", compare_path(prob, run_gpu(prob), prob.oracle()))


def test_viterbi_and_greedy_agree_on_top_k_and_scores(torch_cuda):
    """Only step 5 depends on the path rule: the top-K and the scores of the
    two rules are bit-identical on the same inputs."""
    a = Problem(24, N=2, V=20011, d=512, perturb=True, path_rule=0)
    b = Problem(24, N=2, V=20011, d=512, perturb=True, path_rule=1)
    ga, gb = run_gpu(a), run_gpu(b)
    for k in ("topk_ids", "topk_val", "scores"):
        np.testing.assert_array_equal(ga[k], gb[k])


# ------------------------------------------------------------------ beam walk
@pytest.mark.parametrize("width,topm", [(1, 0), (2, 0), (4, 0), (3, 4)])
def test_beam_batch(torch_cuda, width, topm):
    """Path rule 2 (the DCOCO page's reproduction assessment (2)-(3)):
    decisions equal the oracle's in the kernel's precision on the GPU's scores."""
    prob = Problem(30 + width, N=4, V=20011, d=512, perturb=True, path_rule=2, beam_width=width, beam_topm=topm)
    report(f"beam W={width} m={topm}", compare_path(prob, run_gpu(prob), prob.oracle()))


def test_beam_width_one_equals_greedy(torch_cuda):
    a = Problem(35, N=3, V=20011, d=512, perturb=True, path_rule=0)
    b = Problem(35, N=3, V=20011, d=512, perturb=True, path_rule=2, beam_width=1)
    ga, gb = run_gpu(a), run_gpu(b)
    for k in ("choice", "tokens", "accept_len", "margin"):
        np.testing.assert_array_equal(ga[k], gb[k])


@pytest.mark.parametrize("K", [8, 32])
def test_beam_other_candidate_counts(torch_cuda, K):
    prob = Problem(36 + K, N=2, V=20011, d=512, K=K, planted=8, boost=(8.0, 16.0), path_rule=2, beam_width=4,
                   beam_topm=K // 2)
    report(f"beam K={K}", compare_path(prob, run_gpu(prob), prob.oracle()))


def test_beam_cosine_variant(torch_cuda):
    prob = Problem(37, N=3, V=20011, d=512, variant=1, path_rule=2, beam_width=3)
    report("beam cosine", compare_path(prob, run_gpu(prob), prob.oracle()))


# ------------------------------------------------------------------ stochastic verification
def _stochastic_problem(seed, N, V, B=15, stride=None, u_scale=1.0):
    """Target logits [N, B+1, stride] bf16 with a peaked target; the proposal
    takes each slot's target argmax with probability 0.7, else a random token."""
    rng = np.random.default_rng(seed)
    stride = stride or ((V + 7) // 8) * 8
    tl = synth.make_logits(rng, N, B + 1, V, 2, (14.0, 18.0), stride=stride)  # q(top) ~ 0.3-0.9
    f = synth.bf16_to_f32(tl[:, :, :V])
    top = f.argmax(axis=2)[:, :B]
    toks = np.where(rng.random((N, B)) < 0.7, top, rng.integers(0, V, (N, B))).astype(np.int32)
    u_acc = (rng.random((N, B)) * u_scale).astype(np.float32)
    u_draw = rng.random(N).astype(np.float32)
    return tl, toks, u_acc, u_draw, V


def _check_stochastic(tl, toks, u_acc, u_draw, V, g, tol=1e-5):
    N, B = toks.shape
    near = 0
    for n in range(N):
        al, nt, q = oracle.verify_stochastic(tl[n], toks[n], u_acc[n], float(u_draw[n]), V=V)
        np.testing.assert_allclose(g["q_accept"][n], q, rtol=2e-5, atol=1e-7, err_msg=f"request {n} q")
        ga, gt = int(g["accept_len"][n]), int(g["next_token"][n])
        if ga != al:
            j = min(ga, al)  # the slot where the decisions split must be a near tie
            assert abs(float(u_acc[n, j]) - q[j]) < tol, f"request {n}: accept_len {ga} vs {al}"
            near += 1
            continue
        if gt != nt:
            # the draw split at a near tie: the two tokens are neighbours in the
            # cumulative weight and the threshold sits within tol of their boundary
            row = synth.bf16_to_f32(tl[n, ga if ga < B else B, :V]).astype(np.float64)
            w = np.exp(row - row.max())
            if ga < B:
                w[toks[n, ga]] = 0.0
            c = np.cumsum(w) / w.sum()
            lo, hi = min(gt, nt), max(gt, nt)
            assert np.all(w[lo + 1:hi] == 0.0), f"request {n}: draws {gt} vs {nt} not adjacent"
            assert abs(c[lo] - float(u_draw[n])) < tol, f"request {n}: draw {gt} vs {nt}"
            near += 1
    return near


def _gpu_stochastic(tl, toks, u_acc, u_draw, V, B=15):
    import torch
    import draft_correction_slot_gb300 as dc
    w = synth.make_weights(np.random.default_rng(1), 64)
    corr = dc.Corrector({k: torch.from_numpy(v) for k, v in w.items()}, V, 64, B + 1, 16, max_batch=tl.shape[0])
    try:
        g = corr.verify_stochastic(bf16_tensor(tl), torch.from_numpy(toks).cuda(), torch.from_numpy(u_acc).cuda(),
                                   torch.from_numpy(u_draw).cuda(), target_stride=tl.shape[-1])
        torch.cuda.synchronize()
        assert corr.status() == dc.DCOCO_OK
        return {k: v.cpu().numpy() for k, v in g.items()}
    finally:
        corr.close()


def test_stochastic_verify_qwen_shapes(torch_cuda):
    """DCOCO Core method / Faster Decoding: point-mass proposal, temperature 1."""
    tl, toks, ua, ud, V = _stochastic_problem(70, N=8, V=V_QWEN)
    g = _gpu_stochastic(tl, toks, ua, ud, V)
    print(f"[parity] stochastic verify: accept_len {g['accept_len'].tolist()} near ties "
          f"{_check_stochastic(tl, toks, ua, ud, V, g)}")


def test_stochastic_verify_ragged_and_forced(torch_cuda):
    # ragged vocabulary with a padded stride
    tl, toks, ua, ud, V = _stochastic_problem(71, N=6, V=4099, stride=4112)
    _check_stochastic(tl, toks, ua, ud, V, _gpu_stochastic(tl, toks, ua, ud, V))
    # u_accept = 0: every proposal with target mass is accepted -> bonus draws
    tl, toks, ua, ud, V = _stochastic_problem(72, N=3, V=4099, u_scale=0.0)
    f = synth.bf16_to_f32(tl[:, :, :V])
    toks = f.argmax(axis=2)[:, :15].astype(np.int32)
    g = _gpu_stochastic(tl, toks, ua, ud, V)
    np.testing.assert_array_equal(g["accept_len"], 15)
    _check_stochastic(tl, toks, ua, ud, V, g)
    # u_accept -> 1 with proposals of tiny mass: rejected at slot 1 and redrawn
    tl, toks, ua, ud, V = _stochastic_problem(73, N=3, V=4099)
    f = synth.bf16_to_f32(tl[:, :, :V])
    toks = f.argmin(axis=2)[:, :15].astype(np.int32)
    ua = np.full_like(ua, 0.999999)
    g = _gpu_stochastic(tl, toks, ua, ud, V)
    np.testing.assert_array_equal(g["accept_len"], 0)
    assert np.all(g["next_token"] != toks[:, 0])
    _check_stochastic(tl, toks, ua, ud, V, g)


def test_stochastic_verify_deterministic(torch_cuda):
    tl, toks, ua, ud, V = _stochastic_problem(74, N=5, V=20011)
    a = _gpu_stochastic(tl, toks, ua, ud, V)
    b = _gpu_stochastic(tl, toks, ua, ud, V)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


# ------------------------------------------------------------------ candidate features
def _run_features(prob: Problem):
    import torch
    import draft_correction_slot_gb300 as dc
    corr = dc.Corrector({k: torch.from_numpy(v) for k, v in prob.w.items()}, prob.V, prob.d, prob.slots, prob.K,
                        max_batch=prob.N)
    try:
        E = bf16_tensor(prob.E)
        lg, hd = bf16_tensor(prob.logits), bf16_tensor(prob.hidden)
        tg = torch.from_numpy(prob.targets).cuda()
        with_f = corr.correct(lg, hd, E, tg, out=corr.alloc_outputs(prob.N, lg.device, True, features=True),
                              logits_slot_stride=prob.stride)
        without = corr.correct(lg, hd, E, tg, logits_slot_stride=prob.stride)
        torch.cuda.synchronize()
        assert corr.status() == dc.DCOCO_OK
        return ({k: v.cpu().numpy() for k, v in with_f.items()}, {k: v.cpu().numpy() for k, v in without.items()})
    finally:
        corr.close()


@pytest.mark.parametrize("N,K,V", [(2, 16, V_QWEN), (1, 16, V_QWEN), (3, 8, 4099), (2, 32, 20011), (11, 16, V_QWEN)])
def test_candidate_features(torch_cuda, N, K, V):
    """LiLiCorr App. A: the top-K pass also yields the candidates' log-softmax
    features (one pass; at N = 1 the rows are split into segments whose
    partial sums the last block combines).  Features match the oracle's fp64
    log-sum-exp within fp32 accuracy; the rest of the path is bit-identical
    with and without them."""
    prob = Problem(90 + N + K, N=N, V=V, d=512, K=K, planted=8, boost=(4.0, 12.0),
                   stride=((V + 7) // 8) * 8 + (8 if V % 8 else 0))
    g, plain = _run_features(prob)
    for k in plain:
        np.testing.assert_array_equal(g[k], plain[k], err_msg=k)
    worst = 0.0
    for n in range(N):
        for i in range(prob.B):
            ref = oracle.topk_features(prob.logits[n, i + 1], K, V=V)
            f = g["cand_feat"][n, i]
            worst = max(worst, float(np.abs(f[:, 0] - ref[:, 0]).max()))
            np.testing.assert_allclose(f[:, 0], ref[:, 0], rtol=0, atol=2e-5)
            np.testing.assert_allclose(f[:, 1], ref[:, 1], rtol=5e-5, atol=1e-12)
            np.testing.assert_array_equal(f[:, 2], ref[:, 2].astype(np.float32))
            np.testing.assert_array_equal(f[:, 3], ref[:, 3].astype(np.float32))
            np.testing.assert_array_equal(f[:, 4], ref[:, 4].astype(np.float32))
    print(f"[parity] candidate features N={N} K={K} V={V}: max |log p error| {worst:.2e}")
