"""The allocation-free top-K entry point, dcoco_topk_noalloc.

It exists for callers that cannot allocate device memory (a plugin inside an
engine that owns all device memory, or a latency-critical path where
cudaMalloc is not acceptable).  Its scratch is one fixed array per GPU that
every call reuses, so the tests check it against the oracle call after call,
across shape changes, and on a shape whose segment lists only fit the fixed
array with fewer segments than the handle-based plan would use.  Collected
last, so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import draft_correction_slot_gb300 as dc
    return torch, dc


def _host_logits(seed, N, slots, V, stride):
    rng = np.random.default_rng(seed)
    return synth.make_logits(rng, N, slots, V, 32, (4.0, 12.0), stride=stride)


def _oracle_rows(logits_bits, V, K):
    N, S = logits_bits.shape[:2]
    ids = np.empty((N, S - 1, K), np.int32)
    vals = np.empty((N, S - 1, K), np.float32)
    for n in range(N):
        for i in range(S - 1):
            ids[n, i], vals[n, i] = oracle.topk_row(np.ascontiguousarray(logits_bits[n, i + 1, :V]), K)
    return ids, vals


def _noalloc(torch, dc, logits, N, slots, V, K, stride):
    ids = torch.full((N, slots - 1, K), -1, dtype=torch.int32, device="cuda")
    vals = torch.full((N, slots - 1, K), np.nan, dtype=torch.float32, device="cuda")
    dc.dcoco_topk_noalloc(N, slots, V, K, logits, ids, vals, logits_slot_stride=stride)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), vals.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_topk_matches_oracle_call_after_call(env):
    torch, dc = env
    cases = [(8, 16, 151936, 16, 151936), (3, 9, 4099, 32, 4104)]
    host = {c: _host_logits(100 + i, c[0], c[1], c[2], c[4]) for i, c in enumerate(cases)}
    dev = {c: torch.from_numpy(host[c].view(np.int16)).view(torch.bfloat16).cuda() for c in cases}
    refs = {c: _oracle_rows(host[c], c[2], c[3]) for c in cases}
    # two calls in a row on one shape, another shape, then the first again:
    # the shared scratch keeps each call's leftovers and must not leak them
    for c in (cases[0], cases[0], cases[1], cases[0]):
        ids, vals = _noalloc(torch, dc, dev[c], *c)
        np.testing.assert_array_equal(ids, refs[c][0])
        np.testing.assert_array_equal(vals.view(np.uint32), refs[c][1].view(np.uint32))


def _keys(torch, rows_bf16):
    """(value desc, id asc) as one int64 per element: order16(value) << 32 | (2^32 - 1 - id)."""
    b = rows_bf16.view(torch.int16).to(torch.int64) & 0xFFFF
    b = torch.where(b == 0x8000, torch.zeros_like(b), b)  # -0 == +0
    k16 = torch.where(b >= 0x8000, (~b) & 0xFFFF, b | 0x8000)
    ids = torch.arange(rows_bf16.shape[-1], device=rows_bf16.device, dtype=torch.int64)
    return (k16 << 32) | (0xFFFFFFFF - ids)


@pytest.mark.gpu
def test_noalloc_clamped_segments(env):
    """A call whose plan wants more segments than the fixed list area holds
    runs with fewer: the results must not change.  Every row is checked
    against a full sort of (value, id) keys; sampled rows against the oracle."""
    torch, dc = env
    V, K, slots = 1 << 20, 32, 16
    batch = None
    for b in range(130, 156):
        seg, planned = dc.dcoco_topk_noalloc_plan(b, slots, V, K)
        if seg < planned:
            batch = b
            break
    if batch is None:
        pytest.skip("no batch in range makes this device's plan exceed the list area")
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    x = torch.randn(batch * slots, V, generator=g, device="cuda") * 2.0
    planted = torch.randint(0, V, (batch * slots, 8), generator=g, device="cuda")
    x.scatter_add_(1, planted, torch.rand(batch * slots, 8, generator=g, device="cuda") * 8.0 + 4.0)
    logits = x.to(torch.bfloat16).view(batch, slots, V)
    del x
    ids, vals = _noalloc(torch, dc, logits, batch, slots, V, K, V)
    rows = logits[:, 1:].reshape(-1, V)
    for r0 in range(0, rows.shape[0], 64):
        key = _keys(torch, rows[r0:r0 + 64])
        top = torch.topk(key, K, dim=1, sorted=True).values
        want_ids = (0xFFFFFFFF - (top & 0xFFFFFFFF)).to(torch.int32).cpu().numpy()
        np.testing.assert_array_equal(ids.reshape(-1, K)[r0:r0 + 64], want_ids)
    sample = [(0, 0), (batch // 2, 7), (batch - 1, slots - 2)]
    for n, i in sample:
        row = logits[n, i + 1].view(torch.int16).cpu().numpy().view(np.uint16)
        ri, rv = oracle.topk_row(np.ascontiguousarray(row), K)
        np.testing.assert_array_equal(ids[n, i], ri)
        np.testing.assert_array_equal(vals[n, i].view(np.uint32), rv.view(np.uint32))


def test_noalloc_rejects_oversized_batch_before_cuda():
    """Both size limits answer DCOCO_EBATCH before any CUDA call (runs without a GPU)."""
    import __graft_entry__
    __graft_entry__.build()
    import draft_correction_slot_gb300 as dc
    with pytest.raises(dc.DcocoError) as e:
        dc.dcoco_topk_noalloc_plan(4096 // 15 + 1, 16, 151936, 16)
    assert e.value.status == dc.DCOCO_EBATCH
    # 2400 rows of K = 32 at V = 2^20 need 2400 * 32 * 7 > 522,240 list entries
    with pytest.raises(dc.DcocoError) as e:
        dc.dcoco_topk_noalloc_plan(160, 16, 1 << 20, 32)
    assert e.value.status == dc.DCOCO_EBATCH
    with pytest.raises(dc.DcocoError) as e:
        dc.dcoco_topk_noalloc(160, 16, 1 << 20, 32, 16, 16, 16, logits_slot_stride=1 << 20, stream=0)
    assert e.value.status == dc.DCOCO_EBATCH
