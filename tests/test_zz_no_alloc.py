"""The allocation-free top-K entry point (for callers that cannot allocate
device memory, e.g. inside an engine that owns all device memory) must give
exactly the results of the handle-based dcoco_topk, call after call, even
though every call reuses the same fixed scratch array.  Collected last."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import draft_correction_slot_gb300 as dc
    return torch, dc


def _logits(torch, seed, N, slots, V, stride):
    rng = np.random.default_rng(seed)
    a = synth.make_logits(rng, N, slots, V, 32, (4.0, 12.0), stride=stride)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def _reference(torch, dc, logits, N, slots, V, K, stride):
    h = dc.dcoco_create(V, 64, slots, K, max_batch=N)
    try:
        ids = torch.empty(N, slots - 1, K, dtype=torch.int32, device="cuda")
        vals = torch.empty(N, slots - 1, K, dtype=torch.float32, device="cuda")
        dc.dcoco_topk(h, N, logits, ids, vals, logits_slot_stride=stride)
        torch.cuda.synchronize()
    finally:
        dc.dcoco_destroy(h)
    return ids.cpu().numpy(), vals.cpu().numpy()


def _noalloc(torch, dc, logits, N, slots, V, K, stride):
    ids = torch.full((N, slots - 1, K), -1, dtype=torch.int32, device="cuda")
    vals = torch.full((N, slots - 1, K), np.nan, dtype=torch.float32, device="cuda")
    dc.dcoco_topk_noalloc(N, slots, V, K, logits, ids, vals, logits_slot_stride=stride)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), vals.cpu().numpy()


def test_noalloc_topk_matches_handle_topk(env):
    torch, dc = env
    cases = [(8, 16, 151936, 16, 151936), (3, 9, 4099, 32, 4104)]
    data = {c: _logits(torch, 100 + i, c[0], c[1], c[2], c[4]) for i, c in enumerate(cases)}
    refs = {c: _reference(torch, dc, data[c], *c) for c in cases}
    # two calls in a row on one shape, another shape, then the first again:
    # the shared scratch keeps each call's leftovers and must not leak them
    for c in (cases[0], cases[0], cases[1], cases[0]):
        ids, vals = _noalloc(torch, dc, data[c], *c)
        np.testing.assert_array_equal(ids, refs[c][0])
        np.testing.assert_array_equal(vals.view(np.uint32), refs[c][1].view(np.uint32))


def test_noalloc_rejects_oversized_batch(env):
    torch, dc = env
    limit = 4096 // 15
    x = torch.zeros(1, 16, 64, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(dc.DcocoError) as e:
        dc.dcoco_topk_noalloc(limit + 1, 16, 64, 16, x, ids, ids)
    assert e.value.status == dc.DCOCO_EBATCH
