"""The benchmark's byte and work accounting, pinned to the per-unit figures of
the measurement plan: 6,524,160 bytes per corrected block at K = 16, d = 4096
(15 V bf16 logits + 15 K d bf16 gathered embedding rows), 9,473,280 at K = 32,
d = 5120, and 3584 x 256 GELU elements per block at K = 16."""
import bench


def test_algorithmic_bytes_per_block_and_per_call():
    w = dict(bench.WORKLOAD)
    assert bench.algorithmic_bytes(dict(w, N=1)) == 15 * 151_936 * 2 + 15 * 16 * 4096 * 2 == 6_524_160
    assert bench.algorithmic_bytes(w) == 32 * 6_524_160 == 208_773_120
    assert bench.algorithmic_bytes(dict(w, N=1, K=32, d=5120)) == 9_473_280


def test_stage_model_amounts_and_bounds():
    w = dict(bench.WORKLOAD)
    m = bench.stage_model(w, bench.peaks())
    assert m["topk"][:3] == ("hbm", "GB/s", 32 * 15 * 151_936 * 2)
    assert m["proj"][:3] == ("hbm", "GB/s", 32 * 15 * 16 * 4096 * 2 + 32 * 15 * 4096 * 2)
    assert m["pair_walk"][:3] == ("alu", "Gelem/s", 32 * 3584 * 256)
    assert m["maps"][0] == "tensor"
    # topk + gathered rows: the stage amounts add up to the path's byte floor
    assert m["topk"][2] + m["proj"][2] - 32 * 15 * 4096 * 2 == bench.algorithmic_bytes(w)
