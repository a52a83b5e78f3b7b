"""The benchmark's byte and work accounting, pinned to the per-unit figures of
the measurement plan: 6,524,160 bytes per corrected block at K = 16, d = 4096
(15 V bf16 logits + 15 K d bf16 gathered embedding rows), 9,473,280 at K = 32,
d = 5120, and 3584 x 256 GELU elements per block at K = 16; the maps
kernel's flops are the method's own (1.303 GFLOP at batch 32), not the
three bf16 passes the kernel issues."""
import bench


def test_algorithmic_bytes_per_block_and_per_call():
    w = dict(bench.WORKLOADS["c32"])
    assert bench.algorithmic_bytes(dict(w, N=1)) == 15 * 151_936 * 2 + 15 * 16 * 4096 * 2 == 6_524_160
    assert bench.algorithmic_bytes(w) == 32 * 6_524_160 == 208_773_120
    assert bench.algorithmic_bytes(dict(w, N=1, K=32, d=5120)) == 9_473_280


def test_stage_model_amounts_and_bounds():
    w = dict(bench.WORKLOADS["c32"])
    m = bench.stage_model(w, bench.peaks())
    assert m["topk"][:3] == ("hbm", "GB/s", 32 * 15 * 151_936 * 2)
    assert m["proj"][:3] == ("hbm", "GB/s", 32 * 15 * 16 * 4096 * 2 + 32 * 15 * 4096 * 2)
    assert m["pair_walk"][:3] == ("alu", "Gelem/s", 32 * 3584 * 256)
    assert m["maps"][0] == "tensor"
    # topk + gathered rows: the stage amounts add up to the path's byte floor
    assert m["topk"][2] + m["proj"][2] - 32 * 15 * 4096 * 2 == bench.algorithmic_bytes(w)


def test_maps_flops_are_the_methods_own():
    w = dict(bench.WORKLOADS["c32"])
    N, B, K, r, H = 32, 15, 16, 128, 256
    per_slot = B * r * r + (B - 1) * r * H          # W_fuse[:, r:] g and W1_s s
    per_cand = B * K * (r * r + 2 * r * H)          # W_fuse[:, :r] b, W1_a z, W1_b z
    assert bench.maps_method_flops(w) == 2 * N * (per_slot + per_cand) == 1_303_379_968
    assert bench.stage_model(w, bench.peaks())["maps"][2] == 1_303_379_968


def test_every_workload_has_its_config_shapes():
    W = bench.WORKLOADS
    assert (W["c32"]["N"], W["tiny"]["N"], W["cosine16"]["N"], W["wide32"]["N"]) == (32, 1, 16, 32)
    assert W["cosine16"]["variant"] == 1
    assert (W["wide32"]["d"], W["wide32"]["K"], W["wide32"]["planted"], W["wide32"]["boost"]) == (5120, 32, 8, (8.0, 16.0))
    # every workload's rotating sets exceed the 129 MB L2
    for w in W.values():
        assert w["sets"] * w["N"] * w["slots"] * w["V"] * 2 > 129e6
    assert bench.SWEEP_NS == (1, 2, 4, 8, 16, 32)
    assert [b for _, b in bench.SWEEP_TIERS] == [(2.0, 6.0), (4.0, 12.0), (8.0, 16.0)]
