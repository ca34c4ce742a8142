"""Host-side pieces of bench.py that need no GPU: the per-chunk oracle baseline of the other
reference workloads (timed units, extrapolated to whole chunks)."""
import bench


def test_oracle_per_chunk_covers_the_reference_workloads():
    out = bench._oracle_per_chunk(1)
    assert set(out) == {"tiny_gqa", "mla_recall", "mha_sliding_window", "gqa_recall_sweep"}
    for name, rec in out.items():
        assert rec["us_per_chunk"] > 0, name
        assert rec["sample"], name
    # extrapolation: a whole MLA chunk (27 layers) costs more than the 2-layer tiny chunk
    assert out["mla_recall"]["us_per_chunk"] > out["tiny_gqa"]["us_per_chunk"]


def test_reorder_accounting_matches_the_byte_counts_of_the_workload():
    # the roofline's numerator: 18 placements x 28 layers x 1024 tokens x (K + V rows of 512)
    # bf16 written; each of the 3 canonicals read once; each chunk's orbit patch (14 layers of
    # U [2][1024][32] and V_m^T [32][512 + 512]) read once
    import workloads as wl
    w = wl.config2(device="cpu")
    acc = bench.accounting(w)
    assert acc["written"] == 18 * 28 * 1024 * 1024 * 2 == 1_056_964_608
    assert acc["written"] // 18 == 58_720_256
    assert acc["canon_distinct"] == 3 * 28 * 1024 * 1024 * 2 == 176_160_768
    assert acc["patch"] == 3 * 14 * (2 * 1024 * 32 + 32 * 1024) * 2 == 8_257_536
    assert acc["per_kernel"]["reuse_copy_kernel"] + acc["per_kernel"]["reuse_tile_kernel"] == \
        acc["algorithmic"] + acc["meta"]


def test_spread_gives_the_median_and_nearest_rank_percentiles():
    s = bench.spread([float(x) for x in range(20, 0, -1)])  # 20 runs, 1..20 ms in any order
    assert s["median_ms"] == 10.5 and s["p10_ms"] == 2.0 and s["p90_ms"] == 18.0
    assert s["mean_ms"] == 10.5 and s["runs"] == 20
    one = bench.spread([3.0])
    assert one["median_ms"] == one["p10_ms"] == one["p90_ms"] == 3.0


class _Ev:
    """A recorded event's time in ms; elapsed_time as torch.cuda.Event gives it."""

    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_split_stats_names_the_kernels_of_each_path():
    # two passes of two calls each: (before, between, after planning, after) per call
    passes = [[[_Ev(0), _Ev(1), _Ev(1.25), _Ev(3)], [_Ev(10), _Ev(12), _Ev(12.5), _Ev(14)]],
              [[_Ev(0), _Ev(2), _Ev(2.25), _Ev(4)], [_Ev(10), _Ev(11), _Ev(11.5), _Ev(13)]]]
    p = bench.split_stats(passes, True)
    assert set(p) == {"reuse_copy_kernel", "reuse_plan_kernel", "reuse_persist_kernel"}
    assert p["reuse_copy_kernel"]["median_ms"] == 3.0  # 1 + 2 and 2 + 1
    assert p["reuse_plan_kernel"]["median_ms"] == 0.75
    assert p["reuse_persist_kernel"]["median_ms"] == 3.25
    g = bench.split_stats(passes, False)
    assert set(g) == {"reuse_copy_kernel", "reuse_tile_kernel"}
    assert g["reuse_tile_kernel"]["median_ms"] == 4.0  # (2 + 2) and (2 + 2)


def test_kernel_fracs_times_the_planning_kernel_without_bytes():
    st = {"median_ms": 0.5, "p10_ms": 0.5, "p90_ms": 0.5, "mean_ms": 0.5, "runs": 1}
    out = bench.kernel_fracs({"reuse_plan_kernel": st, "reuse_persist_kernel": st},
                             {"reuse_persist_kernel": 1e9}, peak=1000.0)
    assert "frac" not in out["reuse_plan_kernel"] and out["reuse_plan_kernel"]["ms"] == 0.5
    assert abs(out["reuse_persist_kernel"]["frac"] - 2.0) < 1e-12  # 1 GB in 0.5 ms = 2000 GB/s


def test_config_names_the_l2_flush_of_the_gpu_arm():
    # the GPU arm flushes L2 before every timed step and says so; the oracle arm does not flush
    gpu = bench.config_desc(flushed=True)["l2"]
    cpu = bench.config_desc()["l2"]
    assert gpu.startswith("flushed: a 512 MB write") and "inputs larger than L2" in gpu
    assert "flush" not in cpu and "inputs larger than L2" in cpu
