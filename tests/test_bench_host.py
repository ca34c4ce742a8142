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
