"""bench.py's JSONL provenance records (CPU): one row per measured operation,
each tied to the code (a hash of the CUDA sources and headers), the
workload's shapes and seeds, and the environment."""
import json

import bench
import workloads


def _line():
    c = workloads.case("mxfp8_8192")
    return {
        "ms_per_step": 0.46, "value": 2400.0,
        "config": {"workload": c.name},
        "roofline": {"frac": 0.85},
        "breakdown": {"gemm_ms": 0.34},
        "gemm_only_other_workloads": {
            "mxfp4_8192": {"gemm_ms": 0.17, "tflops": 6500.0,
                           "frac_of_peak": 0.56,
                           "frac_of_instruction_rate": 0.84},
            "w4a16_8192": {"gemm_ms": 0.68, "tflops": 1620.0,
                           "frac_of_peak": 0.84, "gbs": 448.0},
            "proj_layer_aggregate": {"gemms": ["proj_qkv", "proj_out", "proj_up",
                                               "proj_down"],
                                     "gemm_ms": 0.51, "tflops": 3240.0,
                                     "frac_of_peak": 0.84}},
        "fused_epilogue": {"proj_up": {"fused_ms": 0.35, "gemm_ms": 0.19,
                                       "decomposed_ms": 0.91,
                                       "fused_quantize_ms": 0.33,
                                       "fused_tflops": 1570.0}},
        "attention": {"attn_sam_d128": {"ms": 0.2, "tflops": 1365.0,
                                        "frac_of_peak": 0.71,
                                        "unsplit_ms": 0.21}},
        "e2e": {"ms_per_step": 2.7, "value": 400.0},
        "clocks": {"sm_mhz": 2070.0, "reasons": []},
    }


def test_one_row_per_operation_with_shapes_and_seeds():
    rows = bench.provenance_rows(_line())
    ops = [(r["op"], r["workload"]) for r in rows]
    assert ops == [("step", "mxfp8_8192"), ("gemm", "mxfp4_8192"),
                   ("gemm", "w4a16_8192"), ("gemm_aggregate", "proj_layer_aggregate"),
                   ("fused_epilogue", "proj_up"), ("attention", "attn_sam_d128"),
                   ("e2e", "mxfp8_8192")]
    step = rows[0]
    c = workloads.case("mxfp8_8192")
    assert (step["M"], step["N"], step["K"]) == (c.M, c.N, c.K)
    assert (step["seed_a"], step["seed_b"]) == (c.seed_a, c.seed_b)
    a = workloads.attn_case("attn_sam_d128")
    assert (rows[5]["BH"], rows[5]["Lq"], rows[5]["seed"]) == (a.BH, a.Lq, a.seed)
    assert rows[3]["gemms"][0] == "proj_qkv" and rows[3]["tflops"] == 3240.0
    assert rows[1]["frac_of_instruction_rate"] == 0.84
    for r in rows:
        assert len(r["sources"]) == 16 and r["sm_mhz"] == 2070.0
        json.dumps(r)                                  # serialisable


def test_source_hash_tracks_the_sources(tmp_path, monkeypatch):
    h = bench.source_hash()
    assert h == bench.source_hash()                    # deterministic
    # a different tree hashes differently
    (tmp_path / "block_scaled_quantized_mx_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (tmp_path / "block_scaled_quantized_mx_gb300" / "csrc" / "k.cu").write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_hash() != h
