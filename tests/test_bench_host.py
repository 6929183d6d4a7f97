"""Host logic of bench.py that decides what a bench line claims: which roofline a layer is held to, the
algorithmic bytes and FLOPs behind `achieved`, and when a recorded ncu traffic figure still belongs to the
kernel being measured.  No GPU is involved."""
import json

import numpy as np

import bench


def test_code_only_strips_comments_and_layout_but_keeps_strings():
    src = 'int a;  // gone "x"\n/* block\n comment */ const char* s = "// kept /* too */";\nchar q = \'\\\'\';'
    assert bench._code_only(src) == 'int a; const char* s = "// kept /* too */"; char q = \'\\\'\';'
    # a comment-only edit leaves the code unchanged, a code edit does not
    assert bench._code_only("x = 1; // one") == bench._code_only("x = 1;   // uno\n")
    assert bench._code_only("x = 1;") != bench._code_only("x = 2;")


def test_recorded_traffic_is_tied_to_workload_and_kernel_code(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    digest = bench.kernel_source_digest()
    recs = {"records": [
        {"workload": "wl_a", "kernel_sha256": digest, "dram_bytes_per_launch": 123},
        {"workload": "wl_b", "kernel_sha256": "0" * 64, "dram_bytes_per_launch": 456},
    ]}
    (tmp_path / "profiles" / "gate_up_dram_traffic.json").write_text(json.dumps(recs))
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the digest is read from the real sources; only the records file moves
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: digest)
    assert bench.recorded_traffic("wl_a") == 123
    assert bench.recorded_traffic("wl_b") is None       # taken on other kernel code: stale
    assert bench.recorded_traffic("wl_c") is None       # no record for this workload
    monkeypatch.setattr(bench, "ROOT", real_root)


def test_committed_traffic_records_are_well_formed():
    """Every committed DRAM record names a workload, the kernel code it was taken on and the command that took
    it; its per-launch figure is read + write.  (A record whose hash no longer matches the tree is reported as
    null by the bench, not as a claim.)"""
    with open(f"{bench.ROOT}/profiles/gate_up_dram_traffic.json") as f:
        doc = json.load(f)
    assert doc["records"]
    for rec in doc["records"]:
        assert rec["workload"].startswith("moe_layer_T")
        assert len(rec["kernel_sha256"]) == 64
        assert "ncu" in rec["command"] and "--clock-control none" in rec["command"]
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]


def test_algorithmic_bytes_of_the_decode_layer():
    T, E, k, H, I = 1024, 256, 8, 6144, 2048
    counts = np.full(E, T * k // E)
    ab = bench.algorithmic_bytes(counts, T, E, k, H, I)
    w13 = 2 * I * H // 2 + 2 * I * H // 16          # 14,155,776 B per expert
    assert w13 == 14_155_776
    assert ab["gate_up"] == E * w13 + T * k * (3072 + 384) + T * k * (1024 + 128)
    assert ab["gate_up"] == 3_661_627_392
    assert ab["active_experts"] == E
    # an idle expert's weights are not counted
    counts[0] = 0
    assert bench.algorithmic_bytes(counts, T, E, k, H, I)["gate_up"] < ab["gate_up"] - w13 + 1


def _fake_result(T, k, E, H, I, ms):
    counts = np.full(E, T * k // E)
    return {"T": T, "ab": bench.algorithmic_bytes(counts, T, E, k, H, I), "stage_ms": [0.0, 0.0, ms, 0.0]}


def test_layer_roofline_picks_the_bound_by_rows_per_expert():
    E, k, H, I = 256, 8, 6144, 2048
    fp4 = {"peak_tflops": 10_000.0}
    pre = bench.layer_roofline(_fake_result(16384, k, E, H, I, 1.0), k, H, I, fp4, 6790.7, "measured", "wl")
    assert pre["bound"] == "tensor" and pre["unit"] == "TFLOP/s"
    flops = 2.0 * 16384 * k * 2 * I * H
    assert pre["algorithmic_flops_per_launch"] == flops == 6_597_069_766_656
    assert abs(pre["achieved"] - flops / 1e-3 / 1e12) < 1e-6
    assert abs(pre["frac"] - pre["achieved"] / 10_000.0) < 1e-12
    dec = bench.layer_roofline(_fake_result(1024, k, E, H, I, 0.5), k, H, I, fp4, 6790.7, "measured", "wl")
    assert dec["bound"] == "hbm" and dec["unit"] == "GB/s"
    assert abs(dec["achieved"] - 3_661_627_392 / 0.5e-3 / 1e9) < 1e-6
    assert abs(dec["frac"] - dec["achieved"] / 6790.7) < 1e-12


def test_layer_workload_names():
    assert bench.layer_workload_name(16384, 256, 8, 6144, 2048, None) == "moe_layer_T16384_E256_k8_H6144_I2048_uniform"
    assert bench.layer_workload_name(1024, 256, 8, 6144, 2048, 1.1) == "moe_layer_T1024_E256_k8_H6144_I2048_zipf1.1"
