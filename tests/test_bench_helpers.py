"""bench.py's host-side helpers (no GPU): the clock-sample summary and its
throttle reasons, the peaks file and its fallback, the traffic entries that
go null when the kernel source changes, the router's launch count, and
the GPU index mapping under CUDA_VISIBLE_DEVICES."""
import json
import os

import pytest

import bench


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [
        "1400, 2032, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "1350, 2032, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "1500, 2032, 800.0, 0x0, Not Active, Not Active, Not Active, "
        "Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 1400 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    c.lines = ["1000, 2032, 1.0, 0x8, Active, Not Active, Active, "
               "Not Active"]
    assert set(c.summary()["reasons"]) == {"hw_slowdown",
                                           "sw_thermal_slowdown"}
    c.lines = []
    assert c.summary()["sm_mhz"] is None


def test_peaks_measured_then_fallback(tmp_path, monkeypatch):
    d, src = bench.peaks()
    assert src == "measured" and d["hbm_gbs"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d, src = bench.peaks()
    assert src == "fallback" and d == bench.FALLBACK_PEAKS


def test_traffic_entry_goes_null_when_the_source_changes(tmp_path,
                                                        monkeypatch):
    """An entry counts only while the hash of its kernel sources matches:
    a one-byte change to a source makes the bench report traffic null."""
    src_dir = tmp_path / "csrc"
    src_dir.mkdir()
    (tmp_path / "profiles").mkdir()
    (src_dir / "k.cu").write_text("kernel v1\n")
    (src_dir / "common.cuh").write_text("helpers\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    srcs = ["csrc/k.cu", "csrc/common.cuh"]
    entry = {"sources": srcs, "source_hash": bench.source_hash(*srcs),
             "dram_bytes_per_launch": 12345, "how": "test"}
    with open(tmp_path / "profiles" / "ncu_traffic.json", "w") as f:
        json.dump({"k@w": entry}, f)
    assert bench.ncu_traffic("k", "w") == 12345.0
    assert bench.ncu_traffic("k", "other") is None
    (src_dir / "k.cu").write_text("kernel v2\n")
    assert bench.ncu_traffic("k", "w") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    assert {"gemm_up_swiglu@prefill_v3", "gemm_down@prefill_v3",
            "ffn_fp8@decode_v3_fp8"} <= set(d)
    for e in d.values():
        for s in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, s)), s
        assert e["dram_bytes_per_launch"] > 0


@pytest.mark.parametrize("T,extra", [(4096, 2), (16384, 1), (128, 2),
                                     (512, 2), (32768, 1)])
def test_router_extra_launches(T, extra):
    """The weight split always; the split-K sum only when the router's
    tiles (256 experts wide from 1024 tokens, else 64) would fill fewer than
    half of the 148 SMs -- the same decision as the library's, which
    reserves the partial sums in the router workspace exactly then."""
    assert bench.router_extra_launches(T, 7168, 256) == extra
    assert bench.router_extra_launches(T, 7168, 256, presplit=True) == \
        extra - 1
    from deepseekmoe_routing_expert_moe_b300 import ops
    d = ops.dims(T, 7168, 256, 8, 4, 8, 2048, 2048, 0.001)
    ws = ops.workspace_bytes(d, ops.MOE_WS_ROUTER_LOGITS)
    split_parts = 256 + 3 * 256 * 7168 * 2   # status word + the bf16 parts
    assert (ws > split_parts + 4096) == (extra == 2)


@pytest.mark.parametrize("T", [1, 64, 128, 147, 148, 1984, 1985, 4096, 9473,
                               16384])
def test_route_blocks_match_the_library(T):
    """bench.py counts the routing histogram rows in the routing call's
    algorithmic bytes: its block count must be the library's, whose routing
    workspace holds two [blocks, E] int32 tables (histogram, prefixes)."""
    from deepseekmoe_routing_expert_moe_b300 import ops
    E = 256

    def ws(t):
        return ops.workspace_bytes(ops.dims(t, 7168, E, 8, 4, 8, 2048, 2048,
                                            0.001), ops.MOE_WS_ROUTE)

    def up(b):
        return -(-b // 256) * 256
    nb = bench.route_blocks(T)
    assert ws(T) - ws(1) == 2 * (up(nb * E * 4) - up(1 * E * 4))
    assert nb * 64 >= T and (nb < 32 or nb % 148 == 0)


def test_gpu_index_for_smi(monkeypatch):
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.gpu_index_for_smi(3) == 3
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5,2")
    assert bench.gpu_index_for_smi(1) == 2
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-abc")
    assert bench.gpu_index_for_smi(0) == 0
