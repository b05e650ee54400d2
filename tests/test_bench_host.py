"""Host-side logic of bench.py (no GPU): the algorithmic byte and FLOP counts the roofline
divides by, the staleness rule of the recorded ncu traffic, the peak fallback and the
clock-record parsing that decides whether a run is kept.

The expected counts are worked out by hand from the layer's definition (FP8 E4M3 weights,
one FP32 scale per 128x128 block; gate/up = 2I rows of H, down = H rows of I).
"""
import json
import os

import bench


def test_per_expert_bytes_h2048_i768():
    # w13: 2*768*2048 codes + (1536/128)*(2048/128) scales * 4 B
    # w2 : 2048*768 codes + (2048/128)*(768/128) scales * 4 B
    assert bench.per_expert_bytes(2048, 768) == (3_145_728 + 768, 1_572_864 + 384)


def test_algorithmic_decode_step():
    byts, flops, gu_bytes, gu_flops = bench.algorithmic(2048, 768, 128, 8, 1, 8)
    # 8 experts' w13 + the token's codes (2048) + its 16 scales + 8 act rows (768 codes,
    # 6 scales each)
    assert gu_bytes == 8 * 3_146_496 + 2048 + 16 * 4 + 8 * 768 + 8 * 6 * 4 == 25_180_416
    assert gu_flops == 4 * 2048 * 768 * 8
    # whole step: 8 experts' w13 + w2, the BF16 router, hidden in and out, ids + weights
    assert byts == 8 * (3_146_496 + 1_573_248) + 2048 * 128 * 2 + 2048 * 2 * 2 + 8 * 8 == 38_290_496
    # router 2*H*E + gate/up 4*H*I + down 2*H*I per routed row
    assert flops == 2 * 2048 * 128 + 6 * 2048 * 768 * 8 == 76_021_760


def test_launch_count_follows_the_library_modes():
    """The kernels the bench claims per step switch where the library switches modes: the
    pair kernels up to kPairPreferRows routed rows, the one-launch sort up to one sort block
    (kSortBlock pairs), the two-launch sort and the gather above."""
    import re
    src = open(os.path.join(bench.ROOT, "fp8_block_scaled_router_gb300", "csrc", "common.cuh")).read()
    pair = int(re.search(r"constexpr int kPairPreferRows = (\d+);", src).group(1))
    block = int(re.search(r"constexpr int kSortBlock = (\d+);", src).group(1))
    assert (bench.PAIR_ROWS, bench.SORT_BLOCK) == (pair, block)
    assert [bench.launches_per_step(m, 8, 2048, 128) for m in (1, 8, 9, 12, 32, 33, 4096)] == [3, 3, 5, 5, 5, 7, 7]
    assert [bench.launches_per_step(m, 1, 2048, 16) for m in (64, 65, 256, 257)] == [3, 5, 5, 7]


def test_algorithmic_prefill_gate_up_flops():
    _, _, _, gu_flops = bench.algorithmic(2048, 768, 128, 8, 4096, 128)
    assert gu_flops == 206_158_430_208  # 4 * 2048 * 768 * 32768 routed rows


def _fake_root(tmp_path):
    csrc = tmp_path / "fp8_block_scaled_router_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for n, text in (("a.cu", "kernel a"), ("b.cuh", "header b"), ("c.cu", "kernel c")):
        (csrc / n).write_text(text)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_source_hash_is_order_free_and_content_bound(tmp_path, monkeypatch):
    csrc = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h_ab = bench.kernel_source_hash(["a.cu", "b.cuh"])
    assert h_ab == bench.kernel_source_hash(["b.cuh", "a.cu"])
    assert h_ab != bench.kernel_source_hash(["a.cu", "c.cu"])
    (csrc / "a.cu").write_text("kernel a, changed")
    assert h_ab != bench.kernel_source_hash(["a.cu", "b.cuh"])


def test_recorded_traffic_goes_stale_with_its_own_sources_only(tmp_path, monkeypatch):
    csrc = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"prefill": {"gate_up": {"dram_bytes_per_launch": 123, "source_files": ["a.cu", "b.cuh"],
                                   "source_hash": bench.kernel_source_hash(["a.cu", "b.cuh"])}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("gate_up", "prefill") == 123
    assert bench.recorded_traffic("gate_up", "decode") is None
    (csrc / "c.cu").write_text("another kernel changed")  # not a source of this record
    assert bench.recorded_traffic("gate_up", "prefill") == 123
    (csrc / "b.cuh").write_text("header b, changed")
    assert bench.recorded_traffic("gate_up", "prefill") is None


def test_committed_traffic_records_are_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    csrc = os.path.join(bench.ROOT, "fp8_block_scaled_router_gb300", "csrc")
    for wl, kernels in d.items():
        assert wl in bench.WORKLOADS
        for rec in kernels.values():
            assert rec["dram_bytes_per_launch"] > 0
            assert rec["source_files"] and all(os.path.exists(os.path.join(csrc, n)) for n in rec["source_files"])
            assert os.path.exists(os.path.join(bench.ROOT, rec["profile"]))


def test_peaks_fallback_and_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6676.8, "bf16_tflops": 1920.6, "bf16_tflops_sustained": 1700.0}))
    assert bench.load_peaks() == (6676.8, 1920.6, 1700.0, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.load_peaks()[3] == "fallback"


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_parsing():
    s = bench.ClockSampler("0")
    s.proc = _DoneProc()
    s.rows = [["2070", "2070", "900.1", "Not Active", "Not Active", "Not Active", "Active"],
              ["2055", "2070", "950.3", "Not Active", "Not Active", "Not Active", "Not Active"],
              ["2070", "2070", "955.0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    r = s.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]  # kept and noted; no slowdown reason


def test_clock_record_reports_thermal_slowdown():
    s = bench.ClockSampler("0")
    s.proc = _DoneProc()
    s.rows = [["1500", "2070", "1300", "Not Active", "Active", "Not Active", "Not Active"]]
    assert s.stop()["reasons"] == ["hw_thermal_slowdown"]


def test_clock_record_without_nvidia_smi():
    s = bench.ClockSampler("0")
    s.err = "no nvidia-smi"
    r = s.stop()
    assert r["sm_mhz"] is None and r["reasons"] == [] and r["error"] == "no nvidia-smi"
