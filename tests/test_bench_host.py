"""Host-side pieces of bench.py that need no GPU: the DRAM-traffic record built
from an ncu launch list, and the lookup that feeds roofline.traffic."""
import csv
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

_HEADER = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
           "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name",
           "Metric Unit", "Metric Value"]
_KERNELS = {
    "quant": "void unnamed>::inv_rope_fp8_quant_kernel<4>(const unsigned short *)",
    "wo_a": "void unnamed>::block_scaled_gemm_kernel<256, 1, 1, 0, 128, 0>(CUtensorMap_st)",
    "wo_b": "void unnamed>::block_scaled_gemm_kernel<256, 0, 1, 0, 128, 0>(CUtensorMap_st)",
    # the CTA-pair kernel of the large shapes: its first template argument is
    # the epilogue (1: wo_a's re-quantisation), the second whether it is bf16
    "wo_a_pair": "void unnamed>::block_scaled_gemm_pair_kernel<1, 0>(CUtensorMap_st)",
    "wo_b_pair": "void unnamed>::block_scaled_gemm_pair_kernel<0, 0>(CUtensorMap_st)",
}


def _write_launch_list(path, launches):
    with open(path, "w", newline="") as f:
        f.write("==PROF== Connected to process 1\n")   # ncu's own lines come first
        w = csv.writer(f, quoting=csv.QUOTE_ALL)
        w.writerow(_HEADER)
        for i, (kernel, read, write, ns) in enumerate(launches):
            for metric, unit, value in (("dram__bytes_read.sum", "byte", read),
                                        ("dram__bytes_write.sum", "byte", write),
                                        ("gpu__time_duration.sum", "ns", ns)):
                w.writerow([str(i), "1", "python3", "127.0.0.1", _KERNELS[kernel], "1", "7",
                            "(352, 1, 1)", "(152, 1, 1)", "0", "10.3",
                            "Command line profiler metrics", metric, unit, f"{value:,}"])


def test_summarize_traffic_groups_launches_by_kernel(tmp_path):
    # two steps of the three launches, in launch order
    launches = [("quant", 538_000_000, 227_000_000, 128_700),
                ("wo_a", 337_900_000, 54_200_000, 199_400),
                ("wo_b", 408_500_000, 48_300_000, 295_100),
                ("quant", 538_100_000, 229_000_000, 129_000),
                ("wo_a", 337_800_000, 54_300_000, 198_300),
                ("wo_b", 410_200_000, 48_000_000, 301_200)]
    path = tmp_path / "launches.csv"
    _write_launch_list(path, launches)
    lines = bench.summarize_traffic(str(path)).splitlines()
    n_src = len(bench.TRAFFIC_SOURCES)
    assert [l.split()[1] for l in lines[:n_src]] == list(bench.TRAFFIC_SOURCES)
    body = [l.split() for l in lines if l.split()[0] in ("quant", "wo_a", "wo_b")]
    assert [b[0] for b in body] == ["quant", "quant", "wo_a", "wo_a", "wo_b", "wo_b"]
    assert body[0][1:] == ["538.0e6", "227.0e6", "128.7"]
    assert body[5][1:] == ["410.2e6", "48.0e6", "301.2"]


def test_summarize_traffic_names_the_pair_kernels(tmp_path):
    launches = [("wo_a_pair", 300_000_000, 50_000_000, 190_000),
                ("wo_b_pair", 400_000_000, 48_000_000, 280_000)]
    path = tmp_path / "launches.csv"
    _write_launch_list(path, launches)
    body = [l.split() for l in bench.summarize_traffic(str(path)).splitlines()
            if l.split()[0] in ("quant", "wo_a", "wo_b")]
    assert [b[0] for b in body] == ["wo_a", "wo_b"]
    assert body[0][1:] == ["300.0e6", "50.0e6", "190.0"]


def test_recorded_traffic_reads_the_committed_record_format(tmp_path, monkeypatch):
    """The lookup averages read + write over a kernel's lines, and gives None as
    soon as one source hash differs from the files on disk."""
    launches = [("quant", 500_000_000, 200_000_000, 1), ("wo_b", 400_000_000, 50_000_000, 1),
                ("wo_b", 420_000_000, 50_000_000, 1)]
    path = tmp_path / "launches.csv"
    _write_launch_list(path, launches)
    body = bench.summarize_traffic(str(path))
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic_full_T4096.txt").write_text("# comment\n" + body + "\n")
    csrc = tmp_path / "deepseek_v4_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for src in bench.TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "deepseek_v4_attention_gb300", "csrc", src), "rb") as f:
            (csrc / src).write_bytes(f.read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("quant") == 700e6
    assert bench.recorded_traffic("wo_b") == 460e6
    assert bench.recorded_traffic("wo_a") is None          # no lines for it
    (csrc / bench.TRAFFIC_SOURCES[0]).write_bytes(b"// changed\n")
    assert bench.recorded_traffic("wo_b") is None


def test_tensor_peak_rule():
    """Burst cuBLAS bf16 figure for sub-second timed regions, the sustained one
    from a second on; FP8 = 2 x bf16."""
    peaks = {"hbm_gbs": 6663.2, "bf16_tflops": 1902.6, "bf16_tflops_sustained": 1719.6}
    p, rule = bench.tensor_peak(peaks, "measured", 0.013, "e4m3")
    assert p == 2 * 1902.6 and "burst" in rule and "13.0 ms" in rule
    p, rule = bench.tensor_peak(peaks, "measured", 2.5, "e4m3")
    assert p == 2 * 1719.6 and "sustained" in rule
    p, _ = bench.tensor_peak(peaks, "measured", 0.5, "bf16")
    assert p == 1902.6
    p, _ = bench.tensor_peak({"hbm_gbs": 1.0, "bf16_tflops": 100.0}, "fallback", 5.0, "e4m3")
    assert p == 200.0                                  # no sustained figure: burst


def test_add_roofline_clock_matched():
    peaks = {"hbm_gbs": 6663.2, "bf16_tflops": 1902.6, "bf16_tflops_sustained": 1719.6}
    st = {"ms": 0.3, "bound": "tensor", "achieved": 3000.0, "unit": "TFLOP/s"}
    bench.add_roofline(st, peaks, "measured", 0.013, {"sm_mhz": 2000.0}, 152)
    cm = 16384 * 152 * 2000e6 / 1e12
    assert abs(st["clock_matched"]["peak"] - cm) < 1e-9
    assert abs(st["clock_matched"]["frac"] - 3000.0 / cm) < 1e-12
    assert abs(st["tflops_per_ghz"] - 1500.0) < 1e-9
    assert abs(st["frac"] - 3000.0 / (2 * 1902.6)) < 1e-12
    hb = {"ms": 0.1, "bound": "hbm", "achieved": 6000.0, "unit": "GB/s"}
    bench.add_roofline(hb, peaks, "measured", 0.013, {"sm_mhz": None}, 152)
    assert hb["peak"] == 6663.2 and "clock_matched" not in hb


def test_clock_sampler_summary():
    s = bench.ClockSampler(0)
    s.samples = [(2070.0, 900.0, []), (1950.0, 1400.0, ["sw_power_cap"]), (2010.0, None, [])]
    s.max_mhz = 2070.0
    out = s.summary()
    assert out["sm_mhz"] == 2010.0 and out["samples"] == 3 and out["sm_mhz_min"] == 1950.0
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_max"] == 1400.0
