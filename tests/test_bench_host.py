"""Host-side pieces of bench.py: the traffic record built from an ncu log,
the algorithmic bytes of a workload, and the whole-job throughput."""
import json

import numpy as np

import bench
from sparsely_gated_mixture_top_b300 import workloads as wl

CSV = '''==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","unnamed>::ffn_tiles(const int *, int, int, int *)","1","7","(1024, 1, 1)","(1, 1, 1)","0","10.3","m","dram__bytes_read.sum","byte","1,024"
"0","1","python","h","unnamed>::ffn_tiles(const int *, int, int, int *)","1","7","(1024, 1, 1)","(1, 1, 1)","0","10.3","m","dram__bytes_write.sum","byte","0"
"0","1","python","h","unnamed>::ffn_tiles(const int *, int, int, int *)","1","7","(1024, 1, 1)","(1, 1, 1)","0","10.3","m","gpu__time_duration.sum","us","4.5"
"1","1","python","h","void unnamed>::ffn_gemm_tc<256, 4>(x)","1","7","(320, 1, 1)","(148, 1, 1)","0","10.3","m","dram__bytes_read.sum","Mbyte","2.5"
"1","1","python","h","void unnamed>::ffn_gemm_tc<256, 4>(x)","1","7","(320, 1, 1)","(148, 1, 1)","0","10.3","m","dram__bytes_write.sum","Kbyte","3"
"1","1","python","h","void unnamed>::ffn_gemm_tc<256, 4>(x)","1","7","(320, 1, 1)","(148, 1, 1)","0","10.3","m","gpu__time_duration.sum","ns","9000"
'''


def test_traffic_summary_sums_the_captured_launches(tmp_path):
    csv = tmp_path / "t.csv"
    csv.write_text(CSV)
    line = tmp_path / "b.json"
    line.write_text("noise\n" + json.dumps({"roofline": {"algorithmic_per_launch": 123}}) + "\n")
    rec = bench.traffic_summary(str(csv), str(line), wl.WORKLOADS["flat_n256_k4"])
    assert rec["ffn_stage_dram_bytes_per_launch"] == 1024 + 2_500_000 + 3_000
    assert [k["kernel"] for k in rec["kernels"]] == ["unnamed>::ffn_tiles",
                                                    "void unnamed>::ffn_gemm_tc<256, 4>"]
    assert rec["kernels"][0]["duration_ns_cold"] == 4500 and rec["kernels"][1]["duration_ns_cold"] == 9000
    assert rec["algorithmic_bytes_per_launch"] == 123
    assert rec["source_sha256"] == bench.source_digest() and rec["workload"] == "flat_n256_k4"


def test_algorithmic_bytes_and_flops():
    w = wl.Workload("t", T=10, d=64, h=128, n=4, k=2)            # bf16, flat, noisy
    counts = np.array([5, 0, 10, 5])                               # 3 experts hit
    a = bench.algorithmic(w, counts)
    S = 20
    weights = 3 * (2 * 64 * 128 * 2 + 4 * (64 + 128))
    assert a["experts_hit"] == 3
    assert a["flops"] == 4.0 * S * 64 * 128
    # the gate: x (T x d) against the 4 clean and 4 noise columns
    assert a["gate_flops"] == 2.0 * 10 * 64 * 4 * 2
    assert a["layer_flops"] == a["flops"] + a["gate_flops"]
    wh = wl.Workload("h", T=10, d=64, h=128, n=8, k=4, groups=4, k_groups=2)
    # hierarchical: 4 group columns + 2 kept groups x 2 columns each
    assert bench.algorithmic(wh, np.ones(8))["gate_flops"] == 2.0 * 10 * 64 * (4 + 2 * 2) * 2
    # the FFN stage: hit weights and x once; the slot buffer is not algorithmic
    assert a["ffn_bytes"] == weights + 10 * 64 * 2
    assert a["layer_bytes"] == (weights + 2 * 10 * 64 * 2 + 10 * 4 * 4 + 2 * 64 * 4 * 4 +
                                S * 8 + 4 * 8)


def test_job_throughput_single_rank():
    ms, value = bench.job_throughput(2.0, 1000)
    assert ms == 2.0 and value == 1000 / 2e-3


def test_clock_sampler_summary_without_a_gpu():
    # On a machine without NVML or nvidia-smi the sampler reports no source and
    # no numbers instead of failing; with samples injected it reports the
    # median, the minimum, the maximum and every active reason.
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.samples, c.source, c.period = [], "nvml", 0.001
    c._stop = bench.threading.Event()
    c.thread = bench.threading.Thread(target=lambda: None)
    c.thread.start()
    c._take = lambda: None
    c.samples = [(2032.0, 2032.0, 500.0, 0x0), (1900.0, 2032.0, 900.0, 0x4),
                 (2000.0, 2032.0, 800.0, 0x0)]
    r = c.stop()
    assert r["sm_mhz"] == 2000.0 and r["sm_mhz_min"] == 1900.0 and r["sm_max_mhz"] == 2032.0
    assert r["samples"] == 3 and r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 900.0


def test_every_pass_and_workload_parses(monkeypatch):
    import sys
    for which in ("forward", "backward", "balanced", "ep"):
        for name in wl.WORKLOADS:
            monkeypatch.setattr(sys, "argv", ["bench.py", "--pass", which, "--workload", name])
            args = bench.parse()
            assert args.which == which and args.workload == name
            assert args.gpus == 1 and args.warmup >= 3


def test_launch_counts_follow_the_expert_stage_choice():
    """The counts the GPU graph tests confirm: the fused two-layer expert
    kernel (one launch) serves bf16 shapes with d in {256, 512}, h a multiple
    of 256 and at most 128 rows per expert on average; otherwise two GEMMs."""
    W = wl.WORKLOADS
    assert not bench.fused_ffn(W["flat_n256_k4"])            # 256 rows per expert
    assert bench.launches_per_step(W["flat_n256_k4"]) == 8
    assert bench.fused_ffn(W["hier_4096h_16x256"])           # 32 rows per expert
    assert bench.launches_per_step(W["hier_4096h_16x256"]) == 14
    assert bench.fused_ffn(W["sparse_n2048_T32768"])
    assert bench.launches_per_step(W["sparse_n2048_T32768"]) == 7
    assert not bench.fused_ffn(W["skewed_zipf_n64"])          # d = 1024
    assert not bench.fused_ffn(W["tiny_flat_fp32"])           # fp32
    assert bench.backward_launches(W["flat_n256_k4"]) == 29
    assert bench.backward_launches(W["hier_4096h_16x256"]) == 36
