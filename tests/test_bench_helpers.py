"""Host-side helpers of bench.py (no GPU): the recorded-counter key, the all-cores oracle
split, the sweep's coverage of the five workloads, whole-job throughput."""
import os

import numpy as np

import bench
import oracle as orc
import synth


def test_kernel_code_sha_ignores_comments_and_host_code(tmp_path, monkeypatch):
    src, hdr = tmp_path / "k.cu", tmp_path / "k.h"
    mark = bench.HOST_SIDE_MARK
    hdr.write_text("constexpr int kTile = 4;\n")
    src.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n"
                   + mark + "\nvoid launch() { k<<<1, 1>>>(nullptr); }\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    monkeypatch.setattr(bench, "KERNEL_HDR", str(hdr))
    h0 = bench.kernel_code_sha()
    src.write_text("/* another\n header */\n__global__ void k(int* p) {\n    p[0] = 1;\n}\n"
                   + mark + "\nvoid launch() { k<<<2, 1>>>(nullptr); }\n")
    assert bench.kernel_code_sha() == h0          # comments, layout and host code only
    src.write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n" + mark + "\n")
    assert bench.kernel_code_sha() != h0          # a device-code change voids the counters
    src.write_text("__global__ void k(int* p) {\n  p[0] = 1;\n}\n" + mark + "\n")
    assert bench.kernel_code_sha() == h0
    hdr.write_text("constexpr int kTile = 8;\n")
    assert bench.kernel_code_sha() != h0          # so does a change to the shared constants


def test_all_cores_split_gives_the_single_call_result():
    # the all-cores CPU figure cuts the sample into element ranges, one per thread: the
    # pieces must reproduce the single call bit for bit (the collective is elementwise)
    n = 100_003
    xs = [synth.to_numpy(synth.rank_input(2, r, n, "bf16")) for r in range(2)]
    whole = orc.allreduce(orc.BF16, xs, 0.5)[2]
    cuts = [n * t // 7 for t in range(8)]
    parts = [orc.allreduce(orc.BF16, xs, 0.5, cuts[t], cuts[t + 1])[2] for t in range(7)]
    assert np.array_equal(np.concatenate(parts), whole)


def test_sweep_covers_the_five_workloads():
    pts = bench._sweep_points()
    have = {(name, A, dt) for name, A, dt, _, _ in pts}
    assert ("allreduce", 2, "f32") in have                     # workload 1
    assert ("allreduce", 2, "bf16") in have                    # workload 2
    assert {("reduce_scatter", 2, "f32"), ("reduce_scatter", 2, "i32")} <= have   # 3
    assert {("allreduce", 4, "bf16"), ("reduce_scatter", 4, "bf16")} <= have       # 4
    assert {(c, 4, d) for c in ("all_gather", "all_to_all") for d in ("bf16", "i32")} <= have  # 5
    # each sweep group's largest point gets the oracle timed beside it
    assert bench.ORACLE_SWEEP_SAMPLE >= 1 << 20


def test_whole_job_throughput_counts_every_replica():
    # 2 replicas each moving 1 GB per step, 10 steps, slowest rank 20 ms: 1000 GB/s
    assert abs(bench.whole_job_gbs(1e9, 10, 2, 20.0) - 1000.0) < 1e-9
    assert os.path.exists(bench.PROFILE)
