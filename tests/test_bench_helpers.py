"""Host-side helpers of bench.py (no GPU): the recorded-counter key, the all-cores oracle
split, the sweep's coverage of the five workloads, whole-job throughput."""
import os

import numpy as np

import bench
import oracle as orc
import synth


def test_kernel_code_sha_ignores_comments_and_host_code(tmp_path, monkeypatch):
    src, hdr, dev = tmp_path / "k.cu", tmp_path / "k.h", tmp_path / "d.cuh"
    mark = bench.HOST_SIDE_MARK
    hdr.write_text("constexpr int kTile = 4;\n")
    dev.write_text("__device__ int f() { return 1; }  // primitive\n")
    monkeypatch.setattr(bench, "KERNEL_DEV", str(dev))
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
    hdr.write_text("constexpr int kTile = 4;\n")
    assert bench.kernel_code_sha() == h0
    dev.write_text("__device__ int f() { return 2; }\n")
    assert bench.kernel_code_sha() != h0          # and to the shared device primitives


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


def test_reference_arm_bytes_from_the_oracle_plan():
    # the reference arm counts the relay allreduce's pass bytes from the oracle's plan
    # alone; they must equal what the library reports for the same schedule
    import pack_virtual_rank_gb300 as rv
    for count in (1 << 24, 65536, 1 << 20, (1 << 22) + 4099, bench.CPU_SAMPLE):
        g, _ = orc.plan(orc.AR, 2, 8, count, 2, force=orc.FORCE_RELAY)
        p = rv.relay_plan(rv.ALLREDUCE, count, rv.BF16, 2, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
        lib = sum(q["bytes_read"] + q["bytes_written"] for q in rv.relay_plan_passes(p))
        assert bench.relay_allreduce_a2_bytes(g, 2) == lib
    g, _ = orc.plan(orc.AR, 2, 8, 1 << 24, 2)
    assert bench.relay_allreduce_a2_bytes(g, 2) == 68 * g["chunk"] * 2


def test_reference_arm_does_not_load_the_product_library():
    import inspect
    src = inspect.getsource(bench.run_reference)
    assert "pack_virtual_rank_gb300" not in src and "rv." not in src


def test_clock_windows(tmp_path):
    import datetime
    c = bench.Clocks(0, enabled=False)
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5).timestamp()
    lines = []
    for k in range(10):
        ts = datetime.datetime.fromtimestamp(t0 + 0.1 * k).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        reason = "Active" if k == 7 else "Not Active"
        lines.append(f"{ts}, 0, {1900 + k}, 2070, 900.0, 0x0, Not Active, Not Active, "
                     f"Not Active, {reason}")
    c.out.write("\n".join(lines + ["garbage line"]) + "\n")
    c.proc = object()                      # as if nvidia-smi had been started
    w = c.window(t0 + 0.15, t0 + 0.55)      # samples 2..5
    assert w["samples"] == 4 and w["reasons"] == [] and w["sm_mhz"] == 1903.5
    w = c.window(t0, t0 + 1.0)
    assert w["samples"] == 10 and w["reasons"] == ["sw_power_cap"] and w["sm_max_mhz"] == 2070
    assert c.summary()["samples"] == 10


def test_per_workload_points_cover_the_metric():
    pts = bench.per_workload_points()
    have = {(name, A, dt) for _, name, A, dt, _, _ in pts}
    assert ("allreduce", 2, "f32") in have
    assert {("reduce_scatter", 2, "f32"), ("reduce_scatter", 2, "i32")} <= have
    assert {("allreduce", 4, "bf16"), ("reduce_scatter", 4, "bf16")} <= have
    assert {(c, 4, d) for c in ("all_gather", "all_to_all") for d in ("bf16", "i32")} <= have
    odd = [cnt for _, name, _, _, cnt, _ in pts if name == "all_to_all" and cnt % 2 == 1]
    assert len(odd) >= 2          # bf16 and int32 with an odd segmentCount


def test_traffic_record_is_keyed_to_the_kernel_code(tmp_path, monkeypatch):
    import json
    rec = tmp_path / "t.json"
    rec.write_text(json.dumps({"kernel_code_sha256_16": bench.kernel_code_sha(),
                               "traffic_bytes_per_launch": {"group1": 5}}))
    monkeypatch.setattr(bench, "PROFILE", str(rec))
    assert bench._profiled_traffic()[0] == {"group1": 5}
    rec.write_text(json.dumps({"kernel_code_sha256_16": "0" * 16,
                               "traffic_bytes_per_launch": {"group1": 5}}))
    assert bench._profiled_traffic()[0] is None
