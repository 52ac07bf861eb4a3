"""CPU: the benchmark's host-side step construction.  Every timed step must read weights no
recent step has read (the L2 rule): a step that alone exceeds twice the L2 uses one weight
copy per call of a size M, and a step that fits the L2 rotates over enough graphs, each on
other copies, that the bytes between two reads of one copy exceed twice the L2."""
import bench


def _steps(name):
    w = bench.WORKLOADS[name]
    copies = bench._copies_needed(w)
    sets = [[[None] * len(w.projs)] * w.layers] * copies
    calls = bench._calls(w, sets)
    step_bytes = sum(bench._work(w, w.projs[pi].N, w.projs[pi].K, M) for _, _, pi, M in calls)
    return w, copies, calls, step_bytes, bench._rotated_steps(w, calls, copies, step_bytes)


def test_large_steps_are_not_rotated():
    for name in ("mxfp4_mlp_12288x4096", "nvfp4_lm_head_248320x2560", "nvfp4_layer_sweep_5120"):
        w, copies, calls, step_bytes, steps = _steps(name)
        assert len(steps) == 1 and steps[0] == calls
        assert step_bytes > 2 * bench.L2_BYTES, name
        per_copy = sum(bench._algo_bytes(w.fmt, p.N, p.K, 0) for p in w.projs) * w.layers
        if per_copy < 2 * bench.L2_BYTES:
            # a copy smaller than twice the L2: every M of the step streams its own copy
            by_m = {}
            for c, _, _, M in calls:
                by_m.setdefault(M, set()).add(c)
            assert len({frozenset(v) for v in by_m.values()}) == len(w.Ms), name


def test_small_step_rotates_over_cold_copies():
    w, copies, calls, step_bytes, steps = _steps("nvfp4_gemm_2048x1024")
    assert step_bytes < bench.L2_BYTES
    assert len(steps) * step_bytes >= 2 * bench.L2_BYTES
    used = [c for st in steps for c, _, _, _ in st]
    assert len(set(used)) == len(used)  # no copy read twice within one rotation
    assert all(0 <= c < copies for c in used)


def test_traffic_is_dropped_once_the_kernel_source_changes(tmp_path, monkeypatch):
    """The DRAM traffic of a committed capture is reported only while the captured kernel's
    source is unchanged; decode traffic is scaled to the step's average launch."""
    import hashlib
    import json
    import os
    w = bench.WORKLOADS["mxfp4_mlp_12288x4096"]
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    os.makedirs(tmp_path / "profiles")
    rec = {w.name: {"kernel": "k", "source": "k.cu",
                    "source_sha256_16": hashlib.sha256(b"kernel v1\n").hexdigest()[:16],
                    "captured_launch": "one launch", "dram_bytes": 110,
                    "algorithmic_bytes": 100, "summary": "profiles/k.md"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    t = bench._profiled_traffic(w, step_work=4000.0, calls=4)
    assert t["bytes_per_launch"] == 1100 and t["dram_over_algorithmic"] == 1.1
    src.write_text("kernel v2\n")
    assert bench._profiled_traffic(w, step_work=4000.0, calls=4) is None
    assert bench._profiled_traffic(bench.WORKLOADS["nvfp4_gemm_2048x1024"], 1.0, 1) is None


def test_clock_sampler_reads_median_clock_and_throttle_reasons(tmp_path, monkeypatch):
    """The clocks record of the JSON line, from a stand-in nvidia-smi that prints three
    samples: the median SM clock, the highest maximum clock and every reason seen Active."""
    import os
    import stat
    import time
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 1900, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '0, 2010, 2070, 1001.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, 1950, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "exec sleep 30\n")
    fake.chmod(fake.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(1.0)
    rec = s.stop()
    assert rec["sm_mhz"] == 1950 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 4
