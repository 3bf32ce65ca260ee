"""Host-side pieces of bench.py (no GPU): argument parsing, the source files
its profile-staleness hash reads, and the reference arm's oracle pass."""
import os
import sys

import bench
import synthetic as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kernel_sources_exist():
    for cid in (2, 3, 4):
        for L in S.config(cid).layers:
            for f in bench.kernel_sources(L):
                assert os.path.exists(os.path.join(bench.ROOT, f)), f
            assert len(bench.kernel_source_hash(bench.kernel_sources(L))) == 16


def test_only_cases_cover_every_workload():
    assert {c for c, _ in bench.ONLY_CASES.values()} == {1, 2, 3, 4, 5}


def test_oracle_strip_pass_counts_pixels():
    import oracle
    wl = S.config(3, scale={"h": 16, "w": 24})
    assert bench.oracle_net_pass(oracle, wl, 4) == 4 * 24


def test_profiled_traffic_absent_or_stale_is_none():
    assert bench.profiled_traffic("no-such-kernel", "0" * 16) is None


def test_oracle_per_config_covers_every_workload():
    # every workload timed with all threads; 1, 2 and 5 also single-threaded
    r = bench.oracle_per_config(S, min_seconds=0.01)
    assert sorted(r) == ["1", "2", "3", "4", "5"]
    for name, ent in r.items():
        assert ent["openmp"]["mpixel_per_s"] > 0 and ent["openmp"]["calls"] >= 1
        assert ("1 thread" in ent) == (name in ("1", "2", "5"))
        if name != "5":
            assert ent["openmp"]["gflops"] > 0


def test_profile_commands_use_existing_bench_options():
    """Every ncu summary under profiles/ names its command; the bench cases
    and flags it uses must still exist, and the command carries
    --clock-control none."""
    import glob
    flags = {"--steps", "--warmup", "--only", "--no-cpu-baseline", "--no-per-config", "--no-autotune", "--gpus",
             "--impl", "--candidate"}
    seen = 0
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        lines = text.split("\n")
        for i, line in enumerate(lines):
            if not line.lstrip().startswith("ncu --"):
                continue
            cmd = line
            k = i
            while cmd.rstrip().endswith("\\") and k + 1 < len(lines):
                k += 1
                cmd = cmd.rstrip()[:-1] + " " + lines[k]
            assert "--clock-control none" in cmd, path
            assert "python bench.py" in cmd, path
            tail = cmd.split("python bench.py", 1)[1].split()
            for tok in tail:
                if tok.startswith("--"):
                    assert tok in flags, (path, tok)
            if "--only" in tail:
                assert tail[tail.index("--only") + 1] in bench.ONLY_CASES, path
            seen += 1
    assert seen >= 10


def test_per_config_summary_keys_are_unique_and_short():
    pc = {"launch_floor": {"us_per_launch": 0.56},
          "1: 64x64 1->1 3x3": {"ms_mean": 0.0061, "roofline_frac": 0.001, "graph_ms_per_launch": 0.0015,
                                "launch_floor_us": 0.56},
          "3-L3: 1280x720 32->4 3x3": {"ms_mean": 0.05, "roofline_frac": 0.52, "ms_kernel": 0.045,
                                       "roofline_frac_kernel": 0.58},
          "3: 3-layer net replayed as a CUDA graph": {"ms_mean": 0.36},
          "3: 3-layer net, layers 2 and 3 on split-TF32 tensor cores": {"ms_mean": 0.16},
          "4 (tcgen05 TF32)": {"ms_mean": 0.024, "roofline_frac": 0.32},
          "4 (tcgen05 split TF32)": {"ms_mean": 0.064, "roofline_frac": 0.37},
          "3-L2 (tcgen05 BF16, bf16 x/y)": {"ms_mean": 0.035, "roofline_frac": 0.5},
          "_peaks": {"fp32_tflops": 80.5}}
    s = bench.per_config_summary(pc)
    assert s == {"1": [0.0061, 0.001, 0.0015, 0.56], "3-L3": [0.05, 0.52, 0.045, 0.58], "3 graph": [0.36, None],
                 "3 x3 net": [0.16, None], "4 tf32": [0.024, 0.32], "4 x3": [0.064, 0.37],
                 "3-L2 bf16": [0.035, 0.5]}
