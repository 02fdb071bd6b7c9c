"""bench.py host logic without a GPU: the multi-rank reduction (gloo, 2 ranks),
the reference arm's rank handling, and the ncu traffic lookup."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.5, 0.8][rank]
    slowest = bench.max_over_ranks(local_ms, world, "cpu")
    value = bench.job_throughput(2.0 * 4096 ** 3, world, slowest)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 0.8  # the slower rank's time
        assert value == pytest.approx(2 * 2.0 * 4096 ** 3 / 0.8e-3 / 1e12)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--config",
                        "kloop_256x256x1024_f16_abt"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    from dense_gemm_engineering_gb300 import configs

    cfg = configs.BY_NAME["kloop_256x256x1024_f16_abt"]
    assert line["metric"] == bench.metric_for(cfg) and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_metric_names_follow_the_workload():
    from dense_gemm_engineering_gb300 import configs

    assert bench.metric_for(configs.HEADLINE) == bench.METRIC
    every = configs.CONFIGS + configs.FP8_CONFIGS + configs.MX_CONFIGS
    names = {bench.metric_for(c) for c in every}
    assert len(names) == len(every)
    fp8 = configs.FP8_CONFIGS[0]
    assert "E4M3->BF16" in bench.metric_for(fp8)
    peak, basis = bench.peak_for(fp8, {"bf16_tflops": 1910.0})
    assert peak == 3820.0 and "x 2" in basis
    mx = configs.MX_CONFIGS[0]
    assert "block-scaled MX E4M3->BF16" in bench.metric_for(mx)
    assert bench.peak_for(mx, {"bf16_tflops": 1910.0})[0] == 3820.0


def test_reference_arm_runs_the_fp8_oracle():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--config",
                        "fp8_square_4096x4096x4096_e4m3_abt"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and "E4M3" in line["metric"]


def test_reference_arm_runs_the_block_scaled_oracle():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--config",
                        "mx_square_4096x4096x4096_e4m3_abt"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and "MX" in line["metric"]


def test_block_scaled_inputs_and_oracle_rows():
    import oracle
    from dense_gemm_engineering_gb300 import configs

    cfg = configs.MX_CONFIGS[0]
    X = bench.make_inputs(cfg)
    assert len(X) == 4 and X[2].shape == (cfg.M, cfg.K // 32) and X[3].shape == (cfg.N, cfg.K // 32)
    assert 124 <= X[2].min() and X[2].max() <= 130
    rows = bench.oracle_rows(oracle.get(), cfg, X, (5, 7))
    want = oracle.gemm_mx(X[0][5:7], X[1], X[2][5:7], X[3], fmt="e4m3", out_dtype="bf16")
    assert np.array_equal(rows, want)
    assert cfg.min_bytes == 2 * 4096 * 4096 + 2 * 4096 * 4096 + 2 * 4096 * 128


def test_traffic_lookup_matches_only_current_kernel(tmp_path, monkeypatch):
    h = bench.kernel_source_hash()
    assert len(h) == 12
    pdir = tmp_path / "profiles"
    pdir.mkdir()
    (pdir / "x.md").write_text(
        f"bench-traffic: workload=w1 kernel={h} bytes_per_launch=123\n"
        f"bench-traffic: workload=w1 kernel=000000000000 bytes_per_launch=999\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w1", h) == 123
    assert bench.recorded_traffic("w2", h) is None
    assert bench.recorded_traffic("w1", "ffffffffffff") is None


def test_source_hash_ignores_comments_but_not_code():
    code = 'int f(int x) { return x + 1; } // add one\n/* block */ const char* s = "// not a comment";'
    same = 'int  f(int x) {\n  return x + 1;\n}\nconst char* s = "// not a comment"; // note'
    other = 'int f(int x) { return x + 2; }\nconst char* s = "// not a comment";'
    assert bench.strip_c_comments(code) == bench.strip_c_comments(same)
    assert bench.strip_c_comments(code) != bench.strip_c_comments(other)
    assert '"// not a comment"' in bench.strip_c_comments(code)


def test_single_core_oracle_baseline_restores_threads():
    import oracle
    from dense_gemm_engineering_gb300 import configs

    cfg = configs.CONFIGS[0]  # 128 x 128 x 64
    X = bench.make_inputs(cfg)
    before = oracle.get().num_threads()
    ctx = bench.oracle_single_core(cfg, X, rows=16)
    assert oracle.get().num_threads() == before
    assert ctx["cores"] == 1 and ctx["value"] > 0
    assert ctx["extrapolated_full_s"] > 0 and "rows 0..16" in ctx["sample"]


def test_check_rows_against_the_oracle():
    import oracle
    from dense_gemm_engineering_gb300 import configs

    cfg = configs.CONFIGS[0]  # 128 x 128 x 64 FP16
    X = bench.make_inputs(cfg)
    ref = bench.oracle_rows(oracle.get(), cfg, X, (0, 8))
    ok = bench.check_rows(cfg, ref.copy(), ref)
    assert ok["within_tolerance"] and ok["max_abs_err"] == 0.0 and ok["rows"] == 8
    bad = ref.copy()
    bad[3, 5] ^= np.uint16(0x4000)  # flip a high exponent bit
    assert not bench.check_rows(cfg, bad, ref)["within_tolerance"]


# ---- this build's additions: strict row check, in-kernel clock, row sampling -------

def _f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def test_check_rows_strict_bound_accepts_rounding_and_rejects_a_lost_slice():
    from dense_gemm_engineering_gb300 import configs

    cfg = configs.HEADLINE
    exact = np.array([[1.0 + 2 ** -12, -3.25, 0.0, 100.0 + 2 ** -5]])
    sum_abs = np.array([[1024.0, 1024.0, 1024.0, 1024.0]])
    ref = _f16_bits(exact)                        # the one rounding
    ok = bench.check_rows(cfg, ref, ref, exact, sum_abs)
    assert ok["within_tolerance"] and ok["within_strict"] and ok["max_ulp"] <= 0.5
    # a K = 16 slice of U[-1,1) products (|sum| ~ sqrt(16)/3 ~ 1.3) moves one output
    bad = _f16_bits(exact + np.array([[0.0, 0.0, 1.3, 0.0]]))
    chk = bench.check_rows(cfg, bad, ref, exact, sum_abs)
    assert not chk["within_strict"] and chk["max_err_over_strict"] > 1


def test_clock_from_probes():
    rows = [[1000, 10, 1000 + 1800 * 50, 10 + 50_000],   # 1800 MHz over 50 us
            [0, 0, 1700 * 40, 40_000],                   # 1700 MHz
            [5, 5, 5, 5]]                                # no time elapsed: ignored
    c = bench.clock_from_probes(rows)
    assert c["launches"] == 2
    assert c["sm_mhz_min"] == pytest.approx(1700) and c["sm_mhz_max"] == pytest.approx(1800)
    assert bench.clock_from_probes([[1, 1, 1, 1]]) is None


@pytest.mark.parametrize("M", [1, 2, 3, 5, 128, 3000, 8192])
def test_check_row_ranges_are_disjoint_and_inside(M):
    r = bench.check_row_ranges(M)
    assert r and all(0 <= a < b <= M for a, b in r)
    assert all(r[i][1] <= r[i + 1][0] for i in range(len(r) - 1))
    assert r[0][0] == 0 and r[-1][1] == M


def test_options_and_sweep_flags_parse():
    a = bench.parse_args(["--options", '{"raster_group": 8}', "--sweep", "raster",
                          "--no-per-config", "--soak-seconds", "0.5"])
    assert json.loads(a.options) == {"raster_group": 8}
    assert a.sweep == "raster" and a.no_per_config and a.soak_seconds == 0.5
    assert all(o in (1, 2) and g >= 1 and h % 2 == 1 for o, g, h in bench.RASTER_SWEEP)
