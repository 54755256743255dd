"""Host-side logic of bench.py: multi-rank aggregation (gloo, 2 ranks on CPU)
and the reference arm (the CPU oracle on a bounded sample)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed 1e9 bytes in (r + 1) seconds: the job took 2 s for 2e9 bytes
    gbs, t = bench.aggregate_throughput(1e9, float(rank + 1), world)
    q.put((rank, gbs, t, bench.dist_env()))
    bench.barrier()
    dist.destroy_process_group()


def test_aggregation_takes_the_slowest_rank_and_sums_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank, gbs, t, env in res:
        assert t == 2.0
        assert abs(gbs - 1.0) < 1e-12          # 2e9 bytes / 2 s = 1 GB/s
        assert env[0] == 2 and env[1] == rank


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-sample-frac", "0.0002"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better",
              "cpu_baseline", "e2e", "config"):
        assert k in d
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_reference_arm_non_zero_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--warmup", "2"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode != 0


def test_cpu_baseline_all_cores_runs_the_same_sample():
    import bench
    one = bench.cpu_baseline(0.002)
    many = bench.cpu_baseline_all_cores(0.002)
    assert many["sample"] == one["sample"]
    assert many["cores"] == (os.cpu_count() or 1) and many["value"] > 0


def test_cpu_per_config_covers_every_workload():
    """The per-config CPU baseline times the oracle on each configured workload, on one core
    and on all cores, and the 576-slot update for both algorithms and both margins."""
    import bench
    r = bench.cpu_per_config(0.02)
    c = r["compact"]
    assert c["cores"] == (os.cpu_count() or 1)
    for k in ("mlp_activation", "ffn", "grad_quantize", "grad_dequantize", "ragged_12"):
        one, many = c[k]
        assert one > 0 and many > 0
        assert r["configs"][k]["elements_sampled"] > 0
    assert len(c["update_us"]) == 4 and all(u > 0 for u in c["update_us"])
    assert len(json.dumps(c)) < 400          # it rides on the printed line


def test_compact_rows_and_detail_file(tmp_path):
    import bench
    kernels = {"multi_quantize_amax": {"frac_of_peak": 0.95}, "dequantize": {"frac_of_peak": 0.94}}
    other = {"mlp_activation": {"frac_of_peak": 0.9}, "ragged_twelve_tensors": {"frac_of_peak": 1.04}}
    nxt = {"qdq_amax": {"frac_of_peak": 0.99}, "gelu_quantize_amax": {"codes_only": {"frac_of_peak": 0.82}},
           "layernorm_quantize_amax": {"codes_only": {"frac_of_peak": 0.6}},
           "amax_scale_update_ring": {"us": 7.6}}
    rows = bench.compact_rows(kernels, nxt, other, {"ring_update_us_after_dequantize": 2.9})
    assert rows == {"multi_quantize_frac": 0.95, "dequantize_frac": 0.94, "mlp_activation_8192x4096_frac": 0.9,
                    "ragged_12_frac": 1.04, "qdq_frac": 0.99, "gelu_codes_frac": 0.82,
                    "layernorm_codes_frac": 0.6, "ring_update_us": 2.9, "ring_update_us_eager": 7.6}
    assert "ring_update_us" not in bench.compact_rows(kernels, nxt, other)
    other["mlp_activation"]["same_bytes_library"] = {"device_copy": {"frac_of_peak": 0.88}}
    assert bench.compact_rows(kernels, nxt, other)["mlp_same_bytes_copy_frac"] == 0.88
    nxt["layernorm_quantize_amax_wide"] = {"codes_only": {"frac_of_peak": 0.51}}
    assert bench.compact_rows(kernels, nxt, other)["layernorm_12288_codes_frac"] == 0.51
    assert bench.compact_rows(kernels, None, None) == {"multi_quantize_frac": 0.95, "dequantize_frac": 0.94}
    p = tmp_path / "sub" / "detail.json"
    where = bench.write_detail({"a": 1}, str(p))
    assert json.loads(p.read_text()) == {"a": 1} and where.endswith("detail.json")


def test_profile_cases_are_listed_in_the_help():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True,
                         text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0
    import bench
    for case in bench.CASES:
        assert case in out.stdout
