"""Host logic of the multi-rank benchmark on CPU (gloo, world size 2).

The systems are independent, so the only exchange between ranks is a barrier and the
max over ranks of the step timings; the whole-job rate counts every rank's batch.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    r = bench.Ranks("gloo")
    r.barrier()
    got = r.max([1.0 + rank, 10.0 - rank])
    out.put((rank, got))
    r.close()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]


def test_single_rank_needs_no_process_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    r = bench.Ranks("gloo")
    assert (r.world, r.rank) == (1, 0)
    assert r.max([3.5]) == [3.5]
    r.close()


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(65536, 1, 1.0) == pytest.approx(65536e3)
    assert bench.whole_job_rate(65536, 4, 2.0) == pytest.approx(4 * 65536 / 2e-3)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--batch", "256"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "systems/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["n_gpus"] == 2 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("lu_f32_n16")
    # the GPU arm's config for the same workload, batch and world size, key for key
    from gen import workloads as W
    assert d["config"] == bench.config_of(W.WORKLOADS["lu_f32_n16"], 256, 2)
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]


def test_cpu_baseline_reports_all_cores_and_one_core():
    r, check = bench.cpu_baseline("lu_f64_n8", 256, 0.3)
    assert check is None
    assert r["kind"] == "oracle" and r["unit"] == "systems/s" and r["value"] > 0
    assert r["cores"] >= 1 and "256-system batch" in r["sample"]
    assert r["one_core"]["value"] > 0 and "on 1 thread" in r["one_core"]["sample"]


def _oracle_outputs(name, batch):
    import oracle
    from gen import workloads as W
    d = W.make(name, batch)
    w = d["workload"]
    if w.op == "getrf_getrs":
        ref = oracle.getrf_getrs(d["A"], d["B"], w.layout)
        return d, ref, list(ref[:4])
    if w.op == "potrf_potrs":
        ref = oracle.potrf_potrs(d["A"], d["B"], w.layout)
    else:
        ref = oracle.bdsv(d["strips"], d["x"])
    return d, ref, list(ref)


@pytest.mark.parametrize("name,batch", [("lu_f64_n8", 1024), ("lu_f32_n16", 700),
                                        ("chol_f64_n32", 500), ("bdsv_f64_32x8", 40)])
def test_post_timing_check_accepts_the_oracle_and_flags_one_ulp(name, batch):
    """The bench's check after timing: outputs equal to the oracle's pass (planted
    failures included); one output one ulp off in one sampled system is one mismatch."""
    import numpy as np
    d, ref, outs = _oracle_outputs(name, batch)
    fetch = lambda idx: [o[idx] for o in outs]  # noqa: E731
    k = min(64, batch)
    r = bench.verify_sample(d, fetch, ref, k=64)
    assert r["mismatches"] == 0 and r["sampled_systems"] == k
    assert r["bit_identical"] + r["near_tie_exempt"] == k
    idx = np.unique(np.linspace(0, batch - 1, k).astype(np.int64))
    j = next(int(i) for i in idx if outs[-1][i] == 0)          # a system that did not fail
    X = outs[1].copy()
    flat = X[j].reshape(-1)
    flat[0] = np.nextafter(flat[0], np.inf)
    bad = [outs[0], X] + outs[2:]
    r = bench.verify_sample(d, lambda ix: [o[ix] for o in bad], ref, k=64)
    assert r["mismatches"] == 1 or (r["near_tie_exempt"] > 0 and r["mismatches"] <= 1)


def test_problem_outputs_gathers_the_sampled_systems():
    """Problem.outputs gathers systems idx of every output buffer (here CPU tensors
    holding the oracle's results) in the order the check takes."""
    import torch
    d, ref, outs = _oracle_outputs("lu_f64_n8", 1024)
    prob = bench.Problem("lu_f64_n8", None, torch.device("cpu"))
    for dst, src in zip(prob.work + [prob.ipiv, prob.info], outs):
        dst.copy_(torch.from_numpy(src))
    r = bench.verify_sample(prob.d, prob.outputs, ref, k=256)
    assert r == {"sampled_systems": 256, "bit_identical": 256 - r["near_tie_exempt"],
                 "near_tie_exempt": r["near_tie_exempt"], "mismatches": 0}
    import numpy as np
    j = int(np.unique(np.linspace(0, 1023, 256).astype(np.int64))[100])   # a sampled system
    prob.info[j] = 7
    assert bench.verify_sample(prob.d, prob.outputs, ref, k=256)["mismatches"] == 1
    # the CPU leg runs the check on its own last pass over the same batch
    base, check = bench.cpu_baseline("lu_f64_n8", None, 0.2, fetch=prob.outputs)
    assert base["value"] > 0 and check["sampled_systems"] == 256 and check["mismatches"] == 1


def test_bench_interleave_matches_the_generator():
    """bench.interleave_device (torch, on the timed device) lays systems out exactly as
    gen.workloads.interleave does for the parity tests (whole blocks)."""
    import numpy as np
    import torch
    from gen import workloads as W
    rng = np.random.default_rng(5)
    S = rng.standard_normal((96, 16, 4)).astype(np.float32)
    for w in (1, 32, 96):
        got = bench.interleave_device(torch.from_numpy(S), w).numpy()
        assert np.array_equal(got, W.interleave(S, w)), w


def test_traffic_records_point_at_committed_summaries():
    """Every benchmarked row names the kernel sources its traffic record is keyed on, and
    each record in profiles/ncu_traffic.json points at a committed ncu summary."""
    rows = set(bench.KERNEL_SOURCES)
    assert set(bench.W.WORKLOADS) <= rows and set(bench.NEXT_ROWS) <= rows
    for name, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "dense_linear_solvers_gb300", "csrc", f)), f
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as fh:
        records = json.load(fh)
    for name, rec in records.items():
        assert name in rows, name
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), rec["profile"]
        assert rec["dram_bytes_per_launch"] > 0 and rec["captured_batch"] > 0


def test_summary_lines_cover_every_row():
    rf_hbm = {"bound": "hbm", "frac": 0.5, "traffic": 200.0, "algorithmic_bytes_per_launch": 100.0}
    rf_alu = {"bound": "alu", "frac": 0.6, "traffic": None, "algorithmic_bytes_per_launch": 10.0,
              "frac_of_measured": 0.63}
    line = {"config": {"workload": "lu_f32_n16: LU ..."}, "ms_per_step": 0.05, "value": 1e9,
            "roofline": rf_hbm,
            "workloads": {"lu_f32_n16": {}, "chol_f64_n32": {"ms_per_step": 4.0,
                                                             "systems_per_s": 6e7,
                                                             "roofline": rf_alu}},
            "next_rows": {"getrs_f32_n16": {"ms_per_step": 0.03, "systems_per_s": 2e9,
                                            "roofline": rf_hbm}}}
    out = bench.summary_lines(line)
    assert [o.split(":")[0] for o in out] == ["lu_f32_n16", "chol_f64_n32", "getrs_f32_n16"]
    assert "hbm 0.500" in out[0] and "traffic 2.00x" in out[0]
    assert "alu 0.600 (0.630 of measured)" in out[1] and "traffic n/a" in out[1]
