"""Throughput of the batched small dense solvers on GB300: one JSON line.

The headline workload is LU with partial pivoting + solve, FP32, n = 16, nrhs = 4,
batch 65536, row-major (A, B iid N(0,1)). One step = one call of the C ABI over the
whole batch: load, pivot search, interchange, multipliers, Schur update with the
folded forward solve, back substitution and the single store of every output.

Timing: W warm-up steps, then exactly K timed steps. Before every step the inputs are
restored from a pristine device copy and L2 is flushed by writing a 256 MiB buffer;
both happen outside the CUDA events, which bracket the solver launch alone on the
launching stream. ``value`` = systems per second over all ranks (weak scaling: every
rank solves its own batch). ``e2e`` times the same call with pinned host buffers, the
host-to-device copy of A and B and the device-to-host copy of every output inside the
timed region (the host-resident call: chunks copied in, solved and copied out on two
streams). ``cpu_baseline`` (N = 1) is the CPU oracle on this host's cores, with a
one-thread figure beside it; its last pass also gives ``verified``: 256 systems of the
last timed step compared bit for bit with the oracle's results on the same inputs.

``--impl reference`` times the CPU oracle as the reference arm (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from dense_linear_solvers_gb300 import costs  # noqa: E402
from gen import workloads as W  # noqa: E402

METRIC = "systems/sec per (n, dtype, nrhs); achieved HBM GB/s and % of roofline, 1 GB300"
HEADLINE = "lu_f32_n16"
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = {
    "lu_f32_n16": ["lu_rows2.cu", "common.cuh"],
    "lu_f64_n8": ["lu_reg.cuh", "common.cuh"],
    "lu_f64_n64": ["lu_cta.cu", "common.cuh"],
    "chol_f64_n32": ["chol_sys.cu", "common.cuh"],
    "bdsv_f64_32x8": ["bdsv.cu", "common.cuh"],
}
KERNEL_NAMES = {
    "lu_f32_n16": "lu_rows2_kernel", "lu_f64_n8": "lu_reg_kernel", "lu_f64_n64": "lu_cta_kernel",
    "chol_f64_n32": "chol_sys_kernel", "bdsv_f64_32x8": "bdsv_kernel",
}
REASONS = ["clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
           "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


def dtype_tag(dt) -> str:
    return {np.dtype(np.float32): "f32", np.dtype(np.float64): "f64"}[np.dtype(dt)]


def kernel_source_sha(name: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, "dense_linear_solvers_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def ncu_traffic(name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    kernel source that is built now."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(name)
    if not rec or rec.get("kernel_source_sha") != kernel_source_sha(name):
        return None
    return rec.get("dram_bytes_per_launch")


def workload_text(w) -> str:
    return f"{w.name}: {w.text}"


def config_of(w, batch: int, world: int) -> dict:
    """The workload of a bench line; the same dict for the GPU arm and the reference arm."""
    return {
        "workload": workload_text(w), "op": w.op, "n": w.n, "nrhs": w.nrhs,
        "batch_per_gpu": batch, "layout": "row-major" if w.layout == 0 else "column-major",
        "l2": "GPU arm: L2 flushed before every step (256 MiB write), inputs restored from a "
              "pristine device copy, both outside the CUDA events around the solver launch; "
              "reference arm: host memory, inputs regenerated once",
        "parallelism": f"batch shard x{world} (independent systems, no collective)",
    }


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              + ",".join(REASONS))

    def __init__(self, out_path: str | None):
        self.proc = None
        self.path = out_path or os.path.join("/tmp", f"bsolve_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, device_index: int) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9 or parts[0] != str(device_index):
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(REASONS, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name.split(".")[-1])
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def verify_sample(d: dict, fetch, ref, k: int = 256) -> dict:
    """Check after timing: k systems spread over the batch, the outputs of the last timed
    step against the CPU oracle's on the same pristine inputs, bit for bit. ref holds the
    oracle's outputs for the whole batch as it returns them: (LU, X, ipiv, info, near-tie
    step) for LU, (factor, X, info) for Cholesky and bdsv. fetch(idx) returns the timed
    outputs of systems idx as NumPy arrays in the call's order: (A, B, ipiv, info) for LU,
    (A, B, info) for Cholesky, (strips, x, info) for bdsv. LU systems whose pivot search
    met a near tie are counted apart (a legitimate rounding may pick the other row), and a
    failed system's factor is unspecified: its X and info are compared, its factor not."""
    w = d["workload"]
    idx = np.unique(np.linspace(0, d["batch"] - 1, min(k, d["batch"])).astype(np.int64))
    same = lambda x, y: np.array_equal(x, y, equal_nan=True)  # noqa: E731
    exempt = 0
    if w.op == "getrf_getrs":
        LU, X, ipiv, info, tie = (r[idx] for r in ref)
        got = fetch(idx)
        ok_all = []
        for j in range(len(idx)):
            if tie[j] >= 0:
                exempt += 1
                continue
            ok = same(got[1][j], X[j]) and same(got[2][j], ipiv[j]) and got[3][j] == info[j]
            if info[j] == 0:
                ok = ok and same(got[0][j], LU[j])
            ok_all.append(ok)
    else:
        F, X, info = (r[idx] for r in ref)
        got = fetch(idx)
        ok_all = [same(got[1][j], X[j]) and got[2][j] == info[j]
                  and (info[j] != 0 or same(got[0][j], F[j])) for j in range(len(idx))]
    return {"sampled_systems": int(len(idx)), "bit_identical": int(sum(ok_all)),
            "near_tie_exempt": exempt,
            "mismatches": int(len(ok_all) - sum(ok_all))}


# ------------------------------------------------------------------ GPU arm
class Problem:
    """Device buffers of one workload, a pristine copy and the solver call."""

    def __init__(self, name: str, batch: int | None, device):
        import torch
        import dense_linear_solvers_gb300 as bs
        self.bs, self.torch = bs, torch
        self.d = W.make(name, batch)
        self.w = self.d["workload"]
        self.batch = self.d["batch"]
        self.device = device
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        if self.w.op == "bdsv":
            self.inputs = [t(self.d["strips"]), t(self.d["x"])]
        else:
            self.inputs = [t(self.d["A"]), t(self.d["B"])]
        self.work = [x.clone() for x in self.inputs]
        n = self.w.n
        self.info = torch.zeros(self.batch, dtype=torch.int32, device=device)
        self.ipiv = (torch.zeros((self.batch, n), dtype=torch.int32, device=device)
                     if self.w.op == "getrf_getrs" else None)
        elem = np.dtype(self.w.dtype).itemsize
        self.bytes_per_sys, self.flops_per_sys = costs.per_system(
            self.w.op, n, self.w.nrhs, elem, self.w.nbr)

    def call(self, bufs=None, stream=None):
        bs = self.bs
        a, b = bufs if bufs is not None else self.work
        if self.w.op == "getrf_getrs":
            bs.bs_getrf_getrs_batched(a, b, self.ipiv, self.info, self.w.layout, stream)
        elif self.w.op == "potrf_potrs":
            bs.bs_potrf_potrs_batched(a, b, self.info, self.w.layout, bs.BS_LOWER, stream)
        else:
            bs.bs_bdsv_batched(a, b, self.info, stream)

    def restore(self):
        for dst, src in zip(self.work, self.inputs):
            dst.copy_(src)

    def outputs(self, idx):
        """Systems idx of the last call's buffers, gathered on the device and copied to
        the host, in the order verify_sample takes."""
        sel = self.torch.as_tensor(idx, dtype=self.torch.int64, device=self.device)
        outs = list(self.work) + ([self.ipiv] if self.ipiv is not None else []) + [self.info]
        return [x.index_select(0, sel).cpu().numpy() for x in outs]


# The factor / solve halves and the block-tridiagonal matvec, each measured on the inputs of
# the workload it serves (the solves on a factor made once before timing).
NEXT_ROWS = {
    "getrf_f32_n16": ("lu_f32_n16", "getrf"),
    "getrs_f32_n16": ("lu_f32_n16", "getrs"),
    "potrf_f64_n32": ("chol_f64_n32", "potrf"),
    "potrs_f64_n32": ("chol_f64_n32", "potrs"),
    "bdsv_factor_f64_32x8": ("bdsv_f64_32x8", "bdsv_factor"),
    "bdsv_solve_f64_32x8": ("bdsv_f64_32x8", "bdsv_solve"),
    "bdmv_f64_32x8": ("bdsv_f64_32x8", "bdmv"),
    "getrf_getrs_T_f32_n16": ("lu_f32_n16", "getrf_getrs_T"),
    "getrf_getrs_aosoa32_f32_n16": ("lu_f32_n16", "getrf_getrs_il"),
    "potrf_potrs_soa_f64_n32": ("chol_f64_n32", "potrf_potrs_il"),
    "potrf_potrs_f64_n256": ("chol_f64_n256", "potrf_potrs"),
}
# systems per block of the interleaved rows (None: the whole batch, SoA)
IL_WIDTH = {"getrf_getrs_aosoa32_f32_n16": 32, "potrf_potrs_soa_f64_n32": None}
KERNEL_SOURCES.update({
    "getrf_f32_n16": ["lu_rows2.cu", "common.cuh"], "getrs_f32_n16": ["solve.cu", "common.cuh"],
    "potrf_f64_n32": ["chol_sys.cu", "common.cuh"],
    "potrs_f64_n32": ["solve_lane.cu", "common.cuh"],
    "bdsv_factor_f64_32x8": ["bdsv.cu", "common.cuh"],
    "bdsv_solve_f64_32x8": ["bdsv.cu", "common.cuh"], "bdmv_f64_32x8": ["bdmv.cu", "common.cuh"],
    "getrf_getrs_T_f32_n16": ["solve.cu", "lu_rows2.cu", "common.cuh"],
    "getrf_getrs_aosoa32_f32_n16": ["lu_rows2.cu", "common.cuh"],
    "potrf_potrs_soa_f64_n32": ["chol_sys.cu", "common.cuh"],
    "potrf_potrs_f64_n256": ["chol_cluster.cu", "common.cuh"],
})
KERNEL_NAMES["potrf_potrs_f64_n256"] = "chol_cluster_kernel"


def interleave_device(x, w: int):
    """(batch, ...) device tensor -> the flat interleaved layout with w systems per block
    (w divides the batch here): element e of system s at (s // w) * w * size + e * w + s % w."""
    batch = x.shape[0]
    size = x[0].numel()
    return x.reshape(batch // w, w, size).transpose(1, 2).contiguous().reshape(-1)


class SplitProblem(Problem):
    """One of NEXT_ROWS: the inputs of its base workload, the operation alone."""

    def __init__(self, name: str, device, batch: int | None = None):
        import torch
        base, op = NEXT_ROWS[name]
        super().__init__(base, batch, device)
        self.op = op
        bs, w = self.bs, self.w
        a, b = self.inputs
        if op == "getrs":
            LU = a.clone()
            bs.bs_getrf_batched(LU, self.ipiv, self.info, w.layout)
            self.inputs, self.fixed = [b], (LU, self.ipiv)
        elif op == "potrs":
            L = a.clone()
            bs.bs_potrf_batched(L, self.info, w.layout)
            self.inputs, self.fixed = [b], (L,)
        elif op == "bdsv_solve":
            S = a.clone()
            bs.bs_bdsv_factor_batched(S, self.info)
            self.inputs, self.fixed = [b], (S,)
        elif op == "bdmv":
            self.y = torch.zeros_like(b)
            self.inputs, self.fixed = [], (a, b)
        elif op == "getrf_getrs_T":   # the fused call under TDLS's row-major reading
            self.inputs = [a, b]
        elif op == "potrf_potrs":   # the fused call on a workload of its own
            self.inputs = [a, b]
        elif op in ("getrf_getrs_il", "potrf_potrs_il"):   # interleaved batched layout
            self.ilv = IL_WIDTH[name] or self.batch
            if self.batch % self.ilv:
                raise ValueError(f"{name}: batch {self.batch} is not a whole number of blocks "
                                 f"of {self.ilv} systems")
            self.inputs = [interleave_device(a, self.ilv), interleave_device(b, self.ilv)]
            self.ipiv = self.ipiv.reshape(-1) if self.ipiv is not None else None
        else:   # the factor calls mutate A only
            self.inputs = [a]
        torch.cuda.synchronize()
        self.work = [x.clone() for x in self.inputs]
        elem = np.dtype(w.dtype).itemsize
        self.bytes_per_sys, self.flops_per_sys = costs.per_system(op, w.n, w.nrhs, elem, w.nbr)

    def call(self, bufs=None, stream=None):
        bs, w, op = self.bs, self.w, self.op
        if op == "getrf":
            bs.bs_getrf_batched(self.work[0], self.ipiv, self.info, w.layout, stream)
        elif op == "getrs":
            bs.bs_getrs_batched(self.fixed[0], self.fixed[1], self.work[0], w.layout, stream)
        elif op == "potrf":
            bs.bs_potrf_batched(self.work[0], self.info, w.layout, bs.BS_LOWER, stream)
        elif op == "potrs":
            bs.bs_potrs_batched(self.fixed[0], self.work[0], w.layout, bs.BS_LOWER, stream)
        elif op == "bdsv_factor":
            bs.bs_bdsv_factor_batched(self.work[0], self.info, stream)
        elif op == "bdsv_solve":
            bs.bs_bdsv_solve_batched(self.fixed[0], self.work[0], stream)
        elif op == "getrf_getrs_T":
            bs.bs_getrf_getrs_batched_ex(self.work[0], self.work[1], self.ipiv, self.info,
                                         w.layout, 1.0, bs.BS_CONTRACT_DEFAULT,
                                         transposed_factor=1, stream=stream)
        elif op == "getrf_getrs_il":
            bs.bs_getrf_getrs_batched_ex(self.work[0], self.work[1], self.ipiv, self.info,
                                         w.layout, interleave=self.ilv,
                                         shape=(self.batch, w.n, w.nrhs), stream=stream)
        elif op == "potrf_potrs":
            bs.bs_potrf_potrs_batched(self.work[0], self.work[1], self.info, w.layout,
                                      bs.BS_LOWER, stream)
        elif op == "potrf_potrs_il":
            bs.bs_potrf_potrs_batched_ex(self.work[0], self.work[1], self.info, w.layout,
                                         bs.BS_LOWER, interleave=self.ilv,
                                         shape=(self.batch, w.n, w.nrhs), stream=stream)
        else:
            bs.bs_bdmv_batched(self.fixed[0], self.fixed[1], self.y, stream)


def time_device(prob: Problem, steps: int, warmup: int, flush, min_warm_s: float = 0.0):
    torch = prob.torch
    stream = torch.cuda.current_stream()
    t0 = time.time()
    i = 0
    while i < warmup or time.time() - t0 < min_warm_s:
        prob.restore()
        flush.fill_(1.0)
        prob.call(stream=stream)
        i += 1
    torch.cuda.synchronize()
    times = []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for k in range(steps):
        prob.restore()
        flush.fill_(1.0)
        evs[k][0].record(stream)
        prob.call(stream=stream)
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    return times


def time_e2e(prob: Problem, steps: int, warmup: int, chunk: int):
    """The host-resident C-ABI call (bs_*_batched_host): pinned host arrays in, results
    back in them, the copies and the solves pipelined by chunks on two streams, all inside
    the timed region. The pristine inputs are restored into the host arrays between steps,
    outside it."""
    torch = prob.torch
    bs, w = prob.bs, prob.w
    host_in = [x.cpu().pin_memory() for x in prob.inputs]
    host_io = [torch.empty_like(x).pin_memory() for x in host_in]
    ipiv = (torch.empty(prob.ipiv.shape, dtype=torch.int32).pin_memory()
            if prob.ipiv is not None else None)
    info = torch.empty(prob.info.shape, dtype=torch.int32).pin_memory()
    outs = host_io + [x for x in (ipiv, info) if x is not None]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in outs)
    code = bs.BS_FP32 if w.dtype == np.float32 else bs.BS_FP64
    if w.op == "getrf_getrs":
        plan = bs.getrf_getrs_host_plan(code, w.n, w.nrhs, chunk)

        def call():
            bs.bs_getrf_getrs_batched_host(host_io[0], host_io[1], ipiv, info, w.layout,
                                            chunk=chunk, plan=plan, sync=False)
    elif w.op == "potrf_potrs":
        plan = bs.potrf_potrs_host_plan(code, w.n, w.nrhs, chunk)

        def call():
            bs.bs_potrf_potrs_batched_host(host_io[0], host_io[1], info, w.layout, bs.BS_LOWER,
                                            chunk=chunk, plan=plan, sync=False)
    else:
        plan = bs.bdsv_host_plan(code, w.nbr, w.n, chunk)

        def call():
            bs.bs_bdsv_batched_host(host_io[0], host_io[1], info, chunk=chunk, plan=plan,
                                    sync=False)
    s0, s1 = plan.streams
    times = []
    for k in range(warmup + steps):
        for dst, src in zip(host_io, host_in):
            dst.copy_(src)
        torch.cuda.synchronize()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(s0)
        s1.wait_event(e0)
        call()
        e1.record(s1)
        s0.wait_event(e1)
        e2.record(s0)
        e2.synchronize()
        if k >= warmup:
            times.append(e0.elapsed_time(e2))
    return times, h2d, d2h


def roofline(prob: Problem, ms: float, peaks: dict, name: str) -> dict:
    elem = np.dtype(prob.w.dtype).itemsize
    bytes_launch = prob.bytes_per_sys * prob.batch
    flops_launch = prob.flops_per_sys * prob.batch
    hbm = peaks.get("hbm_gbs")
    hbm_src = "measured" if hbm else "fallback"
    hbm = hbm or costs.HBM_FALLBACK_GBS
    alu = costs.alu_peak_tflops(elem)
    t_hbm = bytes_launch / (hbm * 1e9)
    t_alu = flops_launch / (alu * 1e12)
    traffic = ncu_traffic(name)
    if t_hbm >= t_alu:
        ach = bytes_launch / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": traffic,
                "peak_source": f"{hbm_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": bytes_launch}
    ach = flops_launch / (ms * 1e-3) / 1e12
    out = {"bound": "alu", "achieved": round(ach, 4), "peak": round(alu, 4), "unit": "TFLOP/s",
           "frac": round(ach / alu, 4), "traffic": traffic,
           "peak_source": (f"{'FP64' if elem == 8 else 'FP32'} FMA: 152 SMs x "
                           f"{costs.FP64_FMA_PER_CLK_PER_SM if elem == 8 else costs.FP32_FMA_PER_CLK_PER_SM}"
                           " FMA/clk x 2 flops x 2070 MHz (nominal)"),
           "algorithmic_flops_per_launch": flops_launch,
           "algorithmic_bytes_per_launch": bytes_launch,
           "achieved_gbs": round(bytes_launch / (ms * 1e-3) / 1e9, 1)}
    measured = peaks.get("fp64_tflops_measured" if elem == 8 else "fp32_tflops_measured")
    if measured:
        out["measured_peak"] = round(measured, 4)
        out["frac_of_measured"] = round(ach / measured, 4)
    return out


def alu_peaks(device_index: int, seconds: float = 0.3) -> dict:
    """The FP32 and FP64 FMA rates of this GPU, measured: independent FMA chains
    (csrc/fma_peak.cu, built into libbsolve_probe.so) on every SM, each launch sized to
    about `seconds`, the best of five timed with CUDA events, with the SM clock sampled
    while they run. The roofline's nominal FP64 figure is 152 SMs x 2 FMA/clk x 2 flops x
    2070 MHz; the measured one is reported beside it."""
    import ctypes
    import torch
    from dense_linear_solvers_gb300 import _build
    lib = ctypes.CDLL(_build.PROBE_LIB)
    lib.bs_probe_fma_launch.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    lib.bs_probe_fma_flops_per_thread_iter.restype = ctypes.c_int64
    fpt = lib.bs_probe_fma_flops_per_thread_iter()
    sms = torch.cuda.get_device_properties(device_index).multi_processor_count
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(None)
    sampler.start()
    out = {}
    for code, name, tdt in ((0, "fp32", torch.float32), (1, "fp64", torch.float64)):
        best_rate, shape = 0.0, None
        for bps, thr in ((4, 256), (8, 256)):
            blocks = sms * bps
            sink = torch.empty(blocks * thr, dtype=tdt, device=f"cuda:{device_index}")

            def run(iters):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if lib.bs_probe_fma_launch(code, blocks, thr, iters, sink.data_ptr(),
                                           stream.cuda_stream) != 0:
                    raise RuntimeError("FMA probe launch failed")
                e1.record(stream)
                e1.synchronize()
                return e0.elapsed_time(e1)

            iters = 64
            run(iters)
            t = run(iters)                       # calibrate the launch to about `seconds`
            iters = max(64, int(iters * seconds * 1e3 / max(t, 1e-3)))
            best = min(run(iters) for _ in range(5))
            rate = fpt * iters * blocks * thr / (best * 1e-3) / 1e12
            if rate > best_rate:
                best_rate, shape = rate, f"{bps} blocks/SM x {thr} threads, {iters} iterations"
            del sink
        out[f"{name}_tflops_measured"] = round(best_rate, 4)
        out[f"{name}_launch"] = shape
    clocks = sampler.stop(device_index)
    out["sm_mhz_median"] = clocks.get("sm_mhz")
    out["clock_reasons"] = clocks.get("reasons")
    out["how"] = ("independent FMA chains (8 per thread, csrc/fma_peak.cu) on every SM; best of "
                  "5 launches of about 0.3 s, CUDA events; 2 flops per FMA")
    return out


def cpu_baseline(name: str, batch: int | None, seconds: float, fetch=None):
    """The CPU oracle timed on this host's cores over the workload's batch, and on one
    thread over its first systems. With fetch (the timed GPU outputs of given systems),
    the oracle's results of the last pass also check a sample of those outputs
    (verify_sample). Returns (baseline, check or None)."""
    import oracle
    d = W.make(name, batch)
    w = d["workload"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    reps, t0 = 0, time.time()
    while True:
        if w.op == "getrf_getrs":
            res = oracle.getrf_getrs(d["A"], d["B"], w.layout, nthreads=cores)
        elif w.op == "potrf_potrs":
            res = oracle.potrf_potrs(d["A"], d["B"], w.layout, nthreads=cores)
        else:
            res = oracle.bdsv(d["strips"], d["x"], nthreads=cores)
        reps += 1
        el = time.time() - t0
        if el >= seconds:
            break
    out = {"value": round(reps * d["batch"] / el, 1), "unit": "systems/s", "cores": cores,
           "kind": "oracle",
           "sample": f"{reps} passes over the {d['batch']}-system batch of {name} "
                     f"({el:.1f} s wall, oracle built with g++ -O2, systems split over "
                     f"{cores} threads)"}
    # the same oracle on one thread, over the first systems of the batch (a few seconds)
    sub = min(d["batch"], 4096)
    arrays = (d["strips"][:sub], d["x"][:sub]) if w.op == "bdsv" else (d["A"][:sub], d["B"][:sub])
    reps1, t1 = 0, time.time()
    while True:
        if w.op == "getrf_getrs":
            oracle.getrf_getrs(*arrays, w.layout, nthreads=1)
        elif w.op == "potrf_potrs":
            oracle.potrf_potrs(*arrays, w.layout, nthreads=1)
        else:
            oracle.bdsv(*arrays, nthreads=1)
        reps1 += 1
        el1 = time.time() - t1
        if el1 >= min(3.0, seconds / 3):
            break
    out["one_core"] = {"value": round(reps1 * sub / el1, 1), "unit": "systems/s",
                       "sample": f"{reps1} passes over the first {sub} systems on 1 thread "
                                 f"({el1:.1f} s wall)"}
    check = None
    if fetch is not None:
        try:
            check = verify_sample(d, fetch, res)
        except Exception as e:  # reported in the line rather than lost with it
            check = {"error": repr(e)[:200]}
    return out, check


class Ranks:
    """Rank bookkeeping of a torchrun launch (one process per GPU, RANK / LOCAL_RANK /
    WORLD_SIZE / MASTER_* from the environment). The systems are independent, so ranks
    exchange nothing but a barrier and the max over ranks of their timings."""

    def __init__(self, backend: str):
        import torch.distributed as dist
        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.backend = backend
        if self.world > 1:
            dist.init_process_group(backend)

    def barrier(self) -> None:
        if self.world > 1:
            self.dist.barrier()

    def max(self, values, device=None) -> list:
        """Element-wise max over ranks of a list of floats (every rank gets it)."""
        if self.world == 1:
            return [float(v) for v in values]
        import torch
        t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                         device=device if device is not None else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return [float(v) for v in t.cpu()]

    def close(self) -> None:
        if self.world > 1:
            self.dist.destroy_process_group()


def whole_job_rate(batch_per_rank: int, world: int, ms_per_step: float) -> float:
    """Systems per second over all ranks: every rank solves its own batch in a step, and
    a step lasts as long as the slowest rank's."""
    return batch_per_rank * world / (ms_per_step * 1e-3)


def summary_lines(line: dict) -> list:
    """workload: ms per launch, systems/s, the roofline bound and fraction (of the measured
    FMA peak too, for an ALU-bound row) and the DRAM traffic over the algorithmic bytes."""
    rows = [(line["config"]["workload"].split(":")[0], line["ms_per_step"], line["value"],
             line["roofline"])]
    rows += [(k, v["ms_per_step"], v["systems_per_s"], v["roofline"])
             for k, v in line.get("workloads", {}).items() if k != rows[0][0]]
    rows += [(k, v["ms_per_step"], v["systems_per_s"], v["roofline"])
             for k, v in line.get("next_rows", {}).items()]
    out = []
    for name, ms, rate, rf in rows:
        alg = rf.get("algorithmic_bytes_per_launch")
        tr = (f"{rf['traffic'] / alg:.2f}x" if rf.get("traffic") and alg else "n/a")
        meas = f" ({rf['frac_of_measured']:.3f} of measured)" if "frac_of_measured" in rf else ""
        out.append(f"{name}: {ms:.4f} ms, {rate:.3g} sys/s, {rf['bound']} {rf['frac']:.3f}"
                   f"{meas}, traffic {tr}")
    return out


def run_native(args) -> None:
    import torch
    import dense_linear_solvers_gb300 as bs

    ranks = Ranks("nccl")
    world, rank, local = ranks.world, ranks.rank, ranks.local
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    bs.lib()
    peaks = measured_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    prob = Problem(args.workload, args.batch, dev)
    sampler = ClockSampler(os.path.join(args.out, "clocks_bench.csv") if args.out else None)
    sampler.start()
    ranks.barrier()
    torch.cuda.synchronize()
    times = time_device(prob, args.steps, args.warmup, flush, min_warm_s=args.warm_seconds)
    torch.cuda.synchronize()
    ranks.barrier()
    clocks = sampler.stop(local)
    ms = statistics.fmean(times)
    ranks.barrier()                   # the end-to-end steps start together on every rank
    e2e_times, h2d, d2h = time_e2e(prob, max(3, min(args.steps, 20)), 2, args.e2e_chunk)
    ranks.barrier()
    e2e_ms = statistics.fmean(e2e_times)
    ms, e2e_ms = ranks.max([ms, e2e_ms], device=dev)
    if rank != 0:
        ranks.close()
        return
    w = prob.w
    line = {
        "metric": METRIC,
        "value": round(whole_job_rate(prob.batch, world, ms), 1),
        "unit": "systems/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_tag(w.dtype),
        "data": "synthetic (seeded NumPy draws with the workload's distributions)",
        "config": config_of(w, prob.batch, world),
        "ms_per_step_min": round(min(times), 5),
        "ms_per_step_median": round(statistics.median(times), 5),
        "roofline": roofline(prob, ms, peaks, args.workload),
        "e2e": {"value": round(whole_job_rate(prob.batch, world, e2e_ms), 1), "unit": "systems/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "gpu_launches_per_step": -(-prob.batch // args.e2e_chunk),
                "call": "bs_*_batched_host: pinned host arrays, chunks of "
                        f"{args.e2e_chunk} systems on two streams (copies overlap solves)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if world == 1:   # the CPU leg, which also checks a sample of the last timed step
        line["cpu_baseline"], line["verified"] = cpu_baseline(
            args.workload, args.batch, args.cpu_seconds, fetch=prob.outputs)
    if not args.headline_only:
        line["alu_peaks"] = alu_peaks(local)
        peaks = dict(peaks, **{k: v for k, v in line["alu_peaks"].items()
                               if k.endswith("_tflops_measured")})
        extra = {}
        for name in W.WORKLOADS:
            if name == args.workload:
                continue
            p = Problem(name, None, dev)
            tt = time_device(p, min(args.steps, 10), 2, flush)
            m = statistics.fmean(tt)
            extra[name] = {"systems_per_s": round(p.batch / (m * 1e-3), 1), "ms_per_step": round(m, 4),
                           "batch": p.batch, "roofline": roofline(p, m, peaks, name)}
            del p
        extra[args.workload] = {"systems_per_s": line["value"] / world, "ms_per_step": line["ms_per_step"],
                                "batch": prob.batch, "roofline": line["roofline"]}
        line["workloads"] = extra
        nxt = {}
        for name in NEXT_ROWS:
            p = SplitProblem(name, dev)
            tt = time_device(p, min(args.steps, 10), 3, flush)
            m = statistics.fmean(tt)
            nxt[name] = {"op": p.op, "on": p.w.name, "systems_per_s": round(p.batch / (m * 1e-3), 1),
                         "ms_per_step": round(m, 4), "batch": p.batch,
                         "roofline": roofline(p, m, peaks, name)}
            del p
        line["next_rows"] = nxt
        # one short entry per row at the end of the line, where a truncated tail still holds it
        line["summary"] = summary_lines(line)
    print(json.dumps(line), flush=True)
    ranks.close()


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    d = W.make(args.workload, args.batch)
    w = d["workload"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()

    def one():
        if w.op == "getrf_getrs":
            oracle.getrf_getrs(d["A"], d["B"], w.layout, nthreads=cores)
        elif w.op == "potrf_potrs":
            oracle.potrf_potrs(d["A"], d["B"], w.layout, nthreads=cores)
        else:
            oracle.bdsv(d["strips"], d["x"], nthreads=cores)

    for _ in range(args.warmup):
        one()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        times.append((time.perf_counter() - t0) * 1e3)
    ms = statistics.fmean(times)
    value = round(d["batch"] / (ms * 1e-3), 1)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "systems/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_tag(w.dtype),
        "data": "synthetic (seeded NumPy draws with the workload's distributions)",
        "config": config_of(w, d["batch"], int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "systems/s", "cores": cores, "kind": "oracle",
                         "sample": f"the whole {d['batch']}-system batch per step on {cores} "
                                   f"host threads (sequential C++ oracle, g++ -O2)"},
        "e2e": {"value": value, "unit": "systems/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), default=HEADLINE)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (profiling runs on a smaller case)")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the per-workload table of the other four workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--warm-seconds", type=float, default=1.0,
                    help="keep warming up for at least this long (lets the clock sampler "
                         "see the GPU under this load)")
    ap.add_argument("--e2e-chunk", type=int, default=16384,
                    help="systems per chunk of the host-resident call timed as e2e")
    ap.add_argument("--out", default=None, help="folder for the clock samples")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "native":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
