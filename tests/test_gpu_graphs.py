"""The calls capture into CUDA graphs: no call synchronizes or allocates, so a captured
sequence replays with results equal to the eager calls' bit for bit. Also two calls on
two streams at once (the library keeps no per-call state outside the stream)."""
import numpy as np
import pytest
import torch

import dense_linear_solvers_gb300 as bs
from gen import workloads as W
from gen.workloads import COL_MAJOR

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bs.lib()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _same_bits(x, r):
    """Bit-for-bit equality (a failed Cholesky system's factor holds NaN)."""
    if x.dtype in (torch.float32, torch.float64):
        it = torch.int32 if x.dtype == torch.float32 else torch.int64
        return torch.equal(x.view(it), r.view(it))
    return torch.equal(x, r)


def _lu_buffers(name, batch):
    d = W.make(name, batch)
    A0, B0 = _dev(d["A"]), _dev(d["B"])
    n = A0.shape[1]
    return d["workload"], A0, B0, torch.zeros((A0.shape[0], n), dtype=torch.int32,
                                                device="cuda"), \
        torch.zeros(A0.shape[0], dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("name", ["lu_f32_n16", "lu_f64_n64"])
def test_lu_graph_replay(name):
    w, A0, B0, ipiv, info = _lu_buffers(name, 1000)
    A, B = A0.clone(), B0.clone()
    bs.bs_getrf_getrs_batched(A, B, ipiv, info, w.layout)
    ref = [x.clone() for x in (A, B, ipiv, info)]
    Ag, Bg = A0.clone(), B0.clone()
    ipg, infg = torch.zeros_like(ipiv), torch.zeros_like(info)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bs.bs_getrf_getrs_batched(Ag, Bg, ipg, infg, w.layout, stream=s)
    for _ in range(2):
        Ag.copy_(A0)
        Bg.copy_(B0)
        g.replay()
        torch.cuda.synchronize()
        for x, r in zip((Ag, Bg, ipg, infg), ref):
            assert _same_bits(x, r)


def test_cholesky_and_bdsv_graph_replay():
    d = W.make("chol_f64_n32", 500)
    A0, B0 = _dev(d["A"]), _dev(d["B"])
    A, B = A0.clone(), B0.clone()
    info = torch.zeros(500, dtype=torch.int32, device="cuda")
    bs.bs_potrf_potrs_batched(A, B, info, COL_MAJOR, bs.BS_LOWER)
    e = W.make("bdsv_f64_32x8", 100)
    S0, X0 = _dev(e["strips"]), _dev(e["x"])
    S, X = S0.clone(), X0.clone()
    binfo = torch.zeros(100, dtype=torch.int32, device="cuda")
    bs.bs_bdsv_batched(S, X, binfo)
    ref = [x.clone() for x in (A, B, info, S, X, binfo)]
    Ag, Bg, Sg, Xg = A0.clone(), B0.clone(), S0.clone(), X0.clone()
    ig, big = torch.zeros_like(info), torch.zeros_like(binfo)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bs.bs_potrf_potrs_batched(Ag, Bg, ig, COL_MAJOR, bs.BS_LOWER, stream=s)
        bs.bs_bdsv_batched(Sg, Xg, big, stream=s)
    for _ in range(2):
        for dst, src in ((Ag, A0), (Bg, B0), (Sg, S0), (Xg, X0)):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        for x, r in zip((Ag, Bg, ig, Sg, Xg, big), ref):
            assert _same_bits(x, r)


def test_two_streams_at_once():
    w, A0, B0, ipiv, info = _lu_buffers("lu_f32_n16", 4000)
    d = W.make("chol_f64_n32", 3000)
    C0, D0 = _dev(d["A"]), _dev(d["B"])
    A, B, C, D = A0.clone(), B0.clone(), C0.clone(), D0.clone()
    cinfo = torch.zeros(3000, dtype=torch.int32, device="cuda")
    bs.bs_getrf_getrs_batched(A, B, ipiv, info, w.layout)
    bs.bs_potrf_potrs_batched(C, D, cinfo, COL_MAJOR, bs.BS_LOWER)
    torch.cuda.synchronize()
    ref = [x.clone() for x in (A, B, ipiv, info, C, D, cinfo)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    A2, B2, C2, D2 = A0.clone(), B0.clone(), C0.clone(), D0.clone()
    ip2, in2, ci2 = torch.zeros_like(ipiv), torch.zeros_like(info), torch.zeros_like(cinfo)
    torch.cuda.synchronize()
    bs.bs_getrf_getrs_batched(A2, B2, ip2, in2, w.layout, stream=s1)
    bs.bs_potrf_potrs_batched(C2, D2, ci2, COL_MAJOR, bs.BS_LOWER, stream=s2)
    torch.cuda.synchronize()
    for x, r in zip((A2, B2, ip2, in2, C2, D2, ci2), ref):
        assert _same_bits(x, r)


def test_cluster_interleaved_and_split_calls_graph_replay():
    """The cluster Cholesky (a launch with cluster dimensions), the interleaved two-rows LU
    and the row-major reading's two launches capture and replay like the eager calls."""
    rng = np.random.default_rng(5151)
    G = rng.standard_normal((6, 160, 160))
    C0 = _dev(G @ np.swapaxes(G, 1, 2) + 160 * np.eye(160))
    D0 = _dev(rng.standard_normal((6, 3, 160)))                     # column-major B
    w, A0, B0, _, _ = _lu_buffers("lu_f32_n16", 96)
    Ai0 = _dev(W.interleave(A0.cpu().numpy(), 32))
    Bi0 = _dev(W.interleave(B0.cpu().numpy(), 32))
    R0 = _dev(rng.standard_normal((40, 16, 16)).astype(np.float32))
    S0 = _dev(rng.standard_normal((40, 16, 9)).astype(np.float32))

    def calls(bufs, stream=None):
        C, D, ci, Ai, Bi, ipi, ini, R, S, ipr, inr = bufs
        bs.bs_potrf_potrs_batched(C, D, ci, COL_MAJOR, bs.BS_LOWER, stream=stream)
        bs.bs_getrf_getrs_batched_ex(Ai, Bi, ipi, ini, w.layout, interleave=32,
                                     shape=(96, 16, 4), stream=stream)
        bs.bs_getrf_getrs_batched_ex(R, S, ipr, inr, bs.BS_ROW_MAJOR, transposed_factor=1,
                                     stream=stream)

    def fresh():
        return [C0.clone(), D0.clone(), torch.zeros(6, dtype=torch.int32, device="cuda"),
                Ai0.clone(), Bi0.clone(), torch.zeros(96 * 16, dtype=torch.int32, device="cuda"),
                torch.zeros(96, dtype=torch.int32, device="cuda"), R0.clone(), S0.clone(),
                torch.zeros((40, 16), dtype=torch.int32, device="cuda"),
                torch.zeros(40, dtype=torch.int32, device="cuda")]

    ref = fresh()
    calls(ref)
    torch.cuda.synchronize()
    gb = fresh()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(gb, stream=s)
    src = fresh()
    for _ in range(2):
        for dst, x in zip(gb, src):
            dst.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        for x, r in zip(gb, ref):
            assert _same_bits(x, r)
