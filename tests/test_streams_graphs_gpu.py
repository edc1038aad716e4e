"""Streams and CUDA graphs: the library's launches are stream-ordered and
capturable once the stream's workspace has been sized by an ordinary call; a call
that would have to grow the workspace during capture is refused with
SGEMM_ERR_CAPTURE; concurrent calls on different streams use different
workspaces and both stay correct; sgemm_host_async calls on several streams
overlap and each equals the synchronous sgemm_host result bit for bit."""
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu
MODES = ("ffma", "tf32", "3xtf32")


@pytest.fixture(autouse=True)
def _plain_plan():
    pg.load_library()
    pg.force_plan(0, 0)
    yield
    pg.force_plan(0, 0)


def _check(p, mode, A, B, C, out):
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])
    assert res["ok"], (mode, res)


@pytest.mark.parametrize("mode", MODES)
def test_captured_call_replays_on_new_data(mode):
    # split-K shape (workspace for partial sums) plus, for 3xTF32, the split operands
    p = synth.Problem(256, 192, 8192, alpha=1.0, beta=0.5, dist="normal", seed=41)
    A, B, C = synth.make(p)
    s = torch.cuda.Stream()
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    with torch.cuda.stream(s):
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)  # sizes workspace
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    A2, B2, C2 = synth.make(p.with_(seed=42))
    dA.copy_(A2)
    dB.copy_(B2)
    dC.copy_(C2)
    g.replay()
    torch.cuda.synchronize()
    _check(p, mode, A2, B2, C2, dC.cpu())
    dC.copy_(C2)
    g.replay()
    torch.cuda.synchronize()
    _check(p, mode, A2, B2, C2, dC.cpu())
    assert pg.device_status() == 0


def test_workspace_growth_during_capture_is_refused():
    p = synth.Problem(256, 192, 8192, dist="normal", seed=43)
    A, B, C = synth.make(p)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    s = torch.cuda.Stream()  # fresh stream: no workspace yet
    g = torch.cuda.CUDAGraph()
    with pytest.raises(pg.SgemmError) as e:
        with torch.cuda.graph(g, stream=s):
            pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, "3xtf32", s)
    assert e.value.code == 7  # SGEMM_ERR_CAPTURE
    torch.cuda.synchronize()
    # the stream is usable afterwards
    pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, "3xtf32", s)
    torch.cuda.synchronize()
    _check(p, "3xtf32", A, B, C, dC.cpu())


@pytest.mark.parametrize("mode", MODES)
def test_two_streams_run_concurrently(mode):
    p1 = synth.Problem(1024, 768, 4096, alpha=1.0, beta=0.0, dist="normal", seed=51)
    p2 = synth.Problem(640, 1280, 2048, alpha=2.0, beta=1.0, dist="normal", seed=52)
    data = [synth.make(p) for p in (p1, p2)]
    dev = [(A.cuda(), B.cuda(), C.cuda()) for A, B, C in data]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for p, (dA, dB, dC), (A, B, C), s in zip((p1, p2), dev, data, streams):
            with torch.cuda.stream(s):
                dC.copy_(C)  # ordered before the product on the same stream
            pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    torch.cuda.synchronize()
    for p, (dA, dB, dC), (A, B, C) in zip((p1, p2), dev, data):
        _check(p, mode, A, B, C, dC.cpu())


def _pinned_problem(p):
    A, B, C = synth.make(p)
    return A.pin_memory(), B.pin_memory(), C.pin_memory(), C


@pytest.mark.parametrize("same_stream", [False, True])
def test_host_async_calls_overlap_and_match_sync(same_stream):
    # one pipelined (n >= 4096: internal copy streams) and two single-slab problems
    probs = [(synth.Problem(1024, 4608, 640, alpha=1.0, beta=0.75, dist="normal", seed=61), "ffma"),
             (synth.Problem(700, 900, 1000, alpha=-0.5, beta=0.0, dist="normal", seed=62), "tf32"),
             (synth.Problem(2048, 4096, 256, alpha=1.5, beta=1.0, dist="normal", seed=63), "3xtf32")]
    data = [(_pinned_problem(p), p, mode) for p, mode in probs]
    streams = [torch.cuda.Stream()] * 3 if same_stream else [torch.cuda.Stream() for _ in probs]
    outs = []
    for ((A, B, Ch, C), p, mode), s in zip(data, streams):
        out = Ch.clone().pin_memory()
        pg.sgemm_host_async("N", "N", p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, out, p.ldc, mode, s)
        outs.append(out)
    for s in streams:
        s.synchronize()
    for ((A, B, Ch, C), p, mode), out in zip(data, outs):
        ref = Ch.clone().pin_memory()
        pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, ref, p.ldc, mode)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), (p, mode)
        _check(p, mode, A, B, C, out)
    assert pg.device_status() == 0


@pytest.mark.parametrize("mode", ("ffma", "tf32", "3xtf32"))
def test_captured_last_wave_split_replays(mode):
    """A product that splits its last wave along K (arrival counters zeroed by a
    memset before the kernel) captured into a graph: every replay starts from
    zeroed counters and gives the same bits."""
    p = synth.Problem(2500, 2000, 1000, alpha=1.0, beta=0.5, dist="normal", seed=71)
    plan = pg.sgemm_plan("N", "N", p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
    assert plan["tail_split"] > 1, plan
    A, B, C = synth.make(p)
    s = torch.cuda.Stream()
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    with torch.cuda.stream(s):
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    s.synchronize()
    first = dC.cpu()
    _check(p, mode, A, B, C, first)
    g = torch.cuda.CUDAGraph()
    dC.copy_(C)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    for _ in range(3):
        dC.copy_(C)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dC.cpu().view(torch.int32), first.view(torch.int32))
    assert pg.device_status() == 0


@pytest.mark.parametrize("mode,mnk,trans", [("ffma", (1000, 1300, 4000), "NN"), ("ffma", (1500, 1300, 6000), "TT"),
                                            ("3xtf32", (4096, 128, 8192), "NN"), ("3xtf32", (120, 5000, 9000), "TN")])
def test_stream_k_captured_and_replayed(mode, mnk, trans):
    """Stream-K calls (FFMA, and 3xTF32 on single SMs; with transposed operands the
    FFMA path copies them first) are plain stream-ordered launches: once the
    stream's workspace is sized they can be captured into a CUDA graph and
    replayed on new data, matching the oracle each time."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, transa=trans[0], transb=trans[1], alpha=1.25, beta=-0.5, dist="normal", seed=131)
    plan = pg.sgemm_plan(p.transa, p.transb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
    assert plan["sk_ctas"] > 0, plan
    A, B, C = synth.make(p)
    s = torch.cuda.Stream()
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    with torch.cuda.stream(s):
        pg.sgemm(p.transa, p.transb, m, n, k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pg.sgemm(p.transa, p.transb, m, n, k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    for seed in (132, 133):
        A2, B2, C2 = synth.make(p.with_(seed=seed))
        dA.copy_(A2)
        dB.copy_(B2)
        dC.copy_(C2)
        g.replay()
        torch.cuda.synchronize()
        ii, jj = synth.sample_entries(p.m, p.n, count=4096, seed=seed)
        cref, den = H.reference_entries(p, A2, B2, C2, ii, jj)
        res = oracle.check(H.gather(p, dC.cpu(), ii, jj), cref, den, oracle.TOL[mode])
        assert res["ok"], (mode, seed, res)
    assert pg.device_status() == 0
