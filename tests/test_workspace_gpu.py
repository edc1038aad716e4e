"""A workspace given by the caller (sgemm_set_workspace) replaces the library's own:
torch's caching allocator supplies the memory, results match the oracle, a call
on a stream that never had a workspace of the library's can be captured into a
CUDA graph at once (nothing is allocated, so nothing must grow during capture),
a workspace that is too small is refused before anything is launched, and
setting None returns the stream to the library's own workspace."""
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


def _num_sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def _need(p, mode):
    return pg.sgemm_plan(p.transa, p.transb, p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc,
                         mode, num_sms=_num_sms())["workspace_bytes"]


def _check(p, mode, A, B, C, out):
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])
    assert res["ok"], (mode, res)


# Each case needs workspace: an lda that TMA cannot read in place (operand copy),
# a skinny-K product (split-K partial sums), and 3xTF32 on SM pairs (split operands).
CASES = [synth.Problem(600, 520, 1000, lda=601, alpha=1.5, beta=-0.5, dist="normal", seed=81),
         synth.Problem(256, 192, 8192, alpha=1.0, beta=0.5, dist="normal", seed=82)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", range(len(CASES)))
def test_torch_workspace_matches_oracle_and_captures_without_allocating(mode, case):
    p = CASES[case]
    need = _need(p, mode)
    assert need > 0
    A, B, C = synth.make(p)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    s = torch.cuda.Stream()  # a fresh stream: the library never sized a workspace for it
    ws = torch.empty(need // 4 + 1, dtype=torch.float32, device="cuda")
    try:
        pg.set_workspace(ws, stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
        g.replay()
        torch.cuda.synchronize()
        _check(p, mode, A, B, C, dC.cpu())
        # an ordinary call on the stream, and the same again after the workspace's
        # contents were overwritten: nothing in it has to survive between calls
        dC.copy_(C)
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
        s.synchronize()
        first = dC.clone()
        ws.fill_(float("nan"))
        dC.copy_(C)
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
        s.synchronize()
        assert torch.equal(first.view(torch.int32), dC.view(torch.int32))
    finally:
        pg.set_workspace(None, stream=s)
    # back on the library's own workspace
    dC.copy_(C)
    pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    torch.cuda.synchronize()
    _check(p, mode, A, B, C, dC.cpu())
    assert pg.device_status() == 0


@pytest.mark.parametrize("mode", MODES)
def test_workspace_too_small_is_refused_before_launching(mode):
    p = CASES[1]
    need = _need(p, mode)
    A, B, C = synth.make(p)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    s = torch.cuda.Stream()
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    try:
        pg.set_workspace(ws, nbytes=need - 256, stream=s)
        before = pg.launch_count()
        with pytest.raises(pg.SgemmError) as e:
            pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
        assert e.value.code == pg.SGEMM_ERR_WORKSPACE and str(need) in str(e.value)
        assert pg.launch_count() == before
        s.synchronize()
        assert torch.equal(dC.cpu().view(torch.int32), C.view(torch.int32))  # C untouched
    finally:
        pg.set_workspace(None, stream=s)


def test_host_entry_uses_the_given_workspace():
    """sgemm_host's product step takes its workspace from the caller's buffer too."""
    p = synth.Problem(700, 300, 5000, lda=703, ldb=5001, ldc=705, alpha=0.5, beta=1.5, dist="normal", seed=83)
    A, B, C = synth.make(p)
    s = torch.cuda.Stream()
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    Ch = C.clone().pin_memory()
    try:
        pg.set_workspace(ws, stream=s)
        pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, A.pin_memory(), p.lda, B.pin_memory(), p.ldb, p.beta, Ch,
                      p.ldc, "3xtf32", s)
    finally:
        pg.set_workspace(None, stream=s)
    _check(p, "3xtf32", A, B, C, Ch)


def test_set_workspace_refuses_memory_it_cannot_use():
    s = torch.cuda.Stream()
    host = torch.empty(4096, dtype=torch.float32).pin_memory()
    lib = pg.load_library()
    # pinned host memory is not device memory of the current device
    assert lib.sgemm_set_workspace(host.data_ptr(), 4096, s.cuda_stream) == -1
    dev = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    # more bytes than the allocation holds (the caching allocator rounds small
    # blocks up, but never by 1 GiB)
    assert lib.sgemm_set_workspace(dev.data_ptr(), 1 << 30, s.cuda_stream) == -2
    with pytest.raises(ValueError, match="exceeds"):
        pg.set_workspace(dev, nbytes=(1 << 20) + 1, stream=s)
