"""C with more than 2^31 elements (50000 x 45000, 9 GB): in its last columns the
offset j * ldc + i of an entry exceeds the int32 range and its byte offset 2^33,
so every epilogue's index arithmetic and the C tensor maps' coordinates are
exercised where a 32-bit product would wrap.  K = 8 keeps the arithmetic short.
Aligned ldc (TMA stores of C in FFMA) and ldc with a 3-row gap (thread stores);
sampled entries (the corners, the last row and column, tile edges) against the
oracle, the ld gap and a canary run after C untouched.  Only A and B are drawn
on the host (the same seeded draws as the full problem: A, then B); C lives on
the device only, filled with NaN (beta = 0 never reads it)."""
import numpy as np
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu
M, N, K = 50000, 45000, 8
CANARY = 64


@pytest.fixture(scope="module")
def big_c():
    need = (M + 3) * N * 4 + (2 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip("needs %d bytes of free device memory, %d free" % (need, free))
    buf = torch.empty((M + 3) * N + CANARY, dtype=torch.float32, device="cuda")
    yield buf
    del buf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["ffma", "tf32", "3xtf32"])
@pytest.mark.parametrize("pad", [0, 3])
def test_c_beyond_2_31_elements(big_c, mode, pad):
    ldc = M + pad
    assert (N - 1) * ldc + M - 1 >= 2 ** 31
    p = synth.Problem(M, N, K, ldc=ldc, alpha=1.5, beta=0.0, dist="normal", seed=41)
    gen = torch.Generator().manual_seed(p.seed)
    A = synth.storage(*p.a_dims(), p.lda, p.dist, gen)
    B = synth.storage(*p.b_dims(), p.ldb, p.dist, gen)
    dA, dB = A.cuda(), B.cuda()
    C = big_c[: ldc * N]
    big_c.view(torch.int32).fill_(synth.NAN_BITS)
    big_c[ldc * N:].view(torch.int32).fill_(H.CANARY_BITS)
    pg.sgemm("N", "N", M, N, K, p.alpha, dA, p.lda, dB, p.ldb, p.beta, C, ldc, mode)
    torch.cuda.synchronize()
    assert pg.device_status() == 0

    ii, jj = synth.sample_entries(M, N, count=4096, seed=7)
    idx = torch.from_numpy(ii + jj * ldc).cuda()
    got = C[idx].cpu().numpy().astype(np.float64)
    cref, den = H.reference_entries(p, A, B, None, ii, jj)
    res = oracle.check(got, cref, den, oracle.TOL[mode])
    assert res["ok"], res
    assert torch.all(big_c[ldc * N:].view(torch.int32) == H.CANARY_BITS)
    if pad:
        gap = torch.arange(M, ldc, device="cuda")
        cols = torch.tensor([0, N // 2, N - 2, N - 1], device="cuda")
        gap_idx = (gap[None, :] + cols[:, None] * ldc).reshape(-1)
        assert torch.all(C[gap_idx].view(torch.int32) == synth.NAN_BITS)
