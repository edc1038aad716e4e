"""Calls from several host threads at once, each thread on its own stream (the
header allows this).  Four threads repeatedly run a mix of plans that each
need the per-stream workspace in a different way: a K split with its
reduction, FFMA and tensor-core stream-K with their partial blocks, 3xTF32 on
SM pairs with both split pre-passes, 3xTF32 on single SMs with B split by a
pre-pass, operand copies for a misaligned lda, and the host-array entry with
its internal copy streams.  Every result must be bitwise equal to the same
call made alone beforehand (the library is deterministic), and that result is
held to the oracle on sampled entries.  One thread also makes an invalid call:
its error string is its own, and the other threads' calls are unaffected."""
import threading

import numpy as np
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu

CASES = [
    (128, 128, 20000, "ffma", 0),      # K split, reduction
    (2048, 2048, 2048, "ffma", 0),     # FFMA stream-K
    (2048, 64, 4096, "3xtf32", 0),     # single SM, B split by a pre-pass, K split
    (1536, 1536, 1024, "3xtf32", 0),   # SM pairs, both operands split
    (333, 444, 555, "ffma", 1),        # lda misaligned: A copied
    (4096, 128, 8192, "3xtf32", 0),    # tensor-core stream-K
    (700, 900, 3000, "tf32", 0),
    (1000, 1300, 4000, "ffma", 0),     # FFMA stream-K, ragged
]


def _problem(idx):
    m, n, k, mode, pad = CASES[idx]
    p = synth.Problem(m, n, k, alpha=0.75, beta=0.5, dist="normal", seed=600 + idx)
    return p.with_(lda=p.lda + pad), mode


@pytest.fixture(scope="module")
def prepared():
    pg.load_library()
    out = []
    for idx in range(len(CASES)):
        p, mode = _problem(idx)
        A, B, C = synth.make(p)
        dA, dB, dC0 = A.cuda(), B.cuda(), C.cuda()
        dC = dC0.clone()
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode)
        torch.cuda.synchronize()
        ref = dC.cpu()
        ii, jj = synth.sample_entries(p.m, p.n, count=1024, seed=3)
        cref, den = H.reference_entries(p, A, B, C, ii, jj)
        res = oracle.check(H.gather(p, ref, ii, jj), cref, den, oracle.TOL[mode])
        assert res["ok"], (CASES[idx], res)
        out.append((p, mode, dA, dB, dC0, ref))
    assert pg.device_status() == 0
    return out


def test_calls_from_four_threads_match_the_lone_calls(prepared):
    n_threads, rounds = 4, 3
    start = threading.Barrier(n_threads)
    failures = []

    def worker(t):
        try:
            dev_stream = torch.cuda.Stream()
            mine = [(idx, prepared[idx]) for idx in range(len(CASES)) if idx % n_threads == t or (idx + 1) % n_threads == t]
            bufs = {idx: item[4].clone() for idx, item in mine}
            torch.cuda.synchronize()
            start.wait()
            for r in range(rounds):
                for idx, (p, mode, dA, dB, dC0, ref) in mine:
                    C = bufs[idx]
                    with torch.cuda.stream(dev_stream):
                        C.copy_(dC0)
                    pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, C, p.ldc, mode,
                             dev_stream)
                    dev_stream.synchronize()
                    if not torch.equal(C.cpu().view(torch.int32), ref.view(torch.int32)):
                        failures.append(("device", t, r, CASES[idx]))
                # the host-array entry on this thread's stream
                p, mode, dA, dB, dC0, ref = prepared[t]
                hA, hB = dA.cpu().pin_memory(), dB.cpu().pin_memory()
                hC = dC0.cpu().pin_memory()
                pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, hA, p.lda, hB, p.ldb, p.beta, hC, p.ldc, mode,
                              dev_stream)
                if not torch.equal(hC.view(torch.int32), ref.view(torch.int32)):
                    failures.append(("host", t, r, CASES[t]))
                if t == 0:
                    lib = pg.load_library()
                    rc = lib.sgemm(b"N", b"Q", 1, 1, 1, 1.0, None, 1, None, 1, 0.0, None, 1, 0, None)
                    if rc != -2 or "argument 2" not in pg.last_error():
                        failures.append(("error string", rc, pg.last_error()))
        except Exception as exc:  # noqa: BLE001 -- reported below with the thread number
            failures.append(("exception", t, repr(exc)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=600)
    assert not any(th.is_alive() for th in threads), "a thread did not finish"
    assert not failures, failures
    assert pg.device_status() == 0
