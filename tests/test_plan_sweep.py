"""Structural invariants of the planner over a seeded sweep of shapes (CPU only).

The example-based planner tests pin particular choices; this sweep checks what
must hold for every call, whatever the planner picks: the tiles and K blocks
cover the product exactly, no K slice is empty, the kernel fits the SM's
shared memory and thread limits, the launch count and workspace agree with the
plan's own preparation steps, and the operand copies keep every element
(their leading dimension covers the stored rows).  Shapes mix tile multiples,
ragged sizes, skinny and tall products, transposed operands, misaligned
pointers and leading dimensions, and several SM counts.
"""
import numpy as np
import pytest

import precision_gemm_gb300 as pg
from precision_gemm_gb300 import build as pgbuild

SMEM_PER_CTA = 227 * 1024   # largest dynamic shared memory a CTA may request
SMEM_PER_SM = 228 * 1024    # shared memory of one SM, shared by its resident CTAs
THREADS_PER_SM = 2048


@pytest.fixture(scope="module")
def lib():
    pgbuild.build()
    return pg.load_library()


def _cdiv(a, b):
    return -(-a // b)


def _round_up(x, q):
    return _cdiv(x, q) * q


def _shapes(rng, count):
    dims = [1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 777, 1000, 1500, 3000, 4096, 8192, 16384]
    ks = [1, 3, 8, 31, 32, 33, 64, 255, 777, 2048, 4096, 8192, 65536, 262144]
    out = []
    for _ in range(count):
        m = int(rng.choice(dims)) if rng.random() < 0.6 else int(rng.integers(1, 20000))
        n = int(rng.choice(dims)) if rng.random() < 0.6 else int(rng.integers(1, 20000))
        k = int(rng.choice(ks)) if rng.random() < 0.6 else int(rng.integers(1, 40000))
        out.append((m, n, k))
    # the acceptance shapes themselves
    out += [(256, 256, 256), (1024, 1024, 1024), (4096, 4096, 4096), (3000, 1500, 777), (8192, 8192, 8192),
            (16384, 16384, 16384), (16384, 16384, 64), (128, 128, 262144), (8192, 64, 8192)]
    return out


def _check(p, m, n, k, mode, transa, transb, lda, ldb, aligned, sms):
    name = p["kernel_name"]
    tc = mode != "ffma"
    where = "%s %s%s m=%d n=%d k=%d lda=%d ldb=%d aligned=%s sms=%d" % (mode, transa, transb, m, n, k, lda, ldb,
                                                                         aligned, sms)
    # kernel family and tile shape
    assert name == ("ffma" if not tc else ("tc2" if p["bm"] == 256 else "tc")), where
    assert p["mode"] == {"ffma": 0, "tf32": 1, "3xtf32": 2}[mode], where
    if name == "tc2":
        assert m > 128 and p["bn"] in (128, 256, 512), where
    else:
        assert p["bm"] == 128, where
    assert p["bn"] in (64, 128, 256, 512), where
    if p["bn"] == 512:
        assert mode == "tf32" and name == "tc2", where
        assert p["tail_split"] == 1, where  # a 256 x 512 tile's last wave is never split
    # the tiles and the K blocks cover the product exactly
    assert p["tiles_m"] == _cdiv(m, p["bm"]) and p["tiles_n"] == _cdiv(n, p["bn"]), where
    assert p["k_blocks"] == _cdiv(k, p["bk"]), where
    # K slices: at least one, none empty, together covering every K block
    s, per = p["split_k"], p["k_blocks_per_split"]
    assert 1 <= s <= p["k_blocks"], where
    assert s * per >= p["k_blocks"] and (s - 1) * per < p["k_blocks"], where
    # last-wave split: only without split-K, on the kernels that have it, 2..4 (SM pairs) or 2..8 (FFMA)
    # slices of >= 8 K blocks
    if p["tail_split"] > 1:
        assert s == 1 and name in ("tc2", "ffma"), where
        assert 2 <= p["tail_split"] <= (4 if name == "tc2" else 8) and p["tail_split"] * 8 <= p["k_blocks"], where
        tiles = p["tiles_m"] * p["tiles_n"]
        capacity = max(sms // 2, 1) if name == "tc2" else sms * p["ctas_per_sm"]
        assert p["tail_tiles"] == tiles % capacity and 2 * p["tail_tiles"] <= capacity, where
        assert tiles >= capacity, where
    else:
        assert p["tail_split"] == 1, where
    # stream-K: only where the tiles (with their K slices) leave over a tenth of one
    # wave's CTA slots idle and every slot gets at least 4 (FFMA) or 32 (3xTF32)
    # k-blocks; all slots run
    if p["sk_ctas"] > 0:  # FFMA, or 3xTF32 on single SMs
        tiles = p["tiles_m"] * p["tiles_n"]
        capacity = sms * p["ctas_per_sm"]
        assert (name == "ffma" and p["bn"] in (64, 128)) or (name == "tc" and mode == "3xtf32" and p["bn"] == 128), where
        assert s == 1 and p["tail_split"] == 1, where
        min_kb = 4 if name == "ffma" else 32
        assert p["sk_ctas"] == capacity and tiles < capacity and tiles * p["k_blocks"] >= min_kb * capacity, where
    # launch resources fit one SM
    assert 0 < p["smem_bytes"] <= SMEM_PER_CTA, where
    assert p["ctas_per_sm"] * p["smem_bytes"] <= SMEM_PER_SM, where
    assert p["threads"] % 32 == 0 and 0 < p["threads"] <= 1024, where
    assert p["threads"] * p["ctas_per_sm"] <= THREADS_PER_SM, where
    assert p["stages"] >= 2, where
    # operand preparation
    rows_a = m if (transa == "N" or not tc) else k
    rows_b = k if (transb == "N" or not tc) else n
    for op, prep, ld_in, ld_read, rows in (("a", p["prep_a_name"], lda, p["ld_a"], rows_a),
                                            ("b", p["prep_b_name"], ldb, p["ld_b"], rows_b)):
        trans = transa if op == "a" else transb
        if prep == "none":
            assert ld_read == ld_in and ld_in % 4 == 0 and aligned, where
            if not tc:
                assert trans == "N", where  # the FFMA kernel reads A M-major and B K-major only
        else:
            assert ld_read == _round_up(rows, 4), where
            if prep == "transpose":
                assert not tc and trans == "T", where
            if prep == "split":
                assert mode == "3xtf32", where
    if not tc:
        # FFMA copies exactly the operands TMA cannot read as they are
        for prep, trans, ld_in in ((p["prep_a_name"], transa, lda), (p["prep_b_name"], transb, ldb)):
            want = "none" if (trans == "N" and aligned and ld_in % 4 == 0) else ("copy" if trans == "N" else "transpose")
            assert prep == want, where
    if mode == "3xtf32" and name == "tc2":
        assert p["prep_a_name"] == "split" and p["prep_b_name"] == "split", where
    # launches: one per preparation, the GEMM, and the reduction of a K split or the stream-K fix-up
    preps = (p["prep_a_name"] != "none") + (p["prep_b_name"] != "none")
    assert p["launches"] == preps + 1 + (s > 1) + (p["sk_ctas"] > 0), where
    # workspace holds at least the prepared operands and the partial sums
    ws = 0
    for prep, ld_read, rows, elems in ((p["prep_a_name"], p["ld_a"], rows_a, m * k),
                                       (p["prep_b_name"], p["ld_b"], rows_b, k * n)):
        if prep != "none":
            ws += (2 if prep == "split" else 1) * ld_read * (elems // rows) * 4
    if s > 1:
        ws += s * _round_up(m, 4) * n * 4
    if p["tail_split"] > 1:
        ws += p["tail_tiles"] * p["tail_split"] * p["bm"] * p["bn"] * 4
    if p["sk_ctas"] > 0:  # at least one partial block per tile
        ws += p["tiles_m"] * p["tiles_n"] * p["bm"] * p["bn"] * 4
    assert p["workspace_bytes"] >= ws, where
    if preps == 0 and s == 1 and p["tail_split"] == 1 and p["sk_ctas"] == 0:
        assert p["workspace_bytes"] == 0, where


@pytest.mark.parametrize("mode", ["ffma", "tf32", "3xtf32"])
def test_plan_invariants_over_seeded_shapes(lib, mode):
    rng = np.random.default_rng({"ffma": 11, "tf32": 12, "3xtf32": 13}[mode])
    base_a, base_b, base_c = 1 << 20, 1 << 22, 1 << 24
    checked = 0
    for m, n, k in _shapes(rng, 400):
        transa = "T" if rng.random() < 0.25 else "N"
        transb = "T" if rng.random() < 0.25 else "N"
        rows_a = m if transa == "N" else k
        rows_b = k if transb == "N" else n
        pad_a = int(rng.choice([0, 0, 1, 3, 4, 13]))
        pad_b = int(rng.choice([0, 0, 1, 4, 7]))
        aligned = rng.random() < 0.85
        off = 0 if aligned else 4
        sms = int(rng.choice([152, 152, 148, 132, 2]))
        lda, ldb = rows_a + pad_a, rows_b + pad_b
        p = pg.sgemm_plan(transa, transb, m, n, k, 1.0, base_a + off, lda, base_b + off, ldb, 0.0, base_c,
                          m + 5, mode, num_sms=sms)
        _check(p, m, n, k, mode, transa, transb, lda, ldb, aligned, sms)
        checked += 1
    assert checked >= 400


def test_plan_trivial_shapes_launch_nothing_or_scale(lib):
    for mode in ("ffma", "tf32", "3xtf32"):
        for m, n, k, alpha, beta, kernel, launches in (
                (0, 64, 64, 1.0, 0.0, "none", 0), (64, 0, 64, 1.0, 0.0, "none", 0),
                (64, 64, 0, 1.0, 1.0, "none", 0), (64, 64, 0, 1.0, 0.5, "scale", 1),
                (64, 64, 64, 0.0, 1.0, "none", 0), (64, 64, 64, 0.0, 0.0, "scale", 1)):
            p = pg.sgemm_plan("N", "N", m, n, k, alpha, 1 << 20, max(m, 1), 1 << 21, max(k, 1), beta, 1 << 22,
                              max(m, 1), mode)
            assert p["kernel_name"] == kernel and p["launches"] == launches, (mode, m, n, k, alpha, beta)
            assert p["workspace_bytes"] == 0


def _filled(tiles, cap, kb):
    """Share of a grid's CTA-slot waves that its tiles fill, a last wave at most half
    full and split s ways along K (s >= 2) counting as 1/s of a wave."""
    full, rem = divmod(tiles, cap)
    waves = full + (1 if rem else 0)
    if rem and full >= 1 and 2 * rem <= cap:
        s = min(cap // rem, 8, kb // 8)
        if s >= 2:
            waves = full + 1.0 / s
    return tiles / (cap * waves)


@pytest.mark.parametrize("sms", [152, 132, 80])
def test_ffma_tile_width_rules(lib, sms):
    """The FFMA planner's width choices, for n > 64: 128 x 64 tiles (three CTAs per
    SM) when K <= 64; for tiny products (under 2 GFLOP, 128 x 64 tiles filling at
    most half the SMs); when the 128-wide tiles would run stream-K; and, over
    several waves with K >= 2048 (or K >= 512 and two waves of 128 x 64 tiles),
    unless the 128 x 128 grid fills its waves better by more than 0.01.  Otherwise 128 x 128 (two CTAs per SM)."""
    rng = np.random.default_rng(2027 + sms)
    shapes = [(4096, 4096, 4096), (8192, 8192, 8192), (6144, 6144, 6144), (2048, 2048, 2048), (1000, 1300, 4000),
              (16384, 16384, 64), (16384, 16384, 65), (3000, 1500, 777)]
    shapes += [(int(rng.integers(200, 9000)), int(rng.integers(65, 9000)), int(rng.choice([32, 64, 500, 512, 1024, 2048, 5000])))
               for _ in range(120)]
    for m, n, k in shapes:
        p = pg.sgemm_plan("N", "N", m, n, k, 1.0, 256, m, 256, k, 0.0, 256, m, "ffma", num_sms=sms)
        where = (m, n, k, sms, p["bn"])
        assert p["bn"] in (64, 128), where
        assert p["ctas_per_sm"] == (3 if p["bn"] == 64 else 2), where
        if k <= 64:
            assert p["bn"] == 64, where
            continue
        pg.force_plan(128, 0)
        try:
            p128 = pg.sgemm_plan("N", "N", m, n, k, 1.0, 256, m, 256, k, 0.0, 256, m, "ffma", num_sms=sms)
        finally:
            pg.force_plan(0, 0)
        kb = _cdiv(k, 32)
        t128, t64 = _cdiv(m, 128) * _cdiv(n, 128), _cdiv(m, 128) * _cdiv(n, 64)
        long_k = k >= 2048 or (k >= 512 and t64 >= 2 * 3 * sms)
        wave_rule = long_k and t128 >= 2 * sms and _filled(t64, 3 * sms, kb) >= _filled(t128, 2 * sms, kb) - 0.01
        tiny = 2 * t64 <= sms and 2.0 * m * n * k <= 2e9
        want64 = tiny or p128["sk_ctas"] > 0 or wave_rule
        assert (p["bn"] == 64) == want64, (where, p128["sk_ctas"], wave_rule)


@pytest.mark.parametrize("sms", [152, 132, 80])
def test_tf32_pair_tile_width_rule(lib, sms):
    """TF32 on SM pairs with K >= 2048: 256 x 512 tiles when they make at least one
    wave of pairs and 1.8 x their waves (a partial last wave counted whole) is under
    the 256 x 256 grid's waves, a last wave at most half full split s ways counting
    1/s + 0.4; otherwise 256 x 256.  Shorter K keeps 256 x 256."""
    rng = np.random.default_rng(3031 + sms)
    shapes = [(4096, 4096, 4096), (3072, 4096, 4096), (4096, 2560, 4096), (8192, 8192, 2048), (8192, 8192, 1024),
              (3000, 5000, 4096), (2048, 2048, 8192), (16384, 4096, 8192)]
    shapes += [(int(rng.integers(300, 12000)), int(rng.integers(300, 12000)), int(rng.choice([1024, 2048, 3000, 8192])))
               for _ in range(150)]
    pairs = max(sms // 2, 1)
    for m, n, k in shapes:
        p = pg.sgemm_plan("N", "N", m, n, k, 1.0, 256, m, 256, k, 0.0, 256, m, "tf32", num_sms=sms)
        if p["kernel_name"] != "tc2":
            continue
        where = (m, n, k, sms, p["bn"])
        t512, t256 = _cdiv(m, 256) * _cdiv(n, 512), _cdiv(m, 256) * _cdiv(n, 256)
        full, rem = divmod(t256, pairs)
        w256 = full + (1 if rem else 0)
        if rem and full >= 1 and 2 * rem <= pairs:
            sp = min(pairs // rem, 4, _cdiv(k, 32) // 8)
            if sp >= 2:
                w256 = full + 1.0 / sp + 0.4
        want512 = k >= 2048 and t512 >= pairs and 1.8 * _cdiv(t512, pairs) < w256
        if n > 256 and p["split_k"] == 1:
            assert (p["bn"] == 512) == want512, where
        else:
            assert p["bn"] != 512, where
