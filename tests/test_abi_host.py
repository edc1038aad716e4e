"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, rejects invalid arguments with -i before
touching a device, and the planner makes the documented choices."""
import ctypes
import os
import re
import subprocess

import pytest

import precision_gemm_gb300 as pg
from precision_gemm_gb300 import build as pgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "precision_gemm.h")


@pytest.fixture(scope="module")
def lib():
    pgbuild.build()
    return pg.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgemm\w*)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(pg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pg.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if " T " in line)
    assert exported == _declared_functions()


def test_version(lib):
    assert "sm_103a" in pg.version()


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "precision_gemm.h"\nint main(void){ sgemm_plan_t p; (void)p; '
                   'return sgemm_version() == 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c",
                        str(src), "-o", str(tmp_path / "use.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


# Arguments: (transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode)
GOOD = ("N", "N", 64, 48, 32, 1.0, 4096, 64, 8192, 32, 0.0, 16384, 64, 0)


def _call(lib, args):
    ta, tb, m, n, k, al, A, lda, B, ldb, be, C, ldc, mode = args
    return lib.sgemm(ta.encode(), tb.encode(), m, n, k, al, A, lda, B, ldb, be, C, ldc, mode, None)


def _with(**kw):
    names = ("transa", "transb", "m", "n", "k", "alpha", "A", "lda", "B", "ldb", "beta", "C", "ldc", "mode")
    vals = dict(zip(names, GOOD))
    vals.update(kw)
    return tuple(vals[n] for n in names)


@pytest.mark.parametrize("kw,code", [
    (dict(transa="X"), -1), (dict(transb="q"), -2), (dict(m=-1), -3), (dict(n=-5), -4), (dict(k=-2), -5),
    (dict(m=2 ** 31), -3), (dict(A=0), -7), (dict(lda=63), -8), (dict(B=0), -9), (dict(ldb=31), -10),
    (dict(C=0), -12), (dict(ldc=10), -13), (dict(mode=3), -14), (dict(mode=-1), -14),
    (dict(transa="T", lda=31), -8), (dict(transb="T", ldb=47), -10), (dict(lda=0, m=0, transa="N"), -8),
])
def test_invalid_arguments_rejected_before_device_work(lib, kw, code):
    assert _call(lib, _with(**kw)) == code
    assert "argument %d" % -code in pg.last_error()


@pytest.mark.parametrize("entry", ["sgemm_host", "sgemm_host_async", "sgemm_noalloc"])
@pytest.mark.parametrize("kw,code", [(dict(transa="X"), -1), (dict(m=-1), -3), (dict(lda=63), -8),
                                     (dict(ldc=10), -13), (dict(mode=3), -14)])
def test_other_entries_validate_like_sgemm(lib, entry, kw, code):
    ta, tb, m, n, k, al, A, lda, B, ldb, be, C, ldc, mode = _with(**kw)
    fn = getattr(lib, entry)
    assert fn(ta.encode(), tb.encode(), m, n, k, al, A, lda, B, ldb, be, C, ldc, mode, None) == code
    assert "argument %d" % -code in pg.last_error()


def test_argument_order_is_signature_order(lib):
    # both transa and m are bad: the first in signature order is reported
    assert _call(lib, _with(transa="Z", m=-1)) == -1
    assert _call(lib, _with(lda=1, ldc=1)) == -8


def test_null_pointers_allowed_when_unused(lib):
    # alpha == 0 with beta == 1: nothing is read or written, so nulls are fine
    # and the call returns before touching any device.
    assert _call(lib, _with(A=0, B=0, C=0, alpha=0.0, beta=1.0)) == 0
    assert _call(lib, _with(m=0, A=0, B=0, C=0)) == 0
    assert _call(lib, _with(n=0, A=0, B=0, C=0)) == 0


def test_python_binding_raises(lib):
    with pytest.raises(pg.SgemmError) as e:
        pg.sgemm("N", "N", 4, 4, 4, 1.0, 4096, 2, 4096, 4, 0.0, 4096, 4, "ffma", stream=0)
    assert e.value.code == -8


def plan(m, n, k, mode="ffma", transa="N", transb="N", lda=None, ldb=None, ldc=None, A=1 << 20, B=1 << 21,
         C=1 << 22, alpha=1.0, beta=0.0, sms=152):
    ra = m if transa == "N" else k
    rb = k if transb == "N" else n
    return pg.sgemm_plan(transa, transb, m, n, k, alpha, A, lda or max(ra, 1), B, ldb or max(rb, 1), beta, C,
                         ldc or max(m, 1), mode, num_sms=sms)


def test_plan_square_uses_wide_tiles_and_no_split(lib):
    for mode in ("ffma", "tf32", "3xtf32"):
        p = plan(8192, 8192, 8192, mode)
        # FFMA: 128 x 64 tiles, three CTAs per SM (they fill their waves as well as 128 x 128
        # tiles at two per SM, and win the tie); tensor cores on SM pairs: 256 x 512 tiles for
        # TF32 (long K, two waves or more of tiles), 256 x 256 for 3xTF32
        bm, bn = {"ffma": (128, 64), "tf32": (256, 512), "3xtf32": (256, 256)}[mode]
        assert p["bn"] == bn and p["bm"] == bm and p["split_k"] == 1
        assert p["tiles_m"] == 8192 // bm and p["tiles_n"] == 8192 // bn
        assert p["kernel_name"] == ("ffma" if mode == "ffma" else "tc2")
        assert p["ctas_per_sm"] == (3 if mode == "ffma" else 1)
    assert plan(8192, 8192, 8192, "ffma")["prep_a_name"] == "none"
    # 3xTF32 on SM pairs: a split pre-pass per operand, then the GEMM
    x = plan(8192, 8192, 8192, "3xtf32")
    assert x["prep_a_name"] == "split" and x["prep_b_name"] == "split" and x["launches"] == 3
    assert x["workspace_bytes"] >= 4 * 8192 * 8192 * 4  # split parts (+ last-wave partials)
    # narrow shapes (single-SM kernel): the kernel splits A itself (into tensor memory)
    # with one or two groups of four extra warps; B is split on chip too, except with
    # K >= 4096 and four or more rows of tiles sharing B, where a pre-pass splits it once
    t = plan(8192, 64, 8192, "3xtf32")
    assert t["kernel_name"] == "tc" and t["prep_a_name"] == "none" and t["prep_b_name"] == "split"
    assert t["threads"] - plan(8192, 64, 8192, "tf32")["threads"] in (128, 256)
    assert t["launches"] == 2 + (t["split_k"] > 1 or t["sk_ctas"] > 0)  # the reduction or the stream-K fix-up
    assert t["workspace_bytes"] >= 2 * 64 * 8192 * 4
    w = plan(128, 4096, 8192, "3xtf32")
    assert w["kernel_name"] == "tc" and w["prep_a_name"] == "none" and w["prep_b_name"] == "none"
    assert w["launches"] == 1 + (w["split_k"] > 1 or w["sk_ctas"] > 0)
    assert plan(384, 64, 8192, "3xtf32")["prep_b_name"] == "none"    # three rows of tiles
    assert plan(512, 64, 8192, "3xtf32")["prep_b_name"] == "split"   # four
    assert plan(8192, 64, 8192, "tf32")["prep_b_name"] == "none"     # TF32 reads B as stored
    assert plan(1024, 1024, 1024, "3xtf32")["prep_b_name"] == "none"  # short K: the pre-pass costs more


def test_plan_tf32_512_wide_pair_tiles(lib):
    assert plan(6144, 6144, 6144, "tf32")["bn"] == 512
    assert plan(16384, 4096, 8192, "tf32")["bn"] == 512
    assert plan(8192, 8192, 2048, "tf32")["bn"] == 512       # 7 waves against 13 + a split last wave
    assert plan(4096, 4096, 16384, "tf32")["bn"] == 512      # 2 waves against 3 + a split last wave
    assert plan(3072, 4096, 4096, "tf32")["bn"] == 256       # 2 waves of 96 tiles against 3 of 192
    assert plan(4096, 2560, 4096, "tf32")["bn"] == 256       # 2 waves (80 tiles) against 2 + a split
    assert plan(2048, 2048, 8192, "tf32")["bn"] == 256       # 32 tiles of 256 x 512: under one wave
    assert plan(4096, 4096, 2048, "tf32")["bn"] == 512
    assert plan(8192, 8192, 1024, "tf32")["bn"] == 256       # K < 2048
    assert plan(8192, 8192, 8192, "tf32")["tail_split"] == 1  # 256 x 512 tiles do not split a last wave
    assert plan(8192, 8192, 8192, "3xtf32")["bn"] == 256     # 3xTF32 keeps 256 x 256
    assert plan(16384, 16384, 64, "tf32")["bn"] == 256       # skinny K
    # forcing 512 where it does not exist means 256
    pg.force_plan(512, 0)
    try:
        assert plan(8192, 8192, 8192, "3xtf32")["bn"] == 256
        assert plan(8192, 8192, 8192, "ffma")["bn"] == 256
        assert plan(100, 8192, 8192, "tf32")["bn"] == 256
        assert plan(2000, 3000, 700, "tf32")["bn"] == 512
    finally:
        pg.force_plan(0, 0)


def test_plan_last_wave_split(lib):
    # SM pairs: 160 tiles of 256x256 over 76 pairs = 2 full waves + 8 tiles; the last
    # wave's 8 tiles run as 4 K slices each (32 units)
    p = plan(4096, 2560, 4096, "tf32")
    assert p["bn"] == 256 and p["tail_tiles"] == 8 and p["tail_split"] == 4 and p["split_k"] == 1
    assert p["workspace_bytes"] >= 8 * 4 * 256 * 256 * 4
    q = plan(8192, 8192, 8192, "3xtf32")
    assert q["tail_tiles"] == 1024 - 13 * 76 and q["tail_split"] == 2
    # no split when the tiles fill whole waves, the last wave is over half full,
    # K is short, or the problem already uses split-K
    assert plan(256 * 19, 256 * 8, 4096, "tf32")["tail_split"] == 1          # 152 tiles = 2 waves
    assert plan(256 * 10, 256 * 12, 4096, "tf32")["tail_split"] == 1         # 120 tiles: 44 > 76/2
    assert plan(4096, 4096, 96, "tf32")["tail_split"] == 1                  # 3 K blocks
    assert plan(512, 512, 8192, "tf32")["tail_split"] == 1                  # split-K instead
    # FFMA: 2048 tiles of 128x64 over 152 SMs x 3 CTA slots = 4 waves + 224 tiles;
    # the 224 last-wave tiles run as 2 K slices (448 blocks), in the same launch
    f = plan(4096, 4096, 4096, "ffma")
    assert f["bn"] == 64 and f["launches"] == 1
    assert f["tail_tiles"] == 2048 - 4 * 456 and f["tail_split"] == 2
    assert f["workspace_bytes"] >= 224 * 2 * 128 * 64 * 4
    assert plan(8192, 8192, 8192, "ffma")["tail_split"] == 1  # 440-tile last wave: over half full


def test_plan_skinny_k_uses_deterministic_split(lib):
    p = plan(128, 128, 262144, "ffma")
    assert p["bn"] == 128 and p["tiles_m"] * p["tiles_n"] == 1
    assert p["split_k"] > 100 and p["split_k"] * p["k_blocks_per_split"] >= p["k_blocks"]
    assert (p["split_k"] - 1) * p["k_blocks_per_split"] < p["k_blocks"]  # no empty slice
    assert p["launches"] == 2 and p["workspace_bytes"] >= p["split_k"] * 128 * 128 * 4
    tall = plan(8192, 64, 8192, "tf32")
    assert tall["bn"] == 64 and tall["tiles_m"] == 64 and tall["split_k"] == 2


def test_plan_pair_kernel_only_above_128_rows(lib):
    assert plan(128, 8192, 4096, "tf32")["kernel_name"] == "tc"       # one SM tile covers m
    assert plan(129, 8192, 4096, "tf32")["kernel_name"] == "tc2"
    assert plan(4096, 64, 4096, "3xtf32")["kernel_name"] == "tc"      # 64-wide tile: single SM
    # small products whose 128 x 64 tiles fit one wave of SMs run on those (lowest latency)
    small = plan(512, 512, 4096, "tf32")                               # 4 x 8 tiles -> split K over 152 SMs
    assert small["kernel_name"] == "tc" and small["bn"] == 64 and small["tiles_m"] * small["tiles_n"] == 32
    assert small["split_k"] == 152 // 32
    long_k = plan(512, 512, 65536, "tf32")                             # long K: SM pairs, 2 x 2 tiles, split K
    assert long_k["kernel_name"] == "tc2" and long_k["split_k"] == 76 // 4
    # one row of tiles (m <= 128): 128-wide single-SM tiles for 3xTF32 and for TF32 above 4 GFLOP
    for mnk in ((128, 128, 262144), (128, 4096, 8192), (100, 3000, 2000), (64, 8192, 8192)):
        q = plan(*mnk, "3xtf32")
        assert q["kernel_name"] == "tc" and q["bn"] == 128, (mnk, q)
    assert plan(128, 4096, 8192, "tf32")["bn"] == 128
    assert plan(100, 3000, 2000, "tf32")["bn"] == 64                  # 1.2 GFLOP: the 64-wide rule
    assert plan(128, 64, 262144, "3xtf32")["bn"] == 64                 # n <= 64
    assert plan(128, 65536, 4096, "tf32")["bn"] == 256                 # 512 tiles of 128: over one wave
    # 3xTF32 keeps the single-SM kernel at any K (its on-chip split avoids two pre-passes)
    assert plan(8192, 128, 8192, "3xtf32")["kernel_name"] == "tc"
    assert plan(8192, 128, 8192, "tf32")["kernel_name"] == "tc2"
    assert plan(1024, 1024, 1024, "3xtf32")["kernel_name"] == "tc"     # 128 tiles: one wave
    assert plan(1536, 1536, 1536, "3xtf32")["kernel_name"] == "tc2"    # 288 tiles: SM pairs
    pair = plan(1280, 1280, 65536, "tf32")                             # 5 x 5 pair tiles -> split K over 76 pairs
    assert pair["kernel_name"] == "tc2" and pair["tiles_m"] * pair["tiles_n"] == 25
    assert pair["split_k"] == 76 // 25


def test_plan_misaligned_ld_copies_operand(lib):
    p = plan(3000, 1500, 777, "ffma", lda=3013, ldb=784, ldc=3005)
    assert p["prep_a_name"] == "copy" and p["prep_b_name"] == "none"
    assert p["ld_a"] % 4 == 0 and p["ld_b"] == 784
    p2 = plan(64, 64, 64, "tf32", A=(1 << 20) + 4)  # base not 16-byte aligned
    assert p2["prep_a_name"] == "copy"


def test_plan_transposed_operands(lib):
    # FFMA reads A M-major and B K-major only: transposed operands are copied transposed
    p = plan(300, 200, 100, "ffma", transa="T", transb="T")
    assert p["prep_a_name"] == "transpose" and p["prep_b_name"] == "transpose"
    assert p["ld_a"] == 300 and p["ld_b"] == 100
    # the tensor-core kernels read either orientation in place
    t = plan(300, 200, 100, "tf32", transa="T", transb="T", lda=104, ldb=204)
    assert t["prep_a_name"] == "none" and t["prep_b_name"] == "none"
    assert t["ld_a"] == 104 and t["ld_b"] == 204 and t["launches"] == 1
    # 3xTF32 on SM pairs splits them without transposing: ld is the stored row count rounded to 4
    x = plan(3000, 2000, 101, "3xtf32", transa="T", transb="T")
    assert x["kernel_name"] == "tc2" and x["prep_a_name"] == "split" and x["ld_a"] == 104 and x["ld_b"] == 2000
    # the single-SM kernel reads them in place and splits them on chip; a stored
    # row count that is not a multiple of 4 still needs a plain copy, ld rounded up
    y = plan(100, 64, 101, "3xtf32", transa="T", transb="T")
    assert y["kernel_name"] == "tc" and y["prep_a_name"] == "copy" and y["ld_a"] == 104
    assert y["prep_b_name"] == "none" and y["ld_b"] == 64
    # a misaligned transposed operand is copied (not transposed) for the tensor cores
    c = plan(300, 200, 100, "tf32", transa="T", lda=101)
    assert c["prep_a_name"] == "copy" and c["ld_a"] == 100


def test_plan_trivial_cases(lib):
    assert plan(0, 10, 10)["kernel_name"] == "none"
    assert plan(10, 10, 0, beta=0.5)["kernel_name"] == "scale"
    assert plan(10, 10, 10, alpha=0.0, beta=1.0)["kernel_name"] == "none"


def test_force_plan(lib):
    try:
        pg.force_plan(64, 7)
        p = plan(1024, 1024, 4096)
        assert p["bn"] == 64 and p["split_k"] == 7
        with pytest.raises(pg.SgemmError):
            pg.force_plan(96, 0)
    finally:
        pg.force_plan(0, 0)


def test_plan_struct_layout_matches_header(lib, tmp_path):
    """The ctypes mirror of sgemm_plan_t has the C struct's size and offsets."""
    fields = [f for f, _ in pg.sgemm_plan_t._fields_]
    src = tmp_path / "layout.c"
    body = "".join('printf("%%s %%zu\\n", "%s", offsetof(sgemm_plan_t, %s));' % (f, f) for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "precision_gemm.h"\nint main(void){'
                   + body + 'printf("size %zu\\n", sizeof(sgemm_plan_t)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split("\n")
               if line)
    for f in fields:
        assert int(out[f]) == getattr(pg.sgemm_plan_t, f).offset, f
    assert int(out["size"]) == ctypes.sizeof(pg.sgemm_plan_t)


def test_plain_c_caller_links_and_calls_the_library(lib, tmp_path):
    """A C program with no Python or torch in it links the shared library and
    calls it through the header alone: the version, the planner on a device it
    does not touch, an invalid argument answered with -i and a message, a call
    with nothing to do, and the workspace setter's argument checks."""
    src = tmp_path / "caller.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "precision_gemm.h"
int main(void) {
    sgemm_plan_t p;
    if (!strstr(sgemm_version(), "sm_103a")) return 1;
    if (sgemm_plan('N', 'N', 8192, 8192, 8192, 1.0f, (const void *)4096, 8192, (const void *)8192, 8192, 1.0f,
                   (const void *)16384, 8192, SGEMM_TF32, 152, &p) != 0) return 2;
    if (p.kernel != SGEMM_KERNEL_TC2 || p.bm != 256 || p.bn != 512 || p.split_k != 1) return 3;
    if (sgemm_plan('T', 'N', 3000, 1500, 777, 1.5f, (const void *)4100, 777, (const void *)8192, 784, -0.5f,
                   (const void *)16384, 3005, SGEMM_FFMA, 152, &p) != 0) return 4;
    if (p.kernel != SGEMM_KERNEL_FFMA || p.prep_a != SGEMM_PREP_TRANSPOSE || p.prep_b != SGEMM_PREP_NONE) return 5;
    if (sgemm('N', 'N', 64, 48, 32, 1.0f, (const float *)4096, 63, (const float *)8192, 32, 0.0f,
              (float *)16384, 64, SGEMM_FFMA, NULL) != -8) return 6;
    if (!strstr(sgemm_last_error_string(), "argument 8")) return 7;
    if (sgemm_plan('N', 'N', 64, 48, 32, 1.0f, NULL, 64, NULL, 32, 0.0f, NULL, 64, 7, 152, &p) != -7) return 8;
    if (sgemm_plan('N', 'N', 64, 48, 32, 1.0f, (const void *)4096, 64, (const void *)8192, 32, 0.0f,
                   (const void *)16384, 64, 7, 152, &p) != -14) return 10;
    if (sgemm('N', 'N', 0, 48, 32, 1.0f, NULL, 1, NULL, 32, 0.0f, NULL, 1, SGEMM_3XTF32, NULL) != 0) return 9;
    if (sgemm_plan('N', 'N', 64, 48, 32, 1.0f, (const void *)4096, 64, (const void *)8192, 32, 0.0f,
                   (const void *)16384, 64, SGEMM_FFMA, 0, &p) != -15) return 11;
    if (sgemm_plan('N', 'N', 64, 48, 32, 1.0f, (const void *)4096, 64, (const void *)8192, 32, 0.0f,
                   (const void *)16384, 64, SGEMM_FFMA, 152, NULL) != -16) return 12;
    if (sgemm_set_workspace((void *)4112, 64, NULL) != -1) return 13;
    if (!strstr(sgemm_last_error_string(), "argument 1")) return 14;
    if (sgemm_set_workspace(NULL, 64, NULL) != -2) return 15;
    puts("ok");
    return 0;
}
''')
    libdir = os.path.dirname(pg.LIB_PATH)
    libname = os.path.basename(pg.LIB_PATH)
    assert libname.startswith("lib") and libname.endswith(".so")
    exe = tmp_path / "caller"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-l" + libname[3:-3], "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout, run.stderr)
