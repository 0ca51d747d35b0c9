"""CPU proof by enumeration that the block quantizer's scale and reciprocal
quotient code every input as the correctly rounded divisions do.

The quantizer (FP8 GEMM library article, hncyxsy.com/news/241433, sections
2.1-2.2: s = amax/448 per 32x32 block, q = E4M3(x/s)) forms s from the
constant RN(1/448) and x/s from one reciprocal per block, each corrected by
Markstein's method (P. Markstein, IBM J. Res. Develop. 34(1), 1990); the
quotient is taken negated (packed f32x2 form) and the code's sign bit flipped.
Scales below 2^-100 divide.  Both x and amax are bf16, so
quotient_exhaustive.c enumerates every (amax, x) pair in IEEE fp32 with fused
multiply-adds -- the same correctly rounded operations the kernel issues -- and
compares scale, quotient and E4M3 code with those of the correctly rounded
divisions.  The GPU quantizer tests then check the kernel itself against the
oracle."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
AMAX_MAX = 0x7F7F   # largest finite bf16, as bits


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("quotient") / "quotient_exhaustive")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", exe, os.path.join(HERE, "quotient_exhaustive.c"),
                    "-lm", "-lpthread"], check=True)
    return exe


def _run(exe, t_log2, lo, hi):
    nt = max(1, min(32, os.cpu_count() or 1))
    out = subprocess.run([exe, str(t_log2), str(lo), str(hi), str(nt)], check=True, capture_output=True,
                         text=True, timeout=900).stdout.split()
    pairs, bad_q, bad_big, bad_code, bad_scale = (int(v) for v in out)
    return pairs, bad_q, bad_big, bad_code, bad_scale


def _bf16_bits_of(v: float) -> int:
    import struct
    return struct.unpack("<I", struct.pack("<f", v))[0] >> 16


def test_reciprocal_quotient_codes_every_input(prog):
    """Threshold 2^-100: every scale equals RN(amax/448); every quotient of
    size >= 2^-10 is the correctly rounded one and every code agrees, over all
    1.06e9 (amax, x) pairs whose scale takes the reciprocal path."""
    pairs, bad_q, bad_big, bad_code, bad_scale = _run(prog, -100, 1, AMAX_MAX)
    assert pairs > 1_000_000_000
    assert bad_scale == 0
    assert bad_big == 0
    assert bad_code == 0
    # the remaining differences exist (subnormal x, underflowing quotients) and
    # are all below 2^-10, where both codes are +-0
    assert bad_q > 0


def test_enumeration_catches_the_bare_normal_threshold(prog):
    """A planted mistake: admitting every normal scale (2^-126) lets subnormal x
    reach codes that matter, and the enumeration must see code differences.
    Only the block maxima below 448 * 2^-100 are enumerated."""
    hi = _bf16_bits_of(448.0 * 2.0 ** -100)
    pairs, bad_q, bad_big, bad_code, _ = _run(prog, -126, 1, hi)
    assert pairs > 0
    assert bad_big > 0
    assert bad_code > 0
