"""The activation quantisers turn a bf16 element x of a row with scale s into
its code without a division: with r = fp32(1/s),

    q0 = fp32(x r),  rem = fma(-q0, s, x),  q1 = fma(rem, r, q0),
    code = round_half_even(q1)  (by adding and subtracting 1.5 * 2^23),

relying on q1 being the correctly rounded quotient fp32(x / s) (Markstein's
correction step).  The row rule defines the code as
clamp(round_half_even(fp32(x / s)), -127, 127) with s = fp32(amax / 127)
(zhidx TurboT2VA article, section 01 item 3).

This test checks that identity with exact integer arithmetic (every fp32
operation rounded once, to nearest even) for every pair of bf16
significands of amax and x, for x from amax down to 2^-12 amax (below that
|x / s| < 127 * 2^-11 and every code is 0), both signs.  The steps scale
exactly by powers of two, so this covers every row whose values stay normal.
It checks the arithmetic the kernels use, not the kernels: the GPU parity
tests compare their codes with the oracle's division."""
import os
from multiprocessing import get_context

import pytest

SCALE = 200          # values are integers in units of 2^-200
ONE = 1 << SCALE
MAGIC = 3 << (22 + SCALE)   # 1.5 * 2^23


def rn32_ratio(num: int, den: int) -> int:
    """num / den (a real number, den > 0) rounded to 24 significant bits,
    ties to even, in units of 2^-200 (num, den any integers)."""
    if num == 0:
        return 0
    neg = num < 0
    n = abs(num) << SCALE
    q, r = divmod(n, den)
    shift = q.bit_length() - 24
    if shift > 0:
        hi = q >> shift
        low = q - (hi << shift)
        half = 1 << (shift - 1)
        if low > half or (low == half and (r > 0 or hi & 1)):
            hi += 1
        q = hi << shift
    return -q if neg else q


def rn32(v: int) -> int:
    """An exact value in units of 2^-200 rounded to an fp32."""
    return rn32_ratio(v, ONE)


def mul(a: int, b: int) -> int:
    return a * b >> SCALE   # exact: every product here is a multiple of 2^-200


def rne_int(v: int) -> int:
    q, rem = divmod(v, ONE)
    half = ONE >> 1
    if rem > half or (rem == half and q & 1):
        q += 1
    return q


def bf16(sig: int, exp: int) -> int:
    """(1 + sig/128) * 2^exp in units of 2^-200."""
    return (128 + sig) << (SCALE - 7 + exp)


def check_amax(sig_a: int):
    amax = bf16(sig_a, 0)
    s = rn32_ratio(amax, 127 * ONE)
    r = rn32_ratio(ONE, s)
    bad = []
    for k in range(0, 13):
        for sig_x in range(128):
            mag = bf16(sig_x, -k)
            if mag > amax:
                continue
            for x in (mag, -mag):
                u = rn32_ratio(x, s)                              # fp32(x / s)
                ref = max(-127, min(127, rne_int(u)))
                q0 = rn32(mul(x, r))
                rem = rn32(x - mul(q0, s))
                q1 = rn32(q0 + mul(rem, r))
                t = rn32(q1 + MAGIC)
                code = max(-127, min(127, (t - MAGIC) >> SCALE))
                if code != ref:
                    bad.append((sig_a, sig_x, k, x > 0, ref, code))
    return bad


def test_rn32_helper_pins():
    # the helper itself: exact values, ties to even, and a value needing rounding
    assert rn32(ONE) == ONE
    a = (1 << 24) + 1                       # 2^24 + 1: halfway between 2^24 and 2^24 + 2
    assert rn32(a << SCALE) == (1 << 24) << SCALE
    b = (1 << 24) + 3                       # halfway between 2^24 + 2 and 2^24 + 4: to even (2^24 + 4)
    assert rn32(b << SCALE) == ((1 << 24) + 4) << SCALE
    third = rn32_ratio(ONE, 3 * ONE)        # fp32(1/3) = 11184811 * 2^-25
    assert third == 11184811 << (SCALE - 25)
    assert rne_int(ONE // 2) == 0 and rne_int(3 * ONE // 2) == 2 and rne_int(-(ONE // 2)) == 0


def test_correction_step_gives_the_division_codes_for_every_bf16_row():
    ctx = get_context("spawn")
    with ctx.Pool(min(16, os.cpu_count() or 1)) as pool:
        bad = [b for part in pool.map(check_amax, range(128)) for b in part]
    assert not bad, "codes differ from the division rule: %s" % bad[:5]


def test_correction_step_needed():
    # Without the correction step (code = rne(fp32(x r))) some bf16 rows would
    # get a different code: the test above is not vacuous.
    found = 0
    for sig_a in range(128):
        amax = bf16(sig_a, 0)
        s = rn32_ratio(amax, 127 * ONE)
        r = rn32_ratio(ONE, s)
        for sig_x in range(128):
            for k in range(0, 8):
                x = bf16(sig_x, -k)
                if x > amax:
                    continue
                ref = max(-127, min(127, rne_int(rn32_ratio(x, s))))
                naive = max(-127, min(127, rne_int(rn32(mul(x, r)))))
                found += naive != ref
    assert found > 0
