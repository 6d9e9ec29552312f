"""The 4-bit append's rounding rules, emulated on the host (no GPU).

The append epilogue computes each group's scale and codes without a division (csrc/gemm.cu,
int4_store_columns and rne_div).  These tests check the two rules it relies on against
their definitions (the "KV-cache LLM serving" page's 4-bit pages: per group the smallest
fp16 scale with 7 * scale >= max |x|, codes x / scale rounded to nearest, ties to even),
over large seeded samples and the edge cases, in exact fp32 / fp64 emulation:

  * scale: amax * (1/7) in fp32, rounded down to fp16, then raised one fp16 step at a time,
    at most twice, while 7 * scale < amax;
  * code: k = rint(x * inv) in fp32 for any reciprocal inv of the scale within a few fp32
    ulps, then corrected by the exact residual x - k * scale (beyond scale / 2 the
    neighbour on its side, at scale / 2 the even one).
"""
import numpy as np

F32, F16 = np.float32, np.float16


def _smallest_scale(amax):
    """Definition: the smallest finite fp16 h >= 0 with 7 h >= amax (fp64 arithmetic; 7 h is
    exact)."""
    h = F16(amax / 7.0)                          # nearest fp16 to the exact quotient
    while 7.0 * float(h) < amax:
        h = np.nextafter(h, F16(np.inf))
    while h > 0 and 7.0 * float(np.nextafter(h, F16(0))) >= amax:
        h = np.nextafter(h, F16(0))
    return h


def _scale_rule(amax):
    q = F32(F32(amax) * F32(1.0 / 7.0))         # fp32 product, as the kernel
    h = F16(q)                                   # round to nearest, then down if above q
    if F32(h) > q:
        h = np.nextafter(h, F16(-np.inf))
    for _ in range(2):
        if F32(7.0) * F32(h) < F32(amax):        # exact: 7 h has at most 14 bits
            h = np.nextafter(h, F16(np.inf))
    return h


def test_scale_rule_is_the_smallest_fp16_scale():
    rng = np.random.default_rng(2024)
    # log-uniform over the normal and subnormal fp16 range of amax / 7 (amax / 7 below
    # 60000, so that the smallest scale is finite)
    ex = rng.uniform(-26, np.log2(60000.0 * 7) - 1, 200_000)
    amaxes = [float(F32(2.0 ** e * rng.uniform(1, 2))) for e in ex]
    # exact multiples 7 h and their fp32 neighbours
    hs = rng.choice(np.arange(1, 0x7BFF, dtype=np.uint16), 20_000).view(F16)
    for h in hs:
        a = F32(7.0) * F32(h)
        amaxes += [float(a), float(np.nextafter(a, F32(np.inf))), float(np.nextafter(a, F32(0)))]
    amaxes += [0.0, float(np.finfo(F32).tiny), 1e-30, 7 * 6e-8]
    bad = [a for a in amaxes if _scale_rule(a) != _smallest_scale(a)]
    assert not bad, bad[:5]


def _rne_ref(x, s):
    # x / s in fp64 never crosses a half-integer it should not (x has 24 bits, s 11), and
    # a tie x = (k + 1/2) s is exact in fp64
    return int(np.rint(float(x) / float(s)))


def _code_rule(x, s, inv):
    k = F32(np.rint(F32(x) * inv))
    r = float(x) - float(k) * float(s)           # exact, as the kernel's fma
    a2 = 2.0 * abs(r)
    ki = int(k)
    if a2 > float(s) or (a2 == float(s) and (ki & 1)):
        return ki + (1 if r > 0 else -1)
    return ki


def test_code_rule_rounds_to_nearest_even_for_approximate_reciprocals():
    rng = np.random.default_rng(7)
    bits = rng.integers(0x0001, 0x7BFF, 4000).astype(np.uint16)
    scales = bits.view(F16)
    checked = 0
    for s in scales:
        sf = F32(s)
        inv0 = F32(1.0) / sf
        invs = [inv0]
        for n in (1, 2, 4):                      # a reciprocal off by a few fp32 ulps
            up, dn = inv0, inv0
            for _ in range(n):
                up, dn = np.nextafter(up, F32(np.inf)), np.nextafter(dn, F32(0))
            invs += [up, dn]
        xs = [F32(rng.uniform(-7, 7) * sf) for _ in range(8)]
        xs += [F32((k + 0.5) * float(sf)) for k in range(-7, 7)]          # exact ties
        xs += [np.nextafter(x, F32(np.inf)) for x in xs[-14:]]             # just past them
        for x in xs:
            if abs(float(x)) > 7 * float(sf):
                continue
            want = _rne_ref(x, sf)
            for inv in invs:
                assert _code_rule(x, sf, inv) == want, (float(s), float(x), float(inv))
                checked += 1
    assert checked > 200_000
