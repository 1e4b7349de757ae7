"""Pins for the CPU oracle: checks that tie it to something other than itself.

Every check takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch. The same battery runs against the real oracle (it must pass) and
against copies with a planted mistake (one check must fail), so each check
is chosen to catch a plausible slip: a dropped term, a wrong index or sign,
a reordered sum, an extra rounding.

Independent references used here:
* bf16 / fp16 decoding by library routines (torch for bf16, numpy for fp16);
* rounding by brute force: the nearest entry of the sorted table of every
  finite value of the format, ties to the even code;
* binary32 rank-order sums computed with numpy float32 arithmetic;
* the RMSNorm of tiny rows in exact rationals plus 60-digit decimal sqrt;
* hand-worked rows in tests/golden/worked_rows.txt.
"""
from __future__ import annotations

import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

from all_reduce_residual_gb300 import workloads as wlmod

BF16, FP16 = 0, 1
ALLREDUCE, RMSNORM = 0, 1
DT = {"bf16": BF16, "fp16": FP16}
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_rows.txt")

# ---------------------------------------------------------------------------
# Library decoding and the brute-force rounding table
# ---------------------------------------------------------------------------


def lib_decode(dtype: int, codes) -> np.ndarray:
    """Decode 16-bit codes with a library routine (torch bf16 / numpy fp16)."""
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    if dtype == BF16:
        return torch.from_numpy(c.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    with np.errstate(invalid="ignore"):
        return c.view(np.float16).astype(np.float32)


_TABLES = {}


def _table(dtype: int):
    """(values, codes) of every non-negative finite code, ascending, plus a
    final entry 2^(emax+1) standing for +inf (the value overflow rounds to)."""
    if dtype not in _TABLES:
        all_codes = np.arange(0x8000, dtype=np.uint16)
        with np.errstate(invalid="ignore"):
            v = lib_decode(dtype, all_codes).astype(np.float64)
        fin = np.isfinite(v)
        vals, codes = v[fin], all_codes[fin]
        order = np.argsort(vals, kind="stable")
        vals, codes = vals[order], codes[order]
        inf_code = 0x7F80 if dtype == BF16 else 0x7C00
        top = 2.0 ** 128 if dtype == BF16 else 2.0 ** 16
        _TABLES[dtype] = (np.append(vals, top), np.append(codes, np.uint16(inf_code)))
    return _TABLES[dtype]


def nearest_codes(dtype: int, v) -> np.ndarray:
    """Round float64 values to the format by table search, ties to even code."""
    with np.errstate(invalid="ignore", over="ignore"):
        v = np.asarray(v, dtype=np.float64)
    vals, codes = _table(dtype)
    a = np.abs(v)
    sign = np.signbit(v)
    nan = np.isnan(v)
    a_safe = np.where(nan, 0.0, np.minimum(a, vals[-1]))
    hi_i = np.searchsorted(vals, a_safe, side="left")
    hi_i = np.clip(hi_i, 0, len(vals) - 1)
    lo_i = np.clip(hi_i - 1, 0, len(vals) - 1)
    lo, hi = vals[lo_i], vals[hi_i]
    dlo, dhi = a_safe - lo, hi - a_safe
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi_i] % 2 == 0)) | (a_safe == hi)
    out = np.where(pick_hi, codes[hi_i], codes[lo_i]).astype(np.uint16)
    out = np.where(sign, out | np.uint16(0x8000), out).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0 if dtype == BF16 else 0x7E00), out).astype(np.uint16)


def is_nan_code(dtype: int, c) -> np.ndarray:
    c = np.asarray(c, dtype=np.uint16) & np.uint16(0x7FFF)
    return c > (0x7F80 if dtype == BF16 else 0x7C00)


def assert_codes_equal(dtype, got, want, what=""):
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    gn, wn = is_nan_code(dtype, got), is_nan_code(dtype, want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    bad = (~gn) & (got != want)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} codes differ, first at {i}: "
                             f"got {[hex(x) for x in got.ravel()[i]]} want {[hex(x) for x in want.ravel()[i]]}")


# ---------------------------------------------------------------------------
# Converters
# ---------------------------------------------------------------------------


def check_widen(o):
    codes = np.arange(65536, dtype=np.uint16)
    for dtype in (BF16, FP16):
        got, ref = o.widen(dtype, codes), lib_decode(dtype, codes)
        assert np.array_equal(np.isnan(got), np.isnan(ref)), "widen: NaN set differs"
        fin = ~np.isnan(ref)
        assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32)), \
            f"widen dtype={dtype}: decoded values differ from the library decoding"


def check_roundtrip(o):
    codes = np.arange(65536, dtype=np.uint16)
    for dtype in (BF16, FP16):
        back = o.narrow_f32(dtype, o.widen(dtype, codes))
        nan = is_nan_code(dtype, codes)
        assert np.array_equal(back[~nan], codes[~nan]), f"round trip dtype={dtype} changed a code"
        assert is_nan_code(dtype, back[nan]).all(), "NaN did not stay NaN"
        assert ((back[nan] & np.uint16(0x8000)) == (codes[nan] & np.uint16(0x8000))).all(), "NaN sign lost"


def _midpoints(dtype):
    vals, _ = _table(dtype)
    mids = (vals[:-1] + vals[1:]) / 2.0  # exact in float64 and in float32
    return mids


def check_narrow_f32(o, n=1_000_000, seed=1):
    rng = np.random.default_rng(seed)
    for dtype in (BF16, FP16):
        mids = _midpoints(dtype).astype(np.float32)
        near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                               np.nextafter(mids, np.float32(-np.inf))])
        rand_bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
        # values concentrated on the format's own range as well as all bit patterns
        scale = np.float32(2.0) ** rng.integers(-30 if dtype == FP16 else -140, 20 if dtype == FP16 else 130,
                                                size=n).astype(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            ranged = (rng.standard_normal(n).astype(np.float32) * scale).astype(np.float32)
        v = np.concatenate([near, -near, rand_bits, ranged,
                            np.array([0.0, -0.0, np.inf, -np.inf, np.nan], np.float32)])
        got = o.narrow_f32(dtype, v)
        assert_codes_equal(dtype, got, nearest_codes(dtype, v.astype(np.float64)), f"narrow_f32 dtype={dtype}")
        # and a library routine on the finite, non-overflowing values
        if dtype == BF16:
            lib = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        else:
            with np.errstate(over="ignore"):
                lib = v.astype(np.float16).view(np.uint16)
        assert_codes_equal(dtype, got, lib, f"narrow_f32 vs library dtype={dtype}")


def check_narrow_f64(o, n=200_000, seed=2):
    rng = np.random.default_rng(seed)
    for dtype in (BF16, FP16):
        mids = _midpoints(dtype)
        # one binary64 step off each tie: rounding through binary32 first would
        # land on the tie and then go to even, half of the time the wrong way
        off = np.concatenate([np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf), mids])
        lo, hi = (-30, 17) if dtype == FP16 else (-140, 129)
        ranged = rng.standard_normal(n) * 2.0 ** rng.integers(lo, hi, size=n)
        v = np.concatenate([off, -off, ranged])
        assert_codes_equal(dtype, o.narrow_f64(dtype, v), nearest_codes(dtype, v), f"narrow_f64 dtype={dtype}")


# ---------------------------------------------------------------------------
# Worked rows (golden)
# ---------------------------------------------------------------------------


def load_golden(path=GOLDEN):
    cases, cur = [], {}
    for line in open(path):
        line = line.strip()
        if line.startswith("#"):
            continue
        if not line:
            if cur:
                cases.append(cur)
                cur = {}
            continue
        key, _, rest = line.partition(" ")
        cur[key] = rest
    if cur:
        cases.append(cur)
    return cases


def exact_codes(dtype, text):
    """Codes of a list of exact decimals; each must be representable."""
    vals = [Fraction(t) for t in text.split()]
    f = np.array([float(x) for x in vals])
    assert all(Fraction(float(x)) == x for x in vals), f"not exact in binary64: {text}"
    c = nearest_codes(dtype, f)
    back = lib_decode(dtype, c).astype(np.float64)
    assert np.array_equal(back, f), f"value not representable in dtype {dtype}: {text}"
    return c


def check_worked_rows(o):
    for case in load_golden():
        dtype = DT[case["dtype"]]
        pat = ALLREDUCE if case["pattern"] == "allreduce" else RMSNORM
        W = sum(1 for k in case if k.startswith("p") and k[1:].isdigit())
        P = [exact_codes(dtype, case[f"p{r}"])[None, :] for r in range(W)]
        kw = {}
        if pat == RMSNORM:
            kw = dict(residual=exact_codes(dtype, case["residual"])[None, :],
                      gamma=exact_codes(dtype, case["gamma"]), eps=float(case["eps"]))
        out, ro = o.run(pat, P, dtype=dtype, **kw)
        if "expect_residual_out" in case:
            assert_codes_equal(dtype, ro[0], exact_codes(dtype, case["expect_residual_out"]),
                               f"{case['case']} residual_out")
        assert_codes_equal(dtype, out[0], exact_codes(dtype, case["expect_out"]), f"{case['case']} out")


def check_inv_rms_r2(o):
    """The statistic of the R2 row: ss = 25 exactly, inv = 1/sqrt(25/8 + eps)."""
    getcontext().prec = 60
    x = exact_codes(BF16, "3 4 0 0 0 0 0 0")
    eps = np.float32(1e-6)
    inv, ss = o.inv_rms(BF16, x, float(eps))
    assert ss == 25.0, f"sum of squares {ss} != 25"
    ref = 1 / (Decimal(25) / 8 + Decimal(float(eps))).sqrt()
    assert abs(Decimal(inv) - ref) / ref < Decimal("1e-15"), f"inv {inv} vs {ref}"


# ---------------------------------------------------------------------------
# Brute force on tiny inputs, exact arithmetic
# ---------------------------------------------------------------------------


def ref_sum_f32(P32, res32=None):
    """binary32 sum in rank order (numpy float32 ops), then + residual."""
    acc = np.zeros_like(P32[0], dtype=np.float32)
    for p in P32:
        acc = (acc + p).astype(np.float32)
    if res32 is not None:
        acc = (acc + res32).astype(np.float32)
    return acc


def ref_rmsnorm_exact(dtype, x_codes, g_codes, eps32):
    """out codes of RMSNorm over each row, exact rationals + 60-digit sqrt."""
    getcontext().prec = 60
    x = lib_decode(dtype, x_codes).astype(np.float64)
    g = lib_decode(dtype, g_codes).astype(np.float64)
    M, H = x.shape
    out = np.empty((M, H), np.float64)
    e = Fraction(float(eps32))
    for m in range(M):
        ss = sum(Fraction(float(v)) ** 2 for v in x[m])
        ms = ss / H + e
        if ms == 0:
            out[m] = x[m] * np.inf * g
            continue
        inv = 1 / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
        for i in range(H):
            out[m, i] = float(Decimal(float(x[m, i])) * inv * Decimal(float(g[i])))
    return nearest_codes(dtype, out)


def _draw(rng, dtype, shape, sigma):
    return nearest_codes(dtype, rng.standard_normal(shape) * sigma)


def check_exact_tiny(o, trials=150, seed=3):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        dtype = BF16 if t % 2 == 0 else FP16
        W = int(rng.choice([1, 2, 3, 5, 8]))
        M = int(rng.integers(1, 4))
        H = int(rng.choice([1, 3, 8, 13, 16, 24]))
        sigma = float(rng.choice([0.01, 0.5, 3.0, 100.0]))
        eps32 = np.float32(rng.choice([1e-6, 1e-5, 0.1]))
        P = [_draw(rng, dtype, (M, H), sigma) for _ in range(W)]
        if t % 3 == 1:  # ranks of very different magnitude: the sum order matters
            top = 12.0 if dtype == FP16 else 24.0
            P = [_draw(rng, dtype, (M, H), 2.0 ** rng.uniform(-8.0, top)) for _ in range(W)]
        R = _draw(rng, dtype, (M, H), 1.0)
        G = nearest_codes(dtype, 0.5 + rng.random(H))
        if t % 5 == 2 and W >= 3:  # X, -X, then small ranks: exact only in array order
            X = _draw(rng, dtype, (M, H), 2.0 ** (20 if dtype == BF16 else 13))
            P[0], P[1] = X, X ^ np.uint16(0x8000)
            P[2:] = [_draw(rng, dtype, (M, H), 2.0 ** -3) for _ in range(W - 2)]
        if t % 7 == 3:  # integer-valued rows exercise exact cancellation
            P = [nearest_codes(dtype, rng.integers(-64, 65, size=(M, H)).astype(np.float64)) for _ in range(W)]
        P32 = [lib_decode(dtype, p) for p in P]
        # kAllReduce
        want_ar = nearest_codes(dtype, ref_sum_f32(P32).astype(np.float64))
        out, _ = o.run(ALLREDUCE, P, dtype=dtype)
        assert_codes_equal(dtype, out, want_ar, f"tiny trial {t} allreduce")
        # kARResidualRMSNorm
        want_ro = nearest_codes(dtype, ref_sum_f32(P32, lib_decode(dtype, R)).astype(np.float64))
        want_out = ref_rmsnorm_exact(dtype, want_ro, G, eps32)
        out, ro = o.run(RMSNORM, P, R, G, float(eps32), dtype=dtype)
        assert_codes_equal(dtype, ro, want_ro, f"tiny trial {t} residual_out")
        assert_codes_equal(dtype, out, want_out, f"tiny trial {t} out")


def check_one_rounding(o):
    """out is rounded once, from the exact value. Row x = [1, 6, 0, ...] with
    H = 28248, eps = 0 and gamma = 0.5078125 gives out_0 = sqrt(28248/37) *
    0.5078125 = 14.03125047..., 7.5e-6 of a bf16 quantum above the tie
    14.03125: the nearest bf16 is 14.0625, while a pass through binary32 lands
    exactly on the tie and then rounds to the even 14.0. (Found by a search over
    H, x_1 and gamma for a value that close above a tie.)"""
    H = 28248
    x = np.zeros(H, np.float64)
    x[0], x[1] = 1.0, 6.0
    xc = nearest_codes(BF16, x)[None, :]
    gc = nearest_codes(BF16, np.full(H, 0.5078125))
    want = ref_rmsnorm_exact(BF16, xc, gc, np.float32(0.0))
    assert lib_decode(BF16, want[:, :1])[0, 0] == np.float32(14.0625), "search result no longer holds"
    out, _ = o.run(RMSNORM, [xc], np.zeros((1, H), np.uint16), gc, 0.0, dtype=BF16)
    assert_codes_equal(BF16, out, want, "one-rounding row")


# ---------------------------------------------------------------------------
# Invariants on the seeded workloads
# ---------------------------------------------------------------------------

SMALL_M = {"small": None, "llama_tp2": 4, "k3_tp8": 2, "tp4_80mib": 2, "tp16_8mib": 3}


def seeded(name):
    wl = wlmod.WORKLOADS[name]
    inp = wlmod.make_inputs(wl, M=SMALL_M[name])
    P = [wlmod.codes(p) for p in inp.partials]
    return inp.workload, P, wlmod.codes(inp.residual), wlmod.codes(inp.gamma)


def textbook_rmsnorm(dtype, x_codes, g_codes, eps):
    """Ten-line RMSNorm in float64 numpy (pairwise mean, divide by the RMS)."""
    x = lib_decode(dtype, x_codes).astype(np.float64)
    g = lib_decode(dtype, g_codes).astype(np.float64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(np.float32(eps)))
    return nearest_codes(dtype, x / rms * g)


def check_invariants(o, names=tuple(SMALL_M)):
    for name in names:
        wl, P, R, G = seeded(name)
        dtype = DT[wl.dtype]
        zeros = np.zeros_like(R)
        # 1. W=1, residual 0: residual_out == P0 (-0 -> +0) and out == textbook RMSNorm(P0)
        out, ro = o.run(RMSNORM, [P[0]], zeros, G, wl.eps, dtype=dtype)
        p0 = np.where(P[0] == 0x8000, np.uint16(0), P[0])
        assert_codes_equal(dtype, ro, p0, f"{name} inv1 residual_out")
        assert_codes_equal(dtype, out, textbook_rmsnorm(dtype, P[0], G, wl.eps), f"{name} inv1 out")
        out_ar, _ = o.run(ALLREDUCE, [P[0]], dtype=dtype)
        assert_codes_equal(dtype, out_ar, p0, f"{name} W=1 allreduce")
        # 2. RMS(out / gamma) = 1 within 1e-3 where eps does not dominate
        out, ro = o.run(RMSNORM, P, R, G, wl.eps, dtype=dtype)
        y = lib_decode(dtype, out).astype(np.float64) / lib_decode(dtype, G).astype(np.float64)
        x = lib_decode(dtype, ro).astype(np.float64)
        keep = np.mean(x * x, axis=1) >= 100 * wl.eps
        rms = np.sqrt(np.mean(y * y, axis=1))
        assert np.all(np.abs(rms[keep] - 1.0) < 1e-3), f"{name} inv2 RMS(out/gamma) = {rms[keep]}"
        # 3. identical partials: permuting the pointer order changes nothing
        same = [P[0]] * wl.W
        a = o.run(RMSNORM, same, R, G, wl.eps, dtype=dtype)
        b = o.run(RMSNORM, same[::-1], R, G, wl.eps, dtype=dtype)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), f"{name} inv3"
        # 4./5. the sum follows the array order: any order matches the binary32
        # rank-order sum taken in that same order; two ranks commute
        perm = list(np.random.default_rng(7).permutation(wl.W))
        Pp = [P[i] for i in perm]
        out_p, ro_p = o.run(RMSNORM, Pp, R, G, wl.eps, dtype=dtype)
        want = nearest_codes(dtype, ref_sum_f32([lib_decode(dtype, p) for p in Pp],
                                                lib_decode(dtype, R)).astype(np.float64))
        assert_codes_equal(dtype, ro_p, want, f"{name} inv5 permuted residual_out")
        if wl.W == 2:
            assert np.array_equal(ro_p, ro) and np.array_equal(out_p, out), f"{name} inv4 W=2 swap"
        # 6. integer-valued partials sum exactly
        ints = [nearest_codes(dtype, np.round(lib_decode(dtype, p).astype(np.float64) * 16).clip(-128, 128))
                for p in P]
        out_i, _ = o.run(ALLREDUCE, ints, dtype=dtype)
        exact = sum(lib_decode(dtype, p).astype(np.float64) for p in ints)
        rep = lib_decode(dtype, nearest_codes(dtype, exact)).astype(np.float64) == exact
        assert np.array_equal(lib_decode(dtype, out_i)[rep].astype(np.float64), exact[rep]), f"{name} inv6"
        # 7. a zero row gives out = 0 exactly
        zP = [np.zeros_like(p) for p in P]
        out_z, ro_z = o.run(RMSNORM, zP, zeros, G, wl.eps, dtype=dtype)
        assert not out_z.any() and not ro_z.any(), f"{name} inv7 zero row"


# ---------------------------------------------------------------------------
# General layouts: row strides and binary32 partials
# ---------------------------------------------------------------------------


def _widen_rows(a, H, pad, fill):
    """a [M,H] array embedded in a wider [M,H+pad] array filled with `fill`;
    returns the [M,H] column view."""
    M = a.shape[0]
    big = np.full((M, H + pad), fill, dtype=a.dtype)
    big[:, :H] = a
    return big[:, :H], big


def check_strided(o, trials=12, seed=5):
    """Rows embedded in wider buffers (garbage in the padding) give the
    contiguous results, and the padding of the outputs is left untouched."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        dtype = BF16 if t % 2 == 0 else FP16
        W, M, H = int(rng.integers(1, 6)), int(rng.integers(1, 5)), int(rng.choice([1, 5, 8, 24, 40]))
        P = [_draw(rng, dtype, (M, H), 2.0) for _ in range(W)]
        R = _draw(rng, dtype, (M, H), 1.0)
        G = nearest_codes(dtype, 0.5 + rng.random(H))
        for pat in (ALLREDUCE, RMSNORM):
            want = o.run(pat, P, R, G, 1e-6, dtype=dtype)
            pads = [int(x) for x in rng.integers(1, 9, size=4)]
            junk = np.uint16(0x7F81 if dtype == BF16 else 0x7C01)  # NaN codes: any read of them shows
            Ps, bigs = [], []
            for p in P:
                v, b = _widen_rows(p, H, pads[0], junk)
                Ps.append(v)
                bigs.append(b)
            # one shared row stride for all partials
            Ps = [b[:, :H] for b in bigs]
            Rv, _ = _widen_rows(R, H, pads[1], junk)
            Ov, Ob = _widen_rows(np.zeros((M, H), np.uint16), H, pads[2], np.uint16(0x1234))
            ROv, ROb = _widen_rows(np.zeros((M, H), np.uint16), H, pads[3], np.uint16(0x1234))
            out, ro = o.run_general(pat, Ps, Rv, G, 1e-6, dtype=dtype, out=Ov, residual_out=ROv)
            assert_codes_equal(dtype, out, want[0], f"strided trial {t} out")
            assert (Ob[:, H:] == 0x1234).all(), "strided out: padding written"
            if pat == RMSNORM:
                assert_codes_equal(dtype, ro, want[1], f"strided trial {t} residual_out")
                assert (ROb[:, H:] == 0x1234).all(), "strided residual_out: padding written"


def check_f32_partials(o, trials=40, seed=6):
    """binary32 partials: the rank-order sum of numpy float32 values, then the
    residual add, one rounding; out by exact rationals. Odd H included."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        dtype = BF16 if t % 2 == 0 else FP16
        W, M = int(rng.integers(1, 7)), int(rng.integers(1, 4))
        H = int(rng.choice([1, 3, 7, 8, 13, 24]))
        top = 10.0 if dtype == FP16 else 20.0
        P32 = [(rng.standard_normal((M, H)) * 2.0 ** rng.uniform(-6, top)).astype(np.float32) for _ in range(W)]
        if t % 4 == 1 and W >= 3:  # cancellation: exact only in array order
            P32[1] = -P32[0]
        R = _draw(rng, dtype, (M, H), 1.0)
        G = nearest_codes(dtype, 0.5 + rng.random(H))
        eps32 = np.float32(1e-6)
        out, _ = o.run_general(ALLREDUCE, P32, dtype=dtype)
        assert_codes_equal(dtype, out, nearest_codes(dtype, ref_sum_f32(P32).astype(np.float64)),
                           f"f32 trial {t} allreduce")
        out, ro = o.run_general(RMSNORM, P32, R, G, float(eps32), dtype=dtype)
        want_ro = nearest_codes(dtype, ref_sum_f32(P32, lib_decode(dtype, R)).astype(np.float64))
        assert_codes_equal(dtype, ro, want_ro, f"f32 trial {t} residual_out")
        assert_codes_equal(dtype, out, ref_rmsnorm_exact(dtype, want_ro, G, eps32), f"f32 trial {t} out")


def run_battery(o, quick=False):
    """Every pin, in an order that fails fast on the cheap ones."""
    check_worked_rows(o)
    check_inv_rms_r2(o)
    check_one_rounding(o)
    check_exact_tiny(o, trials=40 if quick else 150)
    check_strided(o, trials=6 if quick else 12)
    check_f32_partials(o, trials=16 if quick else 40)
    check_widen(o)
    check_roundtrip(o)
    check_narrow_f32(o, n=100_000 if quick else 1_000_000)
    check_narrow_f64(o, n=20_000 if quick else 200_000)
    check_invariants(o, names=("small", "k3_tp8", "tp16_8mib") if quick else tuple(SMALL_M))
