"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with something other than itself:

* values the pages print (``tests/golden/``),
* closed forms of the matmul (all-zero codes, all-15 codes, identity-like
  weights, ramps) computed here with numpy/fractions from bf16 values decoded
  by torch (a library routine, not the oracle's decoder),
* brute force in exact rational arithmetic on tiny inputs,
* an independent bit-level formulation of bf16 round-to-nearest-even, and
  torch's own float32 -> bfloat16 cast on a sample.

``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on deliberately broken copies of the oracle to show each plausible
mistake is caught by at least one pin.

Citations (page titles; sections in quotes):
  [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
  [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels" model card
"""
from __future__ import annotations

import os
import struct
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
G = 64


# ---- independent helpers (no oracle code) -------------------------------------

def torch_bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns with torch's bfloat16 -> float64 conversion."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def torch_f32_to_bf16(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_bf16_from_f32(u: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even on the float32 bit pattern: add 0x7FFF plus the
    lowest kept bit, then drop the low 16 bits.  NaNs are compared separately."""
    u = u.astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r & 0xFFFF).astype(np.uint16)


def frac_from_bf16(h: int) -> Fraction:
    """Exact value of a finite bf16 pattern (via the float32 it widens to)."""
    return Fraction(struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0])


def frac_to_bf16(v: Fraction) -> int:
    """Exact nearest-even rounding of a rational to bf16 (finite results only)."""
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    sp = Fraction(2) ** (max(e, -126) - 7)
    q = a / sp
    fl = q.numerator // q.denominator
    d = q - fl
    r = fl + 1 if d > Fraction(1, 2) or (d == Fraction(1, 2) and fl % 2 == 1) else fl
    val = r * sp
    if val < Fraction(2) ** -126:
        return sign | int(r)
    e2 = val.numerator.bit_length() - val.denominator.bit_length()
    while Fraction(2) ** e2 > val:
        e2 -= 1
    while Fraction(2) ** (e2 + 1) <= val:
        e2 += 1
    sig = val / Fraction(2) ** (e2 - 7)
    assert sig.denominator == 1 and 128 <= sig < 256
    return sign | ((e2 + 127) << 7) | (int(sig) - 128)


def nibble_bitwise(word: int, i: int) -> int:
    """Code i of a packed word, assembled one bit at a time."""
    q = 0
    for bit in range(4):
        q |= ((word >> (4 * i + bit)) & 1) << bit
    return q


def pack_page_order(codes) -> int:
    """[W2D2 "Packed Storage Layout"]: (h<<28)|(g<<24)|...|(b<<4)|a."""
    word = 0
    for i, c in enumerate(codes):
        word |= (int(c) & 0xF) << (4 * i)
    return word


def bf16_const(v: float) -> int:
    return int(torch_f32_to_bf16(np.array([v], dtype=np.float32))[0])


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def random_bf16(rng, shape, lo=-2.0, hi=2.0) -> np.ndarray:
    return torch_f32_to_bf16(rng.uniform(lo, hi, size=shape).astype(np.float32))


# ---- unpack --------------------------------------------------------------------

def pin_packing_golden(o):
    with open(os.path.join(GOLDEN, "w2d2_packing.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split()
            codes, word = [int(p) for p in parts[:8]], int(parts[8], 16)
            assert pack_page_order(codes) == word, "fixture inconsistent with the page's formula"
            q = o.unpack(np.array([[word]], dtype=np.uint32), 1, 8)
            assert list(q[0]) == codes, f"unpack({word:#x}) = {list(q[0])}, page gives {codes}"


def pin_unpack_exhaustive(o):
    words = []
    expect = []
    for v in range(16):
        for i in range(8):
            words.append(v << (4 * i))
            e = [0] * 8
            e[i] = v
            expect.append(e)
    q = o.unpack(np.array(words, dtype=np.uint32).reshape(-1, 1), len(words), 8)
    assert np.array_equal(q, np.array(expect, dtype=np.uint8)), "single-code words unpack wrongly"
    rng = _rng(11)
    W = rng.integers(0, 2**32, size=(5, 24), dtype=np.uint64).astype(np.uint32)
    q = o.unpack(W, 5, 192)
    for n in range(5):
        for k in range(192):
            assert q[n, k] == nibble_bitwise(int(W[n, k // 8]), k % 8)


# ---- dequant -------------------------------------------------------------------

def pin_dequant_endpoints(o):
    """[W2D2 "Reconstruct a Stored Group"]: both orientations of a signed scale."""
    with open(os.path.join(GOLDEN, "w2d2_dequant_endpoints.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for s, b, q, val, kind in rows:
        sb, bb, q = bf16_const(float(s)), bf16_const(float(b)), int(q)
        w = o.dequant(np.full((1, 8), q * 0x11111111, dtype=np.uint32), np.array([[sb]], dtype=np.uint16),
                      np.array([[bb]], dtype=np.uint16), 1, 64)  # all 64 codes of the group = q
        exact = q * float(torch_bf16_to_f64(np.array([sb]))[0]) + float(torch_bf16_to_f64(np.array([bb]))[0])
        assert np.all(w == exact), f"dequant(q={q}, s={s}, b={b}) = {w[0, 0]}, q*s+b = {exact}"
        if kind == "exact":
            assert w[0, 0] == float(torch_bf16_to_f64(np.array([bf16_const(float(val))]))[0])
        else:
            assert abs(w[0, 0] - float(val)) <= 0.01, f"{w[0, 0]} is not about {val}"
        # orientation: positive scale puts code 15 above code 0, negative below
        w0 = o.dequant(np.zeros((1, 8), dtype=np.uint32), np.array([[sb]], dtype=np.uint16),
                       np.array([[bb]], dtype=np.uint16), 1, 64)[0, 0]
        w15 = o.dequant(np.full((1, 8), 0xFFFFFFFF, dtype=np.uint32), np.array([[sb]], dtype=np.uint16),
                        np.array([[bb]], dtype=np.uint16), 1, 64)[0, 0]
        assert (w15 > w0) == (float(s) > 0)


def pin_dequant_random(o):
    rng = _rng(12)
    N, K = 3, 192
    W = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    S = random_bf16(rng, (N, K // G), -0.05, 0.05)
    B = random_bf16(rng, (N, K // G), -1.0, 1.0)
    w = o.dequant(W, S, B, N, K)
    s64, b64 = torch_bf16_to_f64(S), torch_bf16_to_f64(B)
    for n in range(N):
        for k in range(K):
            q = nibble_bitwise(int(W[n, k // 8]), k % 8)
            assert w[n, k] == q * s64[n, k // G] + b64[n, k // G]


# ---- bf16 ----------------------------------------------------------------------

def pin_bf16_decode_all(o):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = o.bf16_to_f64(h)
    ref = torch_bf16_to_f64(h)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan]), "bf16 decode differs from torch"


def pin_bf16_special(o):
    cases = [(0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3F80), (-2.0, 0xC000), (float("inf"), 0x7F80),
             (float("-inf"), 0xFF80), (2.0**-133, 0x0001), (2.0**-134, 0x0000),  # tie at half the min -> even 0
             (1.5 * 2.0**-134, 0x0001), (2.0**-126, 0x0080), (3.3895313892515355e38, 0x7F7F),
             (3.4e38, 0x7F80),  # rounds past the largest finite bf16
             (1.0 + 2.0**-8, 0x3F80),                 # exact tie -> even
             (1.0 + 3 * 2.0**-8, 0x3F82),             # exact tie -> even (up)
             (1.0 + 2.0**-8 + 2.0**-40, 0x3F81),      # just above a tie: up (a float32 detour would tie)
             (-(1.0 + 2.0**-8 + 2.0**-40), 0xBF81)]
    for v, want in cases:
        got = int(o.bf16_from_f64(np.array([v]))[0])
        assert got == want, f"bf16({v!r}) = {got:#06x}, want {want:#06x}"
    n = int(o.bf16_from_f64(np.array([float("nan")]))[0])
    assert (n & 0x7F80) == 0x7F80 and (n & 0x7F) != 0


def pin_bf16_from_f32_sweep(o):
    """Every float32 high half, with low halves that cover each rounding class."""
    lows = np.array([0x0000, 0x0001, 0x1234, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xBEEF, 0xFFFE, 0xFFFF], dtype=np.uint32)
    hi = np.arange(65536, dtype=np.uint32)
    u = ((hi[:, None] << 16) | lows[None, :]).ravel()
    rng = _rng(13)
    u = np.concatenate([u, rng.integers(0, 2**32, size=1 << 21, dtype=np.uint64).astype(np.uint32)])
    f = u.view(np.float32)
    mine = o.bf16_from_f32(f)
    nan = np.isnan(f)
    ref = bits_bf16_from_f32(u)
    assert np.array_equal(mine[~nan], ref[~nan]), "bf16 RNE differs from the bit-level formulation"
    m = mine[nan]
    assert np.all((m & 0x7F80) == 0x7F80) and np.all((m & 0x7F) != 0), "NaN must stay NaN"
    sample = f[::97]
    ok = ~np.isnan(sample)
    assert np.array_equal(o.bf16_from_f32(sample)[ok], torch_f32_to_bf16(sample)[ok]), "differs from torch"


def pin_bf16_from_f64_exact(o):
    """Direct fp64 -> bf16 rounding against exact rational rounding."""
    rng = _rng(14)
    vals = list(rng.normal(0, 1, 300)) + list(rng.normal(0, 1, 100) * 1e-38) + list(rng.normal(0, 1, 100) * 1e30)
    for i in range(64):  # near-ties that differ only below float32 precision
        base = 1.0 + (2 * i + 1) * 2.0**-8
        vals += [base + 2.0**-40, base - 2.0**-40, -base - 2.0**-45]
    got = o.bf16_from_f64(np.array(vals, dtype=np.float64))
    for v, g in zip(vals, got):
        want = frac_to_bf16(Fraction(float(v)))
        assert int(g) == want, f"bf16({v!r}) = {int(g):#06x}, exact rounding gives {want:#06x}"


def pin_ulp(o):
    cases = [(1.0, 2.0**-7), (1.99, 2.0**-7), (2.0, 2.0**-6), (-3.0, 2.0**-6), (0.75, 2.0**-8),
             (2.0**-126, 2.0**-133), (2.0**-130, 2.0**-133), (0.0, 2.0**-133), (1e30, 2.0**(99 - 7))]
    for v, want in cases:
        got = float(o.ulp_bf16(np.array([v]))[0])
        assert got == want, f"ulp_bf16({v}) = {got}, want {want}"


# ---- matmul closed forms ---------------------------------------------------------

def _group_sums(x64: np.ndarray) -> np.ndarray:
    M, K = x64.shape
    return x64.reshape(M, K // G, G).sum(axis=2)


def _check_close(y, want, absdot, rel=1e-12, what=""):
    err = np.abs(y - want)
    bound = rel * np.maximum(absdot, 1e-300) + 1e-300
    worst = int(np.argmax((err - bound).ravel()))
    assert np.all(err <= bound), f"{what}: err {err.ravel()[worst]:.3e} exceeds bound {bound.ravel()[worst]:.3e}"


def pin_mm_zero_codes(o):
    """All codes 0: y = sum_g b_g * sum_{k in g} x_k  ([W2D2] affine identity with q = 0)."""
    rng = _rng(21)
    for (M, N, K) in [(1, 5, 64), (3, 9, 320), (2, 1, 128)]:
        x = random_bf16(rng, (M, K))
        S = random_bf16(rng, (N, K // G), -0.02, 0.02)
        B = random_bf16(rng, (N, K // G))
        y, ad = o.mm(x, np.zeros((N, K // 8), dtype=np.uint32), S, B, M, N, K)
        want = _group_sums(torch_bf16_to_f64(x)) @ torch_bf16_to_f64(B).T
        _check_close(y, want, ad, what=f"zero codes {M}x{N}x{K}")
        want_abs = np.abs(torch_bf16_to_f64(x)).reshape(M, K // G, G).sum(2) @ np.abs(torch_bf16_to_f64(B)).T
        _check_close(ad, want_abs, ad, what="absdot, zero codes")


def pin_mm_all15(o):
    """All codes 15: y = sum_g (15 s_g + b_g) sum_{k in g} x_k, with signed scales."""
    rng = _rng(22)
    for (M, N, K) in [(1, 4, 64), (4, 7, 256)]:
        x = random_bf16(rng, (M, K))
        S = random_bf16(rng, (N, K // G), -0.1, 0.1)
        B = random_bf16(rng, (N, K // G))
        y, ad = o.mm(x, np.full((N, K // 8), 0xFFFFFFFF, dtype=np.uint32), S, B, M, N, K)
        eff = 15.0 * torch_bf16_to_f64(S) + torch_bf16_to_f64(B)
        want = _group_sums(torch_bf16_to_f64(x)) @ eff.T
        _check_close(y, want, ad, what=f"all-15 codes {M}x{N}x{K}")


def pin_mm_zero_padding(o):
    """K % 512 != 0 runs on the tensor cores as K' = 512 ceil(K / 512) with zero
    activations, scales and biases in the padding groups (any codes there): the
    definition then gains only exact zero terms, so the padded problem's
    outputs and absolute dot products equal the unpadded ones."""
    rng = _rng(26)
    for (M, N, K) in [(1, 3, 64), (3, 5, 576), (2, 4, 2304)]:
        Kp = -(-K // 512) * 512
        x = random_bf16(rng, (M, K))
        W = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
        S = random_bf16(rng, (N, K // G), -0.1, 0.1)
        B = random_bf16(rng, (N, K // G))
        xp = np.zeros((M, Kp), dtype=np.uint16)
        xp[:, :K] = x
        Wp = rng.integers(0, 2**32, size=(N, Kp // 8), dtype=np.uint64).astype(np.uint32)
        Wp[:, :K // 8] = W
        Sp = np.zeros((N, Kp // G), dtype=np.uint16)
        Bp = np.zeros((N, Kp // G), dtype=np.uint16)
        Sp[:, :K // G] = S
        Bp[:, :K // G] = B
        y, ad = o.mm(x, W, S, B, M, N, K)
        yp, adp = o.mm(xp, Wp, Sp, Bp, M, N, Kp)
        assert np.all(y == yp) and np.all(ad == adp), f"padding {M}x{N}x{K} changed the result"


def pin_mm_identity(o):
    """s = 1, b = 0, code 1 on the diagonal: y = x exactly."""
    rng = _rng(23)
    for K in (64, 128):
        N = K
        W = np.zeros((N, K // 8), dtype=np.uint32)
        for n in range(N):
            W[n, n // 8] = 1 << (4 * (n % 8))
        S = np.full((N, K // G), bf16_const(1.0), dtype=np.uint16)
        B = np.zeros((N, K // G), dtype=np.uint16)
        x = random_bf16(rng, (2, K), -100.0, 100.0)
        y, _ = o.mm(x, W, S, B, 2, N, K)
        assert np.array_equal(y, torch_bf16_to_f64(x)), "identity-like weights must reproduce x"
        assert np.array_equal(o.bf16_from_f64(y), x)


def pin_mm_ramp(o):
    """x_k = k/K, codes (k + n) mod 16, s = 1/16, b = -1/2: exact rational sum."""
    for K in (128, 256):
        N = 3
        x = torch_f32_to_bf16((np.arange(K) / K).astype(np.float32))[None, :]
        W = np.zeros((N, K // 8), dtype=np.uint32)
        for n in range(N):
            for k in range(K):
                W[n, k // 8] |= ((k + n) % 16) << (4 * (k % 8))
        S = np.full((N, K // G), bf16_const(1 / 16), dtype=np.uint16)
        B = np.full((N, K // G), bf16_const(-0.5), dtype=np.uint16)
        y, _ = o.mm(x, W, S, B, 1, N, K)
        for n in range(N):
            want = sum(Fraction(k, K) * (Fraction((k + n) % 16, 16) - Fraction(1, 2)) for k in range(K))
            assert Fraction(y[0, n]) == want, f"ramp n={n}: {y[0, n]} != {float(want)}"


def pin_mm_bruteforce(o):
    """Tiny random cases in exact rational arithmetic, including the bf16 rounding."""
    rng = _rng(24)
    for (M, N, K) in [(1, 1, 64), (2, 4, 64), (2, 3, 128), (1, 4, 128)]:
        x = random_bf16(rng, (M, K))
        W = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
        S = random_bf16(rng, (N, K // G), -0.05, 0.05)
        B = random_bf16(rng, (N, K // G), -0.5, 0.5)
        y, ad = o.mm(x, W, S, B, M, N, K)
        yb = o.bf16_from_f64(y)
        for m in range(M):
            for n in range(N):
                tot = Fraction(0)
                tot_abs = Fraction(0)
                for k in range(K):
                    q = nibble_bitwise(int(W[n, k // 8]), k % 8)
                    w = q * frac_from_bf16(int(S[n, k // G])) + frac_from_bf16(int(B[n, k // G]))
                    p = frac_from_bf16(int(x[m, k])) * w
                    tot += p
                    tot_abs += abs(p)
                assert abs(Fraction(y[m, n]) - tot) <= Fraction(1, 2**50) * tot_abs, f"brute force ({m},{n})"
                assert abs(Fraction(ad[m, n]) - tot_abs) <= Fraction(1, 2**50) * tot_abs, "absdot"
                assert int(yb[m, n]) == frac_to_bf16(tot), f"bf16 of ({m},{n})"


def pin_mm_sampled_columns(o):
    """Sampled columns equal the full result; the thread count changes nothing."""
    rng = _rng(25)
    M, N, K = 3, 37, 192
    x = random_bf16(rng, (M, K))
    W = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    S = random_bf16(rng, (N, K // G), -0.05, 0.05)
    B = random_bf16(rng, (N, K // G), -0.5, 0.5)
    y, ad = o.mm(x, W, S, B, M, N, K, threads=1)
    y4, _ = o.mm(x, W, S, B, M, N, K, threads=4)
    assert np.array_equal(y, y4)
    cols = np.array([36, 0, 17, 17, 5])
    ys, ads = o.mm(x, W, S, B, M, N, K, cols=cols)
    assert np.array_equal(ys, y[:, cols]) and np.array_equal(ads, ad[:, cols])
    # row m of an M-row call is the 1-row call on x[m]
    for m in range(M):
        y1, _ = o.mm(x[m:m + 1], W, S, B, 1, N, K)
        assert np.array_equal(y1[0], y[m])


def pin_mm_id(o):
    """Routed experts: per-expert closed form (zero codes), zero rows for bad ids."""
    rng = _rng(26)
    E, N, K, T = 3, 6, 128, 7
    x = random_bf16(rng, (T, K))
    B = random_bf16(rng, (E, N, K // G))
    S = random_bf16(rng, (E, N, K // G), -0.02, 0.02)
    ids = np.array([2, 0, -1, 1, 3, 2, 0], dtype=np.int32)
    y, ad = o.mm_id(x, np.zeros((E, N, K // 8), dtype=np.uint32), S, B, ids, T, N, K, E)
    xs = _group_sums(torch_bf16_to_f64(x))
    for t in range(T):
        if 0 <= ids[t] < E:
            want = xs[t] @ torch_bf16_to_f64(B[ids[t]]).T
            _check_close(y[t], want, ad[t], what=f"mm_id token {t}")
        else:
            assert np.all(y[t] == 0) and np.all(ad[t] == 0), "out-of-range id must give a zero row"
    # random codes: token t equals the plain matmul on expert ids[t]
    W = rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32)
    y, _ = o.mm_id(x, W, S, B, ids, T, N, K, E)
    for t in range(T):
        if 0 <= ids[t] < E:
            e = ids[t]
            ym, _ = o.mm(x[t:t + 1], W[e], S[e], B[e], 1, N, K)
            assert np.array_equal(ym[0], y[t])


def pin_embed(o):
    """Embedding rows: zero codes give bf16(b) and all-15 codes bf16(15 s + b),
    both exactly representable, so element for element the stored bias (resp.
    the exact value); each output row is its id's row; a bad id gives zeros."""
    rng = _rng(27)
    N, K = 5, 256
    S = random_bf16(rng, (N, K // G), -0.02, 0.02)
    B = random_bf16(rng, (N, K // G))
    ids = np.array([4, 0, 7, 2, 2, -3], dtype=np.int32)
    e0 = o.embed(np.zeros((N, K // 8), dtype=np.uint32), S, B, ids, N, K)
    e15 = o.embed(np.full((N, K // 8), 0xFFFFFFFF, dtype=np.uint32), S, B, ids, N, K)
    for t, n in enumerate(ids):
        if 0 <= n < N:
            assert np.array_equal(e0[t], np.repeat(B[n], G)), f"zero codes, token {t}"
            want = 15.0 * torch_bf16_to_f64(S[n]) + torch_bf16_to_f64(B[n])
            got = torch_bf16_to_f64(e15[t].reshape(K // G, G))
            assert np.all(np.abs(got - want[:, None]) <= np.abs(want[:, None]) * 2.0 ** -8), f"all-15 codes, token {t}"
        else:
            assert np.all(e0[t] == 0) and np.all(e15[t] == 0), "out-of-range id must give a zero row"


def pin_group128(o):
    """Group size 128: equal, bit for bit, to group size 64 with every scale and
    bias repeated over the two 64-halves of its group (the same weights, the
    same loop order); zero codes give the closed form sum_g b_g sum_{k in g} x_k;
    dequant's bias follows the 128-group."""
    rng = _rng(28)
    M, N, K = 2, 5, 512
    x = random_bf16(rng, (M, K))
    W = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    S = random_bf16(rng, (N, K // 128), -0.02, 0.02)
    B = random_bf16(rng, (N, K // 128))
    y128, ad128 = o.mm(x, W, S, B, M, N, K, group=128)
    y64, ad64 = o.mm(x, W, np.repeat(S, 2, axis=1), np.repeat(B, 2, axis=1), M, N, K)
    assert np.array_equal(y128, y64) and np.array_equal(ad128, ad64), "group 128 != repeated group 64"
    y0, ad0 = o.mm(x, np.zeros_like(W), S, B, M, N, K, group=128)
    xs = torch_bf16_to_f64(x).reshape(M, K // 128, 128).sum(axis=2)
    _check_close(y0, xs @ torch_bf16_to_f64(B).T, ad0, what="group 128, zero codes")
    w0 = o.dequant(np.zeros_like(W), S, B, N, K, group=128)
    assert np.array_equal(w0, np.repeat(torch_bf16_to_f64(B), 128, axis=1)), "group 128 dequant bias"


# ---- STQ1_0, the ternary format of [HY4] "Notes and gotchas" -------------------

SQW, SQB = 256, 42  # weights and bytes per block


def _stq1_block(codes, signs, dbits: int) -> np.ndarray:
    """One 42-byte block from 64 group codes, 64 sign bits and fp16 bits, laid
    out as the page lists: qs[32] (two codes a byte, group g in byte g/2, low
    nibble for even g), sign[8] (bit g%8 of byte g/8), d little endian."""
    b = np.zeros(SQB, dtype=np.uint8)
    for g in range(64):
        b[g // 2] |= (int(codes[g]) & 0xF) << (4 * (g % 2))
        b[32 + g // 8] |= (int(signs[g]) & 1) << (g % 8)
    b[40], b[41] = dbits & 0xFF, dbits >> 8
    return b


def _fp16(bits: int) -> float:
    """fp16 bits -> float via numpy's float16 (a library decoder)."""
    return float(np.array([bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0])


ONE16 = 0x3C00  # fp16 1.0


def _stq1_group0(o, c: int, s: int) -> list[int]:
    """Lane values of group 0 read back through dequant (the path mm takes):
    every group holds code c and sign s, d = 1; group 0 owns weights 0, 16, 32, 48."""
    w = o.stq1_dequant(_stq1_block([c] * 64, [s] * 64, ONE16), 1, SQW)[0]
    return [int(w[16 * p]) for p in range(4)]


def pin_stq1_codebook(o):
    """The 32 group patterns against what the page fixes: one zero lane, named
    by the code's high bits; three +-1 lanes; a 32-entry codebook whose sign = 1
    half is the negation of the sign = 0 half, i.e. codebook bytes
    q' = 0xAA - q with lane l stored as v + 1 in bits 2l..2l+1; two low code
    bits that each flip one lane's sign; all 32 patterns distinct, which with
    one zero and three unit lanes is every such pattern.  Last the reading of
    which lanes the flips reach (ascending order of the non-zero lanes)."""
    import itertools
    pats = {}
    for s in (0, 1):
        for c in range(16):
            v = _stq1_group0(o, c, s)
            assert v == o.stq1_lanes(c, s), f"dequant and the lane table disagree at code {c}, sign {s}"
            assert v.count(0) == 1 and v.index(0) == c >> 2, f"zero lane of code {c}"
            assert all(abs(t) == 1 for i, t in enumerate(v) if i != c >> 2)
            pats[(c, s)] = v
    byte = {k: sum((v[l] + 1) << (2 * l) for l in range(4)) for k, v in pats.items()}
    for c in range(16):
        assert byte[(c, 1)] == 0xAA - byte[(c, 0)], f"codebook byte identity fails at code {c}"
    every = {p for p in itertools.product((-1, 0, 1), repeat=4) if p.count(0) == 1}
    assert {tuple(v) for v in pats.values()} == every and len(every) == 32
    for z in range(4):
        base = pats[(4 * z, 0)]
        assert all(t in (0, 1) for t in base), "flip bits 00 flip nothing"
        d1 = [i for i in range(4) if pats[(4 * z + 1, 0)][i] != base[i]]
        d2 = [i for i in range(4) if pats[(4 * z + 2, 0)][i] != base[i]]
        d3 = [i for i in range(4) if pats[(4 * z + 3, 0)][i] != base[i]]
        assert len(d1) == 1 and len(d2) == 1 and d1 != d2 and sorted(d1 + d2) == d3, f"flip bits, zero lane {z}"
        nz = [i for i in range(4) if i != z]
        assert d1 == [nz[0]] and d2 == [nz[1]], "reading: bit 0 flips the first non-zero lane, bit 1 the second"


def pin_stq1_layout(o):
    """Where each weight, code, sign bit and scale sits: the page's map
    g = (w/64)*16 + w%16, p = (w%64)/16 seen through zero lanes and a single
    negated group, fp16 scales against numpy's decoder, and the block order
    of a row-major [N][K/256] matrix."""
    w = o.stq1_dequant(_stq1_block([0] * 64, [0] * 64, ONE16), 1, SQW)[0]
    want = np.array([0.0 if (k % 64) // 16 == 0 else 1.0 for k in range(SQW)])
    assert np.array_equal(w, want), "code 0 everywhere: lane 0 (w % 64 < 16) must be the zero lane"
    codes = [12] * 64                 # zero lane 3 everywhere ...
    codes[5] = 0                      # ... but group 5 (an odd group: high nibble of qs[2]) and
    codes[20] = 4                     # group 20 (even: low nibble of qs[10]) zero at lanes 0 and 1
    w = o.stq1_dequant(_stq1_block(codes, [0] * 64, ONE16), 1, SQW)[0]
    zeros = {k for k in range(SQW) if w[k] == 0}
    want_zeros = {(g // 16) * 64 + 48 + g % 16 for g in range(64) if g not in (5, 20)} | {5, 64 + 16 + 4}
    assert zeros == want_zeros, f"zero lanes at {sorted(zeros ^ want_zeros)[:6]} differ from the page's map"
    signs = [0] * 64
    signs[10] = 1                     # bit 2 of sign[1]
    w = o.stq1_dequant(_stq1_block([0] * 64, signs, ONE16), 1, SQW)[0]
    neg = {k for k in range(SQW) if w[k] < 0}
    assert neg == {16 + 10, 32 + 10, 48 + 10}, f"negated weights {sorted(neg)}: group 10 is weights 26, 42, 58"
    for dbits in (0x3555, 0x0001, 0x03FF, 0x0400, 0xBC00, 0x7BFF, 0x1819, 0x251F):
        w = o.stq1_dequant(_stq1_block([0] * 64, [0] * 64, dbits), 1, SQW)[0]
        assert w[16] == _fp16(dbits) and w[0] == 0.0, f"fp16 scale 0x{dbits:04x}"
    ds = [[0x3C00, 0x4000], [0x4200, 0x4400], [0x4500, 0x4600]]  # 1, 2, 3, 4, 5, 6
    blocks = np.stack([np.stack([_stq1_block([0] * 64, [0] * 64, d) for d in row]) for row in ds])
    W = o.stq1_dequant(blocks, 3, 2 * SQW)
    for n in range(3):
        for b in range(2):
            assert W[n, b * SQW + 16] == _fp16(ds[n][b]), f"block ({n}, {b}) out of place"


def pin_stq1_mm(o):
    """y = x W^T against closed forms and against dequant: with code 0 and no
    signs every block adds d * (sum of its lane 1..3 activations); all
    signs set negates it; unit activations read back single columns of W; a
    random case equals numpy's fp64 product of the dequantized matrix, and
    absdot its |x| |W| product; sampled columns equal the full result."""
    rng = _rng(31)
    N, K, M = 3, 512, 2
    dbits = [[int(b) for b in rng.integers(0x1400, 0x3000, size=K // SQW)] for _ in range(N)]
    for sgn in (0, 1):
        blocks = np.stack([np.stack([_stq1_block([0] * 64, [sgn] * 64, d) for d in row]) for row in dbits])
        x = rng.standard_normal((M, K)).astype(np.float32)
        y, ad = o.stq1_mm(x, blocks, M, N, K)
        # weight w = 64 t + 16 p + j of a block is lane p: sum lanes 1..3
        x64 = x.astype(np.float64).reshape(M, K // SQW, 4, 4, 16)[:, :, :, 1:, :].sum(axis=(2, 3, 4))
        dv = np.array([[_fp16(d) for d in row] for row in dbits])
        want = (1 - 2 * sgn) * x64 @ dv.T
        _check_close(y, want, ad, what=f"stq1 closed form, signs {sgn}")
    blocks = rng.integers(0, 256, size=(N, K // SQW, SQB), dtype=np.uint8)
    blocks[:, :, 40:] = np.frombuffer(np.array(rng.uniform(0.002, 0.02, N * (K // SQW)), dtype=np.float16)
                                      .tobytes(), dtype=np.uint8).reshape(N, K // SQW, 2)
    W = o.stq1_dequant(blocks, N, K)
    eye = np.eye(K, dtype=np.float32)[::37]
    y, _ = o.stq1_mm(eye, blocks, eye.shape[0], N, K)
    assert np.array_equal(y, W[:, ::37].T), "unit activations must read back columns of W"
    x = rng.standard_normal((M, K)).astype(np.float32)
    y, ad = o.stq1_mm(x, blocks, M, N, K)
    _check_close(y, x.astype(np.float64) @ W.T, ad, what="stq1 random vs dequant")
    _check_close(ad, np.abs(x.astype(np.float64)) @ np.abs(W).T, ad, what="stq1 absdot")
    ys, _ = o.stq1_mm(x, blocks, M, N, K, cols=np.array([2, 0]))
    assert np.array_equal(ys, y[:, [2, 0]])


def pin_stq1_mm_id(o):
    """Routed STQ1_0: token t equals the plain product on expert ids[t]; a bad
    id gives a zero row; get_rows returns the dequantized rows (zeros for a bad id)."""
    rng = _rng(32)
    E, N, K, T = 3, 4, 256, 6
    blocks = rng.integers(0, 256, size=(E, N, K // SQW, SQB), dtype=np.uint8)
    blocks[..., 41] &= 0x3F  # finite scales
    x = rng.standard_normal((T, K)).astype(np.float32)
    ids = np.array([2, 0, 5, 1, -1, 2], dtype=np.int32)
    y, ad = o.stq1_mm_id(x, blocks, ids, T, N, K, E)
    for t in range(T):
        if 0 <= ids[t] < E:
            ym, am = o.stq1_mm(x[t:t + 1], blocks[ids[t]], 1, N, K)
            assert np.array_equal(ym[0], y[t]) and np.array_equal(am[0], ad[t]), f"token {t}"
        else:
            assert np.all(y[t] == 0) and np.all(ad[t] == 0), "out-of-range id must give a zero row"
    rows = o.stq1_get_rows(blocks[1], np.array([3, 0, 9, 3]), N, K)
    W = o.stq1_dequant(blocks[1], N, K)
    assert np.array_equal(rows[0], W[3].astype(np.float32)) and np.array_equal(rows[1], W[0].astype(np.float32))
    assert np.all(rows[2] == 0) and np.array_equal(rows[3], rows[0])


PINS = [pin_packing_golden, pin_unpack_exhaustive, pin_dequant_endpoints, pin_dequant_random,
        pin_ulp, pin_bf16_special, pin_mm_zero_codes, pin_mm_all15, pin_mm_zero_padding, pin_mm_identity,
        pin_mm_ramp,
        pin_mm_sampled_columns, pin_mm_id, pin_mm_bruteforce, pin_bf16_decode_all,
        pin_bf16_from_f64_exact, pin_bf16_from_f32_sweep, pin_embed, pin_group128,
        pin_stq1_codebook, pin_stq1_layout, pin_stq1_mm, pin_stq1_mm_id]
