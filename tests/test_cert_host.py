"""The certificate of the wide kernels' plain sum (widths 4..8).

From W = 5 (backward) and W = 4 (forward) the main kernels sum the W exact
fp32 products of a value in a fixed tree (pairs by a multiply and a fused
multiply-add, then the pairs' tree) and keep the result when
cert_factor * max_k|w_k| * sum_k|g_k| (formed with upward rounding) <= |sum|;
otherwise the channel is recomputed with the compensated cascade. The claim
is that every kept value, rounded once to the 16-bit type, is within 1 ulp of
the exact sum rounded once (the acceptance bar of the page's gradX).

These CPU tests check the claim by simulation, independently of the kernel's
build: the factors in device_common.cuh are read as text and compared with
the bound they rest on, and the fp32 tree (IEEE round-to-nearest additions;
a fused multiply-add of two exact products rounds once, as a float32 add of
them does) runs in numpy on seeded inputs built for heavy cancellation, where
the certificate is tight. Exact sums come from float64, exact here because
the inputs span a narrow exponent range.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "causal_conv_backward_gb300", "csrc", "device_common.cuh")

# significand bits after the point: fp16 10, bf16 7 (dtype codes: bf16 0, fp16 1)
MBITS = {"fp16": 10, "bf16": 7}


def header_factor(dt: str, W: int) -> float:
    """cert_factor<DT, W>() as written in the header: the return expression
    with its level count kL (itself a function of W) substituted."""
    txt = open(HEADER).read()
    body = txt[txt.index("constexpr float cert_factor()"):]
    body = body[:body.index("\n}")]
    m = re.search(r"kL = W <= (\d+) \? ([\d.]+)f : ([\d.]+)f;", body)
    assert m, "cert_factor's level count not found"
    L = float(m.group(2)) if W <= int(m.group(1)) else float(m.group(3))
    m = re.search(r"DT == 1 \? ([^:]+) : ([^;]+);", body)
    assert m, "cert_factor's expression not found"

    def ev(expr):
        v = 1.0
        for t in expr.split("*"):
            t = t.strip().rstrip("f")
            v *= L if t == "kL" else float(t)
        return v

    return ev(m.group(1) if dt == "fp16" else m.group(2))


def levels(W: int) -> int:
    """Levels of the kernels' tree below the root whose nodes round (see
    tree()): W <= 4 the pairs only; W = 5..8 the pairs and one more."""
    return 1 if W <= 4 else 2


def needed_factor(mbits: int, W: int) -> float:
    """Smallest factor the argument accepts: |s - exact| <= u (L a (1 + 2u)
    + |s|) must stay below (|s| - that) * 2^-(m+1), half the 16-bit relative
    spacing; the last (1 + 2^-20) is margin."""
    u = 2.0 ** -24
    h = 2.0 ** -(mbits + 1)
    q = u / h * (1 + h) / (1 - u / h * (1 + h))
    return levels(W) * q * (1 + 2 * u) * (1 + 2.0 ** -20)


@pytest.mark.parametrize("W", [4, 5, 6, 7, 8])
def test_header_factors_cover_the_bound(W):
    for dt in ("fp16", "bf16"):
        f = header_factor(dt, W)
        need = needed_factor(MBITS[dt], W)
        assert np.float32(f) >= need, (dt, W)
        # and not loose by more than 0.1 %, which would only cost recomputes
        assert f <= 1.001 * need, (dt, W)


def to_bf16(a):
    """float32 -> nearest bf16 (ties to even), as float32 values."""
    b = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32)


def round16(x, dt):
    """Exact float64 x -> nearest 16-bit value (ties to even), normal range."""
    if dt == "fp16":
        return x.astype(np.float16).astype(np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 2.0 ** 8), e - 8)


def ulp16(x, dt):
    m, e = np.frexp(np.abs(x))
    return np.ldexp(np.ones_like(x), e - 1 - MBITS[dt])


def tree(v):
    """The kernels' dot_tree over exact products v[..., 0:W] in float32:
    pairs (2j, 2j+1) rounded once, an odd last product fused into the last
    pair, then the pairs' tree (W = 4: P0 + P1; 5: P0 + (P1 + p4); 6:
    (P0 + P1) + P2; 7: (P0 + P1) + (P2 + p6); 8: (P0 + P1) + (P2 + P3))."""
    f = np.float32
    W = v.shape[1]
    pr = [(v[:, 2 * j] + v[:, 2 * j + 1]).astype(f) for j in range(W // 2)]
    if W % 2:
        pr[-1] = (pr[-1] + v[:, W - 1]).astype(f)
    if len(pr) == 1:
        return pr[0]
    if len(pr) == 2:
        return (pr[0] + pr[1]).astype(f)
    if len(pr) == 3:
        return ((pr[0] + pr[1]).astype(f) + pr[2]).astype(f)
    return ((pr[0] + pr[1]).astype(f) + (pr[2] + pr[3]).astype(f)).astype(f)


def up32(x):
    """float64 x -> the smallest float32 >= x (rounding toward +infinity)."""
    r = x.astype(np.float32)
    lo = r.astype(np.float64) < x
    r[lo] = np.nextafter(r[lo], np.float32(np.inf))
    return r


def operands(rng, n, W, dt, cancel):
    """n rows of W gradY and weight values in the 16-bit type, exponents in
    [-4, 4]; with `cancel`, the last product is set close to minus the sum
    of the others (the cancellation that makes the certificate fail)."""
    conv = (lambda a: a.astype(np.float16).astype(np.float32)) if dt == "fp16" else to_bf16
    g = conv(rng.uniform(1, 2, (n, W)) * 2.0 ** rng.integers(-4, 4, (n, W)) * rng.choice([-1, 1], (n, W)))
    w = conv(rng.uniform(1, 2, (n, W)) * 2.0 ** rng.integers(-4, 4, (n, W)) * rng.choice([-1, 1], (n, W)))
    if cancel:
        rest = (g[:, :-1].astype(np.float64) * w[:, :-1]).sum(1)
        target = -rest * (1 + rng.normal(0, 2.0 ** -rng.integers(4, 20, n)))
        w[:, -1] = conv(np.clip(np.abs(target / g[:, -1]), 2.0 ** -4, 2.0 ** 5)
                        * np.sign(target / g[:, -1]))
    return g, w


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
@pytest.mark.parametrize("W", [4, 5, 6, 7, 8])
def test_every_certified_sum_is_within_one_ulp(dt, W):
    cert = np.float32(header_factor(dt, W))
    rng = np.random.default_rng(1000 * W + (dt == "fp16"))
    kept = failed = 0
    for cancel in (False, True):
        g, w = operands(rng, 60000, W, dt, cancel)
        p32 = g * w                                          # exact in fp32
        p64 = g.astype(np.float64) * w.astype(np.float64)
        assert np.array_equal(p32.astype(np.float64), p64)
        s = tree(p32)
        # kCert * max|w| and sum|g|, each rounded up, and their product
        # rounded up: the kernels' bound, at least kCert * sum|products|
        kmw = up32(np.float64(cert) * np.abs(w).max(1).astype(np.float64))
        gs = up32(np.abs(g).astype(np.float64).sum(1))
        lim = up32(kmw.astype(np.float64) * gs.astype(np.float64))
        assert np.all(lim.astype(np.float64) >= np.float64(cert) * np.abs(p64).sum(1))
        ok = lim <= np.abs(s)
        exact = p64.sum(1)                                   # exact: narrow exponent range
        nz = exact != 0
        ok &= nz
        got = round16(s[ok].astype(np.float64), dt)
        ref = round16(exact[ok], dt)
        err = np.abs(got - ref) / ulp16(ref, dt)
        assert err.max(initial=0) <= 1.0, (dt, W, cancel, err.max())
        kept += int(ok.sum())
        failed += int((~ok & nz).sum())
    # the simulation exercises both outcomes
    assert kept > 60000 and failed > 1000, (kept, failed)


@pytest.mark.parametrize("W", [4, 5, 6, 7, 8])
def test_tree_error_within_the_level_bound(W):
    """The error bound the factor rests on, |s - exact| <= u (L a (1 + 2u)
    + |s|), holds for the tree on random exact products (11-bit by 11-bit
    significands, mixed signs, exponents over 6 binades: float64 sums are
    exact); and with one level fewer it would not (W >= 5), so the level
    count is the one the tree needs."""
    u = 2.0 ** -24
    rng = np.random.default_rng(70 + W)
    worst = worst_fewer = 0.0
    for _ in range(6):
        n = 200000
        sig = rng.integers(1024, 2048, (n, W)).astype(np.float64) * rng.integers(1024, 2048, (n, W))
        p = (sig * 2.0 ** rng.integers(-24, -18, (n, W)) * rng.choice([-1, 1], (n, W))).astype(np.float32)
        assert np.array_equal(p.astype(np.float64), sig * 2.0 ** np.round(np.log2(np.abs(p) / sig))
                              * np.sign(p))                    # products exact in float32
        s = tree(p).astype(np.float64)
        p64 = p.astype(np.float64)
        err, a = np.abs(s - p64.sum(1)), np.abs(p64).sum(1)
        L = levels(W)
        worst = max(worst, float(np.max(err / (u * (L * a * (1 + 2 * u) + np.abs(s))))))
        if L > 1:
            worst_fewer = max(worst_fewer, float(np.max(err / (u * ((L - 1) * a * (1 + 2 * u) + np.abs(s))))))
    assert worst <= 1.0, worst
    assert L == 1 or worst_fewer > 1.0, worst_fewer
