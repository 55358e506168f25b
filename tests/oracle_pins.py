"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the operator page (CANN
"aclnnMaskedCausalConv1dBackward") or the mathematics fixes:

* golden fixtures under ``tests/golden`` (the page's own call example and
  examples worked by hand from its formulas);
* closed forms and shift identities derived by hand from the formulas;
* special cases (mask all zero / all one, S = 1, batch independence);
* brute-force Jacobian transposes of the forward on tiny inputs;
* the adjoint identity <y, gradY> = <x, gradX> = <w, gradWeight>;
* PyTorch's CPU autograd of a float64 depthwise ``conv1d`` (a library routine
  that shares nothing with the oracle);
* sum|terms| of gradWeight (its tolerance scale) summed in numpy;
* numpy's / torch's 16-bit conversions for the oracle's own rounding.

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``, to show that each plausible mistake fails one.
Encoders and decoders used to build expectations here are independent of the
oracle's: numpy ``float16`` and torch ``bfloat16``.
"""
from __future__ import annotations

import glob
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- encoders
def enc(values, dtype: str) -> np.ndarray:
    """16-bit patterns of values by numpy (fp16) / torch (bf16), RNE."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == "fp16":
        return v.astype(np.float16).view(np.uint16)
    # torch rounds float32 -> bfloat16 to nearest even; values reaching here are
    # exactly representable in float32, so this is the direct rounding.
    f32 = v.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), v, equal_nan=True), "value not fp32-exact"
    return torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dec(bits, dtype: str) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        if dtype == "fp16":
            return b.view(np.float16).astype(np.float64)
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bits(rng, shape, dtype, scale=1.0):
    """Random normal values rounded to the 16-bit grid (float32 -> 16-bit RNE
    by numpy for fp16, torch for bf16)."""
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    if dtype == "fp16":
        return v.astype(np.float16).view(np.uint16)
    return torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def small_dyadic_bits(rng, shape, dtype):
    """Values k/4 with |k| <= 16: every product and every short sum is exact."""
    return enc(rng.integers(-16, 17, size=shape) / 4.0, dtype)


def masked_gy(gy_vals, mask, S, B):
    """gradYMasked as [S,B,H] fp64 from values [S,B,H] and mask [B,S] or None."""
    if mask is None:
        return gy_vals.copy()
    return gy_vals * (np.asarray(mask).T != 0)[:, :, None]


# ---------------------------------------------------------------- golden
def _nested(a, dtype):
    return enc(np.array(a, dtype=np.float64), dtype)


def pin_golden(orc):
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    assert files, "no golden fixtures found"
    for f in files:
        with open(f) as fh:
            g = json.load(fh)
        S, B, H, W, dt = g["S"], g["B"], g["H"], g["W"], g["dtype"]
        if g.get("inputs") == {"gradY": "zeros", "x": "zeros", "weight": "zeros", "mask": "zeros"}:
            gy = np.zeros((S, B, H), np.uint16)
            x = np.zeros((S, B, H), np.uint16)
            w = np.zeros((W, H), np.uint16)
            mask = np.zeros((B, S), np.uint8)
            r = orc.bwd(S, B, H, W, dt, gy, x, w, mask)
            assert np.all(dec(r["gx"], dt) == 0), f
            assert np.all(dec(r["gw"], dt) == 0), f
            continue
        gy = _nested(g["gradY"], dt).reshape(S, B, H)
        x = _nested(g["x"], dt).reshape(S, B, H)
        w = _nested(g["weight"], dt).reshape(W, H)
        mask = None if g["mask"] is None else np.array(g["mask"], np.uint8).reshape(B, S)
        r = orc.bwd(S, B, H, W, dt, np.ascontiguousarray(gy), np.ascontiguousarray(x),
                    np.ascontiguousarray(w), mask)
        # the point-wise gradX must give the same bits at every position
        bits, _ = orc.gradx_at(S, B, H, W, dt, np.ascontiguousarray(gy), np.ascontiguousarray(w),
                               mask, np.arange(S * B * H))
        assert np.array_equal(bits.reshape(S, B, H), r["gx"]), f
        if "expected" in g:
            ex_gx = np.array(g["expected"]["gradX"], np.float64).reshape(S, B, H)
            ex_gw = np.array(g["expected"]["gradWeight"], np.float64).reshape(W, H)
            assert np.array_equal(dec(r["gx"], dt), ex_gx), (f, dec(r["gx"], dt), ex_gx)
            assert np.array_equal(dec(r["gw"], dt), ex_gw), (f, dec(r["gw"], dt), ex_gw)
        else:
            ex_gx = np.array(g["expected_bits"]["gradX"], np.uint16).reshape(S, B, H)
            ex_gw = np.array(g["expected_bits"]["gradWeight"], np.uint16).reshape(W, H)
            assert np.array_equal(r["gx"], ex_gx), (f, r["gx"], ex_gx)
            assert np.array_equal(r["gw"], ex_gw), (f, r["gw"], ex_gw)


# ---------------------------------------------------------------- closed forms
def pin_closed_form_ones(orc):
    """mask = null, x = gradY = weight = 1: gradX(i) counts the taps that stay
    inside S (3, then 2 at i = S-2, 1 at i = S-1); gradWeight(k) counts the
    pairs (i, i+2-k) inside S over all batches: B*S, B*(S-1), B*(S-2)."""
    for dt in ("bf16", "fp16"):
        for S in (1, 2, 3, 5, 17):
            for B in (1, 3):
                H = 2
                one = enc(1.0, dt)
                gy = np.full((S, B, H), one, np.uint16)
                x = np.full((S, B, H), one, np.uint16)
                w = np.full((3, H), one, np.uint16)
                r = orc.bwd(S, B, H, 3, dt, gy, x, w, None)
                ex = np.array([min(3, S - i) for i in range(S)], np.float64)
                assert np.array_equal(dec(r["gx"], dt), np.broadcast_to(ex[:, None, None], (S, B, H))), (dt, S, B)
                ex_w = np.array([B * max(S - 2, 0), B * max(S - 1, 0), B * S], np.float64)
                assert np.array_equal(dec(r["gw"], dt), np.broadcast_to(ex_w[:, None], (3, H))), (dt, S, B)


def pin_shift_identities(orc):
    """One-hot weights and inputs isolate single terms of the formulas:
    weight = e2 gives gradX(i) = gYm(i); e1 gives gYm(i+1); e0 gives gYm(i+2)
    (zero past S). x = one-hot at (s, j) gives gradWeight(k) = gYm(s+2-k, j)."""
    rng = np.random.default_rng(7)
    for dt in ("bf16", "fp16"):
        S, B, H = 7, 2, 3
        gy = rand_bits(rng, (S, B, H), dt)
        mask = (rng.random((B, S)) < 0.7).astype(np.uint8)
        gym = masked_gy(dec(gy, dt), mask, S, B)
        x = rand_bits(rng, (S, B, H), dt)
        for tap in range(3):
            w = np.zeros((3, H), np.uint16)
            w[tap, :] = enc(1.0, dt)
            r = orc.bwd(S, B, H, 3, dt, gy, x, w, mask)
            shift = 2 - tap
            ex = np.zeros((S, B, H))
            ex[: S - shift] = gym[shift:]
            assert np.array_equal(dec(r["gx"], dt), ex), (dt, tap)
        w = rand_bits(rng, (3, H), dt)
        for s in range(S):
            for j in range(B):
                xo = np.zeros((S, B, H), np.uint16)
                xo[s, j, :] = enc(1.0, dt)
                r = orc.bwd(S, B, H, 3, dt, gy, xo, w, mask)
                ex = np.zeros((3, H))
                for k in range(3):
                    t = s + 2 - k
                    if t < S:
                        ex[k] = gym[t, j]
                assert np.array_equal(dec(r["gw"], dt), ex), (dt, s, j)


# ---------------------------------------------------------------- special cases
def pin_mask_special_cases(orc):
    """All-zero mask: both gradients exactly zero. All-one mask: bitwise the
    same as mask = nullptr (the optional mask defaults to keeping all)."""
    rng = np.random.default_rng(11)
    for dt in ("bf16", "fp16"):
        S, B, H = 9, 3, 4
        gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                    rand_bits(rng, (3, H), dt))
        r0 = orc.bwd(S, B, H, 3, dt, gy, x, w, np.zeros((B, S), np.uint8))
        assert np.all(dec(r0["gx"], dt) == 0) and np.all(dec(r0["gw"], dt) == 0), dt
        r1 = orc.bwd(S, B, H, 3, dt, gy, x, w, np.ones((B, S), np.uint8))
        rn = orc.bwd(S, B, H, 3, dt, gy, x, w, None)
        assert np.array_equal(r1["gx"], rn["gx"]) and np.array_equal(r1["gw"], rn["gw"]), dt
        # any nonzero byte means keep
        r2 = orc.bwd(S, B, H, 3, dt, gy, x, w, np.full((B, S), 0xA5, np.uint8))
        assert np.array_equal(r2["gx"], rn["gx"]) and np.array_equal(r2["gw"], rn["gw"]), dt


def pin_s1(orc):
    """S = 1 (the page's sample shape): only tap 2 sees a partner, so
    gradWeight(0) = gradWeight(1) = 0, gradWeight(2) = sum_j gYm(0,j) x(0,j)
    and gradX = gYm * weight(2). Products of two 16-bit values are exact in
    float32, so numpy/torch rounding of them is the single rounding."""
    rng = np.random.default_rng(3)
    for dt in ("bf16", "fp16"):
        S, B, H = 1, 2, 384
        gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                    rand_bits(rng, (3, H), dt))
        mask = np.array([[1], [0]], np.uint8)
        r = orc.bwd(S, B, H, 3, dt, gy, x, w, mask)
        gym = masked_gy(dec(gy, dt), mask, S, B)
        ex = dec(enc(gym * dec(w[2], dt)[None, None, :], dt), dt)  # compares +0 == -0
        assert np.array_equal(dec(r["gx"], dt), ex), dt
        assert np.all(dec(r["gw"][:2], dt) == 0), dt
        ex2 = (gym[0] * dec(x, dt)[0]).sum(axis=0)  # B = 2 terms, one of them zero: exact
        assert np.array_equal(dec(r["gw"][2], dt), dec(enc(ex2, dt), dt)), dt


def pin_batch_independence(orc):
    """Changing batch 1 leaves gradX of batch 0 unchanged."""
    rng = np.random.default_rng(5)
    dt, S, B, H = "bf16", 11, 3, 5
    gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                rand_bits(rng, (3, H), dt))
    mask = (rng.random((B, S)) < 0.8).astype(np.uint8)
    r = orc.bwd(S, B, H, 3, dt, gy, x, w, mask)
    gy2, x2 = gy.copy(), x.copy()
    gy2[:, 1] = rand_bits(rng, (S, H), dt)
    x2[:, 1] = rand_bits(rng, (S, H), dt)
    mask2 = mask.copy()
    mask2[1] = 1 - mask2[1]
    r2 = orc.bwd(S, B, H, 3, dt, gy2, x2, w, mask2)
    assert np.array_equal(r["gx"][:, 0], r2["gx"][:, 0])
    assert np.array_equal(r["gx"][:, 2], r2["gx"][:, 2])
    assert not np.array_equal(r["gx"][:, 1], r2["gx"][:, 1])


# ---------------------------------------------------------------- transposes
def pin_jacobian_bruteforce(orc):
    """gradX = J_x^T gradY and gradWeight = J_w^T gradY, with J built column by
    column from the forward evaluated on unit inputs (the forward is linear in
    x for fixed w and in w for fixed x). Small dyadic values keep every sum
    exact, so the comparison is exact. Covers every width the strided calls
    accept, W = 1..8 (widths above S included)."""
    rng = np.random.default_rng(17)
    for dt in ("bf16", "fp16"):
        for W in range(1, 9):
            for S in (1, 2, 3, 4, 5, 6):
                for B in (1, 2):
                    H = 2
                    gy = small_dyadic_bits(rng, (S, B, H), dt)
                    x = small_dyadic_bits(rng, (S, B, H), dt)
                    w = small_dyadic_bits(rng, (W, H), dt)
                    mask = (rng.random((B, S)) < 0.6).astype(np.uint8)
                    r = orc.bwd(S, B, H, W, dt, gy, x, w, mask, want_exact=True)
                    g = dec(gy, dt)
                    one = enc(1.0, dt)
                    gx = np.zeros((S, B, H))
                    for s in range(S):
                        for j in range(B):
                            for h in range(H):
                                e = np.zeros((S, B, H), np.uint16)
                                e[s, j, h] = one
                                col = orc.fwd(S, B, H, W, dt, e, w, mask)
                                gx[s, j, h] = (col * g).sum()
                    assert np.array_equal(gx, r["gx_exact"]), (dt, W, S, B)
                    gw = np.zeros((W, H))
                    for k in range(W):
                        for h in range(H):
                            e = np.zeros((W, H), np.uint16)
                            e[k, h] = one
                            col = orc.fwd(S, B, H, W, dt, x, e, mask)
                            gw[k, h] = (col * g).sum()
                    assert np.array_equal(gw, r["gw_exact"]), (dt, W, S, B)


def pin_adjoint_identity(orc):
    """<y(x,w,mask), gradY> = <x, gradX> = <w, gradWeight> in fp64 (each side
    is the same bilinear form summed in a different order)."""
    rng = np.random.default_rng(23)
    for dt in ("bf16", "fp16"):
        for (S, B, H) in ((1, 1, 3), (2, 2, 4), (37, 3, 8), (130, 2, 16)):
            gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                        rand_bits(rng, (3, H), dt))
            mask = (rng.random((B, S)) < 0.75).astype(np.uint8)
            r = orc.bwd(S, B, H, 3, dt, gy, x, w, mask, want_exact=True)
            y = orc.fwd(S, B, H, 3, dt, x, w, mask)
            a = (y * dec(gy, dt)).sum()
            b = (dec(x, dt) * r["gx_exact"]).sum()
            c = (dec(w, dt) * r["gw_exact"]).sum()
            scale = (np.abs(y) * np.abs(dec(gy, dt))).sum() + 1e-300
            assert abs(a - b) <= 1e-12 * scale and abs(a - c) <= 1e-12 * scale, (dt, S, B, H, a, b, c)


def torch_reference_grads(S, B, H, W, gy_vals, x_vals, w_vals, mask):
    """Gradients of L = sum(mask * conv(x, w) * gradY) by torch autograd in
    float64 on the CPU, with conv the causal depthwise conv1d (left padding
    W-1, groups = H; torch's conv1d is a cross-correlation)."""
    xt = torch.tensor(x_vals, dtype=torch.float64).permute(1, 2, 0).contiguous().requires_grad_(True)
    wt = torch.tensor(w_vals, dtype=torch.float64).t().contiguous().unsqueeze(1).requires_grad_(True)
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (W - 1, 0)), wt, groups=H)
    if mask is not None:
        y = y * torch.tensor(mask != 0, dtype=torch.float64)[:, None, :]
    g = torch.tensor(gy_vals, dtype=torch.float64).permute(1, 2, 0)
    (y * g).sum().backward()
    return xt.grad.permute(2, 0, 1).numpy(), wt.grad.squeeze(1).t().numpy()


def pin_torch_autograd(orc):
    """The oracle's fp64 gradients equal torch's autograd of the masked causal
    depthwise conv1d (fp64, CPU) to rounding; its 16-bit outputs are those
    values rounded once."""
    rng = np.random.default_rng(29)
    for dt in ("bf16", "fp16"):
        for (S, B, H, W) in ((1, 2, 5, 3), (5, 1, 3, 3), (33, 3, 7, 3), (64, 2, 384, 3), (9, 2, 4, 2),
                             (9, 2, 4, 5), (17, 2, 6, 1), (17, 2, 6, 4), (17, 2, 6, 6), (17, 2, 6, 8),
                             (3, 2, 4, 8)):
            gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                        rand_bits(rng, (W, H), dt))
            mask = (rng.random((B, S)) < 0.8).astype(np.uint8)
            r = orc.bwd(S, B, H, W, dt, gy, x, w, mask, want_exact=True)
            tgx, tgw = torch_reference_grads(S, B, H, W, dec(gy, dt), dec(x, dt), dec(w, dt), mask)
            sx = np.abs(dec(gy, dt)).max() * np.abs(dec(w, dt)).max() * W
            assert np.allclose(r["gx_exact"], tgx, rtol=0, atol=1e-12 * sx), (dt, S, B, H, W)
            assert np.allclose(r["gw_exact"], tgw, rtol=0, atol=1e-12 * (r["gw_abs"].max() + 1)), (dt, S, B, H, W)
            # rounding of the oracle's own exact value; equal to rounding torch's
            # value wherever the two fp64 sums agree exactly
            same = r["gx_exact"] == tgx
            if dt == "fp16":
                assert np.array_equal(r["gx"][same], tgx[same].astype(np.float16).view(np.uint16))


def pin_forward_torch(orc):
    """The implied forward y = mask * causal depthwise conv(x, w) equals
    torch's float64 conv1d (left padding W-1, groups = H) on the CPU."""
    rng = np.random.default_rng(41)
    for dt in ("bf16", "fp16"):
        for (S, B, H, W) in ((1, 2, 3, 3), (6, 2, 5, 3), (40, 3, 7, 3), (9, 1, 4, 5), (17, 2, 6, 1),
                             (17, 2, 6, 2), (17, 2, 6, 4), (17, 2, 6, 8), (3, 2, 4, 7)):
            x, w = rand_bits(rng, (S, B, H), dt), rand_bits(rng, (W, H), dt)
            mask = (rng.random((B, S)) < 0.7).astype(np.uint8)
            y = orc.fwd(S, B, H, W, dt, x, w, mask)
            xt = torch.tensor(dec(x, dt)).permute(1, 2, 0)
            wt = torch.tensor(dec(w, dt)).t().contiguous().unsqueeze(1)
            yt = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (W - 1, 0)), wt, groups=H)
            yt = (yt * torch.tensor(mask != 0, dtype=torch.float64)[:, None, :]).permute(2, 0, 1).numpy()
            assert np.allclose(y, yt, rtol=0, atol=1e-12 * (np.abs(yt).max() + 1)), (dt, S, B, H, W)


def pin_forward_rounding(orc):
    """The rounded forward is the fp64 forward rounded once: for fp16 against
    numpy's double -> half rounding, for bf16 against the (separately pinned)
    converter; masked rows are exactly zero."""
    rng = np.random.default_rng(43)
    for dt in ("bf16", "fp16"):
        S, B, H = 33, 3, 16
        x, w = rand_bits(rng, (S, B, H), dt), rand_bits(rng, (3, H), dt)
        mask = (rng.random((B, S)) < 0.7).astype(np.uint8)
        y = orc.fwd(S, B, H, 3, dt, x, w, mask)
        yb = orc.fwd_bits(S, B, H, 3, dt, x, w, mask)
        if dt == "fp16":
            assert np.array_equal(dec(yb, dt), dec(y.astype(np.float16).view(np.uint16), dt))
        else:
            assert np.array_equal(yb, orc.encode(y, dt))
        assert np.all(dec(yb, dt)[(mask.T == 0)] == 0)


def pin_gradw_abs(orc):
    """sum|terms| of gradWeight(k,h), the scale its tolerance is stated
    against, is the sum over j and i of |gYm(i+W-1-k,j,h) * x(i,j,h)| with
    every term of the formula counted once: the shift of the pair, the mask
    and the zero padding past S all as in gradWeight itself. Computed here
    in numpy from independently decoded small dyadic values (every product
    and sum exact), for W = 1..8, with masks and with S shorter than W."""
    rng = np.random.default_rng(47)
    for dt in ("bf16", "fp16"):
        for W in range(1, 9):
            for S in (1, 2, 5, 9):
                for B in (1, 2):
                    H = 3
                    gy = small_dyadic_bits(rng, (S, B, H), dt)
                    x = small_dyadic_bits(rng, (S, B, H), dt)
                    w = small_dyadic_bits(rng, (W, H), dt)
                    mask = (rng.random((B, S)) < 0.6).astype(np.uint8) if B == 2 else None
                    r = orc.bwd(S, B, H, W, dt, gy, x, w, mask, want_gx=False)
                    gym = masked_gy(dec(gy, dt), mask, S, B)
                    xv = dec(x, dt)
                    ex = np.zeros((W, H))
                    for k in range(W):
                        shift = W - 1 - k
                        if shift < S:
                            ex[k] = np.abs(gym[shift:] * xv[: S - shift]).sum(axis=(0, 1))
                    assert np.array_equal(r["gw_abs"], ex), (dt, W, S, B)
    # a case with a closed form: all-ones inputs, no mask, every term +1, so
    # sum|terms| equals gradWeight's pair counts B*(S-(W-1-k)), clamped at 0
    for W in (1, 3, 8):
        S, B, H = 6, 2, 2
        one = enc(1.0, "bf16")
        ones = np.full((S, B, H), one, np.uint16)
        r = orc.bwd(S, B, H, W, "bf16", ones, ones, np.full((W, H), one, np.uint16), None,
                    want_gx=False)
        ex = np.array([B * max(S - (W - 1 - k), 0) for k in range(W)], np.float64)
        assert np.array_equal(r["gw_abs"], np.broadcast_to(ex[:, None], (W, H))), W


# ---------------------------------------------------------------- conversions
def pin_converters(orc):
    """Decoding every 16-bit pattern, and rounding doubles to 16 bits (ties to
    even, gradual underflow, overflow to inf), against numpy float16 and torch
    bfloat16."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("bf16", "fp16"):
        ref = dec(allb, dt)
        got = orc.decode(allb, dt)
        fin = np.isfinite(ref)
        assert np.array_equal(got[fin], ref[fin]), dt
        assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.array_equal(np.isinf(got), np.isinf(ref)), dt
    rng = np.random.default_rng(31)
    # fp16: doubles of every magnitude from below the subnormals to overflow,
    # plus exact ties; numpy rounds double -> half directly.
    v = np.concatenate([
        rng.standard_normal(3000) * 2.0 ** rng.integers(-30, 17, 3000),
        (np.arange(-2048, 2048) + 0.5) * 2.0 ** -24,              # subnormal ties
        (1024 + np.arange(0, 1024) + 0.5) * 2.0 ** -10,           # ties in [1, 2)
        np.array([65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 0.0, -0.0]),
    ])
    got = orc.encode(v, "fp16")
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref), np.nonzero(got != ref)
    # bf16: float32 values (so torch's float32 -> bf16 rounding is the direct one)
    f = np.concatenate([
        (rng.standard_normal(3000) * 2.0 ** rng.integers(-140, 120, 3000)).astype(np.float32),
        ((np.arange(-512, 512) * 2 + 1) * 2.0 ** -9 + 2.0).astype(np.float32),  # ties
        np.array([3.3895313892515355e38, 3.39e38, 1e-45, -1e-45, 0.0], np.float32),
    ]).astype(np.float64)
    got = orc.encode(f, "bf16")
    ref = torch.from_numpy(f.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref), np.nonzero(got != ref)


def pin_gradx_at(orc):
    """The point-wise gradX agrees with the full pass at random positions."""
    rng = np.random.default_rng(37)
    for dt in ("bf16", "fp16"):
        S, B, H = 50, 3, 8
        gy, x, w = (rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt),
                    rand_bits(rng, (3, H), dt))
        mask = (rng.random((B, S)) < 0.7).astype(np.uint8)
        r = orc.bwd(S, B, H, 3, dt, gy, x, w, mask)
        idx = rng.integers(0, S * B * H, 400)
        idx = np.concatenate([idx, np.arange(S * B * H - 2 * B * H, S * B * H)])
        bits, _ = orc.gradx_at(S, B, H, 3, dt, gy, w, mask, idx)
        assert np.array_equal(bits, r["gx"].ravel()[idx]), dt


def pin_thread_independence(orc):
    """The oracle's results (fp64 sums, their roundings, sum|terms|) are the
    same bits on one thread and on every thread: each output is one thread's
    sum in a fixed order, so the parallel runs used at full size are the
    definition, not an approximation of it."""
    rng = np.random.default_rng(37)
    many = orc.threads(0)
    for dt in ("bf16", "fp16"):
        for (S, B, H, W) in ((300, 3, 64, 3), (129, 2, 128, 5), (1000, 1, 64, 1)):
            gy, x = rand_bits(rng, (S, B, H), dt), rand_bits(rng, (S, B, H), dt)
            w = rand_bits(rng, (W, H), dt)
            mask = (rng.random((B, S)) < 0.8).astype(np.uint8)
            one = orc.bwd(S, B, H, W, dt, gy, x, w, mask, want_exact=True, nthreads=1)
            all_ = orc.bwd(S, B, H, W, dt, gy, x, w, mask, want_exact=True, nthreads=many)
            for k in one:
                assert np.array_equal(one[k], all_[k]), (dt, S, B, H, W, k)
            assert np.array_equal(orc.fwd_bits(S, B, H, W, dt, x, w, mask, nthreads=1),
                                  orc.fwd_bits(S, B, H, W, dt, x, w, mask, nthreads=many))


ALL_PINS = [pin_golden, pin_closed_form_ones, pin_shift_identities, pin_mask_special_cases,
            pin_s1, pin_batch_independence, pin_jacobian_bruteforce, pin_adjoint_identity,
            pin_torch_autograd, pin_gradw_abs, pin_forward_torch, pin_forward_rounding, pin_converters,
            pin_gradx_at, pin_thread_independence]
