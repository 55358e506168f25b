"""A CPU model of the kernels' address arithmetic, driven by the real plans.

For the plan ``mcc1d_plan_describe`` reports, this restates how the main
backward kernel and the forward kernel walk their CTA ranges (stages of R
rows, the W-1-row halo, one bulk copy per row or one per tensor on short
B = 1 ranges) and checks, with no GPU: every bulk copy reads inside its
tensor, starts on a 16-byte boundary, moves a multiple of 16 bytes and lands
inside its ring slot; no stage needs more producer lanes than a warp has;
every output element is written exactly once; every partial-sum write stays
inside its slot. From W = 6 the kernels recompute, after a stage, the sums
whose certificate failed from the rows still in shared memory: every such
read must find the row it wants (in this slot, the halo area, or the
previous slot, which the consumers release one stage late). A kernel that broke one of these would fault or corrupt
memory on the GPU; here the mistake fails on the CPU first.
"""
import numpy as np
import pytest

import causal_conv_backward_gb300 as m
from causal_conv_backward_gb300 import build as cbuild

KDEEP = 256   # CTA ranges of at least this many rows copy one row per bulk copy


@pytest.fixture(scope="module", autouse=True)
def lib():
    cbuild.build()
    return m.load()


def ctas_to_check(ncta, full):
    if full:
        return range(ncta)
    pick = {0, 1, 2, ncta // 3, ncta // 2, ncta - 3, ncta - 2, ncta - 1}
    return sorted(c for c in pick if 0 <= c < ncta)


def walk(p, c):
    """Stages of CTA c: (stage index, i, j, hb, n rows)."""
    S, B = p["S"], p["B"]
    N, ncta, R = p["rows_total"], p["ncta"], p["rows_per_stage"]
    r0, r1 = c * N // ncta, (c + 1) * N // ncta
    assert r1 > r0
    bs = B * S
    pos = r0
    hb, rem = divmod(pos, bs)
    j, i = divmod(rem, S)
    stage = 0
    while pos < r1:
        n = min(R, S - i, r1 - pos)
        assert n >= 1
        yield stage, i, j, hb, n
        pos += n
        i += n
        if i == S:
            i = 0
            j += 1
            if j == B:
                j = 0
                hb += 1
        stage += 1


def check_copy(src_elem, nbytes, tensor_elems, dst, slot_bytes):
    assert (2 * src_elem) % 16 == 0 and nbytes % 16 == 0 and nbytes > 0
    assert 0 <= src_elem and 2 * src_elem + nbytes <= 2 * tensor_elems
    assert 0 <= dst and dst + nbytes <= slot_bytes


def model_backward(S, B, H, W, kind, full):
    p = m.mcc1d_plan_describe(S, B, H, W, "bf16", kind)
    R, hbw, vec = p["rows_per_stage"], p["hb_width"], p["vec"]
    E = S * B * H
    rb, sb = p["row_bytes"], p["slot_bytes"]
    cw = p["consumer_warps"]
    contig = B == 1 and p["n_hb"] == 1 and p["rows_total"] // p["ncta"] < KDEEP
    bulk = W == 3 and vec == 8 and rb >= 4096 and p["rows_total"] // p["ncta"] >= 1024
    written = np.zeros(E // vec, np.int32) if full else None
    part_elems = p["nslots"] * W * hbw
    used_slots = set()
    cert = W >= 6 and not bulk
    if cert:
        assert p["stages"] >= 2      # the previous slot is held while this one is read
    for c in ctas_to_check(p["ncta"], full):
        segs = set()
        prev = None
        for stage, i, j, hb, n in walk(p, c):
            head = stage == 0 or i == 0
            hb0 = hb * hbw
            width = min(hbw, H - hb0)
            wbytes = 2 * width
            q0 = 0 if head else W - 1
            q1 = min(n + W - 1, S - i)
            if cert:
                # the fallback for row r reads gradY row i+q, q = r .. r+W-1:
                # slot row q when staged here, else the previous slot's row
                # n_prev + q (same sequence, staged there)
                for r in range(n):
                    for q in range(r, r + W):
                        if i + q >= S:
                            continue            # past the sequence: mask byte 0
                        if head or q >= W - 1:
                            assert q0 <= q < q1
                        else:
                            pi, pj, phb, pn, pq0, pq1 = prev
                            assert (pj, phb) == (j, hb) and pi + pn == i
                            assert pq0 <= pn + q < pq1
            nG = max(0, q1 - q0)
            gy_rows_end = (R + W - 1) * rb          # gradY rows 0 .. R+W-2, then x rows
            if contig:
                if nG:
                    check_copy((i + q0) * H, nG * wbytes, E, q0 * rb, gy_rows_end)
                check_copy(i * H, n * wbytes, E, gy_rows_end, sb)
            else:
                assert nG + n <= 32
                for q in range(q0, q1):
                    check_copy((i + q) * B * H + j * H + hb0, wbytes, E, q * rb, gy_rows_end)
                for q in range(n):
                    check_copy((i + q) * B * H + j * H + hb0, wbytes, E, gy_rows_end + q * rb, sb)
            if bulk:
                # gradX rows leave from the x slot rows, one bulk copy
                # (shared -> global) per row
                for r in range(n):
                    check_copy((i + r) * B * H + j * H + hb0, wbytes, E, gy_rows_end + r * rb, sb)
            # consumer stores of gradX: rows i .. i+n-1, active threads only
            ct = np.arange(cw * 32)
            ct = ct[vec * ct < width]
            for r in range(n):
                e = ((i + r) * B + j) * H + hb0 + vec * ct
                assert e.max() + vec <= E
                if written is not None:
                    np.add.at(written, e // vec, 1)
            segs.add(hb)
            prev = (i, j, hb, n, q0, q1)
        for hb in segs:
            slot = p["slot_base"][hb] + c - p["c_lo"][hb]
            assert 0 <= slot < p["nslots"] and slot not in used_slots
            used_slots.add(slot)
            top = slot * W * hbw + (W - 1) * hbw + vec * (cw * 32 - 1) + vec
            assert top <= part_elems or vec * (cw * 32 - 1) >= hbw
    if written is not None:
        assert written.min() == 1 and written.max() == 1
        assert len(used_slots) == p["nslots"]


def model_forward(S, B, H, W, full):
    p = m.mcc1d_plan_describe(S, B, H, W, "bf16", m.PLAN_FWD)
    R, hbw, vec = p["rows_per_stage"], p["hb_width"], p["vec"]
    E = S * B * H
    rb, sb = p["row_bytes"], p["slot_bytes"]
    cw = p["consumer_warps"]
    contig = B == 1 and p["n_hb"] == 1 and p["rows_total"] // p["ncta"] < KDEEP
    written = np.zeros(E // vec, np.int32) if full else None
    halo = (W - 1) * rb
    bulk = W == 3 and vec == 8 and rb >= 4096 and p["rows_total"] // p["ncta"] >= 1024
    cert = W >= 6 and not bulk
    if cert:
        assert p["stages"] >= 2
    for c in ctas_to_check(p["ncta"], full):
        prev = None
        for stage, i, j, hb, n in walk(p, c):
            hb0 = hb * hbw
            width = min(hbw, H - hb0)
            wbytes = 2 * width
            # slot row r holds x row i+r (r < n); halo row q holds x row
            # i-(W-1)+q, loaded for q in [h0, W-1) at a range's first stage
            # when it starts inside a sequence
            h0 = W - 1
            if stage == 0 and i > 0:
                h0 = 0 if i >= W - 1 else W - 1 - i
            nh = W - 1 - h0
            assert n + nh <= 32
            if cert:
                # the fallback for row r reads x row i+d, d = r-W+1 .. r:
                # slot row d; before the stage, the halo row W-1+d at a head
                # stage (staged, or zero before the sequence start), else
                # the previous slot's row n_prev + d
                head = stage == 0 or i == 0
                for r in range(n):
                    for d in range(r - W + 1, r + 1):
                        if d >= 0:
                            assert d < n
                        elif head:
                            assert W - 1 + d >= h0 or i + d < 0
                        else:
                            pi, pj, phb, pn = prev
                            assert (pj, phb) == (j, hb) and pi + pn == i
                            assert 0 <= pn + d < pn
            if contig:
                check_copy(i * H, n * wbytes, E, 0, sb)
                if nh:
                    check_copy((i - (W - 1) + h0) * H, nh * wbytes, E, h0 * rb, halo)
            else:
                for r in range(n):
                    check_copy((i + r) * B * H + j * H + hb0, wbytes, E, r * rb, sb)
                for q in range(h0, W - 1):
                    check_copy((i - (W - 1) + q) * B * H + j * H + hb0, wbytes, E, q * rb, halo)
            if bulk:
                # y rows leave from the slot rows they were read into, one bulk
                # copy (shared -> global) per row
                for r in range(n):
                    check_copy((i + r) * B * H + j * H + hb0, wbytes, E, r * rb, sb)
            ct = np.arange(cw * 32)
            ct = ct[vec * ct < width]
            for r in range(n):
                e = ((i + r) * B + j) * H + hb0 + vec * ct
                assert e.max() + vec <= E
                if written is not None:
                    np.add.at(written, e // vec, 1)
            prev = (i, j, hb, n)
    if written is not None:
        assert written.min() == 1 and written.max() == 1


SMALL = [(1, 1, 384), (2, 3, 448), (5, 32, 384), (64, 2, 384), (65, 1, 640), (300, 3, 1088), (17, 5, 2112),
         (129, 2, 1984), (9, 2, 24576), (1000, 1, 384), (4096, 1, 384), (777, 3, 1920), (2049, 2, 576)]
LARGE = [(524288, 1, 384), (262144, 2, 384), (16384, 32, 4096), (8192, 4, 24576), (40000, 4, 1920),
         (4096, 8, 2048), (65536, 8, 640), (16384, 32, 24576), (524288, 1, 24576), (13, 32, 24576)]


@pytest.mark.parametrize("S,B,H", SMALL)
def test_backward_model_small_every_cta(S, B, H):
    model_backward(S, B, H, 3, m.PLAN_BWD, full=True)


@pytest.mark.parametrize("S,B,H", LARGE)
def test_backward_model_large_sampled_ctas(S, B, H):
    model_backward(S, B, H, 3, m.PLAN_BWD, full=False)


@pytest.mark.parametrize("W", [1, 2, 4, 5, 6, 7, 8])
def test_backward_model_other_widths(W):
    for (S, B, H) in [(1, 2, 384), (W + 1, 3, 1088), (300, 2, 640), (2049, 1, 2112)]:
        model_backward(S, B, H, W, m.PLAN_BWD_EX, full=True)
    for (S, B, H) in [(524288, 1, 384), (16384, 32, 4096)]:
        model_backward(S, B, H, W, m.PLAN_BWD_EX, full=False)


@pytest.mark.parametrize("W", [1, 2, 3, 4, 6, 7, 8])
def test_forward_model(W):
    for (S, B, H) in SMALL[:8]:
        model_forward(S, B, H, W, full=True)
    for (S, B, H) in LARGE[:5]:
        model_forward(S, B, H, W, full=False)


def test_random_shapes_model():
    rng = np.random.default_rng(11)
    for _ in range(60):
        H = 64 * int(rng.integers(6, 40))
        B = int(rng.integers(1, 9))
        S = int(rng.integers(1, 3000))
        W = int(rng.integers(1, 9))
        model_backward(S, B, H, W, m.PLAN_BWD_EX, full=True)
        model_forward(S, B, H, W, full=True)

