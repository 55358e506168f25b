"""Invariants of the execution plan over the whole valid shape range (no GPU).

``mcc1d_plan_describe`` reports the plan the library would launch; these
checks are the conditions under which the kernels stay inside their buffers
and the hardware's limits: H-blocks that tile H, rows per stage that fit one
producer lane each, shared memory within the per-CTA and per-SM limits, no
more CTAs per SM than threads and registers allow, CTA ranges and partial
slots that cover every row exactly once, and a workspace layout that matches
what the kernels index. A plan that broke one of them would first show as a
fault or a hang on the GPU; here it fails on the CPU.
"""
import numpy as np
import pytest

import causal_conv_backward_gb300 as m
from causal_conv_backward_gb300 import build as cbuild

SMEM_PER_SM = 233472
SMEM_PER_CTA_DYN = 232448 - 1024
RESERVED_PER_CTA = 1024
NUM_SMS = 152
MAX_THREADS = 288
NOALLOC_MAX = 8 * 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def lib():
    cbuild.build()
    return m.load()


def cdiv(a, b):
    return -(-a // b)


def check_common(p, S, B, H, W):
    assert p["S"] == S and p["B"] == B and p["H"] == H and p["W"] == W
    hbw, nhb = p["hb_width"], p["n_hb"]
    assert hbw % 64 == 0 and 1 <= nhb <= 64
    assert nhb * hbw >= H and (nhb - 1) * hbw < H
    assert p["vec"] in (4, 8)
    if p.get("reg_split"):
        # whole consumer warpgroups behind the producer's warpgroup, and the
        # register split (setmaxnreg: producer group 56, consumers 224)
        # within the registers the CTA is launched with (168 per thread)
        assert p["consumer_warps"] == 4 * cdiv(cdiv(hbw // p["vec"], 32), 4)
        assert p["threads"] == 128 + 32 * p["consumer_warps"] <= 384
        assert 168 * p["threads"] >= 56 * 128 + 224 * (p["threads"] - 128)
        # and per scheduler: at most one producer-group warp and two consumer warps
        assert 56 * 32 + 2 * 224 * 32 <= 16384
    else:
        assert p["consumer_warps"] == cdiv(hbw // p["vec"], 32)
        assert p["threads"] == 32 * (p["consumer_warps"] + 1) <= MAX_THREADS
    assert p["row_bytes"] == 2 * hbw and p["row_bytes"] % 16 == 0
    assert p["stages"] >= 2
    cps = p["ctas_per_sm"]
    assert cps >= 1 and cps * p["threads"] <= 2048
    assert p["smem_bytes"] <= SMEM_PER_CTA_DYN
    assert cps * (p["smem_bytes"] + RESERVED_PER_CTA) <= SMEM_PER_SM
    assert p["off_mask"] >= p["stages"] * p["slot_bytes"]
    assert p["off_bar"] >= p["off_mask"] + 32 * p["stages"] and p["off_bar"] % 16 == 0
    # CTA ranges: every row of every H-block in exactly one range, ranges
    # contiguous (CTA c starts at c * rows // ncta)
    rows, ncta = p["rows_total"], p["ncta"]
    assert rows == nhb * B * S
    assert 1 <= ncta <= NUM_SMS * cps
    assert rows // ncta >= 1
    bs = B * S
    for hb in range(nhb):
        lo, hi = p["c_lo"][hb], p["c_hi"][hb]
        assert 0 <= lo <= hi < ncta
        # first CTA holding row hb*bs, last holding row (hb+1)*bs - 1
        assert lo * rows // ncta <= hb * bs < (lo + 1) * rows // ncta
        assert hi * rows // ncta <= (hb + 1) * bs - 1 < (hi + 1) * rows // ncta


def check_bwd(p, S, B, H, W):
    check_common(p, S, B, H, W)
    assert W < 4 or (p["vec"] == 4 and p["hb_width"] <= 1024)
    R = p["rows_per_stage"]
    assert R in ((4, 6, 8, 14) if W == 3 else (10,) if W in (4, 5, 6) else (8,) if W >= 7 else (6,))
    assert W < 5 or W - 1 <= R        # the certified sum's fallback reads the previous slot
    assert p["reg_split"] == (1 if W >= 5 and cdiv(p["hb_width"] // p["vec"], 32) > 4 else 0)
    assert R != 14 or p["vec"] == 4
    assert 2 * R + W - 1 <= 32               # one producer lane per staged row
    assert p["slot_bytes"] == (2 * R + W - 1) * p["row_bytes"]
    assert p["off_mask"] == p["stages"] * p["slot_bytes"]
    assert p["off_outer"] >= p["off_bar"] + 16 * p["stages"] and p["off_outer"] % 16 == 0
    assert p["smem_bytes"] == p["off_outer"] + p["consumer_warps"] * 32 * W * p["vec"] * 4
    # registers: CTAs per SM within the register file at the kernel's bound
    warps_per_sm = 4 * (16384 // (32 * p["regs_bound"]))
    assert p["ctas_per_sm"] * (p["threads"] // 32) <= warps_per_sm
    # partial slots: one per (CTA, H-block) pair, H-blocks contiguous
    base = 0
    for hb in range(p["n_hb"]):
        assert p["slot_base"][hb] == base
        base += p["c_hi"][hb] - p["c_lo"][hb] + 1
    assert p["nslots"] == base
    assert p["ws_part_off"] >= 256 + 4 * p["ncta"] and p["ws_part_off"] % 256 == 0
    assert p["ws_bytes"] == p["ws_part_off"] + p["nslots"] * W * p["hb_width"] * 4
    # reduce: splits x lanes = 512 threads, splits a power of two 8..64, no
    # more splits than the fullest H-block has slots (beyond the minimum)
    assert p["red_splits"] in (8, 16, 32, 64) and p["red_splits"] * p["red_lanes"] == 512
    most = max(p["c_hi"][h] - p["c_lo"][h] + 1 for h in range(p["n_hb"]))
    assert p["red_splits"] == 8 or p["red_splits"] <= most
    assert p["reduce_blocks"] == p["n_hb"] * W * cdiv(p["hb_width"], 4 * p["red_lanes"])


def check_fwd(p, S, B, H, W=3):
    check_common(p, S, B, H, W)
    assert p["rows_per_stage"] + W - 1 <= 32       # one producer lane per staged row
    # slots hold output rows only; one W-1-row halo area follows the slots
    assert p["slot_bytes"] == p["rows_per_stage"] * p["row_bytes"]
    assert p["off_mask"] == p["stages"] * p["slot_bytes"] + (W - 1) * p["row_bytes"]
    assert W == 3 or (p["hb_width"] <= 1024 and p["vec"] == 4)
    assert p["ws_bytes"] == 0


def shapes():
    rng = np.random.default_rng(7)
    out = []
    for H in range(384, 24577, 64):
        for B in (1, 2, 7, 32):
            for S in (1, 3, 17, 1000, 524288 // B):
                out.append((S, B, H))
    for _ in range(2000):
        H = 64 * int(rng.integers(6, 385))
        B = int(rng.integers(1, 33))
        S = int(rng.integers(1, 524288 // B + 1))
        out.append((S, B, H))
    return out


SHAPES = shapes()


def test_backward_plans():
    worst = 0
    for (S, B, H) in SHAPES:
        p = m.mcc1d_plan_describe(S, B, H, 3, "bf16", m.PLAN_BWD)
        check_bwd(p, S, B, H, 3)
        worst = max(worst, p["ws_bytes"])
    # the no-allocation entry point's static scratch holds every valid plan
    assert worst <= NOALLOC_MAX


@pytest.mark.parametrize("W", range(1, 9))
def test_strided_plans_every_width(W):
    for (S, B, H) in SHAPES[::3]:
        p = m.mcc1d_plan_describe(S, B, H, W, "fp16", m.PLAN_BWD_EX)
        check_bwd(p, S, B, H, W)


@pytest.mark.parametrize("W", range(1, 9))
def test_forward_plans(W):
    for (S, B, H) in SHAPES[:: 2 if W == 3 else 5]:
        check_fwd(m.mcc1d_plan_describe(S, B, H, W, "bf16", m.PLAN_FWD), S, B, H, W)


def test_bench_workload_plan():
    """The plan the benchmark's numbers were measured with."""
    p = m.mcc1d_plan_describe(16384, 32, 4096, 3, "fp16", m.PLAN_BWD)
    assert (p["hb_width"], p["vec"], p["rows_per_stage"], p["stages"], p["ncta"], p["threads"]) == \
        (2048, 8, 6, 3, 152, 288)


def test_describe_rejects():
    with pytest.raises(m.Mcc1dError):
        m.mcc1d_plan_describe(64, 2, 384, 4, "bf16", m.PLAN_BWD)      # page calls: W = 3
    with pytest.raises(m.Mcc1dError):
        m.mcc1d_plan_describe(64, 2, 384, 9, "bf16", m.PLAN_BWD_EX)
    with pytest.raises(m.Mcc1dError):
        m.mcc1d_plan_describe(64, 2, 384, 9, "bf16", m.PLAN_FWD)
    with pytest.raises(m.Mcc1dError):
        m.mcc1d_plan_describe(64, 2, 384, 3, "bf16", 7)
