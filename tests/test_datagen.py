"""The seeded input generator: determinism, value laws and mask structure."""
import numpy as np
import pytest

import datagen


def _vals(bits, dtype):
    b = np.asarray(bits, np.uint16)
    if dtype == "fp16":
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_deterministic_and_thread_independent():
    a = np.empty(100_003, np.uint16)
    b = np.empty(100_003, np.uint16)
    datagen.fill_values(a, ("normal", 0.0, 1.0), "bf16", 0, 1, nthreads=1)
    datagen.fill_values(b, ("normal", 0.0, 1.0), "bf16", 0, 1, nthreads=5)
    assert np.array_equal(a, b)
    datagen.fill_values(b, ("normal", 0.0, 1.0), "bf16", 1, 1)
    assert not np.array_equal(a, b)
    datagen.fill_values(b, ("normal", 0.0, 1.0), "bf16", 0, 2)
    assert not np.array_equal(a, b)


@pytest.mark.parametrize("dtype,std", [("bf16", 1.0), ("fp16", 0.5)])
def test_normal_law(dtype, std):
    a = np.empty(1 << 20, np.uint16)
    datagen.fill_values(a, ("normal", 0.0, std), dtype, 0, 2)
    v = _vals(a, dtype)
    assert abs(v.mean()) < 5e-3 * std
    assert abs(v.std() / std - 1) < 5e-3
    assert abs((np.abs(v) < std).mean() - 0.6827) < 3e-3


def test_uniform_law():
    a = np.empty(1 << 20, np.uint16)
    datagen.fill_values(a, ("uniform", -0.5, 0.5), "bf16", 0, 3)
    v = _vals(a, "bf16")
    assert v.min() >= -0.5 and v.max() <= 0.5
    assert abs(v.mean()) < 2e-3 and abs(v.var() - 1 / 12) < 2e-3


def test_to16_rounds_to_nearest_even():
    # values exactly halfway between fp16 neighbours of 1.0
    assert datagen.to16(1 + 2 ** -11, "fp16") == 0x3C00
    assert datagen.to16(1 + 3 * 2 ** -11, "fp16") == 0x3C02
    assert datagen.to16(2 ** -25, "fp16") == 0x0000
    assert datagen.to16(3 * 2 ** -25, "fp16") == 0x0002
    assert datagen.to16(65520.0, "fp16") == 0x7C00
    assert datagen.to16(1 + 2 ** -8, "bf16") == 0x3F80
    assert datagen.to16(1 + 3 * 2 ** -8, "bf16") == 0x3F82
    assert datagen.to16(-2.0, "bf16") == 0xC000
    rng = np.random.default_rng(0)
    v = rng.standard_normal(20000) * 2.0 ** rng.integers(-26, 15, 20000)
    got = np.array([datagen.to16(a, "fp16") for a in v], np.uint16)
    with np.errstate(over="ignore"):
        assert np.array_equal(got, v.astype(np.float16).view(np.uint16))


def test_mask_bernoulli_rate():
    m = np.empty((4, 100_000), np.uint8)
    datagen.fill_mask(m, ("bernoulli", 0.9), 4, 100_000, 0)
    assert abs(m.mean() - 0.9) < 3e-3
    assert set(np.unique(m)) <= {0, 1}


def test_mask_prefix_structure():
    B, S = 8, 4096
    m = np.empty((B, S), np.uint8)
    datagen.fill_mask(m, ("prefix",), B, S, 0)
    L = datagen.prefix_lengths(B, S, 0)
    for j in range(B):
        assert S // 2 <= L[j] <= S
        assert m[j, : L[j]].all() and not m[j, L[j]:].any()


def test_mask_spans_structure():
    B, S = 4, 8192
    m = np.empty((B, S), np.uint8)
    datagen.fill_mask(m, ("spans", 0.2, 64, 1024), B, S, 0)
    for j in range(B):
        zeros = (m[j] == 0).sum()
        assert zeros >= 0.2 * S
        assert zeros < 0.2 * S + 1024  # the last span overshoots by at most one span
        # zeros come in runs; there are no isolated single zeros unless clipped
        edges = np.flatnonzero(np.diff(np.concatenate([[1], m[j], [1]]).astype(int)))
        runs = edges[1::2] - edges[0::2]
        assert runs.min() >= 1 and runs.max() <= S


def test_workloads_registry():
    w = datagen.WORKLOADS["s16384_b32_h4096_fp16"]
    assert w.B * w.S == 512 * 1024
    assert w.algorithmic_bytes() == 12_885_475_328
    assert w.without_mask().algorithmic_bytes() == 12_884_951_040
    d = datagen.generate("s64_b2_h384_bf16")
    assert d["x"].shape == (64, 2, 384) and d["mask"].shape == (2, 64) and d["w"].shape == (3, 384)
    d2 = datagen.generate("s64_b2_h384_bf16")
    assert all(np.array_equal(d[k], d2[k]) for k in d)
