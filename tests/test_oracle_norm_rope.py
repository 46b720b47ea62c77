"""Pins of the oracle's head RMSNorm, RoPE and fused KV write against what
the pages print and what the rotation must satisfy.

None of these tests touch the CUDA library.
"""
import math

import numpy as np
import pytest

import oracle
from oracle_cases import bf16_round, bits, nan_pool, values


def test_rmsnorm_printed_example(golden):
    g = golden("norm_rope_examples.json")["rmsnorm_1_2_3"]
    y = oracle.rmsnorm(g["x"])
    np.testing.assert_array_equal(np.round(y, g["y_decimals"]), g["y"])
    # the common scale is the printed root mean square, and the output's mean square is 1
    assert round(float(np.asarray(g["x"])[0] / y[0]), g["rms_decimals"]) == g["rms"]
    assert math.isclose(float(np.mean(np.square(g["x"]))), g["mean_square"], rel_tol=1e-15)
    assert math.isclose(float(np.mean(np.square(y))), 1.0, rel_tol=1e-12)
    # scaling the input by 10 does not change the output (epsilon ignored)
    np.testing.assert_allclose(oracle.rmsnorm(g["scaled_x"]), y, rtol=1e-14)


def test_rmsnorm_epsilon_and_weight_as_printed(golden):
    # y_i = gamma_i * x_i / sqrt(mean(x^2) + eps), the page's formula (§19.3)
    x = np.array([1e-3, -2e-3, 3e-3, 0.5e-3])
    w = np.array([2.0, 0.5, -1.0, 3.0])
    eps = 1e-6
    ms = (1e-6 + 4e-6 + 9e-6 + 0.25e-6) / 4
    expect = w * x / math.sqrt(ms + eps)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, eps), expect, rtol=1e-13)
    # with eps comparable to mean(x^2) the result is far from the eps-free one
    assert abs(oracle.rmsnorm(x, None, eps)[0] - oracle.rmsnorm(x, None, 0.0)[0]) > 0.05


def test_rope_quarter_turn(golden):
    g = golden("norm_rope_examples.json")["rope_quarter_turn"]
    phi = math.radians(g["degrees"])
    y = oracle.rope_apply(g["pair"], [math.cos(phi), math.sin(phi)])
    np.testing.assert_allclose(y, g["out"], atol=1e-15)


def test_rope_table_closed_form(golden):
    g = golden("norm_rope_examples.json")["rope_frequencies"]
    d, base = g["head_dim"], g["base"]
    t = oracle.rope_cos_sin(base, d, 2000)
    assert t.dtype == np.float32 and t.shape == (2000, d)
    # position 0: every pair unrotated
    np.testing.assert_array_equal(t[0, : d // 2], 1.0)
    np.testing.assert_array_equal(t[0, d // 2:], 0.0)
    p = np.arange(2000)
    # pair 0 turns one radian per position; pair 32 by base^(-1/2) = 1e-3; pair 63 by base^(-126/128)
    for i, w in ((0, 1.0), (32, 1e-3), (63, base ** (-126 / 128))):
        np.testing.assert_allclose(t[:, i], np.cos(p * w).astype(np.float32), atol=2e-7)
        np.testing.assert_allclose(t[:, d // 2 + i], np.sin(p * w).astype(np.float32), atol=2e-7)


def test_rope_pairs_the_two_halves(golden):
    g = golden("norm_rope_examples.json")["rope_pairing"]
    d = g["head_dim"]
    t = oracle.rope_cos_sin(1e6, d, 8)
    for a, b in g["pairs_first"] + [g["pairs_last"]]:
        x = np.zeros(d)
        x[a] = 1.0
        y = oracle.rope_apply(x, t[5])
        others = np.delete(y, [a, b])
        np.testing.assert_array_equal(others, 0.0)        # only the partner feature receives the turn
        assert math.isclose(y[a], float(t[5, a]), rel_tol=1e-7)
        assert math.isclose(y[b], float(t[5, d // 2 + a]), rel_tol=1e-7)


def test_rope_depends_on_relative_position_only():
    rng = np.random.default_rng(11)
    d = 128
    t = oracle.rope_cos_sin(1e6, d, 4096)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for p, j, s in ((3, 10, 100), (700, 40, 1500), (0, 0, 2000)):
        a = oracle.rope_apply(q, t[p]) @ oracle.rope_apply(k, t[j])
        b = oracle.rope_apply(q, t[p + s]) @ oracle.rope_apply(k, t[j + s])
        assert math.isclose(a, b, rel_tol=2e-5, abs_tol=2e-5)
    # each pair keeps its length
    y = oracle.rope_apply(q, t[1234])
    np.testing.assert_allclose(np.hypot(y[:64], y[64:]), np.hypot(q[:64], q[64:]), rtol=1e-6)


def _fused_case(hq=2, hkv=1, d=128, n=5, seed=3):
    rng = np.random.default_rng(seed)
    qkv = bits(rng.standard_normal((n, (hq + 2 * hkv) * d)) * 3.0)
    qw = bits(rng.uniform(0.5, 1.5, d))
    kw = bits(rng.uniform(0.5, 1.5, d))
    pos = np.array([0, 7, 300, 4095, 12][:n], dtype=np.int32)
    cs = oracle.rope_cos_sin(1e6, d, 4096)
    return qkv, qw, kw, pos, cs


def _reference_row(x_bits, w_bits, cs_row, eps):
    """The pages' order for one head, composed from the pinned primitives:
    norm in double, round to bf16, times the bf16 weight, round, RoPE, round."""
    x = values(x_bits)
    if w_bits is not None:
        x = bf16_round(bf16_round(oracle.rmsnorm(x, None, eps)) * values(w_bits))
    return bits(bf16_round(oracle.rope_apply(x, cs_row)))


def test_fused_norm_rope_store_follows_the_pages_order():
    hq, hkv, d, n, eps = 2, 1, 128, 5, 1e-6
    qkv, qw, kw, pos, cs = _fused_case(hq, hkv, d, n)
    kc, vc = nan_pool(4, 4, hkv, d), nan_pool(4, 4, hkv, d)
    slots = np.array([5, -1, 0, 15, 9], dtype=np.int32)
    q_out, rc = oracle.norm_rope_store(qkv, hq, hkv, pos, cs, qw, kw, eps, kc, vc, slots)
    assert rc == oracle.OK
    for t in range(n):
        row = qkv[t]
        for h in range(hq):  # Q heads come first in the fused row
            np.testing.assert_array_equal(q_out[t, h], _reference_row(row[h * d:(h + 1) * d], qw, cs[pos[t]], eps))
        if slots[t] == -1:
            continue
        b, o = divmod(int(slots[t]), 4)
        k_bits = row[hq * d:(hq + 1) * d]
        v_bits = row[(hq + hkv) * d:(hq + 2 * hkv) * d]
        np.testing.assert_array_equal(kc[b, o, 0], _reference_row(k_bits, kw, cs[pos[t]], eps))
        np.testing.assert_array_equal(vc[b, o, 0], v_bits)  # V is stored as it is
    # every other pool row is untouched (still NaN-poisoned)
    live = {int(s) for s in slots if s != -1}
    for s in range(16):
        if s not in live:
            b, o = divmod(s, 4)
            assert (kc[b, o] == 0x7FC0).all() and (vc[b, o] == 0x7FC0).all()


def test_fused_without_head_norm_is_rope_only():
    hq, hkv, d = 2, 1, 128
    qkv, _, _, pos, cs = _fused_case(hq, hkv, d)
    kc, vc = nan_pool(4, 4, hkv, d), nan_pool(4, 4, hkv, d)
    q_out, rc = oracle.norm_rope_store(qkv, hq, hkv, pos, cs, None, None, 1e-6, kc, vc, [0, 1, 2, 3, 4])
    assert rc == oracle.OK
    for t in range(qkv.shape[0]):
        expect = bits(bf16_round(oracle.rope_apply(values(qkv[t, :d]), cs[pos[t]])))
        np.testing.assert_array_equal(q_out[t, 0], expect)


def test_fused_position_zero_is_norm_only():
    hq, hkv, d = 1, 1, 128
    qkv, qw, kw, _, cs = _fused_case(hq, hkv, d)
    kc, vc = nan_pool(2, 4, hkv, d), nan_pool(2, 4, hkv, d)
    pos = np.zeros(qkv.shape[0], dtype=np.int32)
    q_out, _ = oracle.norm_rope_store(qkv, hq, hkv, pos, cs, qw, kw, 0.0, kc, vc, [0, 1, 2, 3, 4])
    x = values(qkv[0, :d])
    np.testing.assert_array_equal(q_out[0, 0], bits(bf16_round(bf16_round(x / math.sqrt(np.mean(x * x))) * values(qw))))


def test_fused_reports_bad_position_and_slot():
    hq, hkv, d = 2, 1, 128
    qkv, qw, kw, pos, cs = _fused_case(hq, hkv, d)
    kc, vc = nan_pool(4, 4, hkv, d), nan_pool(4, 4, hkv, d)
    pos = pos.copy()
    pos[1] = 4096  # one past the table
    _, rc = oracle.norm_rope_store(qkv, hq, hkv, pos, cs, qw, kw, 1e-6, kc, vc, [0, 1, 2, 3, 4])
    assert rc == oracle.BOUNDS
    assert (kc[0, 1] == 0x7FC0).all()  # the skipped token wrote nothing
    _, rc = oracle.norm_rope_store(qkv, hq, hkv, _fused_case()[3], cs, qw, kw, 1e-6, kc, vc, [0, 1, 99, 3, 4])
    assert rc == oracle.BOUNDS
