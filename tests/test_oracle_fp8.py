"""Pins of the oracle's fp8 (E4M3) KV cache: the format against PyTorch's
float8_e4m3fn (a library routine) and its closed forms, and fp8 decode against
the pinned bf16 decode on values both formats hold exactly.  No CUDA."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import bits, nan_pool, values


def test_every_code_decodes_like_the_library():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ours), np.isnan(lib)) and np.isnan(ours).sum() == 2   # 0x7f and 0xff
    np.testing.assert_array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])


def test_format_closed_forms():
    assert oracle.e4m3_value(0x7E) == 448.0                 # largest finite
    assert oracle.e4m3_value(0x08) == 2.0 ** -6             # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9             # smallest subnormal
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0xB8) == -1.0


def test_encode_inverts_decode_and_saturates():
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)
    assert oracle.e4m3_encode(1e4) == 0x7E and oracle.e4m3_encode(-1e4) == 0xFE
    assert oracle.e4m3_encode(464.0) == 0x7E                # past the largest finite: saturated, not NaN
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_encode_rounds_like_the_library():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)]).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    # exact midpoints between neighbouring codes must round to the even code
    vals = np.array([oracle.e4m3_value(c) for c in range(0x00, 0x7E)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(ours, lib)


def test_fp8_store_round_trips_representable_values():
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 0x7E, size=(6, 2, 128)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    k_scale, v_scale = 0.25, 4.0
    kv = np.vectorize(oracle.e4m3_value)(codes)
    k_bits, v_bits = bits(kv * k_scale), bits(kv * v_scale)   # exact in bf16 (4 significant bits)
    kc = np.zeros((2, 4, 2, 128), np.uint8)
    vc = np.zeros_like(kc)
    rc = oracle.store_kvcache_fp8(k_bits, v_bits, k_scale, v_scale, kc, vc, [5, 0, 7, -1, 2, 6])
    assert rc == oracle.OK
    for t, slot in enumerate([5, 0, 7, -1, 2, 6]):
        if slot == -1:
            continue
        b, o = divmod(slot, 4)
        np.testing.assert_array_equal(kc[b, o], codes[t])
        np.testing.assert_array_equal(vc[b, o], codes[t])
    assert (kc[0, 1] == 0).all() and (kc[0, 3] == 0).all()   # untouched slots


def test_fp8_store_error_is_within_half_a_step():
    rng = np.random.default_rng(10)
    x = bits(rng.standard_normal((50, 1, 128)) * 2.0)
    kc = np.zeros((13, 4, 1, 128), np.uint8)
    vc = np.zeros_like(kc)
    scale = 0.03125
    assert oracle.store_kvcache_fp8(x, x, scale, scale, kc, vc, list(range(50))) == oracle.OK
    got = np.vectorize(oracle.e4m3_value)(kc.reshape(-1, 128)[:50]) * scale
    ref = values(x[:, 0, :])
    # relative half-step of a 3-bit mantissa: 2^-4 (normal range); absolute half-step below 2^-6 * scale
    assert (np.abs(got - ref) <= np.maximum(np.abs(ref) * 2.0 ** -4, 2.0 ** -10 * scale) + 1e-12).all()


@pytest.mark.parametrize("hq,hkv", [(16, 8), (4, 1)])
def test_fp8_decode_equals_bf16_decode_on_exact_values(hq, hkv):
    rng = np.random.default_rng(11 + hq)
    bs, nb = 16, 12
    codes_k = rng.integers(0, 0x7E, size=(nb, bs, hkv, 128)).astype(np.uint8) | \
        (rng.integers(0, 2, size=(nb, bs, hkv, 128)) << 7).astype(np.uint8)
    codes_v = rng.integers(0, 0x7E, size=(nb, bs, hkv, 128)).astype(np.uint8)
    ks, vs = 2.0 ** -5, 2.0 ** -3
    dec = np.vectorize(oracle.e4m3_value)
    kb, vb = bits(dec(codes_k) * ks), bits(dec(codes_v) * vs)
    table = rng.permutation(nb).astype(np.int32).reshape(3, 4)
    ctx = np.array([64, 17, 0], np.int32)
    q = bits(rng.standard_normal((3, hq, 128)))
    ref = oracle.decode(q, kb, vb, table, ctx, 1 / math.sqrt(128))
    got = oracle.decode_fp8(q, codes_k, codes_v, ks, vs, table, ctx, 1 / math.sqrt(128))
    np.testing.assert_array_equal(got, ref)
