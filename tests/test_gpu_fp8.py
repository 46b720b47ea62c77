"""fp8 (E4M3) KV cache on the GPU against the oracle, through the C ABI.

The KV write is bit-exact (a quantised code decided in fp32 on both sides).
Decode over the fp8 pool is compared with the oracle's decode over ITS OWN
fp8 pool (built by the oracle's KV write from the same bf16 inputs) within
the attention tolerance; the effect of the format itself (fp8 decode against
the bf16 oracle on the unquantised data) is measured and bounded loosely."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MAX_ABS, MEAN_ABS, Status, assert_close, dev, grow_keys, i32, pa
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _fp8_pools(batch, k_scale, v_scale, hist_rows):
    """(GPU fp8 pools built by pa_store_kvcache_fp8, oracle fp8 pools built by
    the oracle's KV write) holding the batch's bf16 history and its new tokens."""
    d = dev()
    shape = batch.k_cache.shape
    gk = torch.full(shape, 0xAA, dtype=torch.uint8, device=d)
    gv = torch.full(shape, 0xAA, dtype=torch.uint8, device=d)
    ok, ov = np.full(shape, 0xAA, np.uint8), np.full(shape, 0xAA, np.uint8)
    # history rows: pool rows -> pseudo-tokens
    rows = torch.as_tensor(hist_rows.astype(np.int64), device=d)
    hk = batch.k_cache.view(-1, shape[2], shape[3]).index_select(0, rows)
    hv = batch.v_cache.view(-1, shape[2], shape[3]).index_select(0, rows)
    slots = hist_rows.astype(np.int32)
    st = Status(d)
    pa().pa_store_kvcache_fp8(hk, hv, k_scale, v_scale, gk, gv, i32(slots, d), dev_status=st.t)
    pa().pa_store_kvcache_fp8(batch.tokens.k, batch.tokens.v, k_scale, v_scale, gk, gv, i32(batch.slot_mapping, d),
                              dev_status=st.t)
    torch.cuda.synchronize()
    assert int(st.t.item()) == 0
    assert oracle.store_kvcache_fp8(wl.bf16_bits(hk), wl.bf16_bits(hv), k_scale, v_scale, ok, ov, slots) == oracle.OK
    assert oracle.store_kvcache_fp8(wl.bf16_bits(batch.tokens.k), wl.bf16_bits(batch.tokens.v), k_scale, v_scale,
                                    ok, ov, batch.slot_mapping) == oracle.OK
    return gk, gv, ok, ov


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -6])
def test_fp8_store_is_bit_exact(scale):
    batch = wl.paged_batch(wl.SEED_BASE + 80, [33, 100, 7], [33, 100, 7], 16, device=dev())
    gk, gv, ok, ov = _fp8_pools(batch, scale, scale * 2, np.zeros(0, np.int64))
    np.testing.assert_array_equal(gk.cpu().numpy(), ok)   # every byte, untouched rows included
    np.testing.assert_array_equal(gv.cpu().numpy(), ov)


def test_fp8_store_saturates_and_reports_bad_slots():
    d = dev()
    toks = wl.new_tokens(wl.SEED_BASE + 81, 4, device=d)
    big = (toks.k.float() * 1e4).to(torch.bfloat16)            # far past 448 * scale
    gk = torch.zeros((2, 16, 8, 128), dtype=torch.uint8, device=d)
    gv = torch.zeros_like(gk)
    st = Status(d)
    pa().pa_store_kvcache_fp8(big, toks.v, 1.0, 1.0, gk, gv, i32([0, 1, 99, -1], d), dev_status=st.t)
    torch.cuda.synchronize()
    assert int(st.t.item()) == pa().PA_ERR_BOUNDS
    codes = gk.view(-1, 8, 128)[:2].cpu().numpy()
    assert ((codes & 0x7F) <= 0x7E).all()                      # saturated: no NaN codes
    assert ((codes & 0x7F) == 0x7E).mean() > 0.9


def _decode_case(batch, k_scale, v_scale, ctx=None, q=None):
    d = dev()
    hist = wl.history_rows(batch.layout, batch.context_lens - batch.query_lens)
    ctx = batch.context_lens if ctx is None else np.asarray(ctx, np.int32)
    q = batch.tokens.q if q is None else q
    gk, gv, ok, ov = _fp8_pools(batch, k_scale, v_scale, hist)
    max_ctx = int(ctx.max())
    b, hq = len(ctx), batch.num_heads
    ws = torch.empty(max(pa().pa_decode_workspace_bytes(b, hq, 128, max_ctx), 256), dtype=torch.uint8, device=d)
    out = torch.full((b, hq, 128), float("nan"), dtype=torch.bfloat16, device=d)
    st = Status(d)
    pa().pa_decode_paged_fp8(q, gk, gv, k_scale, v_scale, i32(batch.block_tables, d), i32(ctx, d),
                             max_ctx, batch.scale, out, ws, dev_status=st.t)
    torch.cuda.synchronize()
    assert int(st.t.item()) == 0
    q_bits = wl.bf16_bits(q)
    ref = oracle.decode_fp8(q_bits, ok, ov, k_scale, v_scale, batch.block_tables, ctx, batch.scale)
    return out, ref, hist


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (2.0 ** -6, 2.0 ** -5)])
def test_fp8_decode_matches_oracle(k_scale, v_scale):
    batch = wl.decode_batch(device=dev(), num_seqs=64, seed=wl.SEED_BASE + 82)
    out, ref, _ = _decode_case(batch, k_scale, v_scale)
    assert_close(out, ref, "fp8 decode")


def test_fp8_decode_block_size_16_and_padding_rows():
    live = np.array([300, 5, 17, 1000, 1, 9])
    batch = wl.paged_batch(wl.SEED_BASE + 83, live, np.ones_like(live), 16, device=dev())
    ctx = live.copy()
    ctx[[1, 5]] = 0                      # padded rows of a captured batch size
    out, ref, _ = _decode_case(batch, 2.0 ** -6, 2.0 ** -6, ctx=ctx)
    assert_close(out, ref, "fp8 decode bs 16")
    assert (out[[1, 5]].float() == 0).all()


# one sequence of a single token, ragged chunk tails, exact chunks, several
# splits (merged) and a long one; every group size the kernel has (G = 1, 2,
# 4, 8 query heads per KV head, one to eight warps per KV head)
@pytest.mark.parametrize("hq,hkv,bs", [(8, 8, 16), (16, 4, 64), (32, 4, 256), (8, 1, 32), (4, 2, 48)])
def test_fp8_decode_head_layouts(hq, hkv, bs):
    live = np.array([1, 15, 16, 17, 100, 700, 2100, 33])
    batch = wl.paged_batch(wl.SEED_BASE + 85 + hq + 3 * hkv, live, np.ones_like(live), bs, num_heads=hq,
                           num_kv_heads=hkv, device=dev())
    out, ref, _ = _decode_case(batch, 2.0 ** -6, 2.0 ** -5)
    assert_close(out, ref, f"fp8 decode hq={hq} hkv={hkv} bs={bs}")


# scores that grow along the keys (every key = growth * position, q >= 0; K
# scale 2^-3 keeps the largest key, 42, inside E4M3's range): the running
# maximum of each head moves every few chunks (0.02) or rarely (0.002), in
# every lane, for group sizes 2, 8 and 8 with a single KV head
@pytest.mark.parametrize("growth", [0.02, 0.002], ids=["fast_growth", "slow_growth"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 4), (8, 1)])
def test_fp8_decode_growing_scores_rescale(growth, hq, hkv):
    live = np.array([700, 1024, 129, 300, 1600, 17, 2100, 40])
    batch = wl.paged_batch(wl.SEED_BASE + 88 + hq, live, np.ones_like(live), 64, num_heads=hq, num_kv_heads=hkv,
                           device=dev())
    grow_keys(batch, growth)
    out, ref, _ = _decode_case(batch, 2.0 ** -3, 2.0 ** -5)
    assert_close(out, ref, f"fp8 decode, growing scores x {growth}, hq={hq} hkv={hkv}")


# queries far from unit size: a bf16 query of any normal magnitude enters the
# MMA exactly (scaled by a power of two per head, undone on the score)
@pytest.mark.parametrize("qmul", [2.0 ** 12, 2.0 ** -12])
def test_fp8_decode_query_magnitudes(qmul):
    live = np.array([300, 40, 1000, 17])
    batch = wl.paged_batch(wl.SEED_BASE + 86, live, np.ones_like(live), 16, device=dev())
    q = (batch.tokens.q.float() * qmul).to(torch.bfloat16)
    out, ref, _ = _decode_case(batch, 2.0 ** -6, 2.0 ** -6, q=q)
    assert_close(out, ref, f"fp8 decode, queries x {qmul}")


def test_fp8_decode_bad_block_and_long_context_reported():
    d = dev()
    live = np.array([40, 300, 7])
    batch = wl.paged_batch(wl.SEED_BASE + 87, live, np.ones_like(live), 16, device=d)
    hist = wl.history_rows(batch.layout, batch.context_lens - batch.query_lens)
    gk, gv, _, _ = _fp8_pools(batch, 2.0 ** -6, 2.0 ** -6, hist)
    ws = torch.empty(max(pa().pa_decode_workspace_bytes(3, 16, 128, 300), 256), dtype=torch.uint8, device=d)

    def run(tables, max_ctx):
        out = torch.full((3, 16, 128), float("nan"), dtype=torch.bfloat16, device=d)
        st = Status(d)
        pa().pa_decode_paged_fp8(batch.tokens.q, gk, gv, 2.0 ** -6, 2.0 ** -6, i32(tables, d), i32(live, d), max_ctx,
                                 batch.scale, out, ws, dev_status=st.t)
        torch.cuda.synchronize()
        return out, int(st.t.item())

    out, st = run(batch.block_tables, 300)
    assert st == 0 and torch.isfinite(out.float()).all()
    bad = batch.block_tables.copy()
    bad[1, 3] = -1  # inside sequence 1's live context
    out_b, st_b = run(bad, 300)
    assert st_b == pa().PA_ERR_BOUNDS
    assert torch.equal(out_b[[0, 2]].view(torch.int16), out[[0, 2]].view(torch.int16))  # other rows unchanged
    out_l, st_l = run(batch.block_tables, 100)  # a context over the stated maximum
    assert st_l == pa().PA_ERR_BOUNDS
    assert (out_l[1] == 0).all()


def test_fp8_effect_against_the_bf16_oracle():
    # the format's own error: fp8 decode against the bf16 decode of the unquantised data
    batch = wl.decode_batch(device=dev(), num_seqs=64, seed=wl.SEED_BASE + 84)
    k0, v0 = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    out, _, _ = _decode_case(batch, 2.0 ** -6, 2.0 ** -6)
    assert oracle.store_kvcache(wl.bf16_bits(batch.tokens.k), wl.bf16_bits(batch.tokens.v), k0, v0,
                                batch.slot_mapping) == oracle.OK
    ref16 = oracle.decode(wl.bf16_bits(batch.tokens.q), k0, v0, batch.block_tables, batch.context_lens, batch.scale)
    err = np.abs(out.double().cpu().numpy() - ref16)
    print(f"fp8 vs bf16 decode: max-abs {err.max():.4f}, mean-abs {err.mean():.5f}")
    # E4M3 keeps 3 mantissa bits (relative half-step 2^-4 per element); the
    # softmax average over hundreds of keys shrinks it
    assert err.max() < 0.1 and err.mean() < 0.01
