"""Fused head RMSNorm + RoPE + KV write on the GPU against the oracle.

Through the C ABI (binding -> libpa.so).  The V copy and every pool row the
call must not touch are compared bit for bit.  Rotated Q and K are compared
with the oracle's fp64 evaluation of the same steps: each step rounds to bf16,
and fp32 arithmetic changes a rounding only when a value lies within fp32
error of a bf16 rounding boundary, so at most a small fraction of elements
may differ, each by at most 2 bf16 units in the last place (one from the
result's own rounding, one carried from the other rounding) -- except that
a one-unit difference in a normalised input a or b (a legitimate rounding
difference of fp32 against fp64 in the norm step) moves a cos - b sin by up
to one unit of that INPUT, which where the rotation nearly cancels is many
units of the small result.  Hence the bound per element: 2 units of the
result plus 2 units of the row's largest value (which the rotation keeps:
it preserves each pair's length), and at least 99% identical elements.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Status, dev, i32, pa
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ULPS = 2
MIN_IDENTICAL = 0.99


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _values(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_rotated(got_bits, ref_bits, what):
    """Every element within MAX_ULPS bf16 units of the oracle plus MAX_ULPS units
    of its row's largest value; at least MIN_IDENTICAL bit-identical."""
    assert got_bits.shape == ref_bits.shape
    got, ref = _values(got_bits), _values(ref_bits)
    assert np.isfinite(got).all(), f"{what}: non-finite values"

    def ulp(v):
        return np.exp2(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126))) - 7)

    row_max = np.abs(ref).max(axis=-1, keepdims=True)
    allowed = MAX_ULPS * (ulp(ref) + ulp(row_max))
    err = np.abs(got - ref)
    same = float((got_bits == ref_bits).mean())
    worst = float((err / allowed).max())
    assert worst <= 1.0 and same >= MIN_IDENTICAL, f"{what}: worst error {worst:.2f} of the bound, identical {same:.5f}"


def _table(device):
    cs = oracle.rope_cos_sin(wl.ROPE_BASE, 128, 4096)
    return cs, torch.as_tensor(cs, device=device)


def _run(batch, slots, positions, weights=True, eps=wl.RMS_EPS, in_place=False, status=None, seed=21):
    d = dev()
    qw, kw = wl.norm_weights(seed, device=d) if weights else (None, None)
    cs_np, cs = _table(d)
    toks = batch.tokens
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    kc_before, vc_before = wl.bf16_bits(kc), wl.bf16_bits(vc)
    q_out = toks.qkv[:, : batch.num_heads * 128].view(-1, batch.num_heads, 128) if in_place else \
        torch.full((toks.qkv.shape[0], batch.num_heads, 128), float("nan"), dtype=torch.bfloat16, device=d)
    qkv_bits = wl.bf16_bits(toks.qkv)  # read before an in-place call rewrites the Q columns
    pa().pa_norm_rope_store_kvcache(toks.qkv, batch.num_heads, batch.num_kv_heads, i32(positions, d), cs, qw, kw,
                                    eps, q_out, kc, vc, i32(slots, d),
                                    dev_status=None if status is None else status.t)
    torch.cuda.synchronize()
    # oracle on the same inputs
    kc_ref, vc_ref = kc_before.copy(), vc_before.copy()
    q_ref, rc = oracle.norm_rope_store(qkv_bits, batch.num_heads, batch.num_kv_heads, positions, cs_np,
                                       None if qw is None else wl.bf16_bits(qw), None if kw is None else wl.bf16_bits(kw),
                                       eps, kc_ref, vc_ref, slots)
    return (wl.bf16_bits(q_out), q_ref, wl.bf16_bits(kc), kc_ref, wl.bf16_bits(vc), vc_ref, rc)


def _compare(res, slots, what):
    q, q_ref, kc, kc_ref, vc, vc_ref, _ = res
    _check_rotated(q, q_ref, f"{what}: q")
    np.testing.assert_array_equal(vc, vc_ref)  # V and every untouched row: bit-exact
    rows = kc.reshape(-1, kc.shape[2], kc.shape[3])
    rows_ref = kc_ref.reshape(rows.shape)
    live = np.unique(slots[slots != -1])
    dead = np.setdiff1d(np.arange(rows.shape[0]), live)
    np.testing.assert_array_equal(rows[dead], rows_ref[dead])
    _check_rotated(rows[live], rows_ref[live], f"{what}: k")


def test_tiny_batch_matches_oracle():
    batch = wl.paged_batch(wl.SEED_BASE + 60, [7, 33, 64, 100], [7, 33, 64, 100], 16, device=dev())
    slots, pos = batch.slot_mapping, batch.positions
    _compare(_run(batch, slots, pos), slots, "tiny")


def test_prefill_sized_call_with_padding_rows():
    # the varlen-prefill workload's shapes (lengths U[100,1024], block size 256); every 97th token is padding
    lens = wl.varlen_prefill_lengths(budget=4096)
    batch = wl.paged_batch(wl.SEED_BASE + 61, lens, lens, 256, device=dev())
    slots, pos = batch.slot_mapping.copy(), batch.positions
    slots[::97] = -1
    _compare(_run(batch, slots, pos), slots, "prefill-sized")


def test_decode_sized_call_at_late_positions():
    # one new token per sequence at positions up to 4095 (the long-decode workload's range)
    ctx = np.random.default_rng(5).integers(1024, 4096, 256, endpoint=True)
    batch = wl.paged_batch(wl.SEED_BASE + 62, ctx, np.ones(256, int), 256, device=dev())
    slots, pos = batch.slot_mapping, batch.positions
    _compare(_run(batch, slots, pos), slots, "decode-sized")


@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 1), (8, 1), (16, 4), (32, 8), (64, 8)])
def test_head_configurations(hq, hkv):
    """Every supported head count, including the odd row totals of one KV head
    (Hq + 1 rows of Q and K, then one V row), where a K row and a V row are
    processed together."""
    batch = wl.paged_batch(wl.SEED_BASE + 66, [33, 70], [33, 70], 16, num_heads=hq, num_kv_heads=hkv, device=dev())
    slots, pos = batch.slot_mapping, batch.positions
    _compare(_run(batch, slots, pos), slots, f"hq={hq} hkv={hkv}")


def test_rope_only_without_norm_weights():
    batch = wl.paged_batch(wl.SEED_BASE + 63, [50, 77], [50, 77], 16, device=dev())
    slots, pos = batch.slot_mapping, batch.positions
    _compare(_run(batch, slots, pos, weights=False), slots, "rope only")


def test_q_written_in_place():
    batch = wl.paged_batch(wl.SEED_BASE + 64, [40, 90], [40, 90], 32, device=dev())
    slots, pos = batch.slot_mapping, batch.positions
    _compare(_run(batch, slots, pos, in_place=True), slots, "in place")


def test_bad_position_and_slot_reported_and_skipped():
    batch = wl.paged_batch(wl.SEED_BASE + 65, [20, 20], [20, 20], 16, device=dev())
    slots, pos = batch.slot_mapping.copy(), batch.positions.copy()
    pos[3] = 4096          # one past the table
    slots[30] = 1 << 20    # not a row of the pool
    st = Status(dev())
    res = _run(batch, slots, pos, status=st)
    assert int(st.t.item()) == pa().PA_ERR_BOUNDS and res[-1] == oracle.BOUNDS
    q = res[0]
    # the skipped tokens' q_out rows keep their NaN fill; their pool rows are untouched
    assert (q[[3, 30]] & 0x7FFF > 0x7F80).all()
    keep = np.ones(len(pos), bool)
    keep[[3, 30]] = False
    _check_rotated(q[keep], res[1][keep], "q of the other tokens")
    live = slots.copy()
    live[[3, 30]] = -1
    _compare((q[keep], res[1][keep]) + res[2:], live, "other tokens")


def test_host_errors_return_before_launch():
    d = dev()
    batch = wl.paged_batch(wl.SEED_BASE + 66, [8], [8], 16, device=d)
    cs = _table(d)[1]
    q_out = torch.empty((8, 16, 128), dtype=torch.bfloat16, device=d)
    with pytest.raises(pa().PaError) as e:
        pa().pa_norm_rope_store_kvcache(batch.tokens.qkv, 16, 8, i32(batch.positions, d), cs, None, None, -1.0,
                                        q_out, batch.k_cache, batch.v_cache, i32(batch.slot_mapping, d))
    assert e.value.status == pa().PA_ERR_INVALID_ARG


def test_device_table_matches_oracle_table():
    d = dev()
    got = pa().pa_rope_cos_sin_table(wl.ROPE_BASE, 128, 4096, device=d).cpu().numpy()
    ref = oracle.rope_cos_sin(wl.ROPE_BASE, 128, 4096)
    # both evaluate in double and round once to float: equal up to one float unit
    # where the two double evaluations straddle a float rounding boundary
    diff = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    ulp = np.spacing(np.abs(ref)).astype(np.float64)
    assert (diff <= ulp).all() and (got == ref).mean() > 0.999
