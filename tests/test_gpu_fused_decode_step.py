"""pa_norm_rope_store_decode_paged: one layer's decode step in one launch (plus
the split merge) -- head RMSNorm and RoPE of the new token, its KV write and
the paged decode -- against the oracle's norm_rope_store followed by its
decode, through the C ABI.

The attention output must stay within the attention tolerance of the oracle.
The pool rows the call writes: V bit-exact, rotated K within 2 bf16 units of
the oracle's fp64 evaluation of the same steps (plus 2 units of the row's
largest value where the rotation nearly cancels, as for the standalone fused
write); every other pool row untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MAX_ABS, MEAN_ABS, Status, assert_close, compact_pool, dev, i32, pa
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _values(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rows_close(got_bits, ref_bits, what):
    got, ref = _values(got_bits), _values(ref_bits)

    def ulp(v):
        return np.exp2(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126))) - 7)

    allowed = 2 * (ulp(ref) + ulp(np.abs(ref).max(axis=-1, keepdims=True)))
    assert (np.abs(got - ref) <= allowed).all(), f"{what}: rotated K outside 2 bf16 units"


def _run(batch, seqs=None, weights=True, max_positions=4096, seed=31, qkv=None):
    """qkv: one fused QKV row per sequence (the batch's new tokens by default)."""
    d = dev()
    qkv = batch.tokens.qkv if qkv is None else qkv
    hq, hkv = batch.num_heads, batch.num_kv_heads
    qw, kw = wl.norm_weights(seed, device=d) if weights else (None, None)
    cs_np = oracle.rope_cos_sin(wl.ROPE_BASE, 128, max_positions)
    cs = torch.as_tensor(cs_np, device=d)
    ctx = batch.context_lens.astype(np.int32)
    b = len(ctx)
    max_ctx = int(ctx.max())
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    ws = torch.empty(max(pa().pa_decode_workspace_bytes(b, hq, 128, max_ctx), 256), dtype=torch.uint8, device=d)
    out = torch.full((b, hq, 128), float("nan"), dtype=torch.bfloat16, device=d)
    st = Status(d)
    pa().pa_norm_rope_store_decode_paged(qkv, hq, hkv, cs, qw, kw, wl.RMS_EPS, kc, vc,
                                         i32(batch.block_tables, d), i32(ctx, d), max_ctx, batch.scale, out, ws,
                                         dev_status=st.t)
    status = st.value()
    # the oracle: norm + RoPE + KV write, then decode, on the chosen sequences' blocks
    seqs = list(range(b)) if seqs is None else seqs
    bs = batch.layout.block_size
    kb, vb, tables = compact_pool(batch.block_tables, ctx, seqs, batch.k_cache, batch.v_cache, bs)
    meta, rc = oracle.prepare_decode(ctx[seqs], tables, bs, kb.shape[0])
    assert rc == oracle.OK
    qkv_bits = wl.bf16_bits(qkv)[seqs]
    q_ref, rc = oracle.norm_rope_store(qkv_bits, hq, hkv, meta["positions"], cs_np,
                                       None if qw is None else wl.bf16_bits(qw),
                                       None if kw is None else wl.bf16_bits(kw), wl.RMS_EPS, kb, vb,
                                       meta["slot_mapping"])
    ref = oracle.decode(q_ref, kb, vb, tables, meta["context_lens"], batch.scale)
    kg, vg, _ = compact_pool(batch.block_tables, ctx, seqs, kc, vc, bs)
    return out, ref, status, (kg, kb, vg, vb, meta["slot_mapping"]), seqs


def _check_pool(pools, what):
    kg, kb, vg, vb, slots = pools
    np.testing.assert_array_equal(vg, vb)
    rows_g, rows_b = kg.reshape(-1, kg.shape[2], kg.shape[3]), kb.reshape(-1, kb.shape[2], kb.shape[3])
    live = np.unique(slots)
    dead = np.setdiff1d(np.arange(rows_g.shape[0]), live)
    np.testing.assert_array_equal(rows_g[dead], rows_b[dead])
    _rows_close(rows_g[live], rows_b[live], what)


@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 16), (16, 8, 256), (8, 1, 64), (32, 4, 128), (4, 2, 48),
                                       (16, 4, 32)])
def test_fused_step_matches_oracle(hq, hkv, bs):
    ctx = np.array([1, 15, 16, 17, 255, 256, 257, 1000, 33])
    batch = wl.paged_batch(800 + hq + bs, ctx, np.ones_like(ctx), bs, num_heads=hq, num_kv_heads=hkv, device=dev())
    out, ref, status, pools, _ = _run(batch)
    assert status == 0
    assert_close(out, ref, f"fused decode step hq={hq} hkv={hkv} bs={bs}")
    _check_pool(pools, "fused decode step")


def test_fused_step_decode_batch_sampled():
    batch = wl.decode_batch(device=dev())
    ctx = batch.context_lens
    seqs = sorted({0, 1, 2, 63, 64, 127, 128, 200, 254, 255, int(np.argmax(ctx)), int(np.argmin(ctx))})
    out, ref, status, pools, seqs = _run(batch, seqs=seqs)
    assert status == 0
    assert_close(out[torch.as_tensor(seqs, device=out.device)], ref, "fused decode step, decode batch")
    _check_pool(pools, "fused decode step, decode batch")


# Long contexts in a batch large enough for the cluster merge (every sequence
# split over the eight CTAs of one cluster, merged in distributed shared
# memory), with the head norm and RoPE fused: sampled sequences against the oracle.
@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 256), (8, 8, 64)])
def test_fused_step_cluster_merge_sampled(hq, hkv, bs):
    ctx = np.resize(np.array([1, 15, 16, 17, 100, 129, 255, 256, 1000, 2100, 4000, 33]), 96)
    batch = wl.paged_batch(830 + hq + bs, ctx, np.ones_like(ctx), bs, num_heads=hq, num_kv_heads=hkv, device=dev())
    seqs = list(range(12)) + [50, 95]
    out, ref, status, pools, seqs = _run(batch, seqs=seqs, max_positions=4096)
    assert status == 0
    assert_close(out[torch.as_tensor(seqs, device=out.device)], ref, f"fused step, cluster merge hq={hq} hkv={hkv}")
    _check_pool(pools, "fused step, cluster merge")


def test_fused_step_rope_only_and_bad_position():
    ctx = np.array([40, 7, 300, 0])
    batch = wl.paged_batch(811, ctx, np.minimum(ctx, 1), 16, device=dev(), table_width=24)
    qkv = wl.new_tokens(812, 4, device=dev()).qkv  # a row for the padded sequence too
    out, ref, status, pools, _ = _run(batch, seqs=[0, 1, 2], weights=False, qkv=qkv)
    assert status == 0
    assert (out[3] == 0).all()  # a padded sequence (context 0)
    assert_close(out[:3], ref, "RoPE only")
    _check_pool(pools, "RoPE only")
    # a context whose new position is past the table: reported, that sequence's output is 0
    out2, _, status2, _, _ = _run(batch, seqs=[0, 1, 2], weights=False, max_positions=200, qkv=qkv)
    assert status2 == pa().PA_ERR_BOUNDS
    assert (out2[2] == 0).all()
    err = (out2[:2].double() - out[:2].double()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
