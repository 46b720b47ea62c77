"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the
seeded workloads, plus edge cases and invariants.  KV writes are compared
bit for bit over the whole pool; attention within max-abs 2e-2 and mean-abs
2e-3 of the double-precision oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (MAX_ABS, MEAN_ABS, Status, assert_close, compact_pool, dev, gpu_decode, gpu_prefill, gpu_store,
                         grow_keys, i32, oracle_prefill, oracle_store, pa, prefill_workspace)
from oracle_cases import bits
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


# ------------------------------------------------------------------ KV write


@pytest.mark.parametrize("make", [wl.tiny_prefill, wl.varlen_prefill], ids=["tiny", "varlen16k"])
def test_store_bit_exact_whole_pool(make):
    batch = make(device=dev())
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(dev())
    gpu_store(batch, kc, vc, st)
    kb, vb = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    oracle_store(batch, kb, vb)
    assert st.value() == 0
    np.testing.assert_array_equal(wl.bf16_bits(kc), kb)
    np.testing.assert_array_equal(wl.bf16_bits(vc), vb)


@pytest.mark.parametrize("stride_extra", [0, 2, 1], ids=["vec16", "vec4", "vec2"])
def test_store_strides_padding_and_bounds(stride_extra):
    d = dev()
    nb, bs, hkv = 6, 16, 8
    lay = wl.make_layout(5, [40, 9], bs, num_blocks=nb)
    t = 12
    width = hkv * 128 * 2 + stride_extra
    buf = wl.new_tokens(9, t, num_heads=0, num_kv_heads=hkv, device=d).qkv
    full = torch.zeros((t, width), dtype=torch.bfloat16, device=d)
    full[:, : buf.shape[1]] = buf
    k = full[:, : hkv * 128].view(t, hkv, 128) if stride_extra == 0 else \
        torch.as_strided(full, (t, hkv, 128), (width, 128, 1))
    v = torch.as_strided(full, (t, hkv, 128), (width, 128, 1), storage_offset=hkv * 128)
    slots = np.concatenate([lay.slots(0, np.arange(30, 36)), [-1, -1], lay.slots(1, np.arange(0, 3)), [nb * bs + 7]])
    kc = torch.full((nb, bs, hkv, 128), float("nan"), dtype=torch.bfloat16, device=d)
    vc = kc.clone()
    st = Status(d)
    pa().pa_store_kvcache(k, v, kc, vc, i32(slots, d), dev_status=st.t)
    assert st.value() == 4  # the last slot is outside the pool
    kb = np.full((nb, bs, hkv, 128), wl.BF16_NAN_BITS, np.uint16)
    vb = kb.copy()
    rc = oracle.store_kvcache(wl.bf16_bits(k), wl.bf16_bits(v), kb, vb, slots)
    assert rc == oracle.BOUNDS
    np.testing.assert_array_equal(wl.bf16_bits(kc), kb)
    np.testing.assert_array_equal(wl.bf16_bits(vc), vb)


# ------------------------------------------------------------------ prefill


def _prefill_case(batch, paged_and_null=True, seqs=None):
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(kc.device)
    gpu_store(batch, kc, vc, st)
    out = gpu_prefill(batch, kc, vc, paged=True, status=st)
    kb, vb = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    oracle_store(batch, kb, vb)
    ref, rows = oracle_prefill(batch, kb, vb, seqs=seqs)
    assert st.value() == 0
    assert_close(out[torch.as_tensor(rows, device=out.device)], ref, "paged prefill")
    if paged_and_null:
        out_null = gpu_prefill(batch, kc, vc, paged=False, status=st)
        assert st.value() == 0
        assert torch.equal(out.view(torch.int16), out_null.view(torch.int16)), "null vs paged differ"
    return out, kc, vc


def test_prefill_tiny():
    _prefill_case(wl.tiny_prefill(device=dev()))


def test_prefill_varlen_16k():
    _prefill_case(wl.varlen_prefill(device=dev()))


def test_prefill_causal_rows_ignore_the_future():
    """Changing the last 40 tokens of every sequence (their q, k and v) leaves every earlier row's output
    bit-identical: a masked key gets -inf before the row maximum and contributes exactly 0 (the pages' causal-mask
    check, here on the CUDA path)."""
    d = dev()
    batch = wl.varlen_prefill(device=d)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(d)
    gpu_store(batch, kc, vc, st)
    out1 = gpu_prefill(batch, kc, vc, paged=True, status=st)
    cu = batch.cu_seqlens_q
    late = np.concatenate([np.arange(max(cu[b], cu[b + 1] - 40), cu[b + 1]) for b in range(len(cu) - 1)])
    late_t = torch.as_tensor(late, device=d)
    gen = torch.Generator(device="cpu").manual_seed(9)
    qkv = batch.tokens.qkv
    qkv[late_t] = (torch.randn((len(late), qkv.shape[1]), generator=gen) * 3).to(torch.bfloat16).to(d)
    kc2, vc2 = batch.k_cache.clone(), batch.v_cache.clone()
    gpu_store(batch, kc2, vc2, st)
    out2 = gpu_prefill(batch, kc2, vc2, paged=True, status=st)
    assert st.value() == 0
    early = np.setdiff1d(np.arange(int(cu[-1])), late)
    early_t = torch.as_tensor(early, device=d)
    assert torch.equal(out1[early_t].view(torch.int16), out2[early_t].view(torch.int16))
    assert not torch.equal(out1[late_t].view(torch.int16), out2[late_t].view(torch.int16))


def test_prefill_out_aligned_to_16_bytes_only():
    """An output buffer that starts 16 bytes past a 32-byte boundary (allowed:
    the entry point asks for 16) takes the 16-byte-store epilogue instead of
    the 32-byte one; both must give the same bits."""
    batch = wl.varlen_prefill(device=dev())
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(kc.device)
    gpu_store(batch, kc, vc, st)
    ref = gpu_prefill(batch, kc, vc, paged=True, status=st)
    n = ref.numel()
    buf = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device=kc.device)
    out = buf[8:8 + n].view(ref.shape)  # 8 bf16 = 16 bytes in
    assert out.data_ptr() % 32 == 16
    d = kc.device
    max_q, max_k = int(batch.query_lens.max()), int(batch.context_lens.max())
    ws = prefill_workspace(batch.layout.num_seqs, max_q, max_k, 16, 8, d)
    pa().pa_prefill_paged(batch.tokens.q, i32(batch.cu_seqlens_q, d), i32(batch.cu_seqlens_k, d), max_q, max_k,
                          batch.scale, out, workspace=ws, dev_status=st.t, k_cache=kc, v_cache=vc,
                          block_table=i32(batch.block_tables, d))
    assert st.value() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.isnan(buf[:8].float()).all() and torch.isnan(buf[8 + n:].float()).all()


@pytest.mark.parametrize("growth", [0.02, 0.002], ids=["jump_every_tile", "slow_growth"])
@pytest.mark.parametrize("lens", [[700, 1024, 129, 300], [1600]], ids=["batch", "one_long_split"])
def test_prefill_growing_scores_rescale(growth, lens):
    """Scores that grow along the key positions: with q >= 0 and every key
    equal to growth * position, a later key tile's scores exceed the running
    maximum by about 33 (growth 0.02) or 3 (growth 0.002) in log2 units per
    128 keys, so the online softmax moves its maximum and rescales O on nearly
    every tile, inside masked diagonal tiles too, or runs on a stale maximum
    for several tiles.  The single long sequence is a small call whose keys
    are split across CTAs and merged."""
    lens = np.array(lens, dtype=np.int32)
    batch = wl.paged_batch(wl.SEED_BASE + 41, lens, lens, 64, device=dev())
    pos = torch.as_tensor(batch.positions, device=dev(), dtype=torch.float32)
    batch.tokens.q.copy_(batch.tokens.q.abs())
    batch.tokens.k.copy_((growth * pos)[:, None, None].expand_as(batch.tokens.k).to(torch.bfloat16))
    _prefill_case(batch)


@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 16), (8, 8, 32), (8, 1, 64), (32, 4, 128), (4, 2, 256),
                                       (2, 2, 48)])
def test_prefill_shapes_with_cached_prefix(hq, hkv, bs):
    ctx = np.array([1, 70, 129, 300, 64, 200])
    ql = np.array([1, 70, 65, 17, 1, 200])
    batch = wl.paged_batch(300 + hq + bs, ctx, ql, bs, num_heads=hq, num_kv_heads=hkv, device=dev(),
                           num_blocks=64 if bs <= 64 else 40)
    _prefill_case(batch, paged_and_null=False)


def test_prefix_cache_and_chunked_prefill():
    a, b, suffix = wl.prefix_chunk(device=dev())
    kc, vc = a.k_cache.clone(), a.v_cache.clone()
    st = Status(kc.device)
    gpu_store(a, kc, vc, st)
    out_a = gpu_prefill(a, kc, vc, status=st)
    gpu_store(b, kc, vc, st)
    out_b = gpu_prefill(b, kc, vc, status=st)
    assert st.value() == 0
    kb, vb = wl.bf16_bits(a.k_cache).copy(), wl.bf16_bits(a.v_cache).copy()
    oracle_store(a, kb, vb)
    oracle_store(b, kb, vb)
    np.testing.assert_array_equal(wl.bf16_bits(kc), kb)
    # eight of call A's 32 sequences or more: both ends, a spread between, and
    # the longest and shortest suffixes
    ql = a.query_lens
    seqs = sorted({0, 1, 5, 11, 17, 23, 30, 31, int(np.argmax(ql)), int(np.argmin(ql))})
    ref_a, rows_a = oracle_prefill(a, kb, vb, seqs=seqs)
    assert_close(out_a[torch.as_tensor(rows_a, device=out_a.device)], ref_a, "prefix call a")
    ref_b, _ = oracle_prefill(b, kb, vb)
    assert_close(out_b, ref_b, "chunk 2")
    # sequence 0's two chunks equal one call over its whole suffix.  Not bit for
    # bit: a call with few items (the second chunk alone, the whole suffix alone)
    # splits its keys over several CTAs and merges them, a different summation
    # order from the unsplit first call
    s0, c1 = int(suffix[0]), int(a.query_lens[0])
    whole = wl.PagedBatch(wl.PagedLayout(256, a.layout.num_blocks, a.block_tables[:1], np.array([2048 + s0])),
                          np.array([2048 + s0], np.int32), np.array([s0], np.int32),
                          wl.NewTokens(None, torch.cat([a.tokens.q[:c1], b.tokens.q]), None, None),
                          kc, vc)
    out_whole = gpu_prefill(whole, kc, vc, status=st)
    assert st.value() == 0
    chunked = torch.cat([out_a[:c1], out_b])
    err = (out_whole.double() - chunked.double()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    ref_whole, _ = oracle_prefill(whole, kb, vb)
    assert_close(out_whole, ref_whole, "whole suffix in one call")


def test_prefill_block_permutation_bit_identical():
    batch = wl.paged_batch(77, [90, 300, 17], [40, 300, 17], 16, num_blocks=40, device=dev())
    out, kc, vc = _prefill_case(batch, paged_and_null=False)
    perm = torch.as_tensor(np.random.default_rng(1).permutation(40), device=kc.device)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt = batch.block_tables
    bt2 = np.where(bt >= 0, perm.cpu().numpy()[np.maximum(bt, 0)], -1)
    batch2 = wl.PagedBatch(wl.PagedLayout(16, 40, bt2.astype(np.int32), batch.layout.reserve_lens),
                           batch.context_lens, batch.query_lens, batch.tokens, kc2, vc2)
    out2 = gpu_prefill(batch2, kc2, vc2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_prefill_device_errors_are_reported_not_faulted():
    batch = wl.paged_batch(88, [40, 20], [40, 20], 16, num_blocks=8, device=dev())
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    gpu_store(batch, kc, vc)
    bad = batch.block_tables.copy()
    bad[0, 1] = 999  # not a block of the pool
    batch_bad = wl.PagedBatch(wl.PagedLayout(16, 8, bad, batch.layout.reserve_lens), batch.context_lens,
                              batch.query_lens, batch.tokens, kc, vc)
    st = Status(kc.device)
    gpu_prefill(batch_bad, kc, vc, status=st)
    assert st.value() == 4


def test_worked_example_through_gpu():
    """The three-position example (Q = K = V = X, scale 1/sqrt(2)) with head
    dims 2..127 zero: zero dims do not change any dot product."""
    d = dev()
    x = np.zeros((3, 1, 128))
    x[:, 0, :2] = [[1, 0], [0, 1], [1, 1]]
    q = torch.as_tensor(x, dtype=torch.bfloat16, device=d)
    out = torch.empty_like(q)
    cu = i32([0, 3], d)
    pa().pa_prefill_paged(q, cu, cu, 3, 3, 1 / math.sqrt(2), out, k=q, v=q,
                          workspace=prefill_workspace(1, 3, 3, 1, 1, d))
    got = out[:, 0, :2].double().cpu().numpy()
    np.testing.assert_allclose(got[-1], [0.7517, 0.7517], atol=1e-2)
    np.testing.assert_allclose(got[1], [0.3302, 0.6698], atol=1e-2)


# ------------------------------------------------------------------ decode


def _decode_vs_oracle(batch, seqs=None):
    """GPU KV write + decode of the whole batch; the oracle recomputes the
    chosen sequences from the generator's pool (only their blocks, copied to
    the host and renumbered) after its own KV write of their new tokens."""
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(kc.device)
    gpu_store(batch, kc, vc, st)
    out = gpu_decode(batch.tokens.q, kc, vc, batch.block_tables, batch.context_lens, batch.scale, st)
    assert st.value() == 0
    seqs = list(range(batch.layout.num_seqs)) if seqs is None else seqs
    ctx = batch.context_lens[seqs]
    bs = batch.layout.block_size
    kb, vb, tables = compact_pool(batch.block_tables, batch.context_lens, seqs, batch.k_cache, batch.v_cache, bs)
    sub = wl.PagedLayout(bs, kb.shape[0], tables, ctx)
    slots = np.array([sub.slots(i, [c - 1])[0] for i, c in enumerate(ctx)], np.int32)
    rc = oracle.store_kvcache(wl.bf16_bits(batch.tokens.k)[seqs], wl.bf16_bits(batch.tokens.v)[seqs], kb, vb, slots)
    assert rc == oracle.OK
    ref = oracle.decode(wl.bf16_bits(batch.tokens.q)[seqs], kb, vb, tables, ctx, batch.scale)
    assert_close(out[torch.as_tensor(seqs, device=out.device)], ref, "decode")
    return out, kc, vc


def test_decode_tiny_eight_steps():
    d = dev()
    batch = wl.tiny_prefill(device=d)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    kb, vb = wl.bf16_bits(kc).copy(), wl.bf16_bits(vc).copy()
    gpu_store(batch, kc, vc)
    oracle_store(batch, kb, vb)
    st = Status(d)
    for step in range(wl.TINY_DECODE_STEPS):
        toks = wl.tiny_decode_tokens(step, device=d)
        ctx = (batch.context_lens + step + 1).astype(np.int32)
        slots = np.array([batch.layout.slots(b, [c - 1])[0] for b, c in enumerate(ctx)], np.int32)
        gpu_store(batch, kc, vc, st, tokens=toks, slots=slots)
        oracle_store(batch, kb, vb, tokens=toks, slots=slots)
        out = gpu_decode(toks.q, kc, vc, batch.block_tables, ctx, batch.scale, st)
        ref = oracle.decode(wl.bf16_bits(toks.q), kb, vb, batch.block_tables, ctx, batch.scale)
        assert st.value() == 0
        assert_close(out, ref, f"tiny decode step {step}")
    np.testing.assert_array_equal(wl.bf16_bits(kc), kb)


def test_decode_batch_256():
    _decode_vs_oracle(wl.decode_batch(device=dev()))


def test_decode_long_context_512_full_size_sampled():
    batch = wl.long_decode(device=dev())
    ctx = batch.context_lens
    seqs = sorted({0, 1, 2, 37, 100, 128, 200, 255, 256, 301, 384, 400, 450, 500, 510, 511,
                   int(np.argmax(ctx)), int(np.argmin(ctx))})
    out, _, _ = _decode_vs_oracle(batch, seqs=seqs)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 16), (8, 8, 32), (8, 1, 64), (32, 4, 128), (4, 2, 256),
                                       (32, 8, 16), (16, 2, 48)])
def test_decode_shapes(hq, hkv, bs):
    ctx = np.array([1, 15, 16, 17, 255, 256, 257, 1000, 33])
    batch = wl.paged_batch(500 + hq + bs, ctx, np.ones_like(ctx), bs, num_heads=hq, num_kv_heads=hkv,
                           device=dev())
    _decode_vs_oracle(batch)


# Long contexts in a batch large enough that every sequence is split over the
# eight CTAs of one thread-block cluster and merged in distributed shared
# memory: sequences of one token, ragged and exact chunks, sequences with fewer
# splits than the cluster has CTAs, and long ones, for every group size; then
# the fused KV write + decode over the same cluster path, bit-equal to the two
# calls.
@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 256), (8, 1, 64), (32, 4, 16), (4, 2, 48)])
def test_decode_cluster_merge(hq, hkv, bs):
    ctx = np.resize(np.array([1, 15, 16, 17, 100, 129, 255, 256, 1000, 2100, 4000, 33]), 96)
    batch = wl.paged_batch(520 + hq + bs, ctx, np.ones_like(ctx), bs, num_heads=hq, num_kv_heads=hkv,
                           device=dev())
    out, kc, vc = _decode_vs_oracle(batch, seqs=list(range(12)) + [50, 95])
    kf, vf = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(kf.device)
    fused = _store_decode_fused(batch.tokens.q, batch.tokens.k, batch.tokens.v, kf, vf, batch.block_tables,
                                batch.context_lens, batch.scale, st)
    assert st.value() == 0
    assert torch.equal(fused.view(torch.int16), out.view(torch.int16))
    assert torch.equal(kf.view(torch.int16), kc.view(torch.int16)) and torch.equal(vf.view(torch.int16), vc.view(torch.int16))


# Scores that grow along the keys (every key = growth * position, q >= 0):
# with growth 0.02 a 16-token chunk scores about 4 higher (log2 units) than
# the one before, so every decode kernel moves its running maximum (and
# rescales O) every few chunks, in every lane; with 0.002 it runs on a stale
# maximum for many chunks.  The CUDA-core kernel (16 q heads), the tensor-core
# kernel (32 and 64 q heads over 8) and the cluster merge (96 long sequences).
@pytest.mark.parametrize("growth", [0.02, 0.002], ids=["fast_growth", "slow_growth"])
@pytest.mark.parametrize("hq,hkv,nseq", [(16, 8, 8), (32, 8, 8), (64, 8, 8), (16, 8, 96)],
                         ids=["cuda_core", "mma_g4", "mma_g8", "cluster"])
def test_decode_growing_scores_rescale(growth, hq, hkv, nseq):
    ctx = np.resize(np.array([700, 1024, 129, 300, 1600, 17, 2100, 40]), nseq)
    batch = wl.paged_batch(wl.SEED_BASE + 47 + hq + nseq, ctx, np.ones_like(ctx), 64, num_heads=hq,
                           num_kv_heads=hkv, device=dev())
    grow_keys(batch, growth)
    _decode_vs_oracle(batch)


def _store_decode_fused(q, k_new, v_new, kc, vc, tables, ctx, scale, status, max_ctx=None):
    d = kc.device
    b = q.shape[0]
    max_ctx = int(np.max(ctx)) if max_ctx is None else max_ctx
    ws = torch.empty(max(pa().pa_decode_workspace_bytes(b, q.shape[1], 128, max_ctx), 256), dtype=torch.uint8,
                     device=d)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=d)
    pa().pa_store_decode_paged(q, k_new, v_new, kc, vc, i32(tables, d), i32(ctx, d), max_ctx, scale, out, ws,
                               dev_status=status.t)
    return out


@pytest.mark.parametrize("hq,hkv,bs", [(16, 8, 256), (16, 8, 16), (8, 1, 64), (32, 4, 128), (4, 2, 256)])
def test_store_decode_fused_equals_store_then_decode(hq, hkv, bs):
    """pa_store_decode_paged: the same output bits and the same pools (every row) as pa_store_kvcache at the
    decode step's slots followed by pa_decode_paged."""
    if (hq, hkv, bs) == (16, 8, 256):
        batch = wl.decode_batch(device=dev())
    else:
        ctx = np.array([1, 15, 16, 17, 255, 256, 257, 1000, 33])
        batch = wl.paged_batch(700 + hq + bs, ctx, np.ones_like(ctx), bs, num_heads=hq, num_kv_heads=hkv,
                               device=dev())
    d = dev()
    kc1, vc1 = batch.k_cache.clone(), batch.v_cache.clone()
    st1 = Status(d)
    gpu_store(batch, kc1, vc1, st1)
    ref = gpu_decode(batch.tokens.q, kc1, vc1, batch.block_tables, batch.context_lens, batch.scale, st1)
    kc2, vc2 = batch.k_cache.clone(), batch.v_cache.clone()
    st2 = Status(d)
    out = _store_decode_fused(batch.tokens.q, batch.tokens.k, batch.tokens.v, kc2, vc2, batch.block_tables,
                              batch.context_lens, batch.scale, st2)
    assert st1.value() == 0 and st2.value() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "fused output differs"
    assert torch.equal(kc2.view(torch.int16), kc1.view(torch.int16)), "fused K pool differs"
    assert torch.equal(vc2.view(torch.int16), vc1.view(torch.int16)), "fused V pool differs"


def test_store_decode_fused_decode_batch_vs_oracle():
    """pa_store_decode_paged on the decode-batch workload (256 sequences, block size 256), in the launch
    configuration the step uses, against the oracle's KV write + decode on a sample of sequences.  The oracle's
    write slots come from its own decode metadata builder (position context_lens[b] - 1 through the table), not
    from the input generator; the written pool rows are compared too."""
    d = dev()
    batch = wl.decode_batch(device=d)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(d)
    out = _store_decode_fused(batch.tokens.q, batch.tokens.k, batch.tokens.v, kc, vc, batch.block_tables,
                              batch.context_lens, batch.scale, st)
    assert st.value() == 0
    ctx = batch.context_lens
    seqs = sorted({0, 1, 2, 31, 63, 64, 100, 127, 128, 180, 200, 233, 254, 255,
                   int(np.argmax(ctx)), int(np.argmin(ctx))})
    bs = batch.layout.block_size
    kb, vb, tables = compact_pool(batch.block_tables, ctx, seqs, batch.k_cache, batch.v_cache, bs)
    meta, rc = oracle.prepare_decode(ctx[seqs], tables, bs, kb.shape[0])
    assert rc == oracle.OK
    np.testing.assert_array_equal(meta["context_lens"], ctx[seqs])
    rc = oracle.store_kvcache(wl.bf16_bits(batch.tokens.k)[seqs], wl.bf16_bits(batch.tokens.v)[seqs], kb, vb,
                              meta["slot_mapping"])
    assert rc == oracle.OK
    ref = oracle.decode(wl.bf16_bits(batch.tokens.q)[seqs], kb, vb, tables, meta["context_lens"], batch.scale)
    assert_close(out[torch.as_tensor(seqs, device=d)], ref, "fused KV write + decode, decode batch")
    kg, vg, _ = compact_pool(batch.block_tables, ctx, seqs, kc, vc, bs)
    np.testing.assert_array_equal(kg, kb)
    np.testing.assert_array_equal(vg, vb)


# (16, 8): the CUDA-core decode kernel; (32, 4), (64, 8): the tensor-core one
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 4), (64, 8)])
def test_store_decode_fused_padding_rows_and_bad_block(hq, hkv):
    """Padded sequences (context 0) are neither written nor read; a new-token row whose block id is invalid is
    reported (PA_ERR_BOUNDS) and not written."""
    d = dev()
    ctx = np.array([0, 40, 0, 7])
    batch = wl.paged_batch(602, ctx, np.minimum(ctx, 1), 16, device=d, table_width=4, num_heads=hq,
                           num_kv_heads=hkv)
    gen = torch.Generator(device="cpu").manual_seed(5)
    q = torch.randn((4, hq, 128), generator=gen).to(torch.bfloat16).to(d)
    k_new = torch.randn((4, hkv, 128), generator=gen).to(torch.bfloat16).to(d)
    v_new = torch.randn((4, hkv, 128), generator=gen).to(torch.bfloat16).to(d)
    slots = np.array([-1 if c == 0 else batch.layout.slots(b, [c - 1])[0] for b, c in enumerate(ctx)], np.int32)
    kc1, vc1 = batch.k_cache.clone(), batch.v_cache.clone()
    st1 = Status(d)
    pa().pa_store_kvcache(k_new, v_new, kc1, vc1, i32(slots, d), dev_status=st1.t)
    ref = gpu_decode(q, kc1, vc1, batch.block_tables, ctx, batch.scale, st1)
    kc2, vc2 = batch.k_cache.clone(), batch.v_cache.clone()
    st2 = Status(d)
    out = _store_decode_fused(q, k_new, v_new, kc2, vc2, batch.block_tables, ctx, batch.scale, st2)
    assert st1.value() == 0 and st2.value() == 0
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kc2.view(torch.int16), kc1.view(torch.int16))
    assert torch.equal(vc2.view(torch.int16), vc1.view(torch.int16))
    # sequence 3's new token (position 6) lives in table entry 0: make it invalid
    bad = batch.block_tables.copy()
    bad[3, 0] = -1
    kc3, vc3 = batch.k_cache.clone(), batch.v_cache.clone()
    st3 = Status(d)
    _store_decode_fused(q, k_new, v_new, kc3, vc3, bad, ctx, batch.scale, st3)
    assert st3.value() == 4
    row3 = slots[3]
    assert torch.equal(kc3.view(-1, hkv, 128)[row3].view(torch.int16),
                       batch.k_cache.view(-1, hkv, 128)[row3].view(torch.int16)), "row with a bad block id was written"


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 4), (64, 8)])
def test_decode_padded_rows_and_bounds(hq, hkv):
    d = dev()
    ctx = np.array([0, 40, 0, 7])
    batch = wl.paged_batch(601, ctx, np.minimum(ctx, 1), 16, device=d, table_width=4, num_heads=hq,
                           num_kv_heads=hkv)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    gpu_store(batch, kc, vc)
    q = torch.randn((4, hq, 128), device=d).to(torch.bfloat16)
    st = Status(d)
    out = gpu_decode(q, kc, vc, batch.block_tables, ctx, batch.scale, st)
    assert st.value() == 0
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert torch.isfinite(out.float()).all()
    # a context longer than the stated maximum is reported, and its row is 0
    st2 = Status(d)
    out2 = gpu_decode(q, kc, vc, batch.block_tables, ctx, batch.scale, st2, max_ctx=20)
    assert st2.value() == 4
    assert (out2[1] == 0).all()
    # a -1 table entry inside the live context is reported
    bad = batch.block_tables.copy()
    bad[1, 1] = -1
    st3 = Status(d)
    gpu_decode(q, kc, vc, bad, ctx, batch.scale, st3)
    assert st3.value() == 4


def test_decode_equals_prefill_row():
    """Decoding position t over the cache agrees with row t of a causal
    prefill over the same tokens (both against the oracle's tolerance)."""
    d = dev()
    n = 300
    batch = wl.paged_batch(611, [n], [n], 16, device=d, num_blocks=32)
    out, kc, vc = _prefill_case(batch, paged_and_null=False)
    for t in (0, 15, 16, 199, n - 1):
        dec = gpu_decode(batch.tokens.q[t:t + 1], kc, vc, batch.block_tables, [t + 1], batch.scale)
        err = (dec[0].double() - out[t].double()).abs().max().item()
        assert err <= 2e-2


def test_decode_block_permutation_bit_identical():
    batch = wl.decode_batch(device=dev(), num_seqs=32)
    out, kc, vc = _decode_vs_oracle(batch)
    nb = batch.layout.num_blocks
    perm = torch.as_tensor(np.random.default_rng(2).permutation(nb), device=kc.device)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt = batch.block_tables
    bt2 = np.where(bt >= 0, perm.cpu().numpy()[np.maximum(bt, 0)], -1)
    out2 = gpu_decode(batch.tokens.q, kc2, vc2, bt2, batch.context_lens, batch.scale)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("hq,hkv", [(16, 8), (8, 8)])
def test_small_calls_split_keys_and_match_oracle(hq, hkv):
    # one or two long-context sequences: too few items for the GPU, so each
    # item's keys are split over several CTAs and merged
    batch = wl.paged_batch(wl.SEED_BASE + 90 + hq, [3000, 1700], [300, 129], 64, num_heads=hq, num_kv_heads=hkv,
                           device=dev())
    assert pa().pa_prefill_workspace_bytes(2, 300, 3000, hq, hkv) > 0
    out, kc, vc = _prefill_case(batch, paged_and_null=False)
