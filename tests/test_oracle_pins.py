"""Pins of the CPU oracle against values the pages print, closed forms,
brute force on tiny inputs and the invariants the method must satisfy.

None of these tests touch the CUDA library.
"""
import math

import numpy as np
import pytest

import oracle
from oracle_cases import bits, brute_force_attention, nan_pool, values
from paged_kv_cache_110_gb300 import workloads as wl


def _store_seq(kc, vc, k_bits, v_bits, table, block_size):
    n, d = k_bits.shape
    slots = [oracle.slot(np.array(table), block_size, p) for p in range(n)]
    rc = oracle.store_kvcache(k_bits.reshape(n, 1, d), v_bits.reshape(n, 1, d), kc, vc, slots)
    assert rc == oracle.OK
    return slots


def _decode_one(q_vals, k_vals, v_vals, scale, block_size=4, table=(2, 0, 3), num_blocks=4):
    """Decode of one query over len(k_vals) keys stored through a paged pool."""
    k_b, v_b = bits(k_vals), bits(v_vals)
    d = k_b.shape[1]
    kc, vc = nan_pool(num_blocks, block_size, 1, d), nan_pool(num_blocks, block_size, 1, d)
    width = -(-len(k_vals) // block_size)
    bt = np.array([list(table)[:width]], dtype=np.int32)
    _store_seq(kc, vc, k_b, v_b, bt[0], block_size)
    q_b = bits(q_vals).reshape(1, 1, d)
    return oracle.decode(q_b, kc, vc, bt, [len(k_vals)], scale)[0, 0]


def _prefill_one(x_q, x_k, x_v, scale, paged=True, block_size=2, table=(3, 1), num_blocks=4):
    """Full causal prefill of one sequence (Lq = Lk); returns (out, weights per row)."""
    qb, kb, vb = bits(x_q), bits(x_k), bits(x_v)
    n, d = qb.shape
    cu = [0, n]
    kw = {}
    if paged:
        kc, vc = nan_pool(num_blocks, block_size, 1, d), nan_pool(num_blocks, block_size, 1, d)
        bt = np.array([list(table)], dtype=np.int32)
        _store_seq(kc, vc, kb, vb, bt[0], block_size)
        kw = dict(k_cache=kc, v_cache=vc, block_table=bt)
    else:
        kw = dict(k=kb.reshape(n, 1, d), v=vb.reshape(n, 1, d))
    rows = []
    out = None
    for i in range(n):
        out, w = oracle.prefill(qb.reshape(n, 1, d), cu, cu, scale, weights_of=(0, 0, i), **kw)
        rows.append(w)
    return out[:, 0, :], np.array(rows)


# ----------------------------------------------------------------- printed examples


def test_one_dim_head(golden):
    g = golden("attention_examples.json")["one_dim_head"]
    out = _decode_one(g["q"], g["k"], g["v"], g["scale"])
    assert round(out[0], g["out_decimals"]) == g["out"][0]
    _, w = _prefill_one([[0.0], [0.0]] + g["q"], g["k"], g["v"], g["scale"], block_size=2,
                        table=(3, 1))
    np.testing.assert_array_equal(np.round(w[2], g["weights_decimals"]), g["weights"])


def test_softmax_with_temperature(golden):
    g = golden("attention_examples.json")["softmax_of_1_2_3"]
    # scores z_j = scale * q * k_j with q = 1 and k = z: the temperature is 1 / scale
    for case in g["cases"]:
        scale = 1.0 / case["temperature"]
        qs = [[0.0], [0.0], [1.0]]
        _, w = _prefill_one(qs, [[z] for z in g["scores"]], [[0.0]] * 3, scale, block_size=4,
                            table=(1,), num_blocks=2)
        np.testing.assert_array_equal(np.round(w[2], g["weights_decimals"]), case["weights"])


@pytest.mark.parametrize("paged", [True, False])
def test_causal_three_positions(golden, paged):
    g = golden("attention_examples.json")["causal_three_positions"]
    out, w = _prefill_one(g["x"], g["x"], g["x"], g["scale"], paged=paged)
    np.testing.assert_array_equal(np.round(w, g["weights_decimals"]), g["weights"])
    np.testing.assert_array_equal(np.round(out[-1], g["out_decimals"]), g["last_out"])
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)


def test_distinct_v(golden):
    g = golden("attention_examples.json")["distinct_v"]
    out, w = _prefill_one(g["qk"], g["qk"], g["v"], g["scale"])
    np.testing.assert_allclose(w[-1], g["last_weights"], atol=0.6 * 10 ** -g["weights_decimals"])
    np.testing.assert_allclose(out[-1], g["last_out"], atol=0.6 * 10 ** -g["out_decimals"])


def test_future_change(golden):
    g = golden("attention_examples.json")["future_change"]
    x = g["x"]
    y = [x[0], x[1], g["changed_last"]]
    before, _ = _prefill_one(x, x, x, g["scale"])
    after, _ = _prefill_one(y, y, y, g["scale"])
    assert np.abs(after[:2] - before[:2]).max() == g["masked_earlier_delta"]
    # without the mask an earlier row reads all three keys: a one-query call over 3 keys
    delta = max(np.abs(_decode_one(y[i], y, y, g["scale"]) - _decode_one(x[i], x, x, g["scale"])).max()
                for i in range(2))
    assert round(delta, g["delta_decimals"]) == g["unmasked_earlier_delta"]


def test_cached_fourth_position(golden):
    g = golden("attention_examples.json")["cached_fourth_position"]
    x4 = g["x"] + [g["appended"]]
    full, _ = _prefill_one(x4, x4, x4, g["scale"])
    cached = _decode_one(g["appended"], x4, x4, g["scale"], block_size=2, table=(3, 1))
    np.testing.assert_array_equal(np.round(full[-1], g["out_decimals"]), g["last_out"])
    assert np.abs(full[-1] - cached).max() == g["max_error"]


def test_page_merge(golden):
    g = golden("attention_examples.json")["page_merge"]
    # two pages of two keys: scores 0 (exp sum 2) and ln 3 (exp sum 6)
    scale = math.log(3.0)
    k = [[0.0], [0.0], [1.0], [1.0]]
    v = [[0.0], [0.0], [1.0], [1.0]]
    q = [[0.0]] * 3 + [[1.0]]
    out, w = _prefill_one(q, k, v, scale, block_size=2, table=(3, 1), num_blocks=4)
    np.testing.assert_allclose([w[3][:2].sum(), w[3][2:].sum()], g["page_weights"], atol=1e-12)
    np.testing.assert_allclose(out[3][0], g["page_weights"][1], atol=1e-12)


# ----------------------------------------------------------------- slots and sizes


def test_slot_examples(golden):
    g = golden("slot_examples.json")
    for case in g["cases"]:
        table, bs = np.array(case["table"], np.int32), case["block_size"]
        if "positions" in case:
            pos, want = case["positions"], case["slots"]
        else:
            pos = list(range(*case["position_range"]))
            want = list(range(*case["slot_range"]))
        assert [oracle.slot(table, bs, p) for p in pos] == want, case["source"]
    c = g["block_crossing"]
    for p0, p1 in [(3, 9), (40, 2)]:
        got = [oracle.slot(np.array([p0, p1], np.int32), c["block_size"], p) for p in c["positions"]]
        assert got == [p1 * c["block_size"] + o for o in c["slot_offsets_in_p1"]]


def test_kv_bytes_closed_form(golden):
    g = golden("kv_bytes.json")
    for key in ("per_token", "per_position_per_layer"):
        c = g[key]
        assert oracle.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["elem_bytes"]) == c["bytes"]
    t = g["per_token"]
    per_tok = oracle.kv_bytes_per_token(t["layers"], t["kv_heads"], t["head_dim"], t["elem_bytes"])
    assert per_tok * g["per_block"]["block_size"] == g["per_block"]["bytes"]
    assert per_tok * g["per_4096_positions_mib"]["positions"] == g["per_4096_positions_mib"]["mib"] << 20


# ----------------------------------------------------------------- KV write


def test_store_page_example(golden):
    """Second round of the main example: A (table [17,5,23]) writes positions
    512..699 to slots 5888..6075, B (table [11]) positions 0..31 to
    2816..2847; every other row stays poisoned."""
    g = golden("slot_examples.json")["cases"]
    a_slots = list(range(*g[3]["slot_range"]))
    b_slots = list(range(*g[4]["slot_range"]))
    slots = np.array(a_slots + b_slots + [-1, -1], dtype=np.int32)  # two padded rows
    toks = wl.new_tokens(7, len(slots), num_heads=2, num_kv_heads=2, head_dim=8)
    k, v = wl.bf16_bits(toks.k), wl.bf16_bits(toks.v)
    kc, vc = nan_pool(24, 256, 2, 8), nan_pool(24, 256, 2, 8)
    assert oracle.store_kvcache(k, v, kc, vc, slots) == oracle.OK
    flat_k, flat_v = kc.reshape(-1, 2, 8), vc.reshape(-1, 2, 8)
    live = slots[slots >= 0]
    np.testing.assert_array_equal(flat_k[live], k[: len(live)])
    np.testing.assert_array_equal(flat_v[live], v[: len(live)])
    rest = np.setdiff1d(np.arange(flat_k.shape[0]), live)
    assert (flat_k[rest] == wl.BF16_NAN_BITS).all() and (flat_v[rest] == wl.BF16_NAN_BITS).all()


def test_store_out_of_range_slot_reported():
    toks = wl.new_tokens(8, 3, num_heads=1, num_kv_heads=1, head_dim=4)
    k, v = wl.bf16_bits(toks.k), wl.bf16_bits(toks.v)
    kc, vc = nan_pool(2, 4, 1, 4), nan_pool(2, 4, 1, 4)
    assert oracle.store_kvcache(k, v, kc, vc, [1, 8, 5]) == oracle.BOUNDS
    np.testing.assert_array_equal(kc.reshape(-1, 1, 4)[[1, 5]], k[[0, 2]])
    assert oracle.store_kvcache(k, v, kc, vc, [1, -2, 5]) == oracle.BOUNDS


# ----------------------------------------------------------------- masks and heads


def test_prefix_hit_visibility():
    """108 new queries over a 620-key context with table [17, 5, 23]: the
    first sees positions 0..512, the last 0..619."""
    lk, lq, bs = 620, 108, 256
    rng = np.random.default_rng(5)
    d = 4
    x = bits(rng.standard_normal((lk, d)))
    kc, vc = nan_pool(24, bs, 1, d), nan_pool(24, bs, 1, d)
    bt = np.array([[17, 5, 23]], np.int32)
    _store_seq(kc, vc, x, x, bt[0], bs)
    q = x[lk - lq:].reshape(lq, 1, d)
    for i, last in [(0, 512), (lq - 1, 619)]:
        _, w = oracle.prefill(q, [0, lq], [0, lk], 0.5, k_cache=kc, v_cache=vc, block_table=bt,
                              weights_of=(0, 0, i))
        assert (w[: last + 1] > 0).all() and (w[last + 1:] == 0).all()


def test_two_requests_visibility():
    """cu_seqlens_q = [0, 188, 220], cu_seqlens_k = [0, 700, 732]: A's first new
    query (position 512) sees A's 0..512; B's query 0 sees only B's position 0."""
    bs, d = 256, 4
    rng = np.random.default_rng(6)
    kc, vc = nan_pool(24, bs, 1, d), nan_pool(24, bs, 1, d)
    bt = np.array([[17, 5, 23], [11, -1, -1]], np.int32)
    xa, xb = bits(rng.standard_normal((700, d))), bits(rng.standard_normal((32, d)))
    _store_seq(kc, vc, xa, xa, bt[0], bs)
    _store_seq(kc, vc, xb, xb, bt[1], bs)
    q = np.concatenate([xa[512:], xb]).reshape(220, 1, d)
    kw = dict(k_cache=kc, v_cache=vc, block_table=bt)
    _, w = oracle.prefill(q, [0, 188, 220], [0, 700, 732], 0.5, weights_of=(0, 0, 0), **kw)
    assert (w[:513] > 0).all() and (w[513:] == 0).all()
    out, w = oracle.prefill(q, [0, 188, 220], [0, 700, 732], 0.5, weights_of=(1, 0, 0), **kw)
    assert w[0] == 1.0 and (w[1:] == 0).all()
    np.testing.assert_array_equal(out[188, 0], values(xb[0]))


def test_gqa_head_mapping():
    """Q heads of one group share a KV head (Hq=4, Hkv=2: heads 0,1 -> kv 0;
    heads 2,3 -> kv 1).  With V = +1 on kv head 0 and -1 on kv head 1 every
    output is +-1 (up to rounding of the weight sum), whatever the weights."""
    rng = np.random.default_rng(7)
    n, d = 5, 4
    q = bits(rng.standard_normal((n, 4, d)))
    k = bits(rng.standard_normal((n, 2, d)))
    v = bits(np.concatenate([np.ones((n, 1, d)), -np.ones((n, 1, d))], axis=1))
    out = oracle.prefill(q, [0, n], [0, n], 0.3, k=k, v=v)
    np.testing.assert_allclose(out[:, :2], 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:, 2:], -1.0, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- brute force


def _gather_logical(batch, b, kc_bits, vc_bits):
    """Keys 0..ctx-1 of sequence b in logical order, read through the
    generator's own slot bookkeeping."""
    rows = batch.layout.slots(b, np.arange(batch.context_lens[b]))
    kf = kc_bits.reshape(-1, batch.num_kv_heads, batch.head_dim)[rows]
    vf = vc_bits.reshape(-1, batch.num_kv_heads, batch.head_dim)[rows]
    return values(kf), values(vf)


@pytest.mark.parametrize("hq,hkv,bs", [(4, 2, 4), (4, 4, 16), (8, 1, 8), (16, 8, 16)])
def test_oracle_prefill_matches_brute_force(hq, hkv, bs):
    ctx = np.array([5, 17, 1, 33])
    ql = np.array([5, 6, 1, 33])  # a cached prefix on sequence 1
    batch = wl.paged_batch(40 + hq + bs, ctx, ql, bs, num_heads=hq, num_kv_heads=hkv, head_dim=16,
                           num_blocks=40, scale=0.37)
    kc, vc = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    q, k, v = (wl.bf16_bits(t) for t in (batch.tokens.q, batch.tokens.k, batch.tokens.v))
    assert oracle.store_kvcache(k, v, kc, vc, batch.slot_mapping) == oracle.OK
    out = oracle.prefill(q, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.scale, k_cache=kc,
                         v_cache=vc, block_table=batch.block_tables)
    cuq = batch.cu_seqlens_q
    for b in range(len(ctx)):
        kk, vv = _gather_logical(batch, b, kc, vc)
        ref, w = brute_force_attention(values(q[cuq[b]:cuq[b + 1]]), kk, vv, batch.scale)
        np.testing.assert_allclose(out[cuq[b]:cuq[b + 1]], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-12)


@pytest.mark.parametrize("hq,hkv,bs", [(2, 1, 4), (16, 8, 16)])
def test_oracle_decode_matches_brute_force(hq, hkv, bs):
    ctx = np.array([1, 9, 40, 16, 0])
    batch = wl.paged_batch(60 + bs, ctx, np.minimum(ctx, 1), bs, num_heads=hq, num_kv_heads=hkv,
                           head_dim=8, num_blocks=24, table_width=12)
    kc, vc = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    q, k, v = (wl.bf16_bits(t) for t in (batch.tokens.q, batch.tokens.k, batch.tokens.v))
    assert oracle.store_kvcache(k, v, kc, vc, batch.slot_mapping) == oracle.OK
    qd = np.zeros((len(ctx), hq, 8), np.uint16)
    qd[ctx > 0] = q
    out = oracle.decode(qd, kc, vc, batch.block_tables, ctx, batch.scale)
    for b in range(len(ctx)):
        if ctx[b] == 0:
            assert (out[b] == 0).all()
            continue
        kk, vv = _gather_logical(batch, b, kc, vc)
        ref, _ = brute_force_attention(values(qd[b:b + 1]), kk, vv, batch.scale)
        np.testing.assert_allclose(out[b], ref[0], rtol=0, atol=1e-12)


# ----------------------------------------------------------------- invariants


def _store_and_prefill(batch, kc=None, vc=None, tables=None):
    kc = wl.bf16_bits(batch.k_cache).copy() if kc is None else kc
    vc = wl.bf16_bits(batch.v_cache).copy() if vc is None else vc
    q, k, v = (wl.bf16_bits(t) for t in (batch.tokens.q, batch.tokens.k, batch.tokens.v))
    assert oracle.store_kvcache(k, v, kc, vc, batch.slot_mapping) == oracle.OK
    bt = batch.block_tables if tables is None else tables
    return oracle.prefill(q, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.scale, k_cache=kc,
                          v_cache=vc, block_table=bt), kc, vc


def test_block_permutation_invariance():
    """Moving every physical block (data and table entries) leaves the
    outputs bit-identical."""
    batch = wl.paged_batch(71, [30, 50, 7], [10, 50, 7], 8, num_blocks=20, head_dim=16,
                           num_heads=4, num_kv_heads=2)
    out, kc, vc = _store_and_prefill(batch)
    perm = np.random.default_rng(3).permutation(batch.layout.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc  # block i moves to perm[i]
    bt = batch.block_tables
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    q = wl.bf16_bits(batch.tokens.q)
    out2 = oracle.prefill(q, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.scale, k_cache=kc2,
                          v_cache=vc2, block_table=bt2)
    np.testing.assert_array_equal(out, out2)
    ctx = batch.context_lens
    qd = q[batch.cu_seqlens_q[1:] - 1]
    np.testing.assert_array_equal(oracle.decode(qd, kc, vc, bt, ctx, batch.scale),
                                  oracle.decode(qd, kc2, vc2, bt2, ctx, batch.scale))


def test_shared_prefix_equals_private_copy():
    """Sequences whose tables point at the same prefix blocks get the same
    outputs as sequences holding private copies of that prefix."""
    bs, pre = 8, 3
    shared = wl.paged_batch(81, [40, 37], [16, 13], bs, shared_prefix_blocks=pre, head_dim=16,
                            num_heads=4, num_kv_heads=2, num_blocks=16)
    out_shared, kc, vc = _store_and_prefill(shared)
    bt = shared.block_tables.copy()
    used = set(bt[bt >= 0].tolist())
    spare = [i for i in range(shared.layout.num_blocks) if i not in used][:pre]
    bt[1, :pre] = spare
    kc[spare], vc[spare] = kc[bt[0, :pre]], vc[bt[0, :pre]]
    q = wl.bf16_bits(shared.tokens.q)
    out_private = oracle.prefill(q, shared.cu_seqlens_q, shared.cu_seqlens_k, shared.scale,
                                 k_cache=kc, v_cache=vc, block_table=bt)
    np.testing.assert_array_equal(out_shared, out_private)


def test_decode_step_equals_prefill_row():
    """Decoding position t over the cache gives row t of a full causal
    prefill over the same tokens, bit for bit."""
    n = 37
    batch = wl.paged_batch(91, [n], [n], 8, head_dim=16, num_heads=4, num_kv_heads=2, num_blocks=8)
    out, kc, vc = _store_and_prefill(batch)
    q = wl.bf16_bits(batch.tokens.q)
    for t in (0, 1, 8, 17, n - 1):
        dec = oracle.decode(q[t:t + 1], kc, vc, batch.block_tables, [t + 1], batch.scale)
        np.testing.assert_array_equal(dec[0], out[t])


def test_chunked_equals_single_call():
    """A prompt run as two chunks (the second reading the first from the
    cache) gives the same rows as one call over the whole prompt."""
    n, c1 = 45, 19
    whole = wl.paged_batch(95, [n], [n], 8, head_dim=16, num_heads=4, num_kv_heads=2, num_blocks=8)
    out, kc, vc = _store_and_prefill(whole)
    q = wl.bf16_bits(whole.tokens.q)
    bt = whole.block_tables
    kw = dict(k_cache=kc, v_cache=vc, block_table=bt)
    a = oracle.prefill(q[:c1], [0, c1], [0, c1], whole.scale, **kw)
    b = oracle.prefill(q[c1:], [0, n - c1], [0, n], whole.scale, **kw)
    np.testing.assert_array_equal(np.concatenate([a, b]), out)


def test_null_table_equals_paged():
    """Without a cached prefix, reading K/V from the new-token tensors gives the
    same outputs as reading them back from the pool."""
    batch = wl.paged_batch(97, [9, 30, 64], [9, 30, 64], 16, head_dim=16, num_heads=4,
                           num_kv_heads=2, num_blocks=12)
    out, _, _ = _store_and_prefill(batch)
    q, k, v = (wl.bf16_bits(t) for t in (batch.tokens.q, batch.tokens.k, batch.tokens.v))
    out_null = oracle.prefill(q, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.scale, k=k, v=v)
    np.testing.assert_array_equal(out, out_null)


def test_bad_block_id_reported():
    batch = wl.paged_batch(99, [20], [20], 8, head_dim=8, num_heads=2, num_kv_heads=1, num_blocks=4)
    out, kc, vc = _store_and_prefill(batch)
    bt = batch.block_tables.copy()
    bt[0, 1] = 17
    q = wl.bf16_bits(batch.tokens.q)
    with pytest.raises(oracle.OracleError):
        oracle.prefill(q, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.scale, k_cache=kc,
                       v_cache=vc, block_table=bt)
    bt[0, 1] = -1
    with pytest.raises(oracle.OracleError):
        oracle.decode(q[-1:], kc, vc, bt, [20], batch.scale)
