"""Pins of the oracle's step-metadata builder against the batches the pages
work through.  None of these tests touch the CUDA library."""
import numpy as np
import pytest

import oracle


def _ranges(rs):
    return np.concatenate([np.arange(a, b) for a, b in rs]).astype(np.int32)


@pytest.mark.parametrize("case", ["prefill_two_prompts", "prefill_prefix_hit_round_two"])
def test_prefill_metadata_printed(golden, case):
    g = golden("step_metadata_examples.json")[case]
    m, rc = oracle.prepare_prefill(g["seq_lens"], g["num_cached"], g["num_scheduled"], g["block_table"],
                                   g["block_size"], 64)
    assert rc == oracle.OK
    np.testing.assert_array_equal(m["positions"], _ranges(g["positions"]))
    np.testing.assert_array_equal(m["cu_seqlens_q"], g["cu_seqlens_q"])
    np.testing.assert_array_equal(m["cu_seqlens_k"], g["cu_seqlens_k"])
    assert (m["max_seqlen_q"], m["max_seqlen_k"]) == (g["max_seqlen_q"], g["max_seqlen_k"])
    np.testing.assert_array_equal(m["slot_mapping"], _ranges(g["slot_ranges"]))


@pytest.mark.parametrize("case", ["decode_two_prompts", "decode_round_three"])
def test_decode_metadata_printed(golden, case):
    g = golden("step_metadata_examples.json")[case]
    m, rc = oracle.prepare_decode(g["seq_lens"], g["block_table"], g["block_size"], 64)
    assert rc == oracle.OK
    for k in ("positions", "context_lens", "slot_mapping"):
        np.testing.assert_array_equal(m[k], g[k])


def test_lifecycle_prefill_then_decode(golden):
    g = golden("step_metadata_examples.json")["lifecycle_prefill_then_decode"]
    lens = g["prefill_seq_lens"]
    table = [[0], [1]]
    m, rc = oracle.prepare_prefill(lens, [0, 0], lens, table, 256, 4)
    assert rc == oracle.OK
    np.testing.assert_array_equal(m["cu_seqlens_q"], g["cu_seqlens"])
    np.testing.assert_array_equal(m["cu_seqlens_k"], g["cu_seqlens"])
    d, rc = oracle.prepare_decode(g["decode_seq_lens"], table, 256, 4)
    np.testing.assert_array_equal(d["positions"], g["positions"])
    np.testing.assert_array_equal(d["context_lens"], g["context_lens"])


def test_prefix_hit_lengths(golden):
    g = golden("step_metadata_examples.json")["prefix_hit_108_over_620"]
    m, rc = oracle.prepare_prefill([g["seq_len"]], [g["num_cached"]], [g["num_scheduled"]], [[3, 1, 2]], 256, 4)
    assert rc == oracle.OK
    np.testing.assert_array_equal(m["cu_seqlens_q"], g["cu_seqlens_q"])
    np.testing.assert_array_equal(m["cu_seqlens_k"], g["cu_seqlens_k"])
    np.testing.assert_array_equal(m["positions"], np.arange(512, 620))


def test_block_crossing_decode(golden):
    g = golden("step_metadata_examples.json")["block_crossing_decode"]
    p0, p1 = 7, 3
    d, rc = oracle.prepare_decode(g["seq_lens"], [[p0, p1], [p0, p1]], g["block_size"], 8)
    assert rc == oracle.OK
    np.testing.assert_array_equal(d["slot_mapping"], [p1 * 256 + o for o in g["slot_offsets_in_second_block"]])


def test_fully_cached_prompt_recomputes_its_last_token():
    # start = min(num_cached, seqlen - 1): a prompt whose every token is cached still computes the last one
    m, rc = oracle.prepare_prefill([300], [300], [1], [[4, 9]], 256, 16)
    assert rc == oracle.OK
    np.testing.assert_array_equal(m["positions"], [299])
    np.testing.assert_array_equal(m["slot_mapping"], [9 * 256 + 43])
    assert list(m["cu_seqlens_k"]) == [0, 300]


def test_chunk_keys_end_at_the_chunk():
    # a first chunk of 100 of a 300-token prompt: its queries are positions 0..99 and read keys 0..99
    m, rc = oracle.prepare_prefill([300], [0], [100], [[4, 9]], 256, 16)
    assert rc == oracle.OK
    assert list(m["cu_seqlens_k"]) == [0, 100] and m["max_seqlen_k"] == 100
    # its second chunk reads 300 keys
    m, rc = oracle.prepare_prefill([300], [100], [200], [[4, 9]], 256, 16)
    assert list(m["cu_seqlens_q"]) == [0, 200] and list(m["cu_seqlens_k"]) == [0, 300]
    np.testing.assert_array_equal(m["slot_mapping"], np.r_[4 * 256 + np.arange(100, 256), 9 * 256 + np.arange(0, 44)])


def test_metadata_matches_the_slot_rule_on_random_batches():
    # every token's slot equals table[pos // bs] * bs + pos % bs (the pinned slot rule), for fragmented tables
    rng = np.random.default_rng(4)
    for bs in (16, 64, 256):
        b = 9
        lens = rng.integers(1, 900, b)
        cached = np.minimum(rng.integers(0, 900, b), lens)
        start = np.minimum(cached, lens - 1)
        sched = np.array([rng.integers(1, lens[i] - start[i] + 1) for i in range(b)])
        width = int(-(-lens.max() // bs))
        perm = rng.permutation(b * width).astype(np.int32).reshape(b, width)
        m, rc = oracle.prepare_prefill(lens, cached, sched, perm, bs, b * width)
        assert rc == oracle.OK
        k = 0
        for i in range(b):
            for p in range(start[i], start[i] + sched[i]):
                assert m["positions"][k] == p
                assert m["slot_mapping"][k] == oracle.slot(perm[i], bs, p)
                k += 1


def test_padding_and_bad_entries_reported():
    d, rc = oracle.prepare_decode([0, 5], [[1], [-1]], 16, 4)
    assert rc == oracle.BOUNDS
    assert list(d["context_lens"]) == [0, 5] and list(d["slot_mapping"]) == [-1, -1] and d["positions"][0] == 0
    m, rc = oracle.prepare_prefill([20], [0], [20], [[2, -1]], 16, 4)
    assert rc == oracle.BOUNDS and (m["slot_mapping"][16:] == -1).all() and (m["slot_mapping"][:16] >= 0).all()
    _, rc = oracle.prepare_prefill([20], [10], [11], [[2, 3]], 16, 4)  # scheduled past the end of the prompt
    assert rc == oracle.INVALID
