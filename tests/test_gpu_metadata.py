"""Device-built step metadata against the oracle (bit-exact: integer work).

Through the C ABI.  Cases: the pages' worked batches, random batches with
cached prefixes and chunked prompts over fragmented tables (the varlen-prefill
and decode-batch workload shapes), CUDA-graph padding rows, bad table entries
and an output capacity that is too small."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import Status, dev, i32, pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gpu_prefill(lens, cached, sched, table, bs, nb, max_tokens=None, status=None):
    d = dev()
    t = int(np.sum(sched)) if max_tokens is None else max_tokens
    cu_q, cu_k, pos, sl, mx = pa().pa_prepare_prefill(i32(lens, d), i32(cached, d), i32(sched, d), i32(table, d), bs,
                                                      nb, t, dev_status=None if status is None else status.t)
    torch.cuda.synchronize()
    return {"cu_seqlens_q": cu_q.cpu().numpy(), "cu_seqlens_k": cu_k.cpu().numpy(), "positions": pos.cpu().numpy(),
            "slot_mapping": sl.cpu().numpy(), "max_seqlen_q": int(mx[0]), "max_seqlen_k": int(mx[1])}


def _same(got, ref):
    for k, v in ref.items():
        np.testing.assert_array_equal(np.asarray(got[k]), np.asarray(v), err_msg=k)


@pytest.mark.parametrize("case", ["prefill_two_prompts", "prefill_prefix_hit_round_two"])
def test_printed_prefill_batches(golden, case):
    g = golden("step_metadata_examples.json")[case]
    ref, rc = oracle.prepare_prefill(g["seq_lens"], g["num_cached"], g["num_scheduled"], g["block_table"],
                                     g["block_size"], 64)
    assert rc == oracle.OK
    _same(_gpu_prefill(g["seq_lens"], g["num_cached"], g["num_scheduled"], g["block_table"], g["block_size"], 64), ref)


@pytest.mark.parametrize("case", ["decode_two_prompts", "decode_round_three"])
def test_printed_decode_batches(golden, case):
    g = golden("step_metadata_examples.json")[case]
    d = dev()
    pos, ctx, sl = pa().pa_prepare_decode(i32(g["seq_lens"], d), i32(g["block_table"], d), g["block_size"], 64)
    for k, v in (("positions", pos), ("context_lens", ctx), ("slot_mapping", sl)):
        np.testing.assert_array_equal(v.cpu().numpy(), g[k])


def _random_prefill_batch(seed, b, bs, max_len, chunk_first=True):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len, b, endpoint=True)
    cached = (rng.integers(0, 4, b) * bs * rng.integers(0, 2, b))        # whole cached blocks, half the seqs
    cached = np.minimum(cached, lens)
    start = np.minimum(cached, lens - 1)
    sched = lens - start
    if chunk_first:                                                      # only the first sequence is chunked
        sched[0] = max(1, sched[0] // 2)
    width = int(-(-lens.max() // bs))
    table = np.full((b, width + 2), -1, np.int32)
    perm = rng.permutation(b * width).astype(np.int32)
    for i in range(b):
        n = int(-(-lens[i] // bs))
        table[i, :n] = perm[i * width:i * width + n]
    return lens, cached, sched, table, b * width


@pytest.mark.parametrize("bs", [16, 256])
def test_random_prefill_batches(bs):
    for seed, b in ((1, 30), (2, 1), (3, 600), (4, 2100)):  # 2100 > one scan chunk of 1024
        lens, cached, sched, table, nb = _random_prefill_batch(seed, b, bs, 1024)
        ref, rc = oracle.prepare_prefill(lens, cached, sched, table, bs, nb)
        assert rc == oracle.OK
        st = Status(dev())
        _same(_gpu_prefill(lens, cached, sched, table, bs, nb, status=st), ref)
        assert int(st.t.item()) == 0


def test_random_decode_batch_with_graph_padding():
    rng = np.random.default_rng(9)
    b, bs = 512, 256
    lens = rng.integers(1024, 4096, b, endpoint=True).astype(np.int32)
    lens[-37:] = 0                       # spare entries of a captured batch size
    width = 16
    table = rng.permutation(b * width).astype(np.int32).reshape(b, width)
    ref, rc = oracle.prepare_decode(lens, table, bs, b * width)
    assert rc == oracle.OK
    d = dev()
    st = Status(d)
    pos, ctx, sl = pa().pa_prepare_decode(i32(lens, d), i32(table, d), bs, b * width, dev_status=st.t)
    np.testing.assert_array_equal(pos.cpu().numpy(), ref["positions"])
    np.testing.assert_array_equal(ctx.cpu().numpy(), ref["context_lens"])
    np.testing.assert_array_equal(sl.cpu().numpy(), ref["slot_mapping"])
    assert int(st.t.item()) == 0


def test_bad_entries_and_capacity_reported():
    d = dev()
    st = Status(d)
    # a -1 inside the live range: slot -1 and PA_ERR_BOUNDS, the same as the oracle
    ref, rc = oracle.prepare_prefill([40], [0], [40], [[2, -1, 3]], 16, 4)
    got = _gpu_prefill([40], [0], [40], [[2, -1, 3]], 16, 4, status=st)
    assert rc == oracle.BOUNDS and int(st.t.item()) == pa().PA_ERR_BOUNDS
    _same(got, ref)
    # capacity one token short: the last token is not written, the status says so
    st = Status(d)
    got = _gpu_prefill([10, 7], [0, 0], [10, 7], [[0], [1]], 16, 4, max_tokens=16, status=st)
    assert int(st.t.item()) == pa().PA_ERR_BOUNDS
    ref, _ = oracle.prepare_prefill([10, 7], [0, 0], [10, 7], [[0], [1]], 16, 4)
    np.testing.assert_array_equal(got["slot_mapping"], ref["slot_mapping"][:16])
    # scheduled past the end of the prompt
    st = Status(d)
    _gpu_prefill([20], [10], [11], [[2, 3]], 16, 4, max_tokens=11, status=st)
    assert int(st.t.item()) == pa().PA_ERR_INVALID_ARG
