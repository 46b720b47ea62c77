"""A whole decode step of the attention path captured in one CUDA graph and
replayed with new inputs written in place, bit-identical to the same calls
run eagerly; and mixed batches (decode rows and prefill chunks) in one
prefill launch, against the oracle.  Through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (MAX_ABS, MEAN_ABS, Status, assert_close, dev, i32, oracle_prefill, oracle_store, pa,
                         prefill_workspace)
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


class DecodeAttentionStep:
    """One decode step of the attention path for `layers` layers: device-built
    metadata from seq_lens, then per layer the fused head norm + RoPE + KV write
    of each sequence's new token and the paged decode.  All buffers are fixed;
    a step's inputs (seq_lens, the new tokens' qkv) are written in place."""

    def __init__(self, seed, layers, num_seqs, padding, max_len, block_size):
        d = dev()
        self.d, self.layers, self.B, self.max_len, self.bs = d, layers, num_seqs, max_len, block_size
        r = wl.rng(seed)
        lens = r.integers(100, max_len - 8, num_seqs, endpoint=True).astype(np.int32)
        lens[num_seqs - padding:] = 0                      # spare batch entries
        self.lens0 = lens
        layout = wl.make_layout(seed, np.full(num_seqs, max_len), block_size)
        self.nb = layout.num_blocks
        self.tables = torch.as_tensor(layout.block_tables, device=d)
        self.pools = []
        for l in range(layers):
            kc, vc = wl.make_pool(layout, np.maximum(lens - 1, 0), seed + 100 + l, device=d)
            self.pools.append((kc, vc))
        self.seq_lens = torch.as_tensor(lens, device=d)
        self.qkv = [torch.zeros((num_seqs, (wl.HQ + 2 * wl.HKV) * 128), dtype=torch.bfloat16, device=d)
                    for _ in range(layers)]
        self.q_rot = [torch.empty((num_seqs, wl.HQ, 128), dtype=torch.bfloat16, device=d) for _ in range(layers)]
        self.out = [torch.empty((num_seqs, wl.HQ, 128), dtype=torch.bfloat16, device=d) for _ in range(layers)]
        self.cs = pa().pa_rope_cos_sin_table(wl.ROPE_BASE, 128, max_len, device=d)
        self.qw, self.kw = wl.norm_weights(seed + 7, device=d)
        self.ws = torch.empty(max(pa().pa_decode_workspace_bytes(num_seqs, wl.HQ, 128, max_len), 256),
                              dtype=torch.uint8, device=d)

    def run(self):
        p = pa()
        pos, ctx, slots = p.pa_prepare_decode(self.seq_lens, self.tables, self.bs, self.nb)
        for l in range(self.layers):
            kc, vc = self.pools[l]
            p.pa_norm_rope_store_kvcache(self.qkv[l], wl.HQ, wl.HKV, pos, self.cs, self.qw, self.kw, wl.RMS_EPS,
                                         self.q_rot[l], kc, vc, slots)
            p.pa_decode_paged(self.q_rot[l], kc, vc, self.tables, ctx, self.max_len, wl.SCALE, self.out[l], self.ws)

    def set_inputs(self, step):
        """Inputs of step `step` (0, 1, ...): every live sequence grows by one."""
        lens = np.where(self.lens0 > 0, self.lens0 + step, 0).astype(np.int32)
        self.seq_lens.copy_(torch.as_tensor(lens))
        g = torch.Generator(device=self.d).manual_seed(1000 + step)
        for t in self.qkv:
            t.copy_(torch.randn(t.shape, generator=g, device=self.d).to(torch.bfloat16))


@pytest.mark.parametrize("block_size", [256, 16])
def test_graph_replay_equals_eager(block_size):
    eager = DecodeAttentionStep(wl.SEED_BASE + 70, layers=3, num_seqs=64, padding=8, max_len=2048,
                                block_size=block_size)
    graphed = DecodeAttentionStep(wl.SEED_BASE + 70, layers=3, num_seqs=64, padding=8, max_len=2048,
                                  block_size=block_size)
    graphed.set_inputs(0)
    graphed.run()  # first calls outside the capture (library set-up); the state is reset below
    graphed2 = DecodeAttentionStep(wl.SEED_BASE + 70, layers=3, num_seqs=64, padding=8, max_len=2048,
                                   block_size=block_size)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            graphed2.run()
    torch.cuda.current_stream().wait_stream(side)
    for step in range(3):
        eager.set_inputs(step)
        graphed2.set_inputs(step)
        eager.run()
        graph.replay()
        torch.cuda.synchronize()
        for l in range(3):
            assert torch.equal(eager.out[l].view(torch.int16), graphed2.out[l].view(torch.int16)), (step, l)
            for a, b in zip(eager.pools[l], graphed2.pools[l]):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (step, l)
    # padded rows decode to zeros
    assert (eager.out[0][-8:].float() == 0).all()


def test_graph_step_matches_oracle_on_one_layer():
    s = DecodeAttentionStep(wl.SEED_BASE + 71, layers=1, num_seqs=24, padding=3, max_len=1024, block_size=256)
    kc0, vc0 = (wl.bf16_bits(t).copy() for t in s.pools[0])
    s.set_inputs(0)
    s.run()
    torch.cuda.synchronize()
    lens = s.lens0
    meta, rc = oracle.prepare_decode(lens, s.tables.cpu().numpy(), 256, s.nb)
    assert rc == oracle.OK
    qkv = wl.bf16_bits(s.qkv[0])
    cs = oracle.rope_cos_sin(wl.ROPE_BASE, 128, 1024)
    q_rot, rc = oracle.norm_rope_store(qkv, wl.HQ, wl.HKV, meta["positions"], cs, wl.bf16_bits(s.qw),
                                       wl.bf16_bits(s.kw), wl.RMS_EPS, kc0, vc0, meta["slot_mapping"])
    assert rc == oracle.OK
    ref = oracle.decode(q_rot, kc0, vc0, s.tables.cpu().numpy(), meta["context_lens"], wl.SCALE)
    assert_close(s.out[0], ref, "graph step, layer 0")


def test_mixed_decode_rows_and_prefill_chunks_in_one_launch():
    # three decode rows (one query over a long context) and two prefill chunks over a cached prefix
    ctx = np.array([1500, 3000, 777, 900, 2300])
    ql = np.array([1, 1, 1, 300, 130])
    batch = wl.paged_batch(wl.SEED_BASE + 72, ctx, ql, 256, device=dev())
    kc, vc = batch.k_cache, batch.v_cache
    kc_bits, vc_bits = wl.bf16_bits(kc).copy(), wl.bf16_bits(vc).copy()  # the generator's pool, before any write
    d = dev()
    pa().pa_store_kvcache(batch.tokens.k, batch.tokens.v, kc, vc, i32(batch.slot_mapping, d))
    out = torch.empty(batch.tokens.q.shape, dtype=torch.bfloat16, device=d)
    st = Status(d)
    ws = prefill_workspace(len(ctx), int(ql.max()), int(ctx.max()), 16, 8, d)
    pa().pa_prefill_paged(batch.tokens.q, i32(batch.cu_seqlens_q, d), i32(batch.cu_seqlens_k, d), int(ql.max()),
                          int(ctx.max()), batch.scale, out, k_cache=kc, v_cache=vc,
                          block_table=i32(batch.block_tables, d), workspace=ws, dev_status=st.t)
    torch.cuda.synchronize()
    assert int(st.t.item()) == 0
    oracle_store(batch, kc_bits, vc_bits)
    ref, rows = oracle_prefill(batch, kc_bits, vc_bits)
    assert_close(out[rows], ref, "mixed batch")
    # the decode rows equal the decode kernel's answer for the same sequences within the tolerance
    dq = batch.tokens.q[batch.cu_seqlens_q[:3]]
    ws = torch.empty(max(pa().pa_decode_workspace_bytes(3, 16, 128, 3000), 256), dtype=torch.uint8, device=d)
    dout = torch.empty((3, 16, 128), dtype=torch.bfloat16, device=d)
    pa().pa_decode_paged(dq, kc, vc, i32(batch.block_tables[:3], d), i32(ctx[:3], d), 3000, batch.scale, dout, ws)
    torch.cuda.synchronize()
    err = (dout.float() - out[batch.cu_seqlens_q[:3]].float()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
