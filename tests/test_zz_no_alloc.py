"""pa_decode_paged_noalloc: paged decode for callers that cannot allocate
device memory (code inside a framework that owns the device memory pool,
services that must not allocate while serving, C callers without a memory
manager).  Its scratch is a fixed device array inside the library, so it
takes no workspace.

Checked through the C ABI against pa_decode_paged (which takes a caller
workspace) on two calls in a row with different inputs: both run the same
plan and kernels, so the outputs must be identical bit for bit.  The second
batch (mixed lengths, partly single-split, partly multi-split) is also
compared with the CPU oracle within the attention tolerance the other GPU
tests use; and sizes beyond the fixed scratch are refused without a launch.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
SCRATCH_BYTES = 32 << 20  # PA_DECODE_NOALLOC_SCRATCH_BYTES in include/pa.h


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_110_gb300 import binding
    torch.cuda.set_device(0)
    return binding


def _decode_both(pa, batch):
    d = batch.k_cache.device
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    slots = torch.as_tensor(batch.slot_mapping, device=d)
    pa.pa_store_kvcache(batch.tokens.k, batch.tokens.v, kc, vc, slots)
    tables = torch.as_tensor(batch.block_tables, device=d)
    ctx = torch.as_tensor(batch.context_lens, device=d)
    max_ctx = int(batch.context_lens.max())
    b = batch.layout.num_seqs
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(b, 16, 128, max_ctx), 256), dtype=torch.uint8, device=d)
    ref = torch.empty((b, 16, 128), dtype=torch.bfloat16, device=d)
    pa.pa_decode_paged(batch.tokens.q, kc, vc, tables, ctx, max_ctx, batch.scale, ref, ws)
    got = torch.full_like(ref, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=d)
    pa.pa_decode_paged_noalloc(batch.tokens.q, kc, vc, tables, ctx, max_ctx, batch.scale, got, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return got, ref


def test_noalloc_matches_workspace_decode_on_two_calls(pa):
    d = torch.device("cuda:0")
    first = wl.decode_batch(device=d, num_seqs=128, seed=wl.SEED_BASE + 40)
    second = wl.paged_batch(wl.SEED_BASE + 41, np.array([5, 300, 1024, 2000, 17, 640]), np.ones(6, int), 16,
                            device=d)
    for batch in (first, second):
        got, ref = _decode_both(pa, batch)
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    # the second call against the oracle (history rows plus the new token
    # written by the oracle's own KV write)
    kb, vb = wl.bf16_bits(second.k_cache).copy(), wl.bf16_bits(second.v_cache).copy()
    rc = oracle.store_kvcache(wl.bf16_bits(second.tokens.k), wl.bf16_bits(second.tokens.v), kb, vb,
                              second.slot_mapping)
    assert rc == oracle.OK
    want = oracle.decode(wl.bf16_bits(second.tokens.q), kb, vb, second.block_tables, second.context_lens,
                         second.scale)
    err = np.abs(got.double().cpu().numpy() - want)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_noalloc_refuses_sizes_beyond_its_scratch(pa):
    d = torch.device("cuda:0")
    pick = None
    for b in (1024, 2048, 3000, 4000):
        if pa.pa_decode_workspace_bytes(b, 16, 128, 4096) > SCRATCH_BYTES:
            pick = b
            break
    assert pick is not None, "no test size exceeds the fixed scratch"
    q = torch.zeros((pick, 16, 128), dtype=torch.bfloat16, device=d)
    kc = torch.zeros((16, 256, 8, 128), dtype=torch.bfloat16, device=d)
    tables = torch.zeros((pick, 16), dtype=torch.int32, device=d)
    ctx = torch.zeros(pick, dtype=torch.int32, device=d)
    out = torch.empty_like(q)
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_paged_noalloc(q, kc, kc, tables, ctx, 4096, 0.1, out)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
