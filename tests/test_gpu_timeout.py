"""Bounded waits that run out, made to do so on purpose (pa_test_stall_pipelines).

The hook makes one wait of every CTA of the prefill and of the fused norm +
RoPE + KV write wait on a barrier that nothing arrives on, with a short limit
(2^20 SM cycles, about half a millisecond).  The call must then write
PA_ERR_TIMEOUT to its status word, wait for what it issued (those drain waits
keep the default limit), free its tensor memory and return, leaving the
context usable.  With the default limit back, the next
call on the same stream must give the right answer: the prefill is compared
with the oracle, the fused write with the same call made before the timeout.

Nothing here faults, traps or hangs a GPU: every wait is bounded, and the
failure is a status code the host reads.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import Status, assert_close, dev, gpu_prefill, gpu_store, i32, oracle_prefill, oracle_store, pa
from paged_kv_cache_110_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SHORT = 1 << 20  # SM cycles


@pytest.fixture(autouse=True)
def _default_limit_after():
    yield
    pa().pa_test_stall_pipelines(0)


def test_prefill_wait_runs_out_then_next_call_matches_oracle():
    d = dev()
    # cached prefixes and several query tiles per sequence: every role of the kernel has waits to run out
    batch = wl.paged_batch(wl.SEED_BASE + 95, [300, 700, 129, 1000], [300, 200, 129, 500], 64, device=d)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    st = Status(d)
    gpu_store(batch, kc, vc, st)
    assert st.value() == 0
    pa().pa_test_stall_pipelines(SHORT)
    gpu_prefill(batch, kc, vc, status=st)
    assert st.value() == pa().PA_ERR_TIMEOUT
    pa().pa_test_stall_pipelines(0)
    st2 = Status(d)
    out = gpu_prefill(batch, kc, vc, status=st2)
    assert st2.value() == 0
    kb, vb = wl.bf16_bits(batch.k_cache).copy(), wl.bf16_bits(batch.v_cache).copy()
    oracle_store(batch, kb, vb)
    ref, rows = oracle_prefill(batch, kb, vb)
    assert_close(out[torch.as_tensor(rows, device=d)], ref, "prefill after a timed-out call")


def test_norm_rope_store_wait_runs_out_then_next_call_is_unchanged():
    d = dev()
    lens = np.array([200, 300, 150])
    batch = wl.paged_batch(wl.SEED_BASE + 96, lens, lens, 16, device=d)
    cs = pa().pa_rope_cos_sin_table(wl.ROPE_BASE, 128, 4096, device=d)
    qw, kw = wl.norm_weights(21, device=d)
    pos, slots = i32(batch.positions, d), i32(batch.slot_mapping, d)

    def call(status):
        q_out = torch.full((batch.tokens.qkv.shape[0], 16, 128), float("nan"), dtype=torch.bfloat16, device=d)
        kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
        pa().pa_norm_rope_store_kvcache(batch.tokens.qkv, 16, 8, pos, cs, qw, kw, wl.RMS_EPS, q_out, kc, vc, slots,
                                        dev_status=status.t)
        return q_out, kc, vc

    st0 = Status(d)
    before = call(st0)
    assert st0.value() == 0
    pa().pa_test_stall_pipelines(SHORT)
    st1 = Status(d)
    call(st1)
    assert st1.value() == pa().PA_ERR_TIMEOUT
    pa().pa_test_stall_pipelines(0)
    st2 = Status(d)
    after = call(st2)
    assert st2.value() == 0
    for x, y in zip(before, after):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
