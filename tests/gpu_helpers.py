"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the CPU oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from paged_kv_cache_110_gb300 import workloads as wl

# bf16 attention outputs against the double-precision oracle
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def pa():
    from paged_kv_cache_110_gb300 import binding
    return binding


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def i32(a, device):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=device)


def assert_close(gpu_out: torch.Tensor, ref: np.ndarray, what=""):
    got = gpu_out.double().cpu().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"{what}: max-abs {err.max():.3e} mean-abs {err.mean():.3e}"
    return err


class Status:
    def __init__(self, device):
        self.t = torch.zeros(1, dtype=torch.int32, device=device)

    def value(self):
        torch.cuda.synchronize()
        return int(self.t.item())


def gpu_store(batch, kc, vc, status=None, tokens=None, slots=None):
    d = kc.device
    toks = batch.tokens if tokens is None else tokens
    sl = batch.slot_mapping if slots is None else slots
    pa().pa_store_kvcache(toks.k, toks.v, kc, vc, i32(sl, d), dev_status=None if status is None else status.t)


def oracle_store(batch, kc_bits, vc_bits, tokens=None, slots=None):
    toks = batch.tokens if tokens is None else tokens
    sl = batch.slot_mapping if slots is None else slots
    rc = oracle.store_kvcache(wl.bf16_bits(toks.k), wl.bf16_bits(toks.v), kc_bits, vc_bits, sl)
    assert rc == oracle.OK


def prefill_workspace(num_seqs, max_q, max_k, hq, hkv, device):
    """The caller-owned workspace a prefill call asks for (None if it needs none)."""
    n = pa().pa_prefill_workspace_bytes(num_seqs, int(max_q), int(max_k), hq, hkv)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def gpu_prefill(batch, kc, vc, paged=True, status=None, tokens=None):
    d = kc.device
    toks = batch.tokens if tokens is None else tokens
    out = torch.empty(toks.q.shape, dtype=torch.bfloat16, device=d)
    kw = dict(k_cache=kc, v_cache=vc, block_table=i32(batch.block_tables, d)) if paged else dict(k=toks.k, v=toks.v)
    max_q, max_k = int(batch.query_lens.max()), int(batch.context_lens.max())
    ws = prefill_workspace(len(batch.cu_seqlens_q) - 1, max_q, max_k, toks.q.shape[1], kc.shape[2], d)
    pa().pa_prefill_paged(toks.q, i32(batch.cu_seqlens_q, d), i32(batch.cu_seqlens_k, d), max_q, max_k,
                          batch.scale, out, workspace=ws, dev_status=None if status is None else status.t, **kw)
    return out


def oracle_prefill(batch, kc_bits, vc_bits, seqs=None, tokens=None):
    """Oracle rows of the chosen sequences (all by default), in their order."""
    toks = batch.tokens if tokens is None else tokens
    q = wl.bf16_bits(toks.q)
    cuq, cuk = batch.cu_seqlens_q, batch.cu_seqlens_k
    seqs = range(batch.layout.num_seqs) if seqs is None else seqs
    rows = np.concatenate([np.arange(cuq[b], cuq[b + 1]) for b in seqs])
    ql = np.array([cuq[b + 1] - cuq[b] for b in seqs])
    kl = np.array([cuk[b + 1] - cuk[b] for b in seqs])
    sub_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    sub_k = np.concatenate([[0], np.cumsum(kl)]).astype(np.int32)
    out = oracle.prefill(q[rows], sub_q, sub_k, batch.scale, k_cache=kc_bits, v_cache=vc_bits,
                         block_table=batch.block_tables[list(seqs)])
    return out, rows


def gpu_decode(q, kc, vc, tables, ctx, scale, status=None, max_ctx=None):
    d = kc.device
    b = q.shape[0]
    max_ctx = int(np.max(ctx)) if max_ctx is None else max_ctx
    n = pa().pa_decode_workspace_bytes(b, q.shape[1], q.shape[2], max_ctx)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=d)
    out = torch.full((b, q.shape[1], q.shape[2]), float("nan"), dtype=torch.bfloat16, device=d)
    pa().pa_decode_paged(q, kc, vc, i32(tables, d), i32(ctx, d), max_ctx, scale, out, ws,
                         dev_status=None if status is None else status.t)
    return out


def compact_pool(tables, ctx, seqs, kc, vc, block_size):
    """Host copies of only the blocks the chosen sequences use, with their
    tables renumbered into the compact pool (data movement only)."""
    rows, new_tables = [], []
    nxt = 0
    width = tables.shape[1]
    for b in seqs:
        n = -(-int(ctx[b]) // block_size)
        ids = tables[b, :n]
        rows.append(ids)
        t = np.full(width, -1, np.int32)
        t[:n] = np.arange(nxt, nxt + n)
        nxt += n
        new_tables.append(t)
    ids = torch.as_tensor(np.concatenate(rows).astype(np.int64), device=kc.device)
    return (wl.bf16_bits(kc.index_select(0, ids)).copy(), wl.bf16_bits(vc.index_select(0, ids)).copy(),
            np.array(new_tables))


def grow_keys(batch, growth):
    """Scores that grow along the key positions: every query made |q| and every
    key (the history rows in the pool and the new tokens) set to growth times
    its position, in every head, so that each later chunk of keys scores higher
    than the ones before and the online softmax keeps moving its maximum."""
    lay = batch.layout
    rows, pos = [], []
    for b, (c, n) in enumerate(zip(batch.context_lens, batch.query_lens)):
        h = int(c) - int(n)
        rows.append(lay.slots(b, np.arange(h)))
        pos.append(np.arange(h))
    rows, pos = np.concatenate(rows), np.concatenate(pos)
    d = batch.k_cache.device
    kv = batch.k_cache.view(-1, batch.k_cache.shape[2], batch.k_cache.shape[3])
    val = (growth * torch.as_tensor(pos, dtype=torch.float32, device=d))[:, None, None]
    kv[torch.as_tensor(rows, device=d)] = val.expand(-1, kv.shape[1], kv.shape[2]).to(torch.bfloat16)
    new_pos = torch.as_tensor(batch.positions, dtype=torch.float32, device=d)
    batch.tokens.k.copy_((growth * new_pos)[:, None, None].expand_as(batch.tokens.k).to(torch.bfloat16))
    batch.tokens.q.copy_(batch.tokens.q.abs())
