"""Python binding of libpa's C ABI (``include/pa.h``).

Argument marshalling only: each function checks dtypes / devices, reads data
pointers, strides and sizes from torch tensors, and calls the C entry point
of the same name on the current CUDA stream.  All computation happens in the
library's CUDA kernels; there is no fallback.  If ``libpa.so`` has not been
built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "PaError", "lib", "pa_status_string", "pa_abi_version", "pa_kv_bytes_per_token",
    "pa_store_kvcache", "pa_store_kvcache_fp8", "pa_norm_rope_store_kvcache", "pa_rope_cos_sin_table",
    "pa_prepare_prefill", "pa_prepare_decode", "pa_prefill_workspace_bytes", "pa_prefill_paged",
    "pa_decode_workspace_bytes", "pa_decode_paged", "pa_store_decode_paged", "pa_decode_paged_fp8",
    "pa_decode_paged_noalloc", "pa_test_stall_pipelines", "pa_norm_rope_store_decode_paged",
]

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_BOUNDS, PA_ERR_TIMEOUT = range(6)


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {pa_status_string(status)} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(_build.LIB_PATH):
        raise ImportError(f"libpa.so is not built ({_build.LIB_PATH}); run __graft_entry__.build() "
                          "or python -m paged_kv_cache_110_gb300._build")
    L = ctypes.CDLL(_build.LIB_PATH)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_status_string.argtypes = [i32]
    L.pa_abi_version.restype = i32
    L.pa_abi_version.argtypes = []
    L.pa_kv_bytes_per_token.restype = sz
    L.pa_kv_bytes_per_token.argtypes = [i32, i32, i32, i32]
    L.pa_store_kvcache.restype = i32
    L.pa_store_kvcache.argtypes = [vp, i64, vp, i64, i64, i32, i32, vp, vp, i64, i32, vp, vp, vp]
    L.pa_store_kvcache_fp8.restype = i32
    L.pa_store_kvcache_fp8.argtypes = [vp, i64, vp, i64, i64, i32, i32, f32, f32, vp, vp, i64, i32, vp, vp, vp]
    L.pa_decode_paged_fp8.restype = i32
    L.pa_decode_paged_fp8.argtypes = [vp, i64, vp, vp, f32, f32, i64, i32, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                      vp, vp, sz, vp, vp]
    L.pa_prepare_prefill.restype = i32
    L.pa_prepare_prefill.argtypes = [vp, vp, vp, i32, vp, i32, i32, i64, vp, vp, vp, vp, i64, vp, vp, vp]
    L.pa_prepare_decode.restype = i32
    L.pa_prepare_decode.argtypes = [vp, i32, vp, i32, i32, i64, vp, vp, vp, vp, vp]
    L.pa_rope_cos_sin_table.restype = i32
    L.pa_rope_cos_sin_table.argtypes = [ctypes.c_double, i32, i64, vp, vp]
    L.pa_norm_rope_store_kvcache.restype = i32
    L.pa_norm_rope_store_kvcache.argtypes = [vp, i64, i64, i32, i32, i32, vp, vp, i64, vp, vp, f32, vp, i64, vp, vp,
                                             i64, i32, vp, vp, vp]
    L.pa_prefill_paged.restype = i32
    L.pa_prefill_paged.argtypes = [vp, i64, i64, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp, vp, i32, i32, i32,
                                   i32, i32, i32, f32, vp, vp, sz, vp, vp]
    L.pa_prefill_workspace_bytes.restype = sz
    L.pa_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.pa_decode_workspace_bytes.restype = sz
    L.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.pa_decode_paged.restype = i32
    L.pa_decode_paged.argtypes = [vp, i64, vp, vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, i32, f32, vp,
                                  vp, sz, vp, vp]
    L.pa_store_decode_paged.restype = i32
    L.pa_store_decode_paged.argtypes = [vp, i64, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                        f32, vp, vp, sz, vp, vp]
    L.pa_norm_rope_store_decode_paged.restype = i32
    L.pa_norm_rope_store_decode_paged.argtypes = [vp, i64, vp, i64, vp, vp, f32, vp, vp, i64, i32, vp, i32, vp, i32,
                                                  i32, i32, i32, i32, f32, vp, vp, sz, vp, vp]
    L.pa_test_stall_pipelines.restype = None
    L.pa_test_stall_pipelines.argtypes = [ctypes.c_longlong]
    L.pa_decode_paged_noalloc.restype = i32
    L.pa_decode_paged_noalloc.argtypes = [vp, i64, vp, vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                          vp, vp, vp]
    return L


lib = _load()


def pa_status_string(status: int) -> str:
    return lib.pa_status_string(int(status)).decode()


def pa_abi_version() -> int:
    return lib.pa_abi_version()


def pa_kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return lib.pa_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def pa_test_stall_pipelines(cycles: int) -> None:
    """Test hook: later prefill and fused norm + RoPE + KV write calls stall on
    a barrier nothing arrives on and give up after `cycles` SM cycles
    (PA_ERR_TIMEOUT); 0 restores normal operation."""
    lib.pa_test_stall_pipelines(int(cycles))


# ---------------------------------------------------------------- marshalling helpers


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16_rows(t: torch.Tensor, name: str):
    """[N, H, 128] bf16 CUDA tensor with packed heads -> (H, row stride in elements)."""
    if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA bf16 [N, H, D] tensor, got {t.dtype} {tuple(t.shape)} {t.device}")
    if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name}: heads and dims must be packed (strides {t.stride()})")
    return t.shape[1], t.stride(0)


def _cache(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA bf16 [num_blocks, block_size, Hkv, D] tensor")
    return t.shape


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA int32 tensor")
    return t


def _check(status: int, what: str):
    if status != PA_OK:
        raise PaError(status, what)


# ---------------------------------------------------------------- the C entry points


def pa_store_kvcache(k, v, k_cache, v_cache, slot_mapping, dev_status=None, stream=None):
    """KV write: k/v [T, Hkv, 128] bf16 (token stride free), caches
    [NB, bs, Hkv, 128], slot_mapping [T] int32 (-1 skips)."""
    hkv, ks = _bf16_rows(k, "k")
    _, vs = _bf16_rows(v, "v")
    nb, bs, chk, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(slot_mapping, "slot_mapping")
    if slot_mapping.numel() != k.shape[0] or v.shape[0] != k.shape[0] or chk != hkv:
        raise ValueError("pa_store_kvcache: inconsistent shapes")
    _check(lib.pa_store_kvcache(_ptr(k), ks, _ptr(v), vs, k.shape[0], hkv, k.shape[2], _ptr(k_cache),
                                _ptr(v_cache), nb, bs, _ptr(slot_mapping), _ptr(dev_status), _stream(stream)),
           "pa_store_kvcache")


def _cache8(t: torch.Tensor, name: str):
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != 4 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA uint8 / float8_e4m3fn [num_blocks, block_size, Hkv, D]")
    return t.shape


def pa_store_kvcache_fp8(k, v, k_scale, v_scale, k_cache, v_cache, slot_mapping, dev_status=None, stream=None):
    """KV write into E4M3 pools: k, v [T, Hkv, 128] bf16 views; caches uint8 [NB, bs, Hkv, 128]."""
    hkv, ks = _bf16_rows(k, "k")
    _, vs = _bf16_rows(v, "v")
    nb, bs, chk, _ = _cache8(k_cache, "k_cache")
    _cache8(v_cache, "v_cache")
    _i32(slot_mapping, "slot_mapping")
    if slot_mapping.numel() != k.shape[0] or v.shape[0] != k.shape[0] or chk != hkv:
        raise ValueError("pa_store_kvcache_fp8: inconsistent shapes")
    _check(lib.pa_store_kvcache_fp8(_ptr(k), ks, _ptr(v), vs, k.shape[0], hkv, k.shape[2], float(k_scale),
                                    float(v_scale), _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(slot_mapping),
                                    _ptr(dev_status), _stream(stream)),
           "pa_store_kvcache_fp8")


def pa_decode_paged_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, max_context_len, scale, out,
                        workspace, dev_status=None, stream=None):
    """Paged decode over E4M3 pools (see pa_decode_paged for the other arguments)."""
    hq, qs = _bf16_rows(q, "q")
    nb, bs, hkv, d = _cache8(k_cache, "k_cache")
    _cache8(v_cache, "v_cache")
    _i32(block_table, "block_table")
    _i32(context_lens, "context_lens")
    b = q.shape[0]
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (b, hq, d):
        raise ValueError("out must be a contiguous bf16 [B, Hq, D] tensor")
    _check(lib.pa_decode_paged_fp8(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale), nb,
                                   bs, _ptr(block_table), block_table.shape[1], _ptr(context_lens), b,
                                   int(max_context_len), hq, hkv, d, float(scale), _ptr(out), _ptr(workspace),
                                   workspace.numel() if workspace is not None else 0, _ptr(dev_status),
                                   _stream(stream)),
           "pa_decode_paged_fp8")


def pa_prepare_prefill(seq_lens, num_cached, num_scheduled, block_table, block_size, num_blocks, max_tokens,
                       dev_status=None, stream=None):
    """Device-built prefill metadata.  Inputs: CUDA int32 [B] counts and the
    [B, max_blocks] table.  Returns (cu_seqlens_q, cu_seqlens_k, positions,
    slot_mapping, max_seqlens) as CUDA int32 tensors (positions / slots sized
    max_tokens)."""
    for t, n in ((seq_lens, "seq_lens"), (num_cached, "num_cached"), (num_scheduled, "num_scheduled"),
                 (block_table, "block_table")):
        _i32(t, n)
    b = seq_lens.numel()
    if num_cached.numel() != b or num_scheduled.numel() != b or block_table.dim() != 2 or block_table.shape[0] != b:
        raise ValueError("pa_prepare_prefill: inconsistent shapes")
    d = seq_lens.device
    cu_q = torch.empty(b + 1, dtype=torch.int32, device=d)
    cu_k = torch.empty(b + 1, dtype=torch.int32, device=d)
    pos = torch.empty(max(max_tokens, 1), dtype=torch.int32, device=d)
    sl = torch.empty(max(max_tokens, 1), dtype=torch.int32, device=d)
    mx = torch.empty(2, dtype=torch.int32, device=d)
    _check(lib.pa_prepare_prefill(_ptr(seq_lens), _ptr(num_cached), _ptr(num_scheduled), b, _ptr(block_table),
                                  block_table.shape[1], block_size, num_blocks, _ptr(cu_q), _ptr(cu_k), _ptr(pos),
                                  _ptr(sl), max_tokens, _ptr(mx), _ptr(dev_status), _stream(stream)),
           "pa_prepare_prefill")
    return cu_q, cu_k, pos[:max_tokens], sl[:max_tokens], mx


def pa_prepare_decode(seq_lens, block_table, block_size, num_blocks, dev_status=None, stream=None):
    """Device-built decode metadata: (positions, context_lens, slot_mapping), CUDA int32 [B]."""
    _i32(seq_lens, "seq_lens")
    _i32(block_table, "block_table")
    b = seq_lens.numel()
    if block_table.dim() != 2 or block_table.shape[0] != b:
        raise ValueError("pa_prepare_decode: block_table must be [B, max_blocks]")
    d = seq_lens.device
    pos, ctx, sl = (torch.empty(max(b, 1), dtype=torch.int32, device=d) for _ in range(3))
    _check(lib.pa_prepare_decode(_ptr(seq_lens), b, _ptr(block_table), block_table.shape[1], block_size, num_blocks,
                                 _ptr(pos), _ptr(ctx), _ptr(sl), _ptr(dev_status), _stream(stream)),
           "pa_prepare_decode")
    return pos[:b], ctx[:b], sl[:b]


def pa_rope_cos_sin_table(base: float, head_dim: int, max_positions: int, device=None, stream=None) -> torch.Tensor:
    """fp32 [max_positions, head_dim] rotary table on the device (cos half, then sin half)."""
    t = torch.empty((max_positions, head_dim), dtype=torch.float32,
                    device=device if device is not None else torch.device("cuda"))
    _check(lib.pa_rope_cos_sin_table(float(base), head_dim, max_positions, _ptr(t), _stream(stream)),
           "pa_rope_cos_sin_table")
    return t


def pa_norm_rope_store_kvcache(qkv, num_heads, num_kv_heads, positions, cos_sin, q_norm_weight, k_norm_weight,
                               eps, q_out, k_cache, v_cache, slot_mapping, dev_status=None, stream=None):
    """Head RMSNorm + RoPE of Q and K and the KV write.  qkv: CUDA bf16
    [T, (Hq + 2 Hkv) * 128] (token stride free); positions / slot_mapping int32
    [T]; cos_sin fp32 [max_positions, 128]; weights bf16 [128] or None;
    q_out bf16 [T, Hq, 128] (may be a view of qkv's Q columns)."""
    if qkv.dtype != torch.bfloat16 or qkv.dim() != 2 or not qkv.is_cuda or qkv.stride(1) != 1:
        raise TypeError("qkv: expected a CUDA bf16 [T, width] tensor with packed rows")
    nb, bs, hkv, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    if hkv != num_kv_heads or qkv.shape[1] != (num_heads + 2 * num_kv_heads) * d:
        raise ValueError("qkv width or cache heads do not match the head counts")
    hq, qs = _bf16_rows(q_out, "q_out")
    if hq != num_heads or q_out.shape[0] != qkv.shape[0]:
        raise ValueError("q_out must be [T, num_heads, head_dim]")
    _i32(positions, "positions")
    _i32(slot_mapping, "slot_mapping")
    if positions.numel() != qkv.shape[0] or slot_mapping.numel() != qkv.shape[0]:
        raise ValueError("positions and slot_mapping need one entry per token")
    if cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or not cos_sin.is_contiguous() or cos_sin.shape[1] != d:
        raise TypeError("cos_sin: expected a contiguous CUDA fp32 [max_positions, head_dim] tensor")
    for w, name in ((q_norm_weight, "q_norm_weight"), (k_norm_weight, "k_norm_weight")):
        if w is not None and (w.dtype != torch.bfloat16 or w.numel() != d or not w.is_contiguous()):
            raise TypeError(f"{name}: expected a contiguous bf16 [head_dim] tensor or None")
    _check(lib.pa_norm_rope_store_kvcache(_ptr(qkv), qkv.stride(0), qkv.shape[0], num_heads, num_kv_heads, d,
                                          _ptr(positions), _ptr(cos_sin), cos_sin.shape[0], _ptr(q_norm_weight),
                                          _ptr(k_norm_weight), float(eps), _ptr(q_out), qs, _ptr(k_cache),
                                          _ptr(v_cache), nb, bs, _ptr(slot_mapping), _ptr(dev_status),
                                          _stream(stream)),
           "pa_norm_rope_store_kvcache")


def pa_prefill_workspace_bytes(num_seqs, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads) -> int:
    return lib.pa_prefill_workspace_bytes(num_seqs, int(max_seqlen_q), int(max_seqlen_k), num_heads, num_kv_heads)


def pa_prefill_paged(q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale, out, *, k=None, v=None,
                     k_cache=None, v_cache=None, block_table=None, workspace=None, dev_status=None, stream=None):
    """Causal varlen prefill.  With block_table=None keys come from k/v;
    otherwise from the paged caches.  workspace: a CUDA uint8 tensor of at
    least pa_prefill_workspace_bytes(...) bytes (256-byte aligned), owned by
    the caller; nothing is allocated here, and a call that needs a workspace
    and gets none raises."""
    hq, qs = _bf16_rows(q, "q")
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (q.shape[0], hq, q.shape[2]):
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    _i32(cu_seqlens_q, "cu_seqlens_q")
    _i32(cu_seqlens_k, "cu_seqlens_k")
    nseq = cu_seqlens_q.numel() - 1
    if block_table is None:
        hkv, kvs = _bf16_rows(k, "k")
        _, vs = _bf16_rows(v, "v")
        if vs != kvs:
            raise ValueError("k and v must share a token stride")
        if k.shape[0] < q.shape[0] or v.shape[0] < q.shape[0]:
            raise ValueError("k and v need a row per query token")
        args = (_ptr(k), _ptr(v), kvs, None, None, 0, 16, None, 1)
    else:
        nb, bs, hkv, _ = _cache(k_cache, "k_cache")
        _cache(v_cache, "v_cache")
        _i32(block_table, "block_table")
        if block_table.dim() != 2 or block_table.shape[0] != nseq:
            raise ValueError("block_table must be [num_seqs, max_blocks]")
        args = (None, None, 0, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_table), block_table.shape[1])
    need = lib.pa_prefill_workspace_bytes(nseq, int(max_seqlen_q), int(max_seqlen_k), hq, hkv) if nseq > 0 else 0
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        raise ValueError(f"pa_prefill_paged: this call needs a workspace of {need} bytes "
                         "(pa_prefill_workspace_bytes)")
    _check(lib.pa_prefill_paged(_ptr(q), qs, q.shape[0], *args, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), nseq,
                                int(max_seqlen_q), int(max_seqlen_k), hq, hkv, q.shape[2], float(scale), _ptr(out),
                                _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _ptr(dev_status),
                                _stream(stream)),
           "pa_prefill_paged")


def pa_decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int) -> int:
    return lib.pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len)


def pa_decode_paged(q, k_cache, v_cache, block_table, context_lens, max_context_len, scale, out, workspace,
                    dev_status=None, stream=None):
    """Paged decode: q [B, Hq, 128] (seq stride free), out [B, Hq, 128]
    packed, workspace a CUDA uint8 tensor of pa_decode_workspace_bytes."""
    hq, qs = _bf16_rows(q, "q")
    nb, bs, hkv, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(block_table, "block_table")
    _i32(context_lens, "context_lens")
    b = q.shape[0]
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (b, hq, d):
        raise ValueError("out must be a contiguous bf16 [B, Hq, D] tensor")
    if block_table.dim() != 2 or block_table.shape[0] != b or context_lens.numel() != b:
        raise ValueError("block_table / context_lens do not match q")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_decode_paged(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_table),
                               block_table.shape[1], _ptr(context_lens), b, int(max_context_len), hq, hkv, d,
                               float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status),
                               _stream(stream)),
           "pa_decode_paged")


def pa_store_decode_paged(q, k_new, v_new, k_cache, v_cache, block_table, context_lens, max_context_len, scale, out,
                          workspace, dev_status=None, stream=None):
    """The decode step's KV write and decode in one launch: k_new / v_new
    [B, Hkv, 128] (the token at position context_lens[b] - 1, same sequence
    stride) go to that position's pool row, then decode as pa_decode_paged."""
    hq, qs = _bf16_rows(q, "q")
    hk, ks = _bf16_rows(k_new, "k_new")
    hv, vs = _bf16_rows(v_new, "v_new")
    nb, bs, hkv, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(block_table, "block_table")
    _i32(context_lens, "context_lens")
    b = q.shape[0]
    if hk != hkv or hv != hkv or ks != vs or k_new.shape[0] != b or v_new.shape[0] != b:
        raise ValueError("k_new / v_new must be [B, Hkv, D] bf16 with one sequence stride")
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (b, hq, d):
        raise ValueError("out must be a contiguous bf16 [B, Hq, D] tensor")
    if block_table.dim() != 2 or block_table.shape[0] != b or context_lens.numel() != b:
        raise ValueError("block_table / context_lens do not match q")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_store_decode_paged(_ptr(q), qs, _ptr(k_new), _ptr(v_new), ks, _ptr(k_cache), _ptr(v_cache), nb,
                                     bs, _ptr(block_table), block_table.shape[1], _ptr(context_lens), b,
                                     int(max_context_len), hq, hkv, d, float(scale), _ptr(out), _ptr(workspace),
                                     ws_bytes, _ptr(dev_status), _stream(stream)),
           "pa_store_decode_paged")


def pa_norm_rope_store_decode_paged(qkv, num_heads, num_kv_heads, cos_sin, q_norm_weight, k_norm_weight, eps, k_cache,
                                    v_cache, block_table, context_lens, max_context_len, scale, out, workspace,
                                    dev_status=None, stream=None):
    """One layer's decode step from the fused QKV output: qkv [B, (Hq + 2 Hkv) * 128] bf16 (sequence stride free);
    head norm + RoPE of the new token at position context_lens[b] - 1, its K/V to that position's pool row, then
    decode as pa_decode_paged.  out [B, Hq, 128] packed; workspace as for pa_decode_paged."""
    if qkv.dtype != torch.bfloat16 or qkv.dim() != 2 or not qkv.is_cuda or qkv.stride(1) != 1:
        raise TypeError("qkv: expected a CUDA bf16 [B, (Hq + 2 Hkv) * D] tensor with packed columns")
    nb, bs, hkv, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    if hkv != num_kv_heads or qkv.shape[1] != (num_heads + 2 * num_kv_heads) * d:
        raise ValueError("qkv columns do not match num_heads / num_kv_heads and the cache")
    if cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or not cos_sin.is_contiguous() or cos_sin.shape[1] != d:
        raise TypeError("cos_sin: expected a contiguous CUDA fp32 [max_positions, head_dim] tensor")
    for w, name in ((q_norm_weight, "q_norm_weight"), (k_norm_weight, "k_norm_weight")):
        if w is not None and (w.dtype != torch.bfloat16 or w.numel() != d or not w.is_contiguous()):
            raise TypeError(f"{name}: expected a contiguous bf16 [head_dim] tensor or None")
    _i32(block_table, "block_table")
    _i32(context_lens, "context_lens")
    b = qkv.shape[0]
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (b, num_heads, d):
        raise ValueError("out must be a contiguous bf16 [B, Hq, D] tensor")
    if block_table.dim() != 2 or block_table.shape[0] != b or context_lens.numel() != b:
        raise ValueError("block_table / context_lens do not match qkv")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_norm_rope_store_decode_paged(_ptr(qkv), qkv.stride(0), _ptr(cos_sin), cos_sin.shape[0],
                                               _ptr(q_norm_weight), _ptr(k_norm_weight), float(eps), _ptr(k_cache),
                                               _ptr(v_cache), nb, bs, _ptr(block_table), block_table.shape[1],
                                               _ptr(context_lens), b, int(max_context_len), num_heads, hkv, d,
                                               float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                               _stream(stream)),
           "pa_norm_rope_store_decode_paged")


def pa_decode_paged_noalloc(q, k_cache, v_cache, block_table, context_lens, max_context_len, scale, out,
                            dev_status=None, stream=None):
    """Paged decode for callers that cannot allocate device memory: no
    workspace argument; the library's fixed device scratch is used instead
    (see include/pa.h).  Calls that overlap on the GPU must not be issued."""
    hq, qs = _bf16_rows(q, "q")
    nb, bs, hkv, d = _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(block_table, "block_table")
    _i32(context_lens, "context_lens")
    b = q.shape[0]
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.shape != (b, hq, d):
        raise ValueError("out must be a contiguous bf16 [B, Hq, D] tensor")
    if block_table.dim() != 2 or block_table.shape[0] != b or context_lens.numel() != b:
        raise ValueError("block_table / context_lens do not match q")
    _check(lib.pa_decode_paged_noalloc(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_table),
                                       block_table.shape[1], _ptr(context_lens), b, int(max_context_len), hq, hkv,
                                       d, float(scale), _ptr(out), _ptr(dev_status), _stream(stream)),
           "pa_decode_paged_noalloc")
