"""CPU oracle for attention over a block-paged KV cache (test infrastructure).

This package is the slow, obviously correct definition that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
product path never does, and it imports nothing from the product package.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, one key at a
time through ``block_table``).  This module only builds that file with gcc and
marshals numpy arrays into it.  bf16 tensors are passed as their raw uint16
bits; outputs come back as float64.

Sources: "大模型推理入门与 nano-vLLM 源码详解" §4.4, §9.2, §9.5, §11.2, §11.4,
§13.1, §13.5, §19.1, §19.6; "大模型推理引擎入门 ... 对着日志读懂 nano-vllm"
§2.7; Pico-vLLM log #6 ("VLLM on Fain的Blog").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")

_lib = None
_lock = threading.Lock()

OK, INVALID, BOUNDS = 0, 1, 4


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library with gcc (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PA_ORACLE_LIB lets the mutation tests load a deliberately broken build
            override = os.environ.get("PA_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.orc_kv_bytes_per_token.restype = i64
            lib.orc_kv_bytes_per_token.argtypes = [i32, i32, i32, i32]
            lib.orc_slot.restype = i64
            lib.orc_slot.argtypes = [vp, i32, i64]
            lib.orc_num_threads.restype = i32
            lib.orc_set_num_threads.argtypes = [i32]
            lib.orc_store_kvcache.restype = i32
            lib.orc_store_kvcache.argtypes = [vp, i64, vp, i64, i64, i32, i32, vp, vp, i64, i32, vp]
            pre = [vp, i64, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp, vp, i32, i32, i32, i32, dbl, vp]
            lib.orc_prefill.restype = i32
            lib.orc_prefill.argtypes = pre
            lib.orc_prefill_weights.restype = i32
            lib.orc_prefill_weights.argtypes = pre + [i32, i32, i32, vp]
            lib.orc_decode.restype = i32
            lib.orc_decode.argtypes = [vp, i64, vp, vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, dbl, vp]
            lib.orc_rmsnorm.restype = None
            lib.orc_rmsnorm.argtypes = [vp, i32, vp, dbl, vp]
            lib.orc_rope_cos_sin.restype = None
            lib.orc_rope_cos_sin.argtypes = [dbl, i32, i64, vp]
            lib.orc_rope_apply.restype = None
            lib.orc_rope_apply.argtypes = [vp, i32, vp, vp]
            lib.orc_e4m3_value.restype = dbl
            lib.orc_e4m3_value.argtypes = [i32]
            lib.orc_e4m3_encode.restype = i32
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_store_kvcache_fp8.restype = i32
            lib.orc_store_kvcache_fp8.argtypes = [vp, i64, vp, i64, i64, i32, i32, ctypes.c_float, ctypes.c_float,
                                                  vp, vp, i64, i32, vp]
            lib.orc_decode_fp8.restype = i32
            lib.orc_decode_fp8.argtypes = [vp, i64, vp, vp, dbl, dbl, i64, i32, vp, i32, vp, i32, i32, i32, i32, dbl,
                                           vp]
            lib.orc_prepare_prefill.restype = i32
            lib.orc_prepare_prefill.argtypes = [vp, vp, vp, i32, vp, i32, i32, i64, vp, vp, vp, vp, vp, vp]
            lib.orc_prepare_decode.restype = i32
            lib.orc_prepare_decode.argtypes = [vp, i32, vp, i32, i32, i64, vp, vp, vp]
            lib.orc_norm_rope_store.restype = i32
            lib.orc_norm_rope_store.argtypes = [vp, i64, i64, i32, i32, i32, vp, vp, i64, vp, vp, dbl, vp, i64,
                                                vp, vp, i64, i32, vp]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(a: np.ndarray, name: str):
    """Validate a [T, H, d] bf16-bits array whose last two axes are packed;
    return (array, token stride in elements)."""
    if a.dtype != np.uint16 or a.ndim != 3:
        raise OracleError(f"{name}: expected uint16 [T, H, d], got {a.dtype} {a.shape}")
    if a.strides[2] != 2 or a.strides[1] != 2 * a.shape[2]:
        a = np.ascontiguousarray(a)
    if a.strides[0] % 2:
        raise OracleError(f"{name}: token stride is not a whole number of elements")
    return a, a.strides[0] // 2


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what}: status {rc}")


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return _load().orc_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def slot(block_table_row, block_size: int, pos: int) -> int:
    row = _i32(block_table_row)
    return _load().orc_slot(_ptr(row), block_size, pos)


def store_kvcache(k, v, k_cache, v_cache, slot_mapping):
    """In-place KV write into (k_cache, v_cache) [NB, bs, Hkv, d] (uint16 bits).
    Returns the oracle status (0, or 4 if some slot was out of range)."""
    k, ks = _rows(k, "k")
    v, vs = _rows(v, "v")
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or c.ndim != 4 or not c.flags.c_contiguous:
            raise OracleError("cache must be a C-contiguous uint16 [NB, bs, Hkv, d] array")
    slots = _i32(slot_mapping)
    nb, bs, hkv, d = k_cache.shape
    return _load().orc_store_kvcache(_ptr(k), ks, _ptr(v), vs, k.shape[0], hkv, d,
                                     _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(slots))


def prefill(q, cu_seqlens_q, cu_seqlens_k, scale, *, k=None, v=None, k_cache=None, v_cache=None,
            block_table=None, weights_of=None):
    """Causal varlen prefill; returns float64 [T, Hq, d] (and the weights of
    row ``weights_of=(b, h, i)`` if asked).  With ``block_table=None`` keys come
    from the contiguous ``k``/``v``; otherwise from the paged cache."""
    q, qs = _rows(q, "q")
    t, hq, d = q.shape
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    nseq = len(cu_q) - 1
    if block_table is None:
        k, kvs = _rows(k, "k")
        v, vs2 = _rows(v, "v")
        if kvs != vs2:
            raise OracleError("k and v must share a token stride")
        hkv = k.shape[1]
        bt, mb, nb, bs, kc, vc = None, 0, 0, 1, None, None
    else:
        bt = _i32(block_table)
        mb = bt.shape[1]
        kc, vc = k_cache, v_cache
        nb, bs, hkv, _ = kc.shape
        kvs = 0
        k = v = None
    out = np.zeros((t, hq, d), dtype=np.float64)
    lib = _load()
    args = [_ptr(q), qs, _ptr(k), _ptr(v), kvs, _ptr(kc), _ptr(vc), nb, bs, _ptr(bt), mb,
            _ptr(cu_q), _ptr(cu_k), nseq, hq, hkv, d, float(scale), _ptr(out)]
    if weights_of is None:
        _check(lib.orc_prefill(*args), "orc_prefill")
        return out
    b, h, i = weights_of
    w = np.zeros(int(cu_k[b + 1] - cu_k[b]), dtype=np.float64)
    _check(lib.orc_prefill_weights(*args, b, h, i, _ptr(w)), "orc_prefill_weights")
    return out, w


def decode(q, k_cache, v_cache, block_table, context_lens, scale):
    """Paged decode: q [B, Hq, d] bits; returns float64 [B, Hq, d]."""
    q, qs = _rows(q, "q")
    b, hq, d = q.shape
    bt, ctx = _i32(block_table), _i32(context_lens)
    nb, bs, hkv, _ = k_cache.shape
    out = np.zeros((b, hq, d), dtype=np.float64)
    _check(_load().orc_decode(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(bt),
                              bt.shape[1], _ptr(ctx), b, hq, hkv, d, float(scale), _ptr(out)),
           "orc_decode")
    return out


def rmsnorm(x, weight=None, eps: float = 0.0) -> np.ndarray:
    """x * 1/sqrt(mean(x^2) + eps) [* weight], in double (no rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = None if weight is None else np.ascontiguousarray(weight, dtype=np.float64)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_ptr(x), x.size, _ptr(w), float(eps), _ptr(y))
    return y


def rope_cos_sin(base: float, head_dim: int, max_positions: int) -> np.ndarray:
    """[max_positions, head_dim] float32: cos(p * inv_freq) then sin(p * inv_freq)."""
    t = np.empty((max_positions, head_dim), dtype=np.float32)
    _load().orc_rope_cos_sin(float(base), head_dim, max_positions, _ptr(t))
    return t


def rope_apply(x, cos_sin_row) -> np.ndarray:
    """Rotate one head vector (double) by one table row; pairs (i, i + d/2)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    cs = np.ascontiguousarray(cos_sin_row, dtype=np.float32)
    y = np.empty_like(x)
    _load().orc_rope_apply(_ptr(x), x.size, _ptr(cs), _ptr(y))
    return y


def norm_rope_store(qkv, num_heads, num_kv_heads, positions, cos_sin, q_weight, k_weight, eps,
                    k_cache, v_cache, slot_mapping):
    """Head RMSNorm + RoPE of Q and K and the KV write.  qkv: uint16 [T, (Hq + 2 Hkv) * d]
    (any token stride); k_cache / v_cache uint16 [NB, bs, Hkv, d], written in place.
    Returns q_out uint16 [T, Hq, d]."""
    if qkv.dtype != np.uint16 or qkv.ndim != 2 or qkv.strides[1] != 2:
        raise OracleError("qkv: expected uint16 [T, width] with packed rows")
    d = cos_sin.shape[1]
    t = qkv.shape[0]
    if qkv.shape[1] != (num_heads + 2 * num_kv_heads) * d:
        raise OracleError("qkv width does not match the head counts")
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags.c_contiguous or c.ndim != 4 or c.shape[2:] != (num_kv_heads, d):
            raise OracleError("caches: expected contiguous uint16 [NB, bs, Hkv, d]")
    q_out = np.zeros((t, num_heads, d), dtype=np.uint16)
    pos, sl = _i32(positions), _i32(slot_mapping)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    qw = None if q_weight is None else np.ascontiguousarray(q_weight, dtype=np.uint16)
    kw = None if k_weight is None else np.ascontiguousarray(k_weight, dtype=np.uint16)
    rc = _load().orc_norm_rope_store(_ptr(qkv), qkv.strides[0] // 2, t, num_heads, num_kv_heads, d, _ptr(pos),
                                     _ptr(cs), cs.shape[0], _ptr(qw), _ptr(kw), float(eps), _ptr(q_out),
                                     num_heads * d, _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                     k_cache.shape[1], _ptr(sl))
    if rc not in (OK, BOUNDS):
        raise OracleError(f"norm_rope_store: status {rc}")
    return q_out, rc


def _table2d(block_table, num_seqs):
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim != 2 or bt.shape[0] != num_seqs:
        raise OracleError("block_table must be [num_seqs, max_blocks]")
    return bt


def prepare_prefill(seq_lens, num_cached, num_scheduled, block_table, block_size, num_blocks):
    """Step metadata of a prefill batch; returns a dict of int32 arrays / ints and the status."""
    sl, nc, ns = _i32(seq_lens), _i32(num_cached), _i32(num_scheduled)
    b = sl.size
    bt = _table2d(block_table, b)
    t = int(ns.sum())
    cu_q, cu_k = np.zeros(b + 1, np.int32), np.zeros(b + 1, np.int32)
    pos, slots = np.zeros(t, np.int32), np.zeros(t, np.int32)
    mq, mk = ctypes.c_int32(), ctypes.c_int32()
    rc = _load().orc_prepare_prefill(_ptr(sl), _ptr(nc), _ptr(ns), b, _ptr(bt), bt.shape[1], block_size, num_blocks,
                                     _ptr(cu_q), _ptr(cu_k), _ptr(pos), _ptr(slots), ctypes.byref(mq),
                                     ctypes.byref(mk))
    return {"cu_seqlens_q": cu_q, "cu_seqlens_k": cu_k, "positions": pos, "slot_mapping": slots,
            "max_seqlen_q": mq.value, "max_seqlen_k": mk.value}, rc


def prepare_decode(seq_lens, block_table, block_size, num_blocks):
    sl = _i32(seq_lens)
    b = sl.size
    bt = _table2d(block_table, b)
    pos, ctx, slots = np.zeros(b, np.int32), np.zeros(b, np.int32), np.zeros(b, np.int32)
    rc = _load().orc_prepare_decode(_ptr(sl), b, _ptr(bt), bt.shape[1], block_size, num_blocks, _ptr(pos), _ptr(ctx),
                                    _ptr(slots))
    return {"positions": pos, "context_lens": ctx, "slot_mapping": slots}, rc


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code (NaN for 0x7f / 0xff)."""
    return _load().orc_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code of a float32 value (ties to even, saturating to +-448)."""
    return _load().orc_e4m3_encode(float(np.float32(x)))


def store_kvcache_fp8(k, v, k_scale, v_scale, k_cache, v_cache, slot_mapping):
    """KV write into uint8 E4M3 pools [NB, bs, Hkv, d] (in place); returns the status."""
    k, ks = _rows(k, "k")
    v, vs = _rows(v, "v")
    for c in (k_cache, v_cache):
        if c.dtype != np.uint8 or not c.flags.c_contiguous or c.ndim != 4:
            raise OracleError("fp8 caches: expected contiguous uint8 [NB, bs, Hkv, d]")
    sl = _i32(slot_mapping)
    return _load().orc_store_kvcache_fp8(_ptr(k), ks, _ptr(v), vs, k.shape[0], k.shape[1], k.shape[2],
                                         float(k_scale), float(v_scale), _ptr(k_cache), _ptr(v_cache),
                                         k_cache.shape[0], k_cache.shape[1], _ptr(sl))


def decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, scale):
    """Decode over E4M3 pools; out [B, Hq, d] double."""
    q, qs = _rows(q, "q")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    ctx = _i32(context_lens)
    b, hq, d = q.shape
    out = np.zeros((b, hq, d), dtype=np.float64)
    rc = _load().orc_decode_fp8(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale),
                                k_cache.shape[0], k_cache.shape[1], _ptr(bt), bt.shape[1], _ptr(ctx), b, hq,
                                k_cache.shape[2], d, float(scale), _ptr(out))
    _check(rc, "decode_fp8")
    return out
