"""The C-ABI library builds, loads and exports every symbol include/pa.h
declares; host-side argument checks reject bad calls before any CUDA work.
No kernel is launched here (no GPU is needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_110_gb300 import _build
    _build.build()
    from paged_kv_cache_110_gb300 import binding
    return binding.lib


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pa_store_kvcache", "pa_prefill_paged", "pa_decode_paged", "pa_decode_workspace_bytes",
              "pa_status_string", "pa_kv_bytes_per_token", "pa_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from paged_kv_cache_110_gb300 import binding as pa
    assert pa.pa_status_string(0) == "ok"
    assert pa.pa_status_string(4) == "index out of bounds"
    assert pa.pa_status_string(99) == "unknown status"
    assert pa.pa_abi_version() >= 100


def test_kv_bytes_closed_form(lib):
    from paged_kv_cache_110_gb300 import binding as pa
    assert pa.pa_kv_bytes_per_token(28, 8, 128, 2) == 114688
    assert pa.pa_kv_bytes_per_token(28, 8, 128, 2) * 256 == 29360128
    assert pa.pa_kv_bytes_per_token(0, 8, 128, 2) == 0


FAKE = 0x10000  # a 16-byte aligned non-null value; never dereferenced by the host checks below


def test_store_host_checks(lib):
    f = lib.pa_store_kvcache
    ok = dict(k=FAKE, ks=1024, v=FAKE, vs=1024, n=4, hkv=8, d=128, kc=FAKE, vc=FAKE, nb=4, bs=16, slot=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["k"], a["ks"], a["v"], a["vs"], a["n"], a["hkv"], a["d"], a["kc"], a["vc"], a["nb"], a["bs"],
                 a["slot"], None, None)

    assert call(d=64) == 2
    assert call(hkv=3) == 2
    assert call(bs=24) == 2
    assert call(n=-1) == 1
    assert call(n=0) == 0          # nothing to do, nothing launched
    assert call(k=None) == 1
    assert call(slot=None) == 1
    assert call(ks=512) == 1       # stride shorter than a row


def test_prefill_host_checks(lib):
    f = lib.pa_prefill_paged

    def call(q=FAKE, qs=2048, nt=16, k=None, v=None, kvs=0, kc=FAKE, vc=FAKE, nb=4, bs=16, bt=FAKE, mb=2,
             cuq=FAKE, cuk=FAKE, ns=2, mq=8, mk=8, hq=16, hkv=8, d=128, out=FAKE):
        return f(q, qs, nt, k, v, kvs, kc, vc, nb, bs, bt, mb, cuq, cuk, ns, mq, mk, hq, hkv, d,
                 ctypes.c_float(0.1), out, None, 0, None, None)

    assert call(d=64) == 2
    assert call(hq=12, hkv=8) == 2
    assert call(hq=32, hkv=2) == 2   # 16 query heads per KV head is not built
    assert call(ns=0) == 0
    assert call(mq=0) == 0
    assert call(q=None) == 1
    assert call(bt=None) == 1                               # no table and no k / v
    assert call(bt=None, k=FAKE, v=FAKE, kvs=1024, mk=9) == 1  # null table needs max_seqlen_k == max_seqlen_q
    assert call(qs=100) == 1
    assert call(nt=-1) == 1
    assert call(nt=0) == 0                                  # no query rows: nothing to do
    assert call(nt=1 << 31) == 2


def test_decode_host_checks(lib):
    f = lib.pa_decode_paged

    def call(q=FAKE, qs=2048, kc=FAKE, vc=FAKE, nb=4, bs=16, bt=FAKE, mb=2, ctx=FAKE, ns=2, mctx=32, hq=16,
             hkv=8, d=128, out=FAKE, ws=None, wsb=0):
        return f(q, qs, kc, vc, nb, bs, bt, mb, ctx, ns, mctx, hq, hkv, d, ctypes.c_float(0.1), out, ws, wsb,
                 None, None)

    assert call(d=256) == 2
    assert call(hkv=16, hq=16) == 2
    assert call(bs=8) == 2
    assert call(ns=0) == 0
    assert call(ns=-1) == 1
    assert call(ctx=None) == 1
    assert call(q=FAKE + 2) == 1   # q must be 16-byte aligned


def test_store_decode_host_checks(lib):
    f = lib.pa_store_decode_paged

    def call(q=FAKE, qs=2048, kn=FAKE, vn=FAKE, ks=1024, kc=FAKE, vc=FAKE, nb=4, bs=16, bt=FAKE, mb=2, ctx=FAKE,
             ns=2, mctx=32, hq=16, hkv=8, d=128, out=FAKE):
        return f(q, qs, kn, vn, ks, kc, vc, nb, bs, bt, mb, ctx, ns, mctx, hq, hkv, d, ctypes.c_float(0.1), out,
                 None, 0, None, None)

    assert call(kn=None) == 1
    assert call(vn=None) == 1
    assert call(kn=FAKE + 8) == 1  # k_new must be 16-byte aligned
    assert call(ks=1000) == 1      # stride below Hkv * D
    assert call(ks=1028) == 1      # stride not a multiple of 8
    assert call(d=256, ks=2048) == 2  # then the decode checks apply
    assert call(ns=0) == 0


def test_decode_workspace_follows_the_split_plan(lib):
    """The decode workspace holds fp32 partials [seqs, splits, heads, 128] (256-byte aligned) and a (max, sum)
    pair per (seq, split, head); the keys are split for about 64 CTAs per SM (152 SMs, the GB300 count the
    library assumes when no GPU is visible) into runs of at least 128 tokens (256 from 32 query heads on),
    rounded up to 64; one split needs no workspace."""
    from paged_kv_cache_110_gb300 import binding as pa

    def expect(seqs, heads, ctx, sms=152):
        per_seq = -(-64 * sms // seqs)
        length = max(-(-(-(-ctx // per_seq)) // 64) * 64, 256 if heads >= 32 else 128)
        splits = -(-ctx // length)
        if splits <= 1:
            return 0
        n = seqs * splits * heads
        return -(-n * 512 // 256) * 256 + n * 8

    for seqs, heads, ctx in [(256, 16, 1024), (512, 16, 4096), (1, 16, 32768), (64, 16, 100), (1000, 8, 3000),
                             (3, 32, 129), (256, 64, 1024), (256, 32, 1024), (512, 64, 4096)]:
        assert pa.pa_decode_workspace_bytes(seqs, heads, 128, ctx) == expect(seqs, heads, ctx), (seqs, heads, ctx)
    assert pa.pa_decode_workspace_bytes(256, 16, 128, 1024) == 256 * 8 * 16 * 520   # 8 splits of 128 tokens
    assert pa.pa_decode_workspace_bytes(512, 16, 128, 4096) == 512 * 16 * 16 * 520  # 16 splits of 256 tokens
    assert pa.pa_decode_workspace_bytes(64, 16, 128, 128) == 0                       # one split
    assert pa.pa_decode_workspace_bytes(256, 64, 128, 1024) == 256 * 4 * 64 * 520   # 4 splits of 256 tokens


def test_norm_rope_store_host_checks(lib):
    f = lib.pa_norm_rope_store_kvcache

    def call(qkv=FAKE, qs=4096, nt=4, hq=16, hkv=8, d=128, pos=FAKE, cs=FAKE, mp=64, qw=None, kw=None, eps=1e-6,
             qo=FAKE, qos=2048, kc=FAKE, vc=FAKE, nb=4, bs=16, sl=FAKE):
        return f(qkv, qs, nt, hq, hkv, d, pos, cs, mp, qw, kw, ctypes.c_float(eps), qo, qos, kc, vc, nb, bs, sl,
                 None, None)

    assert call(d=64) == 2
    assert call(hq=12) == 2
    assert call(bs=8) == 2
    assert call(nt=0) == 0
    assert call(nt=-1) == 1
    assert call(pos=None) == 1
    assert call(cs=None) == 1
    assert call(mp=0) == 1
    assert call(qs=4000) == 1          # shorter than a fused row
    assert call(qos=1024) == 1         # shorter than the Q heads
    assert call(eps=-1.0) == 1
    assert call(qw=FAKE + 8) == 1      # weight not 16-byte aligned


def test_rope_table_host_checks(lib):
    f = lib.pa_rope_cos_sin_table
    assert f(1e6, 127, 16, FAKE, None) == 1   # odd head_dim
    assert f(1.0, 128, 16, FAKE, None) == 1   # base must exceed 1
    assert f(1e6, 128, -1, FAKE, None) == 1
    assert f(1e6, 128, 0, FAKE, None) == 0    # nothing to fill
    assert f(1e6, 128, 16, None, None) == 1


def test_metadata_host_checks(lib):
    pf = lib.pa_prepare_prefill

    def pre(sl=FAKE, nc=FAKE, ns=FAKE, b=3, bt=FAKE, mb=4, bs=16, nb=8, cq=FAKE, ck=FAKE, pos=FAKE, slots=FAKE,
            mt=100, mx=FAKE):
        return pf(sl, nc, ns, b, bt, mb, bs, nb, cq, ck, pos, slots, mt, mx, None, None)

    assert pre(b=0) == 0
    assert pre(b=-1) == 1
    assert pre(sl=None) == 1
    assert pre(mx=None) == 1
    assert pre(mb=0) == 1
    assert pre(nb=1 << 30, bs=256) == 1   # pool rows past int32
    assert pre(mt=-5) == 1
    pd = lib.pa_prepare_decode

    def dec(sl=FAKE, b=3, bt=FAKE, mb=4, bs=16, nb=8, pos=FAKE, ctx=FAKE, slots=FAKE):
        return pd(sl, b, bt, mb, bs, nb, pos, ctx, slots, None, None)

    assert dec(b=0) == 0
    assert dec(b=-2) == 1
    assert dec(ctx=None) == 1
    assert dec(bs=0) == 1
