"""The C-ABI library: it loads, exports every declared symbol, and its host-side
validation (no kernel launches, no GPU needed) returns the documented codes and
leaves the cache descriptor unchanged on error."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import sizes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")

kvq = pytest.importorskip("quantized_kv_cache_quant_gb300.kvq", reason="libkvq.so not built")

ALIGNED = 1 << 20  # a fake, 256-byte aligned address: validation never dereferences it


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"KVQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) == 29
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(kvq.EXPORTED)


def test_status_strings():
    for code, name in kvq.STATUS.items():
        assert kvq.kvq_status_string(code)
    assert kvq.kvq_status_string(0) == "ok"


@pytest.mark.parametrize("b,h,hq,d,kb,vb,r,t", [
    (1, 2, 2, 64, 2, 2, 128, 272),
    (8, 32, 32, 128, 2, 2, 128, 4097),
    (32, 8, 64, 128, 4, 4, 128, 8193),
    (4, 8, 64, 128, 2, 2, 128, 131584),
    (2, 3, 6, 64, 2, 4, 0, 100),
])
def test_cache_sizes_match_layout(b, h, hq, d, kb, vb, r, t):
    cfg = kvq.make_config(b, h, hq, d, kb, vb, r, t)
    got = kvq.kivi_cache_sizes(cfg)
    want = sizes.kivi_buffer_bytes(b, h, d, kb, vb, r, t)
    assert got == [want[n] for n in ("k_codes", "k_meta", "v_codes", "v_meta", "k_res", "v_res")]
    ws = kvq.kv_decode_workspace_bytes(cfg)
    counters = -(-b * hq * 4 // 256) * 256
    assert ws == 256 + counters + b * hq * 64 * (d + 2) * 4


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, "KVQ_ERR_UNSUPPORTED"),
    ("k_bits", 3, "KVQ_ERR_UNSUPPORTED"),
    ("v_bits", 8, "KVQ_ERR_UNSUPPORTED"),
    ("group_size", 64, "KVQ_ERR_UNSUPPORTED"),
    ("residual_len", 100, "KVQ_ERR_ARG"),
    ("residual_len", -32, "KVQ_ERR_ARG"),
    ("q_heads", 12, "KVQ_ERR_SHAPE"),
    ("q_heads", 144, "KVQ_ERR_UNSUPPORTED"),
    ("batch", 0, "KVQ_ERR_ARG"),
    ("max_tokens", 0, "KVQ_ERR_ARG"),
])
def test_bad_config(field, value, code):
    cfg = kvq.make_config(2, 8, 64, 128, 2, 2, 128, 1024)
    setattr(cfg, field, value)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_cache_sizes(cfg)
    assert e.value.name == code
    assert kvq.kv_decode_workspace_bytes(cfg) == 0


def _fake_cache(n_grouped=0, n_resid=0, **kw):
    args = dict(batch=2, kv_heads=2, q_heads=4, head_dim=64, k_bits=2, v_bits=2, residual_len=128, max_tokens=512)
    args.update(kw)
    cfg = kvq.make_config(**args)
    cache = kvq.kivi_cache_init(cfg, [ALIGNED * (i + 1) for i in range(6)])
    cache.n_grouped, cache.n_resid = n_grouped, n_resid
    return cfg, cache


def test_init_checks_pointers():
    cfg = kvq.make_config(2, 2, 4, 64, 2, 2, 128, 512)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_cache_init(cfg, [ALIGNED, ALIGNED, None, ALIGNED, ALIGNED, ALIGNED])
    assert e.value.name == "KVQ_ERR_NULL"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_cache_init(cfg, [ALIGNED, ALIGNED + 16, ALIGNED, ALIGNED, ALIGNED, ALIGNED])
    assert e.value.name == "KVQ_ERR_ALIGN"
    _, cache = _fake_cache()
    assert (cache.groups_cap, cache.res_cap, cache.n_grouped, cache.n_resid) == (16, 128, 0, 0)
    _, c0 = _fake_cache(residual_len=0)
    assert c0.res_cap == 32


def _snapshot(cache):
    return (cache.n_grouped, cache.n_resid, cache.k_codes, cache.v_res)


def test_prefill_validation_leaves_state():
    _, cache = _fake_cache(64, 10)
    before = _snapshot(cache)
    for args, code in [((ALIGNED, ALIGNED, 513), "KVQ_ERR_CAPACITY"),
                       ((ALIGNED, ALIGNED, -1), "KVQ_ERR_ARG"),
                       ((None, ALIGNED, 10), "KVQ_ERR_NULL"),
                       ((ALIGNED + 2, ALIGNED, 10), "KVQ_ERR_ALIGN")]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.kv_quant_prefill(cache, *args, stream=0)
        assert e.value.name == code
        assert _snapshot(cache) == before


def test_append_capacity_and_state():
    _, cache = _fake_cache(384, 128)   # 512 tokens = max_tokens
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_append_token(cache, ALIGNED, ALIGNED, stream=0)
    assert e.value.name == "KVQ_ERR_CAPACITY"
    assert (cache.n_grouped, cache.n_resid) == (384, 128)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_append_token(cache, None, ALIGNED, stream=0)
    assert e.value.name == "KVQ_ERR_NULL"


def test_corrupt_descriptor_is_rejected():
    _, cache = _fake_cache(40, 0)       # not a multiple of 32
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_flush_residual(cache, stream=0)
    assert e.value.name == "KVQ_ERR_ARG"
    _, cache = _fake_cache(0, 129)      # window over capacity
    with pytest.raises(kvq.KvqError):
        kvq.kv_append_token(cache, ALIGNED, ALIGNED, stream=0)


def test_flush_noop_when_window_short():
    _, cache = _fake_cache(64, 31)
    kvq.kv_flush_residual(cache, stream=0)   # fewer than 32 tokens: nothing to do, no launch
    assert (cache.n_grouped, cache.n_resid) == (64, 31)


def test_decode_validation():
    cfg, cache = _fake_cache(0, 0)
    ws = kvq.kv_decode_workspace_bytes(cfg)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention(cache, ALIGNED, ALIGNED, True, 0.0, ALIGNED, ws, stream=0)
    assert e.value.name == "KVQ_ERR_ARG"                  # empty cache
    _, cache = _fake_cache(64, 3)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention(cache, ALIGNED, ALIGNED, True, 0.0, ALIGNED, ws - 1, stream=0)
    assert e.value.name == "KVQ_ERR_WORKSPACE"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention(cache, ALIGNED, ALIGNED, True, 0.0, None, ws, stream=0)
    assert e.value.name == "KVQ_ERR_WORKSPACE"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention(cache, ALIGNED, ALIGNED, True, float("nan"), ALIGNED, ws, stream=0)
    assert e.value.name == "KVQ_ERR_ARG"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention(cache, ALIGNED + 8, ALIGNED, True, 0.0, ALIGNED, ws, stream=0)
    assert e.value.name == "KVQ_ERR_ALIGN"


def test_fp8_validation():
    """Host-side checks of the FP8 calls: pool descriptors (role, format, scale
    granularity, shape), capacity, workspace, alignment; the decode refuses
    swapped or mismatched pools with KVQ_ERR_ARG."""
    assert kvq.fp8_pool_bytes(6, 2, 128) == 6 * 2 * 16 * 128 and kvq.fp8_pool_bytes(6, 2, 96) == 0
    for args, code in [((2, 0, 0, 6, 2, 128), "KVQ_ERR_ARG"), ((0, 2, 0, 6, 2, 128), "KVQ_ERR_ARG"),
                       ((0, 0, 2, 6, 2, 128), "KVQ_ERR_ARG"), ((0, 0, 0, 0, 2, 128), "KVQ_ERR_ARG"),
                       ((0, 0, 0, 6, 2, 96), "KVQ_ERR_UNSUPPORTED")]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.fp8_pool_init(*args, ALIGNED, ALIGNED * 2)
        assert e.value.name == code, args
    with pytest.raises(kvq.KvqError) as e:
        kvq.fp8_pool_init(kvq.ROLE_KEY, 0, 0, 6, 2, 128, ALIGNED, ALIGNED + 4)
    assert e.value.name == "KVQ_ERR_ALIGN"
    k = kvq.fp8_pool_init(kvq.ROLE_KEY, 0, 0, 6, 2, 128, ALIGNED, ALIGNED * 2)
    v = kvq.fp8_pool_init(kvq.ROLE_VALUE, 0, 0, 6, 2, 128, ALIGNED * 3, ALIGNED * 4)
    q = dict(x=ALIGNED, batch=2, seq_len=40, block_table=ALIGNED, max_blocks=3, static_scale=False, ws=ALIGNED,
             ws_bytes=kvq.fp8_quantize_workspace_bytes(2, 2, 40, 128))
    for change, code in [(dict(max_blocks=2), "KVQ_ERR_CAPACITY"), (dict(ws_bytes=8), "KVQ_ERR_WORKSPACE"),
                         (dict(x=None), "KVQ_ERR_NULL"), (dict(block_table=ALIGNED + 4), "KVQ_ERR_ALIGN"),
                         (dict(seq_len=0), "KVQ_ERR_ARG")]:
        args = dict(q, **change)
        with pytest.raises(kvq.KvqError) as e:
            kvq.fp8_kv_quantize(k, **args, stream=0)
        assert e.value.name == code, change
    d = dict(q=ALIGNED, block_table=ALIGNED, seq_lens=ALIGNED, batch=2, q_heads=8, max_blocks=3, max_seq_len=40,
             out=ALIGNED, out_fp32=True, softmax_scale=0.0, ws=ALIGNED, ws_bytes=kvq.fp8_decode_workspace_bytes(2, 8, 128))

    def dec(kk, vv, **change):
        args = dict(d, **change)
        qq = args.pop("q")
        with pytest.raises(kvq.KvqError) as e:
            kvq.fp8_decode_attention(qq, kk, vv, **args, stream=0)
        return e.value.name

    for change, code in [(dict(q_heads=7), "KVQ_ERR_SHAPE"), (dict(max_seq_len=49), "KVQ_ERR_CAPACITY"),
                         (dict(q_heads=32), "KVQ_ERR_UNSUPPORTED"), (dict(ws_bytes=100), "KVQ_ERR_WORKSPACE"),
                         (dict(seq_lens=None), "KVQ_ERR_NULL"), (dict(q_fp8=2), "KVQ_ERR_ARG"),
                         (dict(ws_bytes=kvq.kv_decode_workspace_bytes(kvq.make_config(2, 8, 8, 128, 2, 2, 128, 32))),
                          "KVQ_ERR_WORKSPACE")]:
        assert dec(k, v, **change) == code, change
    assert dec(v, k) == "KVQ_ERR_ARG"                        # roles swapped
    assert dec(k, k) == "KVQ_ERR_ARG"
    v5 = kvq.fp8_pool_init(kvq.ROLE_VALUE, 1, 0, 6, 2, 128, ALIGNED * 3, ALIGNED * 4)
    assert dec(k, v5) == "KVQ_ERR_ARG"                       # formats differ
    vph = kvq.fp8_pool_init(kvq.ROLE_VALUE, 0, 1, 6, 2, 128, ALIGNED * 3, ALIGNED * 4)
    assert dec(k, vph) == "KVQ_ERR_ARG"                      # scale granularities differ
    v7 = kvq.fp8_pool_init(kvq.ROLE_VALUE, 0, 0, 7, 2, 128, ALIGNED * 3, ALIGNED * 4)
    assert dec(k, v7) == "KVQ_ERR_SHAPE"


# ---------------------------------------------------------------------------
# paged, variable-length cache
# ---------------------------------------------------------------------------

PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "kvq.h"
#define F(T, m) printf("%s.%s %zu\n", #T, #m, offsetof(T, m));
int main(void) {
  printf("kivi_config %zu\n", sizeof(kivi_config));
  printf("kivi_cache %zu\n", sizeof(kivi_cache));
  printf("kivi_paged_config %zu\n", sizeof(kivi_paged_config));
  printf("kivi_paged_cache %zu\n", sizeof(kivi_paged_cache));
  printf("nvfp4_pool %zu\n", sizeof(nvfp4_pool));
  printf("fp8_pool %zu\n", sizeof(fp8_pool));
  F(fp8_pool, role) F(fp8_pool, fp8_format) F(fp8_pool, per_head) F(fp8_pool, head_dim) F(fp8_pool, pool)
  F(fp8_pool, scale)
  F(nvfp4_pool, role) F(nvfp4_pool, head_dim) F(nvfp4_pool, pool) F(nvfp4_pool, tensor_scale)
  printf("KVQ_ROLE_KEY %d\n", KVQ_ROLE_KEY);
  printf("KVQ_ROLE_VALUE %d\n", KVQ_ROLE_VALUE);
  F(kivi_cache, k_codes) F(kivi_cache, v_res) F(kivi_cache, groups_cap) F(kivi_cache, n_resid)
  F(kivi_paged_config, num_blocks)
  F(kivi_paged_cache, pool) F(kivi_paged_cache, v_res) F(kivi_paged_cache, block_table)
  F(kivi_paged_cache, groups_cap) F(kivi_paged_cache, res_cap) F(kivi_paged_cache, n_grouped)
  F(kivi_paged_cache, n_resid)
  printf("KVQ_PAGED_MAX_SEQS %d\n", KVQ_PAGED_MAX_SEQS);
  return 0;
}
"""


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes descriptors have the sizes and field offsets a C compiler
    gives the header's structs."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src, exe = tmp_path / "probe.c", tmp_path / "probe"
    src.write_text(PROBE)
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                       text=True).stdout.splitlines())
    want = {"kivi_config": ctypes.sizeof(kvq.kivi_config), "kivi_cache": ctypes.sizeof(kvq.kivi_cache),
            "kivi_paged_config": ctypes.sizeof(kvq.kivi_paged_config),
            "kivi_paged_cache": ctypes.sizeof(kvq.kivi_paged_cache), "KVQ_PAGED_MAX_SEQS": kvq.PAGED_MAX_SEQS,
            "nvfp4_pool": ctypes.sizeof(kvq.nvfp4_pool), "fp8_pool": ctypes.sizeof(kvq.fp8_pool),
            "KVQ_ROLE_KEY": kvq.ROLE_KEY,
            "KVQ_ROLE_VALUE": kvq.ROLE_VALUE}
    for key, val in got.items():
        if "." in key:
            t, m = key.split(".")
            want[key] = getattr(getattr(kvq, t), m).offset
        assert int(val) == want[key], key


def _pcfg(batch=3, num_blocks=40, **kw):
    args = dict(batch=batch, kv_heads=2, q_heads=4, head_dim=64, k_bits=2, v_bits=2, residual_len=128,
                max_tokens=512)
    args.update(kw)
    return kvq.kivi_paged_config(kvq.make_config(**args), num_blocks)


def _fake_paged(grouped=(), resid=(), **kw):
    pcfg = _pcfg(**kw)
    cache = kvq.kivi_paged_cache_init(pcfg, [ALIGNED * (i + 1) for i in range(3)], ALIGNED * 8)
    for b, n in enumerate(grouped):
        cache.n_grouped[b] = n
    for b, n in enumerate(resid):
        cache.n_resid[b] = n
    return pcfg, cache


def _pstate(cache, n):
    return [(cache.n_grouped[b], cache.n_resid[b]) for b in range(n)]


@pytest.mark.parametrize("b,h,d,kb,vb,r,t,nb", [(3, 2, 64, 2, 2, 128, 512, 40), (256, 8, 128, 4, 2, 0, 100, 7),
                                                (5, 3, 128, 2, 4, 64, 4097, 1)])
def test_paged_sizes_match_layout(b, h, d, kb, vb, r, t, nb):
    from oracle import paged
    pcfg = kvq.kivi_paged_config(kvq.make_config(b, h, 2 * h, d, kb, vb, r, t), nb)
    got = kvq.kivi_paged_cache_sizes(pcfg)
    rec = paged.PagedKiviCache(1, h, d, kb, vb, r, nb, np.zeros((1, 1), np.int32)).record_bytes()
    res_cap = r if r > 0 else 32
    want = [nb * h * sum(rec.values())] + [b * h * res_cap * d * 2] * 2
    assert got == want
    assert kvq.kv_paged_decode_workspace_bytes(pcfg) == kvq.kv_decode_workspace_bytes(pcfg.cfg)


def test_paged_config_limits():
    for pcfg, code in [(_pcfg(batch=257), "KVQ_ERR_UNSUPPORTED"), (_pcfg(num_blocks=0), "KVQ_ERR_ARG"),
                       (_pcfg(head_dim=96), "KVQ_ERR_UNSUPPORTED"), (_pcfg(q_heads=3), "KVQ_ERR_SHAPE")]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.kivi_paged_cache_sizes(pcfg)
        assert e.value.name == code
        assert kvq.kv_paged_decode_workspace_bytes(pcfg) == 0
    kvq.kivi_paged_cache_sizes(_pcfg(batch=256))


def test_paged_init_checks_pointers():
    pcfg = _pcfg()
    bufs = [ALIGNED] * 3
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_paged_cache_init(pcfg, bufs, None)
    assert e.value.name == "KVQ_ERR_NULL"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_paged_cache_init(pcfg, bufs, ALIGNED + 4)
    assert e.value.name == "KVQ_ERR_ALIGN"
    with pytest.raises(kvq.KvqError) as e:
        kvq.kivi_paged_cache_init(pcfg, [ALIGNED] * 2 + [None], ALIGNED)
    assert e.value.name == "KVQ_ERR_NULL"
    _, cache = _fake_paged()
    assert (cache.groups_cap, cache.res_cap, cache.pcfg.num_blocks) == (16, 128, 40)
    assert _pstate(cache, 3) == [(0, 0)] * 3


def test_paged_prefill_validation_leaves_state():
    _, cache = _fake_paged((64, 0, 32), (10, 5, 128))
    before = _pstate(cache, 3)
    for args, code in [((ALIGNED, ALIGNED, 100, [10, 101, 0]), "KVQ_ERR_ARG"),
                       ((ALIGNED, ALIGNED, 600, [10, 513, 0]), "KVQ_ERR_CAPACITY"),
                       ((ALIGNED, ALIGNED, 100, [10, -1, 0]), "KVQ_ERR_ARG"),
                       ((None, ALIGNED, 100, [10, 1, 0]), "KVQ_ERR_NULL"),
                       ((ALIGNED + 2, ALIGNED, 100, [10, 1, 0]), "KVQ_ERR_ALIGN")]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.kv_paged_prefill(cache, *args, stream=0)
        assert e.value.name == code
        assert _pstate(cache, 3) == before


def test_paged_prefill_of_empty_sequences_launches_nothing():
    """Zero tokens everywhere: no pointer is needed, nothing is enqueued, every
    sequence is emptied."""
    _, cache = _fake_paged((64, 0, 32), (10, 5, 128))
    kvq.kv_paged_prefill(cache, None, None, 0, [0, 0, 0], stream=0)
    assert _pstate(cache, 3) == [(0, 0)] * 3


def test_paged_append_capacity_and_state():
    _, cache = _fake_paged((0, 384, 32), (3, 128, 0))   # sequence 1 holds max_tokens
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_paged_append(cache, ALIGNED, ALIGNED, stream=0)
    assert e.value.name == "KVQ_ERR_CAPACITY"
    assert _pstate(cache, 3) == [(0, 3), (384, 128), (32, 0)]
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_paged_append(cache, ALIGNED, None, stream=0)
    assert e.value.name == "KVQ_ERR_NULL"


def test_paged_corrupt_descriptor_is_rejected():
    for grouped, resid in [((40, 0, 0), (0, 0, 0)), ((0, 0, 0), (0, 129, 0)), ((0, 0, -32), (0, 0, 0)),
                           ((512, 0, 0), (1, 0, 0))]:
        _, cache = _fake_paged(grouped, resid)
        with pytest.raises(kvq.KvqError) as e:
            kvq.kv_paged_flush(cache, stream=0)
        assert e.value.name == "KVQ_ERR_ARG"
    _, cache = _fake_paged((0, 0, 0), (0, 32, 0), residual_len=0)  # an R = 0 stage is never left full
    with pytest.raises(kvq.KvqError):
        kvq.kv_paged_flush(cache, stream=0)


def test_paged_flush_noop_when_windows_short():
    _, cache = _fake_paged((64, 0, 32), (31, 0, 5))
    kvq.kv_paged_flush(cache, stream=0)
    assert _pstate(cache, 3) == [(64, 31), (0, 0), (32, 5)]


def test_paged_decode_validation():
    pcfg, cache = _fake_paged((64, 0, 32), (3, 1, 0))
    ws = kvq.kv_paged_decode_workspace_bytes(pcfg)
    for args, code in [((ALIGNED, ALIGNED, True, 0.0, ALIGNED, ws - 1), "KVQ_ERR_WORKSPACE"),
                       ((ALIGNED, ALIGNED, True, 0.0, None, ws), "KVQ_ERR_WORKSPACE"),
                       ((ALIGNED, ALIGNED, True, float("inf"), ALIGNED, ws), "KVQ_ERR_ARG"),
                       ((ALIGNED, None, True, 0.0, ALIGNED, ws), "KVQ_ERR_NULL"),
                       ((ALIGNED + 64, ALIGNED, True, 0.0, ALIGNED, ws), "KVQ_ERR_ALIGN")]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.kv_paged_decode_attention(cache, *args, stream=0)
        assert e.value.name == code
    _, cache = _fake_paged((64, 0, 32), (3, 0, 0))         # sequence 1 is empty
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_paged_decode_attention(cache, ALIGNED, ALIGNED, True, 0.0, ALIGNED, ws, stream=0)
    assert e.value.name == "KVQ_ERR_ARG"


def test_fp8_decode_workspace_holds_the_query():
    """The FP8 decode workspace is the split-K layout followed by the E4M3 query
    (rounded to 256 bytes), its scale slot and 1 KiB of amax partials."""
    for b, hq, d in [(2, 8, 128), (64, 32, 128), (3, 5, 64)]:
        base = kvq.kv_decode_workspace_bytes(kvq.make_config(b, hq, hq, d, 2, 2, 128, 32))
        assert kvq.fp8_decode_workspace_bytes(b, hq, d) == base + -(-b * hq * d // 256) * 256 + 256 + 1024


def test_nvfp4_validation():
    """Host-side checks of the NVFP4 calls: roles, shapes, alignment, workspace;
    the decode refuses a value pool given as keys (and the reverse)."""
    assert kvq.nvfp4_pool_bytes(10, 8, 128) == 10 * 8 * 9 * 128
    assert kvq.nvfp4_pool_bytes(10, 8, 96) == 0
    with pytest.raises(kvq.KvqError) as e:
        kvq.nvfp4_pool_init(2, 4, 2, 128, ALIGNED, ALIGNED * 2)
    assert e.value.name == "KVQ_ERR_ARG"
    with pytest.raises(kvq.KvqError) as e:
        kvq.nvfp4_pool_init(kvq.ROLE_KEY, 4, 2, 96, ALIGNED, ALIGNED * 2)
    assert e.value.name == "KVQ_ERR_UNSUPPORTED"
    with pytest.raises(kvq.KvqError) as e:
        kvq.nvfp4_pool_init(kvq.ROLE_KEY, 4, 2, 128, ALIGNED + 16, ALIGNED * 2)
    assert e.value.name == "KVQ_ERR_ALIGN"
    k = kvq.nvfp4_pool_init(kvq.ROLE_KEY, 4, 2, 128, ALIGNED, ALIGNED * 2)
    v = kvq.nvfp4_pool_init(kvq.ROLE_VALUE, 4, 2, 128, ALIGNED * 3, ALIGNED * 4)
    wsb = kvq.nvfp4_decode_workspace_bytes(2, 4, 128)

    def dec(kk, vv, **kw):
        args = dict(q=ALIGNED * 5, block_table=ALIGNED * 6, seq_lens=ALIGNED * 7, batch=2, q_heads=4, max_blocks=2,
                    max_seq_len=32, out=ALIGNED * 8, out_fp32=True, softmax_scale=0.0, ws=ALIGNED * 9, ws_bytes=wsb)
        args.update(kw)
        with pytest.raises(kvq.KvqError) as e:
            kvq.nvfp4_decode_attention(args["q"], kk, vv, args["block_table"], args["seq_lens"], args["batch"],
                                       args["q_heads"], args["max_blocks"], args["max_seq_len"], args["out"],
                                       args["out_fp32"], args["softmax_scale"], args["ws"], args["ws_bytes"], stream=0)
        return e.value.name

    assert dec(v, k) == "KVQ_ERR_ARG"          # roles swapped
    assert dec(k, k) == "KVQ_ERR_ARG"
    v2 = kvq.nvfp4_pool_init(kvq.ROLE_VALUE, 5, 2, 128, ALIGNED * 3, ALIGNED * 4)
    assert dec(k, v2) == "KVQ_ERR_SHAPE"
    assert dec(k, v, q_heads=3) == "KVQ_ERR_SHAPE"
    assert dec(k, v, q_heads=18) == "KVQ_ERR_UNSUPPORTED"
    assert dec(k, v, max_seq_len=33) == "KVQ_ERR_CAPACITY"
    assert dec(k, v, ws_bytes=wsb - 1) == "KVQ_ERR_WORKSPACE"
    assert dec(k, v, out=ALIGNED + 4) == "KVQ_ERR_ALIGN"

    def quant(pool, **kw):
        args = dict(x=ALIGNED * 5, batch=2, seq_len=40, block_table=ALIGNED * 6, max_blocks=3, static_scale=False,
                    ws=ALIGNED * 7, ws_bytes=kvq.nvfp4_quantize_workspace_bytes())
        args.update(kw)
        with pytest.raises(kvq.KvqError) as e:
            kvq.nvfp4_kv_quantize(pool, args["x"], args["batch"], args["seq_len"], args["block_table"],
                                  args["max_blocks"], args["static_scale"], args["ws"], args["ws_bytes"], stream=0)
        return e.value.name

    assert quant(k, max_blocks=2) == "KVQ_ERR_CAPACITY"
    assert quant(k, ws=None) == "KVQ_ERR_WORKSPACE"
    assert quant(k, ws_bytes=16) == "KVQ_ERR_WORKSPACE"
    assert quant(k, x=None) == "KVQ_ERR_NULL"
    assert quant(k, seq_len=0) == "KVQ_ERR_ARG"


def test_noalloc_status_needs_a_host_word():
    # the pointer check comes before any device access
    assert kvq._lib.kv_decode_noalloc_status(None, 0, None) == 1
