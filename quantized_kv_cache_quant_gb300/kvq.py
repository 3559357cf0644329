"""Python binding of libkvq (the C ABI declared in include/kvq.h).

Argument marshalling only: every function here forwards to the C function of
the same name through ctypes; all work runs in the library's CUDA kernels.
PyTorch supplies device memory and the current CUDA stream. Importing this
module raises ImportError when the library has not been built — there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libkvq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libkvq.so not found at {LIB_PATH}; build it with "
        "`python -m quantized_kv_cache_quant_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

c_i32, c_sz, c_vp, c_f32 = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float

EXPORTED = (
    "kvq_status_string", "kivi_cache_sizes", "kivi_cache_init", "kv_quant_prefill", "kv_append_token",
    "kv_flush_residual", "kv_decode_workspace_bytes", "kv_decode_attention", "kv_decode_attention_noalloc",
    "kv_decode_noalloc_status", "kivi_paged_cache_sizes", "kivi_paged_cache_init", "kv_paged_prefill", "kv_paged_append", "kv_paged_flush",
    "kv_paged_decode_workspace_bytes", "kv_paged_decode_attention",
    "fp8_pool_bytes", "fp8_pool_init", "fp8_quantize_workspace_bytes",
    "fp8_kv_quantize", "fp8_decode_workspace_bytes", "fp8_decode_attention",
    "nvfp4_pool_bytes", "nvfp4_pool_init", "nvfp4_quantize_workspace_bytes", "nvfp4_kv_quantize",
    "nvfp4_decode_workspace_bytes", "nvfp4_decode_attention",
)

STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_NULL", 2: "KVQ_ERR_ARG", 3: "KVQ_ERR_SHAPE", 4: "KVQ_ERR_CAPACITY",
          5: "KVQ_ERR_WORKSPACE", 6: "KVQ_ERR_UNSUPPORTED", 7: "KVQ_ERR_CUDA", 8: "KVQ_ERR_TIMEOUT",
          9: "KVQ_ERR_ALIGN"}
WS_STATUS_TIMEOUT = 1


class KvqError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({_lib.kvq_status_string(code).decode()})")


class kivi_config(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("batch", "kv_heads", "q_heads", "head_dim", "k_bits", "v_bits",
                                    "group_size", "residual_len", "max_tokens")]


class kivi_cache(ctypes.Structure):
    _fields_ = [("cfg", kivi_config), ("k_codes", c_vp), ("k_meta", c_vp), ("v_codes", c_vp), ("v_meta", c_vp),
                ("k_res", c_vp), ("v_res", c_vp), ("groups_cap", c_i32), ("res_cap", c_i32),
                ("n_grouped", c_i32), ("n_resid", c_i32)]


PAGED_MAX_SEQS = 256


class kivi_paged_config(ctypes.Structure):
    _fields_ = [("cfg", kivi_config), ("num_blocks", c_i32)]


class kivi_paged_cache(ctypes.Structure):
    _fields_ = [("pcfg", kivi_paged_config), ("pool", c_vp), ("k_res", c_vp), ("v_res", c_vp), ("block_table", c_vp),
                ("groups_cap", c_i32), ("res_cap", c_i32),
                ("n_grouped", c_i32 * PAGED_MAX_SEQS), ("n_resid", c_i32 * PAGED_MAX_SEQS)]


ROLE_KEY, ROLE_VALUE = 0, 1


class nvfp4_pool(ctypes.Structure):
    _fields_ = [("role", c_i32), ("num_blocks", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32), ("pool", c_vp),
                ("tensor_scale", c_vp)]


class fp8_pool(ctypes.Structure):
    _fields_ = [("role", c_i32), ("fp8_format", c_i32), ("per_head", c_i32), ("num_blocks", c_i32),
                ("kv_heads", c_i32), ("head_dim", c_i32), ("pool", c_vp), ("scale", c_vp)]


_P_NV = ctypes.POINTER(nvfp4_pool)
_P_F8 = ctypes.POINTER(fp8_pool)
_P_CFG, _P_CACHE = ctypes.POINTER(kivi_config), ctypes.POINTER(kivi_cache)
_P_PCFG, _P_PCACHE = ctypes.POINTER(kivi_paged_config), ctypes.POINTER(kivi_paged_cache)
_SIG = {
    "kvq_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "kivi_cache_sizes": ([_P_CFG, ctypes.POINTER(c_sz)], ctypes.c_int),
    "kivi_cache_init": ([_P_CACHE, _P_CFG, ctypes.POINTER(c_vp)], ctypes.c_int),
    "kv_quant_prefill": ([_P_CACHE, c_vp, c_vp, c_i32, c_vp], ctypes.c_int),
    "kv_append_token": ([_P_CACHE, c_vp, c_vp, c_vp], ctypes.c_int),
    "kv_flush_residual": ([_P_CACHE, c_vp], ctypes.c_int),
    "kv_decode_workspace_bytes": ([_P_CFG], c_sz),
    "kv_decode_attention": ([_P_CACHE, c_vp, c_vp, c_i32, c_f32, c_vp, c_sz, c_vp], ctypes.c_int),
    "kv_decode_attention_noalloc": ([_P_CACHE, c_vp, c_vp, c_i32, c_f32, c_vp], ctypes.c_int),
    "kv_decode_noalloc_status": ([ctypes.POINTER(ctypes.c_uint32), c_i32, c_vp], ctypes.c_int),
    "kivi_paged_cache_sizes": ([_P_PCFG, ctypes.POINTER(c_sz)], ctypes.c_int),
    "kivi_paged_cache_init": ([_P_PCACHE, _P_PCFG, ctypes.POINTER(c_vp), c_vp], ctypes.c_int),
    "kv_paged_prefill": ([_P_PCACHE, c_vp, c_vp, c_i32, ctypes.POINTER(c_i32), c_vp], ctypes.c_int),
    "kv_paged_append": ([_P_PCACHE, c_vp, c_vp, c_vp], ctypes.c_int),
    "kv_paged_flush": ([_P_PCACHE, c_vp], ctypes.c_int),
    "kv_paged_decode_workspace_bytes": ([_P_PCFG], c_sz),
    "kv_paged_decode_attention": ([_P_PCACHE, c_vp, c_vp, c_i32, c_f32, c_vp, c_sz, c_vp], ctypes.c_int),
    "fp8_pool_bytes": ([c_i32, c_i32, c_i32], c_sz),
    "fp8_pool_init": ([_P_F8, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp], ctypes.c_int),
    "fp8_quantize_workspace_bytes": ([c_i32, c_i32, c_i32, c_i32], c_sz),
    "fp8_kv_quantize": ([_P_F8, c_vp, c_i32, c_i32, c_vp, c_i32, c_i32, c_vp, c_sz, c_vp], ctypes.c_int),
    "fp8_decode_workspace_bytes": ([c_i32, c_i32, c_i32], c_sz),
    "fp8_decode_attention": ([c_vp, _P_F8, _P_F8, c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_i32, c_f32,
                              c_vp, c_sz, c_vp], ctypes.c_int),
    "nvfp4_pool_bytes": ([c_i32, c_i32, c_i32], c_sz),
    "nvfp4_pool_init": ([_P_NV, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp], ctypes.c_int),
    "nvfp4_quantize_workspace_bytes": ([], c_sz),
    "nvfp4_kv_quantize": ([_P_NV, c_vp, c_i32, c_i32, c_vp, c_i32, c_i32, c_vp, c_sz, c_vp], ctypes.c_int),
    "nvfp4_decode_workspace_bytes": ([c_i32, c_i32, c_i32], c_sz),
    "nvfp4_decode_attention": ([c_vp, _P_NV, _P_NV, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_i32, c_f32, c_vp,
                                c_sz, c_vp], ctypes.c_int),
}
for _name, (_args, _res) in _SIG.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def _ptr(x) -> Optional[int]:
    """A device/host address from a torch tensor, an int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != 0:
        raise KvqError(code, where)


# ---------------------------------------------------------------------------
# thin wrappers, same names as the C ABI
# ---------------------------------------------------------------------------

def kvq_status_string(code: int) -> str:
    return _lib.kvq_status_string(code).decode()


def make_config(batch, kv_heads, q_heads, head_dim, k_bits=2, v_bits=2, residual_len=128, max_tokens=0,
                group_size=32) -> kivi_config:
    return kivi_config(batch, kv_heads, q_heads, head_dim, k_bits, v_bits, group_size, residual_len, max_tokens)


def kivi_cache_sizes(cfg: kivi_config) -> list:
    out = (c_sz * 6)()
    _check(_lib.kivi_cache_sizes(ctypes.byref(cfg), out), "kivi_cache_sizes")
    return list(out)


def kivi_cache_init(cfg: kivi_config, bufs: Sequence) -> kivi_cache:
    cache = kivi_cache()
    arr = (c_vp * 6)(*[_ptr(b) for b in bufs])
    _check(_lib.kivi_cache_init(ctypes.byref(cache), ctypes.byref(cfg), arr), "kivi_cache_init")
    return cache


def kv_quant_prefill(cache: kivi_cache, k, v, seq_len: int, stream=None) -> None:
    _check(_lib.kv_quant_prefill(ctypes.byref(cache), _ptr(k), _ptr(v), seq_len, _stream(stream)), "kv_quant_prefill")


def kv_append_token(cache: kivi_cache, k_new, v_new, stream=None) -> None:
    _check(_lib.kv_append_token(ctypes.byref(cache), _ptr(k_new), _ptr(v_new), _stream(stream)), "kv_append_token")


def kv_flush_residual(cache: kivi_cache, stream=None) -> None:
    _check(_lib.kv_flush_residual(ctypes.byref(cache), _stream(stream)), "kv_flush_residual")


def kv_decode_workspace_bytes(cfg: kivi_config) -> int:
    return int(_lib.kv_decode_workspace_bytes(ctypes.byref(cfg)))


def kv_decode_attention(cache: kivi_cache, q, out, out_fp32: bool, softmax_scale: float, ws, ws_bytes: int,
                        stream=None) -> None:
    _check(_lib.kv_decode_attention(ctypes.byref(cache), _ptr(q), _ptr(out), int(bool(out_fp32)),
                                    float(softmax_scale), _ptr(ws), ws_bytes, _stream(stream)),
           "kv_decode_attention")


def kv_decode_attention_noalloc(cache: kivi_cache, q, out, out_fp32: bool, softmax_scale: float,
                                stream=None) -> None:
    """kv_decode_attention without a workspace, for callers that cannot allocate
    device memory: the scratch is a fixed device array inside the library."""
    _check(_lib.kv_decode_attention_noalloc(ctypes.byref(cache), _ptr(q), _ptr(out), int(bool(out_fp32)),
                                            float(softmax_scale), _stream(stream)), "kv_decode_attention_noalloc")


def kv_decode_noalloc_status(clear: bool = False, stream=None) -> int:
    """The status word of kv_decode_attention_noalloc's scratch array on the
    current device (bit 0: a device wait timed out); waits for `stream`.
    Returns the word; KVQ_ERR_TIMEOUT is reported through the word, not raised."""
    word = ctypes.c_uint32(0)
    code = _lib.kv_decode_noalloc_status(ctypes.byref(word), int(bool(clear)), _stream(stream))
    if code not in (0, 8):
        raise KvqError(code, "kv_decode_noalloc_status")
    return int(word.value)


def kivi_paged_cache_sizes(pcfg: kivi_paged_config) -> list:
    out = (c_sz * 3)()
    _check(_lib.kivi_paged_cache_sizes(ctypes.byref(pcfg), out), "kivi_paged_cache_sizes")
    return list(out)


def kivi_paged_cache_init(pcfg: kivi_paged_config, bufs: Sequence, block_table) -> kivi_paged_cache:
    cache = kivi_paged_cache()
    arr = (c_vp * 3)(*[_ptr(b) for b in bufs])
    _check(_lib.kivi_paged_cache_init(ctypes.byref(cache), ctypes.byref(pcfg), arr, _ptr(block_table)),
           "kivi_paged_cache_init")
    return cache


def kv_paged_prefill(cache: kivi_paged_cache, k, v, max_seq_len: int, seq_lens: Sequence[int], stream=None) -> None:
    lens = (c_i32 * len(seq_lens))(*[int(x) for x in seq_lens])
    _check(_lib.kv_paged_prefill(ctypes.byref(cache), _ptr(k), _ptr(v), max_seq_len, lens, _stream(stream)),
           "kv_paged_prefill")


def kv_paged_append(cache: kivi_paged_cache, k_new, v_new, stream=None) -> None:
    _check(_lib.kv_paged_append(ctypes.byref(cache), _ptr(k_new), _ptr(v_new), _stream(stream)), "kv_paged_append")


def kv_paged_flush(cache: kivi_paged_cache, stream=None) -> None:
    _check(_lib.kv_paged_flush(ctypes.byref(cache), _stream(stream)), "kv_paged_flush")


def kv_paged_decode_workspace_bytes(pcfg: kivi_paged_config) -> int:
    return int(_lib.kv_paged_decode_workspace_bytes(ctypes.byref(pcfg)))


def kv_paged_decode_attention(cache: kivi_paged_cache, q, out, out_fp32: bool, softmax_scale: float, ws,
                              ws_bytes: int, stream=None) -> None:
    _check(_lib.kv_paged_decode_attention(ctypes.byref(cache), _ptr(q), _ptr(out), int(bool(out_fp32)),
                                          float(softmax_scale), _ptr(ws), ws_bytes, _stream(stream)),
           "kv_paged_decode_attention")


def fp8_pool_bytes(num_blocks, kv_heads, head_dim) -> int:
    return int(_lib.fp8_pool_bytes(num_blocks, kv_heads, head_dim))


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def fp8_pool_init(role: int, fp8_format: int, per_head: bool, num_blocks: int, kv_heads: int, head_dim: int, buf,
                  scale) -> fp8_pool:
    desc = fp8_pool()
    _check(_lib.fp8_pool_init(ctypes.byref(desc), role, int(fp8_format), int(per_head), num_blocks, kv_heads,
                              head_dim, _ptr(buf), _ptr(scale)), "fp8_pool_init")
    return desc


def fp8_quantize_workspace_bytes(batch, kv_heads, seq_len, head_dim) -> int:
    return int(_lib.fp8_quantize_workspace_bytes(batch, kv_heads, seq_len, head_dim))


def fp8_kv_quantize(pool: fp8_pool, x, batch, seq_len, block_table, max_blocks, static_scale: bool, ws,
                    ws_bytes: int, stream=None) -> None:
    _check(_lib.fp8_kv_quantize(ctypes.byref(pool), _ptr(x), batch, seq_len, _ptr(block_table), max_blocks,
                                int(bool(static_scale)), _ptr(ws), ws_bytes, _stream(stream)), "fp8_kv_quantize")


def fp8_decode_workspace_bytes(batch, q_heads, head_dim) -> int:
    return int(_lib.fp8_decode_workspace_bytes(batch, q_heads, head_dim))


def fp8_decode_attention(q, k: fp8_pool, v: fp8_pool, block_table, seq_lens, batch, q_heads, max_blocks,
                         max_seq_len, out, out_fp32: bool, softmax_scale: float, ws, ws_bytes: int, stream=None,
                         q_fp8: bool = False) -> None:
    _check(_lib.fp8_decode_attention(_ptr(q), ctypes.byref(k), ctypes.byref(v), int(q_fp8), _ptr(block_table),
                                     _ptr(seq_lens), batch, q_heads, max_blocks, max_seq_len, _ptr(out),
                                     int(bool(out_fp32)), float(softmax_scale), _ptr(ws), ws_bytes, _stream(stream)),
           "fp8_decode_attention")


def nvfp4_pool_bytes(num_blocks, kv_heads, head_dim) -> int:
    return int(_lib.nvfp4_pool_bytes(num_blocks, kv_heads, head_dim))


def nvfp4_pool_init(role: int, num_blocks: int, kv_heads: int, head_dim: int, buf, tensor_scale) -> nvfp4_pool:
    desc = nvfp4_pool()
    _check(_lib.nvfp4_pool_init(ctypes.byref(desc), role, num_blocks, kv_heads, head_dim, _ptr(buf),
                                _ptr(tensor_scale)), "nvfp4_pool_init")
    return desc


def nvfp4_quantize_workspace_bytes() -> int:
    return int(_lib.nvfp4_quantize_workspace_bytes())


def nvfp4_kv_quantize(pool: nvfp4_pool, x, batch, seq_len, block_table, max_blocks, static_scale: bool, ws,
                      ws_bytes: int, stream=None) -> None:
    _check(_lib.nvfp4_kv_quantize(ctypes.byref(pool), _ptr(x), batch, seq_len, _ptr(block_table), max_blocks,
                                  int(bool(static_scale)), _ptr(ws), ws_bytes, _stream(stream)), "nvfp4_kv_quantize")


def nvfp4_decode_workspace_bytes(batch, q_heads, head_dim) -> int:
    return int(_lib.nvfp4_decode_workspace_bytes(batch, q_heads, head_dim))


def nvfp4_decode_attention(q, k: nvfp4_pool, v: nvfp4_pool, block_table, seq_lens, batch, q_heads, max_blocks,
                           max_seq_len, out, out_fp32: bool, softmax_scale: float, ws, ws_bytes: int,
                           stream=None) -> None:
    _check(_lib.nvfp4_decode_attention(_ptr(q), ctypes.byref(k), ctypes.byref(v), _ptr(block_table), _ptr(seq_lens),
                                       batch, q_heads, max_blocks, max_seq_len, _ptr(out), int(bool(out_fp32)),
                                       float(softmax_scale), _ptr(ws), ws_bytes, _stream(stream)),
           "nvfp4_decode_attention")


# ---------------------------------------------------------------------------
# torch-owned buffers around the descriptors (allocation only; no compute)
# ---------------------------------------------------------------------------

def _alloc_bytes(n: int, device):
    import torch
    # 256-byte aligned: the caching allocator hands out 512-byte aligned blocks
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


class KiviCache:
    """One layer's KIVI cache in device memory owned by PyTorch."""

    NAMES = ("k_codes", "k_meta", "v_codes", "v_meta", "k_res", "v_res")

    def __init__(self, batch, kv_heads, q_heads, head_dim, k_bits=2, v_bits=2, residual_len=128, max_tokens=0,
                 device="cuda"):
        import torch
        self.cfg = make_config(batch, kv_heads, q_heads, head_dim, k_bits, v_bits, residual_len, max_tokens)
        sizes = kivi_cache_sizes(self.cfg)
        self.buffers = {n: _alloc_bytes(s, device) for n, s in zip(self.NAMES, sizes)}
        self.desc = kivi_cache_init(self.cfg, [self.buffers[n] for n in self.NAMES])
        self.ws_bytes = kv_decode_workspace_bytes(self.cfg)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)

    @property
    def n_grouped(self) -> int:
        return self.desc.n_grouped

    @property
    def n_resid(self) -> int:
        return self.desc.n_resid

    def prefill(self, k, v, stream=None):
        kv_quant_prefill(self.desc, k, v, k.shape[2], stream)

    def append(self, k_new, v_new, stream=None):
        kv_append_token(self.desc, k_new, v_new, stream)

    def flush(self, stream=None):
        kv_flush_residual(self.desc, stream)

    def decode(self, q, out=None, out_fp32=True, softmax_scale=0.0, stream=None):
        import torch
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else torch.float16, device=q.device)
        kv_decode_attention(self.desc, q, out, out_fp32, softmax_scale, self.ws, self.ws_bytes, stream)
        return out

    def status(self) -> int:
        """Status word of the workspace (bit 0: a device wait timed out). Synchronizes."""
        return int(self.ws[:4].view(__import__("torch").int32).item())

    def grouped_view(self, name: str):
        """Device bytes of one grouped record as ``[B, H, groups_cap, bytes]`` (uint8)."""
        cfg = self.cfg
        per = {"k_codes": 32 * cfg.head_dim * cfg.k_bits // 8, "k_meta": 4 * cfg.head_dim,
               "v_codes": 32 * cfg.head_dim * cfg.v_bits // 8, "v_meta": 128}[name]
        return self.buffers[name][: cfg.batch * cfg.kv_heads * self.desc.groups_cap * per].view(
            cfg.batch, cfg.kv_heads, self.desc.groups_cap, per)

    def residual_view(self, name: str):
        cfg = self.cfg
        n = cfg.batch * cfg.kv_heads * self.desc.res_cap * cfg.head_dim * 2
        return self.buffers[name][:n].view(__import__("torch").float16).view(
            cfg.batch, cfg.kv_heads, self.desc.res_cap, cfg.head_dim)


class PagedKiviCache:
    """One layer's paged, variable-length KIVI cache: pools, windows and the
    block table in device memory owned by PyTorch. The block table
    (int32 ``[B, groups_cap]``) is filled by the caller (``table`` below)."""

    NAMES = ("pool", "k_res", "v_res")
    RECORDS = ("k_codes", "k_meta", "v_codes", "v_meta")   # back to back in each (block, kv head) entry

    def __init__(self, batch, kv_heads, q_heads, head_dim, k_bits=2, v_bits=2, residual_len=128, max_tokens=0,
                 num_blocks=1, device="cuda"):
        import torch
        self.pcfg = kivi_paged_config(make_config(batch, kv_heads, q_heads, head_dim, k_bits, v_bits,
                                                  residual_len, max_tokens), num_blocks)
        self.cfg = self.pcfg.cfg
        sizes = kivi_paged_cache_sizes(self.pcfg)
        self.buffers = {n: _alloc_bytes(s, device) for n, s in zip(self.NAMES, sizes)}
        groups_cap = -(-max_tokens // 32)
        self.table = torch.zeros((batch, groups_cap), dtype=torch.int32, device=device)
        self.desc = kivi_paged_cache_init(self.pcfg, [self.buffers[n] for n in self.NAMES], self.table)
        self.ws_bytes = kv_paged_decode_workspace_bytes(self.pcfg)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)

    def n_grouped(self, b: int) -> int:
        return self.desc.n_grouped[b]

    def n_resid(self, b: int) -> int:
        return self.desc.n_resid[b]

    def prefill(self, k, v, seq_lens, stream=None):
        kv_paged_prefill(self.desc, k, v, k.shape[2], seq_lens, stream)

    def append(self, k_new, v_new, stream=None):
        kv_paged_append(self.desc, k_new, v_new, stream)

    def flush(self, stream=None):
        kv_paged_flush(self.desc, stream)

    def decode(self, q, out=None, out_fp32=True, softmax_scale=0.0, stream=None):
        import torch
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else torch.float16, device=q.device)
        kv_paged_decode_attention(self.desc, q, out, out_fp32, softmax_scale, self.ws, self.ws_bytes, stream)
        return out

    def status(self) -> int:
        """Status word of the workspace (bit 0: a device wait timed out). Synchronizes."""
        return int(self.ws[:4].view(__import__("torch").int32).item())

    def record_bytes(self) -> dict:
        cfg = self.cfg
        return {"k_codes": 32 * cfg.head_dim * cfg.k_bits // 8, "k_meta": 4 * cfg.head_dim,
                "v_codes": 32 * cfg.head_dim * cfg.v_bits // 8, "v_meta": 128}

    def pool_view(self, name: str = None):
        """Device bytes of the pool as ``[num_blocks, H, entry bytes]`` (uint8), or
        of one of its records, ``[num_blocks, H, record bytes]``."""
        cfg, rec = self.cfg, self.record_bytes()
        entry = sum(rec.values())
        pool = self.buffers["pool"][: self.pcfg.num_blocks * cfg.kv_heads * entry].view(
            self.pcfg.num_blocks, cfg.kv_heads, entry)
        if name is None:
            return pool
        off = 0
        for n in self.RECORDS:
            if n == name:
                return pool[:, :, off:off + rec[n]]
            off += rec[n]
        raise KeyError(name)

    def residual_view(self, name: str):
        cfg = self.cfg
        n = cfg.batch * cfg.kv_heads * self.desc.res_cap * cfg.head_dim * 2
        return self.buffers[name][:n].view(__import__("torch").float16).view(
            cfg.batch, cfg.kv_heads, self.desc.res_cap, cfg.head_dim)


def default_softmax_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


class Nvfp4Pool:
    """One NVFP4 pool (keys or values) with its tensor scale, in device memory
    owned by PyTorch."""

    def __init__(self, role: int, num_blocks: int, kv_heads: int, head_dim: int, device="cuda"):
        import torch
        self.buf = _alloc_bytes(nvfp4_pool_bytes(num_blocks, kv_heads, head_dim), device)
        self.scale = torch.ones(64, dtype=torch.float32, device=device)  # [0] is the tensor scale (256-byte slot)
        self.desc = nvfp4_pool_init(role, num_blocks, kv_heads, head_dim, self.buf, self.scale)
        self.ws_bytes = nvfp4_quantize_workspace_bytes()
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)

    def quantize(self, x, block_table, max_blocks, static_scale=False, stream=None):
        nvfp4_kv_quantize(self.desc, x, x.shape[0], x.shape[2], block_table, max_blocks, static_scale, self.ws,
                          self.ws_bytes, stream)

    def view(self):
        """Device bytes as ``[num_blocks, H, 9 * D]`` (uint8)."""
        d = self.desc
        return self.buf[: d.num_blocks * d.kv_heads * 9 * d.head_dim].view(d.num_blocks, d.kv_heads, 9 * d.head_dim)


class Fp8Pool:
    """One FP8 pool (keys or values) with its scale(s), in device memory owned by PyTorch."""

    def __init__(self, role: int, num_blocks: int, kv_heads: int, head_dim: int, fp8_format: int = 0,
                 per_head: bool = False, device="cuda"):
        import torch
        self.buf = _alloc_bytes(fp8_pool_bytes(num_blocks, kv_heads, head_dim), device)
        n = kv_heads if per_head else 1
        self.scale_buf = torch.ones(max(64, -(-n // 64) * 64), dtype=torch.float32, device=device)
        self.scale = self.scale_buf[:n]
        self.desc = fp8_pool_init(role, fp8_format, per_head, num_blocks, kv_heads, head_dim, self.buf, self.scale_buf)
        self.ws = None

    def quantize(self, x, block_table, max_blocks, static_scale=False, stream=None):
        import torch
        b, h, s, d = x.shape
        wsb = fp8_quantize_workspace_bytes(b, h, s, d)
        if self.ws is None or self.ws.numel() < wsb:
            self.ws = torch.zeros(wsb, dtype=torch.uint8, device=x.device)
        fp8_kv_quantize(self.desc, x, b, s, block_table, max_blocks, static_scale, self.ws, wsb, stream)

    def view(self):
        """Device bytes as ``[num_blocks, H, 16 * D]`` (uint8)."""
        d = self.desc
        return self.buf[: d.num_blocks * d.kv_heads * 16 * d.head_dim].view(d.num_blocks, d.kv_heads,
                                                                             16 * d.head_dim)
