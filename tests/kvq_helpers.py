"""Shared helpers of the GPU parity tests: device copies, oracle caches, and the
parity bars (bit-exact bytes; attention within max-abs 2e-3 and relative L2
1e-3 of the float64 oracle on the same dequantized values)."""
import numpy as np

from oracle import attention, kivi, layout

MAX_ABS = 2e-3
REL_L2 = 1e-3


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def oracle_cache(cfg_like, k, v):
    c = kivi.KiviCache(k.shape[0], k.shape[1], k.shape[3], cfg_like["k_bits"], cfg_like["v_bits"],
                       cfg_like["residual"], cfg_like.get("max_tokens"))
    c.prefill(k, v)
    return c


def assert_grouped_bytes_equal(gpu_cache, ocache, groups=None):
    """Bit-exact comparison of the packed grouped region (all or the listed groups)."""
    ng = ocache.n_grouped // 32
    assert gpu_cache.n_grouped == ocache.n_grouped
    packed = layout.pack_cache(ocache) if groups is None else _pack_groups(ocache, groups)
    for name, want in packed.items():
        got = host(gpu_cache.grouped_view(name))
        got = got[:, :, :ng] if groups is None else got[:, :, groups]
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            raise AssertionError(f"{name}: {len(bad)} bytes differ, first at {bad[:5].tolist()}")


def assert_all_grouped_bytes_equal(gpu_cache, ocache, rows_per_chunk=1):
    """Bit-exact comparison of every group of every (batch row, kv head), the
    oracle packed a few batch rows at a time (bounded host memory)."""
    ng = ocache.n_grouped // 32
    assert gpu_cache.n_grouped == ocache.n_grouped
    got = {name: host(gpu_cache.grouped_view(name))[:, :, :ng] for name in
           ("k_codes", "k_meta", "v_codes", "v_meta")}
    for b0 in range(0, ocache.B, rows_per_chunk):
        rows = slice(b0, b0 + rows_per_chunk)
        want = {
            "k_codes": layout.pack_key_codes(ocache.k_codes[rows], ocache.k_bits),
            "k_meta": layout.pack_key_meta(ocache.k_scale[rows], ocache.k_zero[rows]),
            "v_codes": layout.pack_value_codes(ocache.v_codes[rows], ocache.v_bits),
            "v_meta": layout.pack_value_meta(ocache.v_scale[rows], ocache.v_zero[rows]),
        }
        for name, w in want.items():
            g = got[name][rows]
            if not np.array_equal(g, w):
                bad = np.argwhere(g != w)
                raise AssertionError(f"{name} rows {b0}+: {len(bad)} bytes differ, first at {bad[:5].tolist()}")


def _pack_groups(ocache, groups):
    g = np.asarray(groups)
    return {
        "k_codes": layout.pack_key_codes(ocache.k_codes[:, :, g], ocache.k_bits),
        "k_meta": layout.pack_key_meta(ocache.k_scale[:, :, g], ocache.k_zero[:, :, g]),
        "v_codes": layout.pack_value_codes(ocache.v_codes[:, :, g], ocache.v_bits),
        "v_meta": layout.pack_value_meta(ocache.v_scale[:, :, g], ocache.v_zero[:, :, g]),
    }


def assert_residual_equal(gpu_cache, ocache):
    n = ocache.n_resid
    assert gpu_cache.n_resid == n
    for name, want in (("k_res", ocache.k_res), ("v_res", ocache.v_res)):
        got = host(gpu_cache.residual_view(name))[:, :, :n]
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), name


def oracle_attention(ocache, q, scale, heads=None):
    return attention.decode_attention(q, ocache.keys_hat, ocache.values_hat, ocache.H, scale, heads)


def assert_attention_close(got, ref, heads=None, fp16_out=False):
    got = np.asarray(got, np.float64)
    if heads is not None:
        idx = tuple(np.array(heads).T)
        got, ref = got[idx], ref[idx]
    err = np.abs(got - ref)
    tol = MAX_ABS
    if fp16_out:
        # fp16 output: the bar plus half an fp16 ulp of the reference value
        ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
        tol = MAX_ABS + 0.5 * ulp
    assert np.all(err <= tol), f"max abs err {err.max():.3g}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2, f"relative L2 err {rel:.3g}"
    return err.max(), rel
