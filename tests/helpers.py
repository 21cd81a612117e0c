"""Shared helpers for the parity tests: run the oracle on a workload and
compare a GPU result with it at the acceptance tolerances.

Acceptance (bf16 outputs against the fp64 oracle): max-abs <= 1e-2 and
mean-abs <= 1e-3; fp32 lse within 1e-4 * max(1, |lse|).  An lse of -inf
(no visible key, no sink) must be -inf on both sides.

A bf16 output cannot sit closer to the exact value than half a unit in the
last place, and a value near a rounding boundary may round either way, so
for |out| >= 2 (where one bf16 ulp exceeds 1e-2) the per-element bound is
one bf16 ulp of the exact value instead of 1e-2.
"""
import numpy as np
import torch

import oracle

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_REL = 1e-4


def oracle_kv(w, cache):
    cache = cache.cpu()
    if w.indices is not None:
        return oracle.KV.sparse(cache, w.indices.cpu())
    if w.page_table is not None:
        return oracle.KV.paged(cache, w.page_table.cpu())
    return oracle.KV.contiguous(cache)


def oracle_result(w, sample=None, sink=None, threads=None):
    """fp64 oracle output for workload w (optionally only sampled pairs)."""
    k = oracle_kv(w, w.k_cache)
    v = k if w.v_cache is None else oracle_kv(w, w.v_cache)
    if sink is None:
        sink = None if w.sink is None else w.sink.cpu()
    return oracle.attention(w.q.cpu(), k, v, w.kv_len.cpu(), group=w.group, scale=w.scale,
                            dim_v=w.dim_v, sink=sink, causal=w.causal,
                            q_row_offsets=None if w.q_row_offsets is None
                            else w.q_row_offsets.cpu(),
                            sample=sample, threads=threads)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_close(out, lse, ref_o, ref_l, what=""):
    o = out.float().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out)
    err = np.abs(o.astype(np.float64) - ref_o)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    tol = np.maximum(OUT_MAX_ABS, bf16_ulp(ref_o))
    worst = np.argmax(err - tol)
    assert np.all(err <= tol), (f"{what}: max-abs {err.flat[worst]:.3g} at |ref| "
                                f"{abs(ref_o.flat[worst]):.3g} (bound {tol.flat[worst]:.3g})")
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3g}"
    if lse is not None:
        lg = lse.cpu().numpy().astype(np.float64) if isinstance(lse, torch.Tensor) else lse
        ninf = np.isneginf(ref_l)
        assert np.array_equal(np.isneginf(lg), ninf), f"{what}: -inf lse mismatch"
        fin = ~ninf
        if fin.any():
            rel = np.abs(lg[fin] - ref_l[fin]) / np.maximum(1.0, np.abs(ref_l[fin]))
            assert rel.max() <= LSE_REL, f"{what}: lse rel {rel.max():.3g}"


def bits_equal(a, b):
    if a is None or b is None:
        return a is None and b is None
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))
