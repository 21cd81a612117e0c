"""Shared helpers for the parity tests: run the oracle on a workload and
compare a GPU result with it at the acceptance tolerances.

Acceptance (bf16 outputs against the fp64 oracle), element by element:

    |out - exact| <= max(1e-2, ulp(|exact| + eps) / 2 + eps)

with mean-abs <= 1e-3 over the whole output, and fp32 lse within
1e-4 * max(1, |lse|) (an lse of -inf, no visible key and no sink, must be
-inf on both sides).  The 1e-2 is the acceptance figure; a bf16 output can
only be within half a unit in the last place (ulp) of the exact value, which
is above 1e-2 from |exact| = 4 on.  eps bounds the distance between the
exact value and the fp32 value the kernel rounds to bf16; it is derived per
element (error_bound below) from the arithmetic every tensor-core kernel
here shares:

* Each weight p_j = 2^(s_j - m) enters the P.V product rounded to bf16
  (relative error at most u = 2^-8), after the approximate exp2 of the
  special-function unit (at most 2^-22 relative) of a score carrying its own
  fp32 error.  Output and
  partials are normalised by the sum of the weights actually multiplied, so
  the output is a convex combination with perturbed weights and its error is
  sum_j d_j (v_j - out) / Z (d_j the weight errors): at most
  c/(1-c) * sum_j w_j |v_j - out| <= c/(1-c) * sd, sd = sqrt(sum_j w_j
  (v_j - out)^2) being the weighted spread of V around the exact output.
  With split-K every slice is a normalised average over its keys, merged
  with exact weights; by Jensen's inequality the sum of the slices' spreads
  (each around its own average) stays below sd, so the bound holds for any
  partition of the keys, the balanced MLA split included.
* The fp32 accumulations (P.V in the tensor core, 16 keys per step, the
  weight sums, the rescales by the running maximum, the split-K merge) add
  at most (2 ceil(n/16) + 32) 2^-23 * sum_j w_j |v_j| for n visible keys.
* A score is an fp32 MMA sum of dim_qk / 16 steps of 16 exact products, then
  scaled to base 2: its error is at most (ceil(dim_qk/16) + 2) 2^-23
  * max_j scale sum_c |q_c k_jc| + 6 * 2^-24 max_j |s_j| (rho), and it moves
  each weight by a relative 2 rho (1 + 2 rho) at most (score and maximum).

The oracle returns sd, sum_j w_j |v_j| and the score magnitudes
(oracle.spread); oracle_result attaches the resulting eps to the exact
output it returns.  A comparison of two GPU results (split-K P > 1 against
P = 1) checks each against the exact value and their distance against
ulp(|exact| + eps) + 2 eps (two roundings of values within eps of it).
"""
import json
import os

import numpy as np
import torch

import oracle

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_REL = 1e-4
U_BF16 = 2.0 ** -8           # bf16 unit roundoff (8 significant bits)

# Elements that needed more than 1e-2, over the whole session (reported by
# the terminal summary in conftest.py).
STATS = {"comparisons": 0, "elements": 0, "above_1e2": 0, "worst": None}


class ExactOut(np.ndarray):
    """The oracle's fp64 output with its per-element error bound (.eps)."""

    def __new__(cls, out, eps):
        obj = np.asarray(out, dtype=np.float64).view(cls)
        obj.eps = np.asarray(eps, dtype=np.float64)
        return obj

    def __array_finalize__(self, obj):
        self.eps = getattr(obj, "eps", None)


def error_bound(sd, am, stats, dim_qk):
    """eps per output element from the oracle's spread statistics (see the
    module docstring for the derivation)."""
    nvis = stats[..., 0:1]
    sabs = stats[..., 1:2]
    smax = stats[..., 2:3]
    rho = (np.ceil(dim_qk / 16.0) + 2.0) * 2.0 ** -23 * sabs + 6.0 * 2.0 ** -24 * smax
    ds = 2.0 * rho * (1.0 + 2.0 * rho)
    c = U_BF16 + 2.0 ** -22 + ds
    c_acc = (2.0 * np.ceil(nvis / 16.0) + 32.0) * 2.0 ** -23
    return c / (1.0 - c) * sd + c_acc * am


def oracle_kv(w, cache):
    cache = cache.cpu()
    if w.indices is not None:
        return oracle.KV.sparse(cache, w.indices.cpu())
    if w.page_table is not None:
        return oracle.KV.paged(cache, w.page_table.cpu())
    return oracle.KV.contiguous(cache)


def oracle_result(w, sample=None, sink=None, threads=None):
    """fp64 oracle output for workload w (optionally only sampled pairs):
    (ExactOut out carrying eps, lse)."""
    k = oracle_kv(w, w.k_cache)
    v = k if w.v_cache is None else oracle_kv(w, w.v_cache)
    if sink is None:
        sink = None if w.sink is None else w.sink.cpu()
    kw = dict(group=w.group, scale=w.scale, dim_v=w.dim_v, sink=sink, causal=w.causal,
              q_row_offsets=None if w.q_row_offsets is None else w.q_row_offsets.cpu(),
              sample=sample, threads=threads)
    q = w.q.cpu()
    kvl = w.kv_len.cpu()
    out, lse = oracle.attention(q, k, v, kvl, **kw)
    sd, am, st = oracle.spread(q, k, v, kvl, **kw)
    return ExactOut(out, error_bound(sd, am, st, w.dim_qk)), lse


def full_rows_sample(row_lengths, num_heads, heads_per_row, seed):
    """(rows, heads) for a full-size oracle check: every head of four rows
    (the two longest, the median and the shortest) and heads_per_row random
    heads of every other row."""
    lens = np.asarray(row_lengths)
    order = np.argsort(lens, kind="stable")
    full = sorted({int(order[-1]), int(order[-2]), int(order[len(order) // 2]), int(order[0])})
    rng = np.random.default_rng(seed)
    rows, heads = [], []
    for r in range(len(lens)):
        hs = (np.arange(num_heads) if r in full
              else np.sort(rng.choice(num_heads, heads_per_row, replace=False)))
        rows.extend([r] * len(hs))
        heads.extend(hs.tolist())
    return np.asarray(rows), np.asarray(heads)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def _host(t):
    if isinstance(t, torch.Tensor):
        return t.float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def _record(what, err, ref, bound):
    STATS["comparisons"] += 1
    STATS["elements"] += int(err.size)
    over = err > OUT_MAX_ABS
    STATS["above_1e2"] += int(over.sum())
    if over.any():
        i = int(np.argmax(np.where(over, err, -1.0)))
        worst = STATS["worst"]
        if worst is None or err.flat[i] - OUT_MAX_ABS > worst["excess"]:
            STATS["worst"] = {"what": str(what), "excess": float(err.flat[i] - OUT_MAX_ABS),
                              "err": float(err.flat[i]), "ref": float(ref.flat[i]),
                              "bound": float(bound.flat[i])}
    path = os.environ.get("ATTN_TOL_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": str(what), "n": int(err.size),
                                "max_err": float(err.max()), "mean_err": float(err.mean()),
                                "above_1e2": int(over.sum()),
                                "max_err_over_bound": float((err / bound).max())}) + "\n")


def _check_lse(lse, ref_l, what, rel=LSE_REL):
    lg = lse.cpu().numpy().astype(np.float64) if isinstance(lse, torch.Tensor) else lse
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(lg), ninf), f"{what}: -inf lse mismatch"
    fin = ~ninf
    if fin.any():
        d = np.abs(lg[fin] - ref_l[fin]) / np.maximum(1.0, np.abs(ref_l[fin]))
        assert d.max() <= rel, f"{what}: lse rel {d.max():.3g}"


def assert_close(out, lse, ref_o, ref_l, what=""):
    """out (bf16) within max(1e-2, ulp(|exact| + eps)/2 + eps) of the oracle's
    ref_o element by element, mean-abs <= 1e-3; lse within 1e-4 relative."""
    eps = getattr(ref_o, "eps", None)
    if eps is None:
        raise ValueError(f"{what}: the reference must come from oracle_result (it carries eps)")
    ref = np.asarray(ref_o, dtype=np.float64).view(np.ndarray)
    o = _host(out)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref)
    bound = np.maximum(OUT_MAX_ABS, 0.5 * bf16_ulp(np.abs(ref) + eps) + eps)
    _record(what, err, ref, bound)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"{what}: error {err.flat[worst]:.3g} at |ref| "
                                  f"{abs(ref.flat[worst]):.3g} (bound {bound.flat[worst]:.3g}, "
                                  f"eps {eps.flat[worst]:.3g})")
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3g}"
    if lse is not None:
        _check_lse(lse, ref_l, what)


def assert_pair(a, la, b, lb, ref_o, ref_l, what=""):
    """Two GPU results of the same problem (e.g. split-K P > 1 and P = 1):
    each within the acceptance bound of the exact value, and their distance
    within two roundings of values eps from it, max(1e-2, ulp(|exact| + eps)
    + 2 eps), mean-abs <= 1e-3; lse within 2e-4 relative of each other."""
    assert_close(a, la, ref_o, ref_l, f"{what} (first)")
    assert_close(b, lb, ref_o, ref_l, f"{what} (second)")
    ref = np.asarray(ref_o, dtype=np.float64).view(np.ndarray)
    eps = ref_o.eps
    d = np.abs(_host(a) - _host(b))
    bound = np.maximum(OUT_MAX_ABS, bf16_ulp(np.abs(ref) + eps) + 2.0 * eps)
    worst = int(np.argmax(d - bound))
    assert np.all(d <= bound), (f"{what}: pair distance {d.flat[worst]:.3g} at |ref| "
                                f"{abs(ref.flat[worst]):.3g} (bound {bound.flat[worst]:.3g})")
    assert d.mean() <= OUT_MEAN_ABS, f"{what}: pair mean-abs {d.mean():.3g}"
    if la is not None and lb is not None:
        _check_lse(la, _host(lb), f"{what} (pair lse)", rel=2 * LSE_REL)


def assert_consistent(a, la, b, lb, eps, what=""):
    """Two GPU results of the same problem compared on outputs whose exact
    values were not all computed (full-size batches, where the oracle checks
    samples): a consistency check between the two paths, with eps the
    largest error bound of the sampled exact values, max(1e-2, ulp + 2 eps)
    per element and mean-abs <= 1e-3.  The accuracy claim rests on the oracle
    comparisons of the samples."""
    x = _host(a)
    y = _host(b)
    assert np.all(np.isfinite(x)) and np.all(np.isfinite(y)), f"{what}: non-finite output"
    d = np.abs(x - y)
    bound = np.maximum(OUT_MAX_ABS, bf16_ulp(np.maximum(np.abs(x), np.abs(y))) + 2.0 * eps)
    worst = int(np.argmax(d - bound))
    assert np.all(d <= bound), (f"{what}: distance {d.flat[worst]:.3g} (bound "
                                f"{bound.flat[worst]:.3g})")
    assert d.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {d.mean():.3g}"
    if la is not None and lb is not None:
        _check_lse(la, _host(lb), f"{what} (lse)", rel=2 * LSE_REL)


def bits_equal(a, b):
    if a is None or b is None:
        return a is None and b is None
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))
