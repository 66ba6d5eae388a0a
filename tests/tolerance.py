"""Error metrics for comparing a GEMM result with the fp64 oracle.

The bar: every element within 2 ulps of the output type at |ref| plus an
absolute 1e-3, and a relative Frobenius error of at most 1e-3.  The ulp is
the spacing of the output format in the binade of |ref|:
  fp16:  2^(floor(log2|x|) - 10) for |x| >= 2^-14, else 2^-24;
  bf16:  2^(floor(log2|x|) - 7)  for |x| >= 2^-126, else 2^-133.

Reading of the Frobenius bound for bf16: rounding the exact result once to
bf16 (8 significant bits) already leaves a relative Frobenius error of about
1.6e-3, above the 1e-3 bound, so no bf16 output can meet it literally.  For
bf16 the Frobenius error is therefore measured against the oracle's result
correctly rounded to bf16 (the error the computation adds beyond the one
unavoidable output rounding); fp16 is checked literally against the exact
result.
"""
from __future__ import annotations

import numpy as np

_FMT = {"f16": (10, -14), "bf16": (7, -126), "f32": (23, -126)}

ULPS = 2.0
ABS = 1e-3
FROB = 1e-3


def ulp(x, dtype: str) -> np.ndarray:
    mant, emin = _FMT[dtype]
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        _, e = np.frexp(a)                  # a = f * 2^e, f in [0.5, 1)
    floor_log2 = e.astype(np.int64) - 1
    q = np.where(a >= np.ldexp(1.0, emin), floor_log2 - mant, emin - mant)
    return np.ldexp(1.0, q)


def rounded_reference(ref, dtype: str) -> np.ndarray:
    import oracle
    return oracle.decode(oracle.round_to(ref, dtype), dtype)


def compare(got, ref, dtype: str, ulps: float = ULPS, abs_tol: float = ABS):
    """Return a dict of error statistics; `ok` is the pass/fail verdict."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if g.size == 0:
        return {"ok": True, "max_abs": 0.0, "max_ulp": 0.0, "frob": 0.0, "bad": 0}
    err = np.abs(g - r)
    u = ulp(r, dtype)
    bound = ulps * u + abs_tol
    finite = np.isfinite(g)
    bad = (~finite) | (err > bound)
    nr = np.linalg.norm(r)
    frob_base = r if dtype in ("f16", "f32") else rounded_reference(r, dtype)
    diff = np.where(finite, g - frob_base, np.inf)
    frob = float(np.linalg.norm(diff) / nr) if nr > 0 else float(np.linalg.norm(diff))
    frob_exact = float(np.linalg.norm(np.where(finite, g - r, np.inf)) / nr) if nr > 0 else 0.0
    return {
        "ok": bool((not bad.any()) and frob <= FROB),
        "frob_vs_exact": frob_exact,
        "max_abs": float(np.max(np.where(finite, err, np.inf))),
        "max_ulp": float(np.max(np.where(finite, err / u, np.inf))),
        "frob": frob,
        "bad": int(bad.sum()),
        "first_bad": (tuple(int(i) for i in np.argwhere(bad)[0]) if bad.any() else None),
    }


def compare_rows(got_rows, ref, dtype: str, chunk: int = 512, ulps: float = ULPS,
                 abs_tol: float = ABS):
    """compare() over a large matrix, a block of `chunk` rows at a time.

    got_rows(r0, r1) returns the decoded GPU rows [r0, r1) as float64; ref is
    the oracle's full fp64 result.  The per-element bound and the Frobenius
    norms are the ones compare() uses; the norms are accumulated as sums of
    squares over the blocks, so no temporary larger than one block exists."""
    r = np.asarray(ref)
    M = r.shape[0]
    bad = 0
    first_bad = None
    max_abs = max_ulp = 0.0
    num = num_exact = den = 0.0
    for r0 in range(0, M, chunk):
        r1 = min(M, r0 + chunk)
        g = np.asarray(got_rows(r0, r1), dtype=np.float64)
        rr = np.asarray(r[r0:r1], dtype=np.float64)
        assert g.shape == rr.shape, (g.shape, rr.shape)
        finite = np.isfinite(g)
        err = np.where(finite, np.abs(g - rr), np.inf)
        u = ulp(rr, dtype)
        b = (~finite) | (err > ulps * u + abs_tol)
        if b.any():
            bad += int(b.sum())
            if first_bad is None:
                i, j = np.argwhere(b)[0]
                first_bad = (int(i) + r0, int(j))
        max_abs = max(max_abs, float(err.max()) if err.size else 0.0)
        max_ulp = max(max_ulp, float((err / u).max()) if err.size else 0.0)
        base = rr if dtype in ("f16", "f32") else rounded_reference(rr, dtype)
        num += float(np.sum(np.where(finite, g - base, np.inf) ** 2))
        num_exact += float(np.sum(np.where(finite, g - rr, np.inf) ** 2))
        den += float(np.sum(rr * rr))
    nr = np.sqrt(den)
    frob = float(np.sqrt(num) / nr) if nr > 0 else float(np.sqrt(num))
    return {
        "ok": bool(bad == 0 and frob <= FROB),
        "frob_vs_exact": float(np.sqrt(num_exact) / nr) if nr > 0 else 0.0,
        "max_abs": max_abs,
        "max_ulp": max_ulp,
        "frob": frob,
        "bad": bad,
        "first_bad": first_bad,
        "elements": int(r.size),
    }
