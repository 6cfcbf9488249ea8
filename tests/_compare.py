"""The parity bar between the CUDA path and the oracle.

* ue8m0 scales and slot placement: bit-exact (every byte of the cache outside
  the written slots keeps its previous value, every scale word is identical);
* e4m3 codes: at most one code apart, in at most 0.1% of elements (two
  fp32 LayerNorm evaluations in different summation orders may straddle an
  e4m3 rounding boundary);
* q codes: the q side has one fp32 rounding sequence (bf16 -> fp32 exact, the
  fixed FMA form of RoPE, an exact power-of-two scale), so they must match
  exactly;
* gate weights: within 1e-6 relative (both zero when the reference is zero).
"""
import numpy as np

from _run import cache_views, code_distance

CODE_FRAC = 1e-3
WEIGHT_RTOL = 1e-6


def compare(inp, gpu, ref, q_exact=True):
    rep = {}
    if "q_fp8" in gpu:
        d = code_distance(gpu["q_fp8"], ref["q_fp8"])
        rep["q_max_dist"] = int(d.max()) if d.size else 0
        rep["q_diff"] = int((d > 0).sum())
        wr, wg = ref["weights"].astype(np.float64), gpu["weights"].astype(np.float64)
        bad = np.abs(wg - wr) > WEIGHT_RTOL * np.abs(wr)
        rep["weights_bad"] = int(bad.sum())
        rep["weights_max_rel"] = float(np.max(np.abs(wg - wr) / np.maximum(np.abs(wr), 1e-45))) \
            if wr.size else 0.0
    cg, sg = cache_views(inp, gpu["cache"])
    cr, sr = cache_views(inp, ref["cache"])
    rep["scale_mismatch"] = int(np.sum(sg.view(np.uint32) != sr.view(np.uint32)))
    d = code_distance(cg, cr)
    rep["k_max_dist"] = int(d.max()) if d.size else 0
    rep["k_diff"] = int((d > 0).sum())
    n_k = max(1, inp.T * 128)
    ok = rep["scale_mismatch"] == 0 and rep["k_max_dist"] <= 1 and rep["k_diff"] <= CODE_FRAC * n_k
    if "q_fp8" in gpu:
        n_q = max(1, gpu["q_fp8"].size)
        ok = ok and rep["weights_bad"] == 0 and rep["q_max_dist"] <= 1 \
            and rep["q_diff"] <= CODE_FRAC * n_q
        if q_exact:
            ok = ok and rep["q_diff"] == 0
    rep["ok"] = bool(ok)
    return rep


def assert_parity(inp, gpu, ref, q_exact=True):
    rep = compare(inp, gpu, ref, q_exact=q_exact)
    assert rep["ok"], rep
    return rep
