"""Comparison of GPU results with the fp64 oracle under the parity rules.

  greedy   accepted lengths and token ids bit-exact.
  sampling decisions identical except where the oracle flags a near tie
           (|u - p/q| < 1e-6 at an accept test it evaluated, or a residual
           CDF boundary within 1e-6 of the final uniform); such requests are
           counted and reported, never silently passed.
           p_j(x_j) within 1e-5 relative; the residual mass R and the drawn
           token's probability r(v*)/R within 1e-5 relative plus an absolute
           allowance of 4e-7 / R: r = p - q is a difference of two
           probabilities, so the fp32 rounding of p (about 2^-22 relative)
           becomes an absolute error in r that a relative bound cannot cover
           when p and q are close.
"""
from __future__ import annotations

import json
import os

import numpy as np

REL = 1e-5
REPORT = {}


def record(name, info):
    REPORT[name] = info
    path = os.environ.get("SV_PARITY_REPORT")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1, sort_keys=True, default=float)
    print(f"[parity] {name}: {info}")


def split_rows(row_offsets):
    ro = np.asarray(row_offsets, dtype=np.int64)
    return [(int(ro[b]), int(ro[b + 1])) for b in range(len(ro) - 1)]


def compare_greedy(name, row_offsets, gpu_out, gpu_al, orc):
    gpu_out = np.asarray(gpu_out)
    gpu_al = np.asarray(gpu_al)
    assert np.array_equal(gpu_al, orc["accept_len"]), f"{name}: accept lengths differ"
    assert np.array_equal(gpu_out, orc["out_tokens"]), f"{name}: tokens differ"
    record(name, {"requests": len(gpu_al), "mismatch": 0, "mean_al": float(gpu_al.mean())})


def compare_sampling(name, row_offsets, gpu_out, gpu_al, gpu_diag, orc, max_tie_mismatch_frac=0.05):
    gpu_out = np.asarray(gpu_out)
    gpu_al = np.asarray(gpu_al)
    rows = split_rows(row_offsets)
    B = len(rows)
    n_draft = rows[-1][1] - B
    mism, tie_mism, ties = [], 0, 0
    for b, (r0, r1) in enumerate(rows):
        tie = orc["near_tie_accept"][b] > 0 or orc["near_tie_sample"][b] > 0
        ties += int(tie)
        same = gpu_al[b] == orc["accept_len"][b] and np.array_equal(gpu_out[r0:r1], orc["out_tokens"][r0:r1])
        if not same:
            if tie:
                tie_mism += 1
            else:
                mism.append(b)
    info = {"requests": B, "mismatch": len(mism), "near_ties": ties, "near_tie_mismatch": tie_mism,
            "mean_al": float(gpu_al.mean())}
    if gpu_diag is not None:
        d = np.asarray(gpu_diag, dtype=np.float64)
        po = orc["p_draft"]
        ev = ~np.isnan(po)
        pg = d[:n_draft][ev]
        rel_p = np.abs(pg - po[ev]) / np.maximum(np.abs(po[ev]), 1e-30)
        info["p_max_rel_err"] = float(rel_p.max()) if rel_p.size else 0.0
        assert info["p_max_rel_err"] <= REL, f"{name}: p(x) rel err {info['p_max_rel_err']}"
        same_tok = np.array([gpu_al[b] == orc["accept_len"][b] and
                             np.array_equal(gpu_out[r0:r1], orc["out_tokens"][r0:r1])
                             for b, (r0, r1) in enumerate(rows)])
        Rg = d[n_draft::2][:B]
        rg = d[n_draft + 1::2][:B]
        Ro = orc["residual_mass"]
        ro_ = orc["residual_prob"]
        ok = same_tok & ~np.isnan(Ro)
        if ok.any():
            relR = np.abs(Rg[ok] - Ro[ok]) / np.maximum(Ro[ok], 1e-30)
            info["R_max_rel_err"] = float(relR.max())
            # r(v*) = p(v*) - q(v*): fp32 rounding of p (~2^-22 p) is absolute in r
            err_r = np.abs(rg[ok] - ro_[ok])
            allow = REL * np.abs(ro_[ok]) + 4e-7 / np.maximum(Ro[ok], 1e-30)
            info["r_max_rel_err"] = float((err_r / np.maximum(np.abs(ro_[ok]), 1e-30)).max())
            assert np.all(relR <= REL + 4e-7 / np.maximum(Ro[ok], 1e-30)), f"{name}: residual mass off"
            assert np.all(err_r <= allow), f"{name}: residual probability off"
    record(name, info)
    assert not mism, f"{name}: {len(mism)} requests differ without a near tie, e.g. {mism[:5]}"
    assert tie_mism <= max(2, max_tie_mismatch_frac * B), f"{name}: too many near-tie mismatches {tie_mism}"
    return info
