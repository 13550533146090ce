"""Shared helpers of the parity tests: seeded workloads, gap search, comparisons."""
from __future__ import annotations

import numpy as np

import oracle
from quantized_routed_expert_fn_gb300 import synth

TOL = 2e-3  # max |gpu - oracle| <= TOL * RMS(oracle MoE row)
GAP = 1e-3  # logits of the k-th and (k+1)-th expert differ by at least this


def topk_gap(logits: np.ndarray, k: int) -> float:
    s = np.sort(logits.astype(np.float32))[::-1]
    return float(s[k - 1] - s[k]) if k < len(s) else np.inf


def layer_gaps_ok(oracle_layer, x) -> bool:
    r = oracle.route(oracle_layer, x)
    k = oracle_layer.src.top_k
    return all(topk_gap(r["logits"][b], k) >= GAP for b in range(x.shape[0]))


def find_x(oracle_layer, nb, seed, rho=0.0, tries=64):
    """First x (seeded) whose rows all have a top-k gap >= GAP."""
    H = oracle_layer.src.hidden
    for s in range(seed, seed + tries):
        x = synth.make_x(np.random.default_rng(s), nb, H, rho)
        if layer_gaps_ok(oracle_layer, x):
            return x, s
    raise RuntimeError("no seed with the required top-k gap")


def find_x_union(oracle_layer, nb, seed, target_u, tries=200):
    """Rows x_b = sqrt(rho) c + sqrt(1-rho) z_b with rho chosen by bisection so
    that the union holds about target_u experts; top-k gaps >= GAP."""
    H = oracle_layer.src.hidden
    best = None
    for s in range(seed, seed + tries):
        lo, hi = 0.0, 1.0
        for _ in range(14):
            rho = 0.5 * (lo + hi)
            x = synth.make_x(np.random.default_rng(s), nb, H, rho)
            U = len(oracle.route(oracle_layer, x)["union"])
            if U == target_u:
                break
            if U > target_u:
                lo = rho
            else:
                hi = rho
        if U == target_u and layer_gaps_ok(oracle_layer, x):
            return x, s, rho
        if best is None or abs(U - target_u) < abs(best[3] - target_u):
            if layer_gaps_ok(oracle_layer, x):
                best = (x, s, rho, U)
    if best is None:
        raise RuntimeError("no union-controlled seed found")
    return best[0], best[1], best[2]


def assert_gaps(ref, k):
    for b in range(ref["logits"].shape[0]):
        assert topk_gap(ref["logits"][b], k) >= GAP, "input does not keep the top-k gap"


def rms_rows(a: np.ndarray) -> np.ndarray:
    return np.sqrt((a.astype(np.float64) ** 2).mean(axis=-1))


def assert_close_rows(got, ref_out, ref_moe, tol=TOL, what=""):
    """max |got - ref_out| <= tol * RMS(ref_moe) row by row."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref_out).max(axis=-1)
    bound = tol * rms_rows(ref_moe)
    bad = err > bound
    assert not bad.any(), f"{what}: rows {np.nonzero(bad)[0].tolist()} err {err[bad]} > bound {bound[bad]}"
    return float((err / bound).max())


def check_routing(gpu_idx, gpu_w, ref, logits_ref, k, what=""):
    """Ids: same set per row, GPU order descending in the oracle's logits;
    weights within 1e-5 of the oracle's."""
    nb = gpu_idx.shape[0]
    for b in range(nb):
        gi = [int(v) for v in gpu_idx[b][:k]]
        ri = [int(v) for v in ref["idx"][b]]
        assert sorted(gi) == sorted(ri), f"{what} row {b}: ids {gi} vs {ri}"
        lv = logits_ref[b][gi]
        assert np.all(np.diff(lv) <= 1e-5), f"{what} row {b}: order not descending"
        if gpu_w is not None:
            wref = {int(e): float(w) for e, w in zip(ref["idx"][b], ref["w"][b])}
            for e, w in zip(gi, gpu_w[b][:k]):
                assert abs(float(w) - wref[e]) < 1e-5, f"{what} row {b}: weight of {e}"


def check_union(slot_row, wmap_row, ref, eaddr, nb, what=""):
    U = len(ref["union"])
    assert int(slot_row[62]) == U and int(slot_row[63]) == U, f"{what}: union size"
    addr_to_e = {int(a): e for e, a in enumerate(eaddr)}
    gu = [addr_to_e[int(slot_row[j])] for j in range(U)]
    assert sorted(gu) == sorted(ref["union"].tolist()), f"{what}: union set"
    assert list(gu) == ref["union"].tolist(), f"{what}: union order (first seen)"
    for b in range(nb):
        for j, e in enumerate(gu):
            want = ref["wmap"][b][list(ref["union"]).index(e)]
            assert abs(float(wmap_row[b][j]) - want) < 1e-5, f"{what}: wmap[{b}][{j}]"
        assert np.all(wmap_row[b][U:] == 0)
    for b in range(nb, 4):
        assert np.all(wmap_row[b] == 0)
