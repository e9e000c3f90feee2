"""Host-side logic of bench.py that needs no GPU: the routing report of the CPU-baseline leg
(selection flips against the oracle, clamped Taylor weights) and the CPU description."""
import numpy as np
import torch

import bench
import oracle
from workloads import Workload, make_qkv, to_f64


def lists_from_selection(sel):
    """Compacted ascending lists [B, H, NQB, NKB] + counts, as the route kernel writes them."""
    B, H, nq, nk = sel.shape
    idx = np.zeros((B, H, nq, nk), dtype=np.int32)
    cnt = sel.sum(-1).astype(np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                lst = np.flatnonzero(sel[b, h, i])
                idx[b, h, i, :lst.size] = lst
    return {"sel_idx": torch.from_numpy(idx), "sel_cnt": torch.from_numpy(cnt)}


def test_routing_report_counts_flips_and_clamps():
    w = Workload("t", B=1, H=2, Sq=1000, Skv=1000, d=64, seed=3, q_std=0.5, k_std=0.5, block=64, beta=0.5)
    q, k, v = make_qkv(w, device="cpu")
    qh, kh, vh = to_f64(q), to_f64(k), to_f64(v)
    qp, kp, vp = (oracle.block_pool(x, w.block) for x in (qh, kh, vh))
    rt = oracle.route(qp, kp, vp, w.Sq, w.block, w.scale, w.beta)
    # the oracle's own selection: no flips, and the clamp count equals the oracle's
    _, rep = bench.routing_report(q, k, v, w, lists_from_selection(rt["sel"]))
    assert rep["near_tau_flips"] == 0 and rep["flips_outside_1e-4_band"] == 0
    assert rep["clamped_taylor_weights"] == rt["n_clamped"]
    assert rep["selected_blocks_gpu"] == rep["selected_blocks_oracle"] == int(rt["sel"].sum())
    # one block dropped from a list (far from tau): counted as a flip outside the band
    sel = rt["sel"].copy()
    cand = [(i, j) for i in range(sel.shape[2]) for j in np.flatnonzero(sel[0, 1, i])
            if j != rt["proxy"][0, 1, i].argmax() and abs(rt["proxy"][0, 1, i, j] - rt["tau"][0, 1, i]) > 1e-3]
    assert cand
    sel[0, 1, cand[0][0], cand[0][1]] = False
    _, rep = bench.routing_report(q, k, v, w, lists_from_selection(sel))
    assert rep["near_tau_flips"] == 1 and rep["flips_outside_1e-4_band"] == 1


def test_cpu_model_names_the_machine():
    name = bench.cpu_model()
    assert "(" in name and name.endswith(")")
