"""Sharding one sequence along T over ranks, with one exchange step: the
combine of the design for multi-GPU prefill, checked among CPU ranks (gloo)
against the fp64 oracle of the whole sequence.

Every call of the GPU path runs on one GPU, so this validates the design
(the algebra of the exchange), with the oracle as each rank's local scan:

1. rank s scans its segment [t_s, t_{s+1}) from a zero state, with the token
   t_s - 1 as the previous token of the trapezoidal beta term, giving y_loc
   and the local end state g_s (complex frame);
2. the recurrence is linear in the incoming state h_in, and its homogeneous
   part over a segment is a per-(b, h) decay and a per-pair rotation
   (Mamba-3 summary page, §3.2, Proposition 3.2.1: the rotations of one pair
   commute): h'_t = y-free local part + prod_{i=t_s}^{t} alpha_i *
   Rot(sum_{i=t_s}^{t} theta_i) h_in.  So the ranks all-gather
   (a_s = prod alpha, phi_s = sum theta, g_s) and each folds the earlier
   ranks' pairs: h_in(s + 1) = a_s Rot(phi_s) h_in(s) + g_s;
3. rank s corrects its outputs: y_t += C_t^T a_{t_s..t} Rot(phi_{t_s..t}) h_in(s).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rot_rows(h, phi):
    """Rotate the row pairs (2k, 2k+1) of h[..., N, P] by phi[..., k]:
    (a, b) -> (a cos - b sin, a sin + b cos), the complex frame's e^{i phi}."""
    c, s = np.cos(phi)[..., None], np.sin(phi)[..., None]
    a, b = h[..., 0::2, :], h[..., 1::2, :]
    out = np.empty_like(h)
    out[..., 0::2, :] = a * c - b * s
    out[..., 1::2, :] = a * s + b * c
    return out


def _problem(R):
    from selective_state_space_131_b300 import inputs
    shape = inputs.ScanShape(batch=2, seqlen=96, heads=2, headdim=8, dstate=8, rank=R, chunk=16, dtype="f32")
    inp = inputs.make_scan_inputs(shape, 31 + R)
    return {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}


def _worker(rank, world, port, R, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        p = _problem(R)
        T = p["x"].shape[1]
        seg = T // world
        t0, t1 = rank * seg, (rank + 1) * seg
        sl = lambda a: a[:, t0:t1]
        # 1. local scan from zero; the token before the segment carries the beta term
        prevB = p["B"][:, t0 - 1] if t0 > 0 else None
        prevx = p["x"][:, t0 - 1] if t0 > 0 else None
        y_loc, g = oracle.scan(sl(p["x"]), sl(p["dt"]), p["A"], sl(p["B"]), sl(p["C"]), sl(p["lam"]),
                               sl(p["theta"]), prevB=prevB, prevx=prevx)
        # the segment's homogeneous propagator: prefix decays and angles from t_s
        log_a = np.cumsum(sl(p["dt"]) * p["A"][None, None, :], axis=1)    # [b, seg, h]
        phi = np.cumsum(sl(p["theta"]), axis=1)                             # [b, seg, h, K]
        # 2. all-gather (a_s, phi_s, g_s) and fold the earlier ranks' pairs
        mine = torch.from_numpy(np.concatenate([np.exp(log_a[:, -1]).ravel(), phi[:, -1].ravel(), g.ravel()]))
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        b, H = log_a.shape[0], log_a.shape[2]
        K, N, P = phi.shape[-1], g.shape[-2], g.shape[-1]
        h_in = np.zeros((b, H, N, P))
        for s in range(rank):
            v = got[s].numpy()
            a_s = v[:b * H].reshape(b, H)
            phi_s = v[b * H:b * H + b * H * K].reshape(b, H, K)
            g_s = v[b * H + b * H * K:].reshape(b, H, N, P)
            h_in = a_s[..., None, None] * _rot_rows(h_in, phi_s) + g_s
        # 3. correct the outputs and the end state with the propagated h_in
        y = y_loc.copy()
        for t in range(t1 - t0):
            ht = np.exp(log_a[:, t])[..., None, None] * _rot_rows(h_in, phi[:, t])   # [b, h, N, P]
            y[:, t] += np.einsum("bhrn,bhnp->bhrp", sl(p["C"])[:, t], ht)
        h_end = np.exp(log_a[:, -1])[..., None, None] * _rot_rows(h_in, phi[:, -1]) + g
        out[rank] = (y, h_end)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,R", [(2, 1), (4, 2)])
def test_tsharded_scan_matches_the_whole_sequence(world, R):
    import oracle
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, R, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == set(range(world))
    p = _problem(R)
    y_ref, h_ref = oracle.scan(p["x"], p["dt"], p["A"], p["B"], p["C"], p["lam"], p["theta"])
    y = np.concatenate([res[r][0] for r in range(world)], axis=1)
    assert np.abs(y - y_ref).max() <= 1e-12 * np.abs(y_ref).max()
    # the last rank's end state is the sequence's final state
    assert np.abs(res[world - 1][1] - h_ref).max() <= 1e-12 * np.abs(h_ref).max()


def test_dropping_the_boundary_beta_term_is_detected():
    """Without the previous token's beta term at the segment start, the
    sharded result is not the sequence's: the exchange must carry it."""
    import oracle
    p = _problem(1)
    T = p["x"].shape[1]
    t0 = T // 2
    sl = lambda a: a[:, t0:]
    _, h_ref = oracle.scan(p["x"], p["dt"], p["A"], p["B"], p["C"], p["lam"], p["theta"])
    _, h_half = oracle.scan(p["x"][:, :t0], p["dt"][:, :t0], p["A"], p["B"][:, :t0], p["C"][:, :t0],
                            p["lam"][:, :t0], p["theta"][:, :t0])
    _, g = oracle.scan(sl(p["x"]), sl(p["dt"]), p["A"], sl(p["B"]), sl(p["C"]), sl(p["lam"]), sl(p["theta"]))
    log_a = np.sum(sl(p["dt"]) * p["A"][None, None, :], axis=1)
    phi = np.sum(sl(p["theta"]), axis=1)
    h_wrong = np.exp(log_a)[..., None, None] * _rot_rows(h_half, phi) + g
    assert np.abs(h_wrong - h_ref).max() > 1e-6 * np.abs(h_ref).max()
