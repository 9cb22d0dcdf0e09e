"""The fp32 arithmetic the acceptance kernel uses for the draft-q rule keeps
its decisions inside the oracle's tie band (1e-5 relative).  The kernel's
steps are written out here in numpy float32 (softmax at T, the residual pair
(c, F) with c <- c + F, r = max(p - c q, 0) / F, accept iff u < min(1, r / q));
the exponential is numpy's, not the GPU's, whose relative error is of the same
order.  On random star trees with long rejection chains, every decision the
oracle does not flag as a near tie must agree with the fp64 oracle's."""
import numpy as np
import pytest

import oracle as O

f32 = np.float32


def _fp32_decision(pz, qz, toks, us, T):
    invT = f32(1.0) / f32(T)
    y = (pz.astype(f32) * invT).astype(f32)
    yd = (qz.astype(f32) * invT).astype(f32)
    ep = np.exp((y - y.max()).astype(f32), dtype=f32)
    eq = np.exp((yd - yd.max()).astype(f32), dtype=f32)
    p = (ep * (f32(1) / ep.sum(dtype=f32))).astype(f32)
    q = (eq * (f32(1) / eq.sum(dtype=f32))).astype(f32)
    c, F = f32(0), f32(1)
    for k, (x, u) in enumerate(zip(toks, us)):
        r = f32(max(np.float64(p[x]) - np.float64(c) * np.float64(q[x]), 0.0)) / F
        ratio = f32(1) if q[x] <= 0 else min(f32(1), f32(r / q[x]))
        if u < ratio:
            return k
        c1 = f32(c + F)
        F1 = np.maximum((p.astype(np.float64) - np.float64(c1) * q.astype(np.float64)).astype(f32), f32(0)).sum(dtype=f32)
        if F1 > 0:
            c, F = c1, F1
    return -1


@pytest.mark.parametrize("kmin,kmax,squeezes,cases,seed", [(2, 10, (1.0, 0.1, 0.01), 250, 5),
                                                          (10, 30, (0.01, 0.001), 80, 6)])
def test_draftq_fp32_decisions_stay_in_the_tie_band(kmin, kmax, squeezes, cases, seed):
    rng = np.random.default_rng(seed)
    checked = 0
    for _ in range(cases):
        V = int(rng.choice([50, 500, 4000]))
        k = int(rng.integers(kmin, kmax + 1))
        T = float(rng.choice([0.7, 1.0, 1.3]))
        pz = np.empty(V, np.float32)
        pz[rng.permutation(V)] = (-1.2 * np.log(np.arange(1, V + 1)) + rng.standard_normal(V)).astype(np.float32)
        qz = (pz + rng.uniform(0.3, 1.5) * rng.standard_normal(V)).astype(np.float32)
        toks = rng.choice(V, k, p=O.softmax_t(qz, T))  # children drawn i.i.d. from q
        us = (1.0 - (1.0 - rng.random(k)) * rng.choice(squeezes)).astype(np.float32)
        cfg = O.TreeCfg(B=1, V=V, depth=1, topk=k, m=1, n=k, temperature=T)
        res = O.verify_accept(cfg, O.STOCH_DRAFTQ, np.array([[0] + list(toks)], np.int32),
                              np.array([[-1] + [0] * k], np.int32), np.arange(-1, k, dtype=np.int32)[None],
                              np.stack([pz] * (k + 1)), None, uniforms=np.array([[0.5] + list(us)], np.float32),
                              draft_table=np.stack([qz] * (k + 1)))
        if any(what == "accept" for _, what, _ in res.near_ties):
            continue
        want = int(res.path[0, 1]) - 1 if res.accept_len[0] > 0 else -1
        assert _fp32_decision(pz, qz, toks, us, T) == want
        checked += 1
    assert checked >= int(0.95 * cases)
