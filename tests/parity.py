"""Helpers for GPU-vs-oracle parity: run the CUDA path through the C ABI and the fp64 oracle
on the same seeded inputs, and compare with the magnitude-relative metric.

Tolerances (max relative error against max(|oracle|, magnitude companion)): 1e-5 for fp32
I/O and 2e-2 for bf16 I/O, for y and for the final state.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_153_b300 import gen, ssm

TOL = {"f32": 1e-5, "bf16": 2e-2}


def to_dev(inp, dev="cuda"):
    out = {}
    for k, v in inp.items():
        out[k] = v.to(dev) if isinstance(v, torch.Tensor) else v
    return out


def gpu_scan(inp, stream=None, workspace=None, discretization="euler"):
    g = to_dev(inp)
    y, h = ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                  delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                                  return_last_state=True, stream=stream, workspace=workspace,
                                  discretization=discretization)
    torch.cuda.synchronize()
    return y, h


def oracle_scan(inp, channels=None, nthreads=8, zoh=False):
    """Oracle on all channels, or on a list of (b, d) pairs (then packed [nch, ...])."""
    f = gen.as_f64
    if channels is None:
        return oracle.selective_scan(f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]),
                                     D=f(inp["D"]), z=f(inp["z"]), delta_bias=f(inp["delta_bias"]),
                                     delta_softplus=inp["delta_softplus"], with_mag=True, nthreads=nthreads,
                                     zoh=zoh)
    ch = np.asarray(channels, dtype=np.int64).reshape(-1, 2)
    bs, ds = ch[:, 0], ch[:, 1]

    def rows(t):
        if t is None:
            return None
        return t[torch.as_tensor(bs), torch.as_tensor(ds), :].to(torch.float64).numpy()

    A = f(inp["A"])[ds]
    D = None if inp["D"] is None else f(inp["D"])[ds]
    bias = None if inp["delta_bias"] is None else f(inp["delta_bias"])[ds]
    return oracle.scan_rows(rows(inp["u"]), rows(inp["delta"]), A, f(inp["B"]), f(inp["C"]), bs, D=D,
                            z=rows(inp["z"]), delta_bias=bias, delta_softplus=inp["delta_softplus"],
                            with_mag=True, nthreads=nthreads, zoh=zoh)


def compare_scan(inp, y_gpu, h_gpu, channels=None, tol=None, nthreads=8, zoh=False):
    io = inp["cfg"].io
    tol = TOL[io] if tol is None else tol
    yo, ho, ym, hm = oracle_scan(inp, channels, nthreads, zoh=zoh)
    if channels is None:
        yg = y_gpu.float().cpu().double().numpy()
        hg = h_gpu.cpu().double().numpy()
    else:
        ch = np.asarray(channels, dtype=np.int64).reshape(-1, 2)
        yg = y_gpu[ch[:, 0], ch[:, 1], :].float().cpu().double().numpy()
        hg = h_gpu[ch[:, 0], ch[:, 1], :].cpu().double().numpy()
    ey = oracle.rel_err(yg, yo, ym)
    eh = oracle.rel_err(hg, ho, hm)
    assert ey <= tol, f"y parity {ey:.3e} > {tol}"
    assert eh <= tol, f"state parity {eh:.3e} > {tol}"
    return ey, eh


def sample_channels(Bt, Dm, k, seed=0):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (Bt - 1, Dm - 1), (0, Dm - 1), (Bt - 1, 0)}
    while len(picks) < min(k, Bt * Dm):
        picks.add((int(rng.integers(Bt)), int(rng.integers(Dm))))
    return sorted(picks)
