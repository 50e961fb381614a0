"""Gradients of the selective scan for the backward parity tests.

TEST INFRASTRUCTURE, like the rest of oracle/: only tests/, the smoke check and the
benchmark's CPU baseline may import it; the CUDA path never does.

The forward is the per-timestep loop of section 3.2 of "From RNN to Mamba: state-space
model principles and long-sequence modelling in practice" (lmnt.cn), written with plain
PyTorch CPU ops in float64 (dt = softplus(delta + bias) with PyTorch's defaults, A_bar =
exp(dt*A), B_bar = dt*B, h = A_bar*h + B_bar*u, y = sum_n C*h + D*u, y *= SiLU(z)); the
gradients are PyTorch autograd of that loop for a given upstream gradient dy (and, if given,
a gradient of the final state). Section 2.2 of the same page: training differentiates
through the parallel form of this recurrence; the loop and its autograd are the plain
definition the GPU kernel must match. The forward is checked against the C oracle and the
gradients against central finite differences of the C oracle (tests/oracle_pins.py).
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch


def scan_forward_torch(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
    """Float64 torch forward: u, delta, z [Bt, D, L]; A [D, N]; B, C [Bt, N, L]; D, bias [D].
    Returns (y [Bt, D, L], last_state [Bt, D, N])."""
    Bt, Dm, L = u.shape
    N = A.shape[1]
    v = delta + (delta_bias[None, :, None] if delta_bias is not None else 0.0)
    dt = torch.nn.functional.softplus(v) if delta_softplus else v
    h = torch.zeros(Bt, Dm, N, dtype=torch.float64)
    ys = []
    for t in range(L):
        a = torch.exp(dt[:, :, t, None] * A[None, :, :])
        h = a * h + dt[:, :, t, None] * B[:, None, :, t] * u[:, :, t, None]
        yt = (h * C[:, None, :, t]).sum(-1)
        if D is not None:
            yt = yt + D[None, :] * u[:, :, t]
        ys.append(yt)
    y = torch.stack(ys, -1)
    if z is not None:
        y = y * torch.nn.functional.silu(z)
    return y, h


def scan_backward(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                  dy=None, dlast=None) -> Dict[str, Optional[np.ndarray]]:
    """Gradients (float64 numpy) of sum(y * dy) + sum(last_state * dlast) with respect to
    u, delta, A, B, C, D, z and delta_bias (None where the input is absent)."""
    def t64(x):
        return None if x is None else torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)
    tu, tdl, tA, tB, tC = t64(u), t64(delta), t64(A), t64(B), t64(C)
    tD, tz, tb = t64(D), t64(z), t64(delta_bias)
    y, h = scan_forward_torch(tu, tdl, tA, tB, tC, tD, tz, tb, delta_softplus)
    loss = (y * torch.as_tensor(np.asarray(dy, dtype=np.float64))).sum()
    if dlast is not None:
        loss = loss + (h * torch.as_tensor(np.asarray(dlast, dtype=np.float64))).sum()
    loss.backward()
    g = lambda t: None if t is None else t.grad.detach().numpy()  # noqa: E731
    return {"u": g(tu), "delta": g(tdl), "A": g(tA), "B": g(tB), "C": g(tC), "D": g(tD),
            "z": g(tz), "delta_bias": g(tb)}
