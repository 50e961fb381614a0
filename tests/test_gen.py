"""The seeded generator: deterministic, the documented shapes, dtypes and distributions."""
import math

import numpy as np
import torch

from selective_state_space_153_b300 import gen


def test_deterministic_and_seeded():
    a = gen.scan_inputs(gen.BLOCK512)
    b = gen.scan_inputs(gen.BLOCK512)
    c = gen.scan_inputs(gen.BLOCK512, seed=99)
    for k in ("u", "delta", "B", "C", "z", "D", "delta_bias"):
        assert torch.equal(a[k], b[k]), k
        assert not torch.equal(a[k], c[k]), k


def test_shapes_dtypes():
    for cfg in (gen.TINY, gen.BLOCK512):
        x = gen.scan_inputs(cfg)
        io = torch.float32 if cfg.io == "f32" else torch.bfloat16
        assert x["u"].shape == (cfg.Bt, cfg.D, cfg.L) and x["u"].dtype == io
        assert x["B"].shape == (cfg.Bt, cfg.N, cfg.L) and x["C"].dtype == io
        assert x["A"].shape == (cfg.D, cfg.N) and x["A"].dtype == torch.float32
        assert torch.equal(x["A"][0], -torch.arange(1, cfg.N + 1, dtype=torch.float32))
        assert (x["z"] is not None) == cfg.gate


def test_step_bias_range():
    x = gen.scan_inputs(gen.BLOCK512)
    sp = np.logaddexp(0.0, x["delta_bias"].double().numpy())
    assert sp.min() >= 1e-3 * (1 - 1e-5) and sp.max() <= 1e-1 * (1 + 1e-5)
    # log-uniform: the median of log(softplus(bias)) is near the middle of the range
    mid = 0.5 * (math.log(1e-3) + math.log(1e-1))
    assert abs(np.median(np.log(sp)) - mid) < 0.3


def test_ar1_input():
    x = gen.scan_inputs(gen.LONG128K, D=8, L=20000)
    u = x["u"].double().numpy()[0]
    r = (u[:, 1:] * u[:, :-1]).mean() / (u * u).mean()
    assert abs(r - 0.9) < 0.02 and abs(u.var() - 1.0) < 0.15


def test_decode_inputs():
    d = gen.decode_inputs(Bt=4, D=16, steps=3)
    assert d["x"].shape == (3, 4, 16) and d["B"].shape == (3, 4, 16)
    assert d["state0"].dtype == torch.float32 and d["dt"].dtype == torch.bfloat16
    assert float(d["dt"].float().min()) > 0


def test_per_channel_A_recipes():
    """``scaled`` and ``random`` give every channel its own row of A (so that a kernel reading
    A[n] for A[d, n] fails parity), negative, and leave every other array unchanged."""
    base = gen.scan_inputs(gen.BLOCK512)
    for kind in ("scaled", "random"):
        x = gen.scan_inputs(gen.BLOCK512, a_kind=kind)
        A = x["A"].double().numpy()
        assert A.shape == (512, 16) and x["A"].dtype == torch.float32
        assert (A < 0).all()
        assert len({tuple(r) for r in A}) == 512, "rows must differ between channels"
        for k in ("u", "delta", "B", "C", "z", "D", "delta_bias"):
            assert torch.equal(x[k], base[k]), k
    sc = gen.scan_inputs(gen.BLOCK512, a_kind="scaled")["A"].double().numpy()
    ratio = sc / sc[:, :1]
    assert np.allclose(ratio, np.arange(1, 17)[None, :], rtol=1e-6)   # (n+1) * a_d
    d = gen.decode_inputs(Bt=2, D=8, steps=1, a_kind="random")
    assert len({tuple(r) for r in d["A"].numpy()}) == 8
