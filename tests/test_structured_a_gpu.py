"""Structured-A fast path of the forward scan (A[d, n] == (n + 1) * A[d, 0]: the decays of a
warp's states come from powers of exp(dt * A[d, 0])), through the C ABI, against the fp64
oracle. The oracle evaluates exp(dt * A[d, n]) per state whatever A is, so agreement pins the
power form; the general path's output is the second witness: warps that fail the test must
reproduce it bit for bit, warps that pass must not (they take the other arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_scan, gpu_scan, sample_channels, to_dev
from selective_state_space_153_b300 import build, gen, ssm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    ssm.load()


@pytest.fixture(autouse=True)
def _detect_on():
    prev = ssm.set_structured_a(True)
    yield
    ssm.set_structured_a(prev)


def _both(inp, **kw):
    """(y, h) with the structured-A test on, then off."""
    ssm.set_structured_a(True)
    on = gpu_scan(inp, **kw)
    ssm.set_structured_a(False)
    off = gpu_scan(inp, **kw)
    ssm.set_structured_a(True)
    return on, off


def test_switch_returns_previous_setting():
    assert ssm.set_structured_a(False) is True   # the fixture switched it on
    assert ssm.set_structured_a(False) is False
    assert ssm.set_structured_a(True) is False


CASES = [
    # Bt, D, L, N, io, gate, dskip, states per lane (KS), chunks (0 = planner's choice)
    (1, 3, 200, 4, "f32", False, "ones", "4", 0),        # one lane per channel pair
    (2, 70, 520, 8, "bf16", True, "normal", "4", 0),
    (1, 100, 1000, 16, "f32", False, "ones", "4", 3),
    (2, 67, 136, 8, "f32", True, None, "8", 0),
    (3, 45, 1000, 16, "f32", True, "ones", "8", 2),
    (1, 50, 776, 32, "bf16", True, "normal", "8", 0),
    (1, 40, 2000, 64, "f32", False, "ones", "8", 5),     # the long-sequence lane split, chunked
    (1, 20, 520, 128, "bf16", True, "ones", "8", 4),
    (2, 33, 40, 128, "f32", False, "normal", "8", 1),    # a short ragged tile
    (1, 40, 2000, 64, "f32", False, "ones", "16", 5),    # sixteen states per lane
]


@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,ks,chunks", CASES)
def test_structured_shapes(Bt, D, L, N, io, gate, dskip, ks, chunks):
    cfg = gen.ScanConfig("st", Bt, D, L, N, io=io, gate=gate, dskip=dskip, seed=31 * L + N)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(pair_states_per_lane=int(ks), chunks=chunks):
        (y, h), (y0, h0) = _both(inp)
    compare_scan(inp, y, h)
    # the fast path ran: the fp32 final state differs from the general path's in rounding
    assert not torch.equal(h, h0)


def test_scaled_structured_a():
    """A[d, n] = (n + 1) * a_d with a per-channel a_d (exact products): still structured."""
    cfg = gen.ScanConfig("sc", 2, 40, 300, 16, io="f32", gate=True, dskip="normal", seed=5)
    inp = gen.scan_inputs(cfg)
    a = torch.tensor([0.25, 0.5, 1.5, 2.0] * 10, dtype=torch.float32)
    inp["A"] = -(a[:, None] * torch.arange(1, 17, dtype=torch.float32)[None, :])
    (y, h), (y0, h0) = _both(inp)
    compare_scan(inp, y, h)
    assert not torch.equal(h, h0)


def test_unstructured_a_takes_general_path():
    cfg = gen.ScanConfig("un", 1, 64, 500, 16, io="f32", gate=True, dskip="ones", seed=9)
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(9)
    inp["A"] = torch.from_numpy(-rng.uniform(0.2, 4.0, (64, 16)).astype(np.float32))
    (y, h), (y0, h0) = _both(inp)
    assert torch.equal(y, y0) and torch.equal(h, h0)
    compare_scan(inp, y, h)


def test_one_broken_channel_falls_back_alone():
    """One channel whose A misses the pattern by one ulp: its warp takes the general path (bit
    for bit), the other warps keep the fast path, and everything matches the oracle."""
    cfg = gen.ScanConfig("mx", 1, 256, 600, 64, io="f32", gate=False, dskip="ones", seed=12)
    inp = gen.scan_inputs(cfg)
    bad = 77
    inp["A"][bad, 5] = float(np.nextafter(np.float32(inp["A"][bad, 5]), np.float32(0.0)))
    (y, h), (y0, h0) = _both(inp)
    assert torch.equal(y[0, bad], y0[0, bad]) and torch.equal(h[0, bad], h0[0, bad])
    assert not torch.equal(h, h0)
    compare_scan(inp, y, h)


def test_padded_states_take_general_path():
    """dstate 24 with eight states per lane pads the lane's states to 32: no warp qualifies."""
    cfg = gen.ScanConfig("pd", 2, 30, 400, 24, io="f32", gate=True, dskip="normal", seed=4)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(pair_states_per_lane=8):
        (y, h), (y0, h0) = _both(inp)
    assert torch.equal(y, y0) and torch.equal(h, h0)
    compare_scan(inp, y, h)


def test_zero_a_is_structured_prefix_sum():
    """A = 0 passes the test (0 == (n+1)*0): the decays are exactly 1 and h is a prefix sum."""
    cfg = gen.ScanConfig("za", 1, 16, 256, 16, io="f32", gate=False, dskip=None, seed=6)
    inp = gen.scan_inputs(cfg)
    inp["A"] = torch.zeros(16, 16)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


@pytest.mark.parametrize("N,io,chunks", [(16, "f32", 0), (64, "bf16", 3)])
def test_structured_zoh(N, io, chunks):
    cfg = gen.ScanConfig("sz", 2, 40, 720, N, io=io, gate=True, dskip="ones", seed=N + 1)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(chunks=chunks):
        (y, h), (y0, h0) = _both(inp, discretization="zoh")
    compare_scan(inp, y, h, zoh=True)
    assert not torch.equal(h, h0)


def test_structured_conv_front():
    Bt, D, L, N, K = 2, 48, 640, 16, 4
    cfg = gen.ScanConfig("scv", Bt, D, L, N, io="f32", gate=True, dskip="ones", seed=21)
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(22)
    w = torch.from_numpy(rng.standard_normal((D, K)).astype(np.float32) * 0.5)
    cb = torch.from_numpy(rng.standard_normal(D).astype(np.float32) * 0.2)
    g = to_dev(inp)
    y, h = ssm.conv_selective_scan_fwd(g["u"], w.cuda(), cb.cuda(), g["delta"], g["A"], g["B"], g["C"], D=g["D"],
                                       z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True,
                                       return_last_state=True)
    torch.cuda.synchronize()
    u = oracle.conv_silu(gen.as_f64(inp["u"]), np.broadcast_to(w.double().numpy(), (Bt, D, K)),
                         np.broadcast_to(cb.double().numpy(), (Bt, D)))
    ref = dict(inp)
    ref["u"] = torch.from_numpy(u)
    compare_scan(ref, y, h)


def test_long128k_structured_sampled():
    """The long-sequence workload (1 x 1536 x 131072 x 64, bf16) on the fast path, sampled
    channels over the whole length."""
    inp = gen.scan_inputs(gen.LONG128K)
    y, h = gpu_scan(inp)
    assert torch.isfinite(y.float()).all()
    compare_scan(inp, y, h, channels=sample_channels(1, 1536, 10, seed=11))


def test_m130_structured_sampled():
    inp = gen.scan_inputs(gen.M130)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h, channels=sample_channels(8, 1536, 32, seed=2))
