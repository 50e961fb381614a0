"""GPU (C ABI) against the fp64 oracle, element by element, on seeded inputs."""
import os

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, compare_scan, gpu_scan, sample_channels, to_dev
from selective_state_space_153_b300 import build, gen, ssm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    ssm.load()


@pytest.fixture(autouse=True)
def _general_path():
    """The generators' A = -(n+1) passes the structured-A test; these cases check the general
    path, so the test is kept off around each of them (it is off by default). The fast path
    has its own module (test_structured_a_gpu.py)."""
    prev = ssm.set_structured_a(False)
    yield
    ssm.set_structured_a(prev)


# ---- the workloads ------------------------------------------------------------------------
def test_tiny_fp32():
    inp = gen.scan_inputs(gen.TINY)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


def test_block512_bf16_full():
    inp = gen.scan_inputs(gen.BLOCK512)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


def test_m130_full_size_sampled():
    inp = gen.scan_inputs(gen.M130)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h, channels=sample_channels(8, 1536, 48))


def test_long128k_full_size_sampled():
    inp = gen.scan_inputs(gen.LONG128K)
    y, h = gpu_scan(inp)
    assert torch.isfinite(y.float()).all()
    compare_scan(inp, y, h, channels=sample_channels(1, 1536, 12, seed=3))


@pytest.mark.parametrize("a_kind", ["scaled", "random"])
def test_long128k_per_channel_A_sampled(a_kind):
    """The full-size long-sequence launch (its chunks, carries and combine) with a different
    row of A in every channel, checked on sampled channels over the whole sequence."""
    inp = gen.scan_inputs(gen.LONG128K, a_kind=a_kind)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h, channels=sample_channels(1, 1536, 8, seed=11))


def test_m130_per_channel_A_sampled():
    inp = gen.scan_inputs(gen.M130, a_kind="random")
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h, channels=sample_channels(8, 1536, 24, seed=12))


# ---- shapes and options -------------------------------------------------------------------
CASES = [
    # Bt, D, L, N, io, gate, dskip, bias, softplus
    (1, 1, 1, 1, "f32", False, "ones", True, True),
    (1, 5, 7, 3, "f32", True, "normal", True, True),
    (2, 37, 33, 16, "f32", True, None, False, False),
    (1, 3, 100, 17, "bf16", False, "ones", True, True),
    (3, 9, 129, 64, "bf16", True, "normal", True, True),
    (1, 40, 257, 100, "f32", True, "ones", True, True),
    (2, 33, 96, 128, "bf16", False, None, True, True),
    (1, 130, 64, 8, "bf16", True, "ones", True, False),
    (2, 64, 1000, 32, "f32", True, "normal", True, True),
    (1, 7, 4097, 4, "f32", False, "ones", True, True),
]


# A recipe per case: the s4d row shared by every channel, a per-channel scaled row, or an
# independent random value per (channel, state)
A_KINDS = ("s4d", "scaled", "random")


@pytest.mark.parametrize("a_kind", A_KINDS)
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,sp", CASES)
def test_shapes(Bt, D, L, N, io, gate, dskip, bias, sp, a_kind):
    cfg = gen.ScanConfig("case", Bt, D, L, N, io=io, gate=gate, dskip=dskip, bias=bias, softplus=sp, seed=L + N,
                         a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    if not sp:  # without the softplus the raw step itself must be a positive step
        inp["delta"] = (inp["delta"].float().abs() * 0.2).to(inp["delta"].dtype)
        if inp["delta_bias"] is not None:
            inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


# ---- the channel-pair kernel: every lane split, ragged tails, partial channel blocks ------
PAIR_CASES = [
    # Bt, D, L, N, io, gate, dskip, states per lane (KS), chunks (0 = planner's choice)
    (1, 3, 200, 4, "f32", False, "ones", "4", 0),        # KS 4, one lane per pair
    (2, 70, 520, 8, "bf16", True, "normal", "4", 0),     # KS 4, two lanes per pair
    (1, 100, 1000, 16, "bf16", False, "ones", "4", 3),   # KS 4, four lanes per pair
    (2, 67, 136, 7, "f32", True, None, "8", 0),          # KS 8, one lane per pair
    (3, 45, 1000, 16, "bf16", True, "ones", "8", 2),     # KS 8, two lanes per pair
    (1, 50, 776, 24, "bf16", True, "normal", "8", 0),    # KS 8, four lanes per pair
    (1, 40, 2000, 64, "bf16", False, "ones", "8", 5),    # KS 8, eight lanes per pair
    (3, 9, 136, 50, "f32", True, "normal", "8", 0),      # KS 8, eight lanes, padded states
    (1, 20, 520, 100, "bf16", True, "ones", "8", 4),     # KS 8, sixteen lanes per pair
    (2, 33, 40, 128, "f32", False, "normal", "8", 1),    # KS 8, sixteen lanes, a short ragged tile
    (1, 40, 2000, 64, "f32", False, "ones", "16", 5),    # KS 16, four lanes per pair
    (1, 24, 8192, 16, "bf16", True, "normal", "4", 100),  # 86 chunks, 384 pairs: the grouped combine
    (1, 24, 8192, 64, "f32", False, "ones", "16", 200),   # 128 chunks (the cap at L/64), grouped
    (2, 70, 520, 48, "bf16", True, "normal", "16", 3),   # KS 16, padded states, partial channel block
    (3, 9, 136, 40, "f32", True, "ones", "16", 0),       # KS 16, padded states, planner's chunks
]


@pytest.mark.parametrize("a_kind", A_KINDS)
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,ks,chunks", PAIR_CASES)
def test_pair_kernel_shapes(Bt, D, L, N, io, gate, dskip, ks, chunks, a_kind):
    cfg = gen.ScanConfig("pair", Bt, D, L, N, io=io, gate=gate, dskip=dskip, seed=Bt * 1000 + L + N, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(pair_states_per_lane=int(ks), chunks=chunks):
        y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


# ---- backward: gradients against float64 autograd of the loop (oracle/backward.py) --------
BWD_CASES = [
    # Bt, D, L, N, io, gate, dskip, bias, dlast, A recipe
    (1, 4, 64, 4, "f32", False, "ones", True, False, "s4d"),
    (2, 7, 100, 16, "f32", True, "normal", True, True, "random"),
    (1, 5, 40, 64, "f32", True, "ones", False, False, "scaled"),
    (1, 3, 33, 100, "f32", False, None, True, True, "random"),
    (2, 9, 70, 16, "bf16", True, "normal", True, False, "scaled"),
    (1, 40, 48, 8, "f32", False, "ones", True, False, "random"),
    (3, 33, 130, 32, "f32", True, "normal", True, True, "scaled"),
    (2, 37, 96, 16, "bf16", True, "ones", True, True, "random"),   # bf16 rows of whole 16-byte pieces
]


def _grad_err(got, ref):
    """Element-wise relative error with a magnitude floor: max_i |g_i - r_i| / max(|r_i|, f),
    f = 1e-3 * max|r|. An element 100x smaller than the largest is held to its own size
    (a max-normalised metric would let it be entirely wrong); the floor only keeps elements
    that are zero up to cancellation from dividing by ~0."""
    floor = 1e-3 * max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,dlast,a_kind", BWD_CASES)
def test_backward_gradients(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind):
    _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind)


@pytest.mark.parametrize("q", [2, 4])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,dlast,a_kind", [c for c in BWD_CASES if c[3] <= 32])
def test_backward_gradients_forced_split(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind, q):
    """Both lane splits of the backward on every case that has both (the planner takes two
    states per lane for small channel counts, four otherwise)."""
    with ssm.plan_override(bwd_states_per_lane=q):
        _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind)


@pytest.mark.parametrize("cfg", [gen.M130, gen.BWD_LONG], ids=["m130", "bwd_long"])
def test_backward_full_size_sampled_channels(cfg):
    """The bench's backward workloads at full size, in the launch configuration the planner
    gives them (8 x 1536 x 2048 x 16 unsplit; 1 x 1536 x 16384 x 16 split into 37 chunks):
    the gradients that belong to one channel -- du, ddelta, dz over every batch row and step,
    and dA, dD, dbias -- for sampled channels, against the float64 oracle run on those
    channels alone (the channels of the scan are independent given B and C). dB and dC sum
    over every channel, so they are compared at the small sizes above."""
    from oracle import backward as obwd
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(cfg.L)
    dy = torch.from_numpy(rng.standard_normal((cfg.Bt, cfg.D, cfg.L)).astype(np.float32)).to(inp["u"].dtype)
    g = to_dev(inp)
    got = ssm.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.cuda(), D=g["D"], z=g["z"],
                                 delta_bias=g["delta_bias"], delta_softplus=True)
    torch.cuda.synchronize()
    f = gen.as_f64
    for d in (0, 777, cfg.D - 1):
        sl = slice(d, d + 1)
        ref = obwd.scan_backward(f(inp["u"][:, sl]), f(inp["delta"][:, sl]), f(inp["A"][sl]), f(inp["B"]), f(inp["C"]),
                                 D=f(inp["D"][sl]), z=f(inp["z"][:, sl]), delta_bias=f(inp["delta_bias"][sl]),
                                 delta_softplus=True, dy=f(dy[:, sl]))
        for k, gk in (("u", got["u"][:, sl]), ("delta", got["delta"][:, sl]), ("z", got["z"][:, sl]),
                      ("A", got["A"][sl]), ("D", got["D"][sl]), ("delta_bias", got["delta_bias"][sl])):
            err = _grad_err(gk.double().cpu().numpy(), ref[k])
            assert err <= 5e-2, f"channel {d}, d{k}: element-wise error {err:.3e}"


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,dlast,a_kind", BWD_CASES[:5])
def test_backward_without_softplus(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind, chunks):
    """delta_softplus = 0: dt = delta + bias directly, so ddelta = ddt (no sigmoid factor)."""
    with ssm.plan_override(bwd_chunks=chunks):
        _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind, softplus=False)


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward_rows_off_pair_alignment(io, chunks):
    """Even length with every input one element off a 2-element boundary: the rows are read
    one step per load instead of two (also under a time split)."""
    with ssm.plan_override(bwd_chunks=chunks):
        _check_backward(2, 9, 70, 16, io, True, "normal", True, True, "scaled", odd_offset=True)


@pytest.mark.parametrize("chunks", [2, 3, 7])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,dlast,a_kind", BWD_CASES)
def test_backward_gradients_time_split(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind, chunks):
    """The sequence cut into chunks of whole 8-step segments (the last one ragged where the
    segments do not divide evenly; 7 is clamped to the segment count on the shortest cases):
    chunk-local checkpoints corrected by the combined chunk states, adjoint carries from the
    aggregate pass."""
    with ssm.plan_override(bwd_chunks=chunks):
        _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind)


def test_backward_empty_sequence():
    """seqlen = 0: no step contributes, so the parameter gradients (dA, dD, d bias) come back
    as zeros and nothing else is touched."""
    g = {"u": torch.empty((2, 5, 0), dtype=torch.float32, device="cuda"),
         "delta": torch.empty((2, 5, 0), dtype=torch.float32, device="cuda"),
         "A": -torch.ones((5, 4), dtype=torch.float32, device="cuda"),
         "B": torch.empty((2, 4, 0), dtype=torch.float32, device="cuda"),
         "C": torch.empty((2, 4, 0), dtype=torch.float32, device="cuda"),
         "D": torch.ones(5, dtype=torch.float32, device="cuda"),
         "bias": torch.zeros(5, dtype=torch.float32, device="cuda")}
    dy = torch.empty((2, 5, 0), dtype=torch.float32, device="cuda")
    got = ssm.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, D=g["D"], delta_bias=g["bias"])
    torch.cuda.synchronize()
    for k in ("A", "D", "delta_bias"):
        assert torch.equal(got[k], torch.zeros_like(got[k])), k
    assert ssm.stream_status() == ssm.SSM_OK


@pytest.mark.parametrize("L,chunks", [(560, 40), (512, 64), (560, 100)])
def test_backward_time_split_many_chunks(L, chunks):
    """Many chunks of one or two 8-step segments: 32 to 64 chunks take the combine's warp scan
    (560 steps, 40 asked: 35 chunks of 2 segments, lanes past the last chunk; 512 steps: 64
    chunks, every lane two), more than 64 its loop (560 steps, 100 asked: 70 chunks)."""
    with ssm.plan_override(bwd_chunks=chunks):
        _check_backward(2, 9, L, 16, "bf16", True, "normal", True, True, "scaled")


@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,bias,dlast,a_kind", [c for c in BWD_CASES if c[3] <= 32])
def test_backward_time_split_two_states_per_lane(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind):
    with ssm.plan_override(bwd_chunks=3, bwd_states_per_lane=2):
        _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind)


def test_backward_planner_time_split():
    """One channel block over 2048 steps: the planner cuts the sequence into 16 chunks by
    itself (fewer than two CTAs per SM otherwise)."""
    _check_backward(1, 32, 2048, 16, "bf16", True, "ones", True, True, "random")


def _odd_offset(t):
    """t's values at a storage offset of one element (no 2-element alignment)."""
    if t is None:
        return None
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


def _check_backward(Bt, D, L, N, io, gate, dskip, bias, dlast, a_kind, odd_offset=False, softplus=True):
    from oracle import backward as obwd
    cfg = gen.ScanConfig("bwd", Bt, D, L, N, io=io, gate=gate, dskip=dskip, bias=bias, seed=3 * L + N,
                         a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    if not softplus:  # the raw step is the step itself: keep it positive
        inp["delta"] = (inp["delta"].float().abs() * 0.2).to(inp["delta"].dtype)
        if inp["delta_bias"] is not None:
            inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    rng = np.random.default_rng(L + N)
    dy = torch.from_numpy(rng.standard_normal((Bt, D, L)).astype(np.float32)).to(inp["u"].dtype)
    dl = torch.from_numpy(rng.standard_normal((Bt, D, N)).astype(np.float32)) if dlast else None
    g = to_dev(inp)
    dyd = dy.cuda()
    if odd_offset:
        for k in ("u", "delta", "B", "C", "z"):
            g[k] = _odd_offset(g[k])
        dyd = _odd_offset(dyd)
    got = ssm.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dyd, D=g["D"], z=g["z"],
                                 delta_bias=g["delta_bias"], delta_softplus=softplus,
                                 dlast_state=None if dl is None else dl.cuda())
    torch.cuda.synchronize()
    f = gen.as_f64
    ref = obwd.scan_backward(f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), D=f(inp["D"]),
                             z=f(inp["z"]), delta_bias=f(inp["delta_bias"]), delta_softplus=softplus, dy=f(dy),
                             dlast=None if dl is None else f(dl))
    # fp32: sums of up to L*N*D terms in fp32 with atomics, compared element by element;
    # bf16: the rounding of the bf16 inputs' products at 2^-9
    tol = 1e-3 if io == "f32" else 5e-2
    for k, r in ref.items():
        if r is None:
            assert got[k] is None
            continue
        err = _grad_err(got[k].double().cpu().numpy(), r)
        assert err <= tol, f"d{k}: element-wise error {err:.3e} (tol {tol})"


# ---- conv1d + SiLU front fused in the scan (lmnt.cn sections 3.1-3.2) --------------------
CONV_CASES = [
    # Bt, D, L, N, io, gate, dskip, K, forced chunks (0 = planner)
    (1, 4, 64, 4, "f32", False, "ones", 4, 0),
    (2, 37, 1000, 16, "bf16", True, "normal", 4, 0),
    (1, 50, 2000, 64, "bf16", False, "ones", 4, 5),
    (3, 20, 520, 32, "f32", True, "ones", 3, 3),
    (2, 33, 136, 16, "f32", True, None, 2, 4),
    (1, 16, 96, 8, "bf16", False, "ones", 1, 2),
]


def _conv_case(Bt, D, L, N, io, gate, dskip, K, seed, a_kind="s4d"):
    cfg = gen.ScanConfig("conv", Bt, D, L, N, io=io, gate=gate, dskip=dskip, seed=seed, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(seed + 1)
    w = torch.from_numpy(rng.standard_normal((D, K)).astype(np.float32) * 0.5)
    cb = torch.from_numpy(rng.standard_normal(D).astype(np.float32) * 0.2)
    return inp, w, cb


@pytest.mark.parametrize("a_kind", ["s4d", "random"])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,K,chunks", CONV_CASES)
def test_conv_front_shapes(Bt, D, L, N, io, gate, dskip, K, chunks, a_kind):
    inp, w, cb = _conv_case(Bt, D, L, N, io, gate, dskip, K, 13 * L + N + K, a_kind)
    g = to_dev(inp)
    with ssm.plan_override(chunks=chunks):
        y, h = ssm.conv_selective_scan_fwd(g["u"], w.cuda(), cb.cuda(), g["delta"], g["A"], g["B"], g["C"],
                                           D=g["D"], z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True,
                                           return_last_state=True)
    torch.cuda.synchronize()
    # oracle: the conv + SiLU span, then the scan on its output (same rows in double)
    u = oracle.conv_silu(gen.as_f64(inp["u"]), np.broadcast_to(w.double().numpy(), (Bt, D, K)),
                         np.broadcast_to(cb.double().numpy(), (Bt, D)))
    ref = dict(inp)
    ref["u"] = torch.from_numpy(u)
    compare_scan(ref, y, h)


@pytest.mark.parametrize("L,io", [(1001, "bf16"), (77, "f32")])
def test_conv_front_ragged_rows(L, io):
    """Rows that are not 16-byte multiples: padded copies in the workspace, then the fused
    conv front and scan; equal to the oracle. With a caller workspace too small for the
    copies the call returns SSM_ERR_WORKSPACE."""
    inp, w, cb = _conv_case(2, 9, L, 16, io, True, "ones", 4, 7 * L, "random")
    g = to_dev(inp)
    y, h = ssm.conv_selective_scan_fwd(g["u"], w.cuda(), cb.cuda(), g["delta"], g["A"], g["B"], g["C"], D=g["D"],
                                       z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True,
                                       return_last_state=True)
    torch.cuda.synchronize()
    u = oracle.conv_silu(gen.as_f64(inp["u"]), np.broadcast_to(w.double().numpy(), (2, 9, 4)),
                         np.broadcast_to(cb.double().numpy(), (2, 9)))
    ref = dict(inp)
    ref["u"] = torch.from_numpy(u)
    compare_scan(ref, y, h)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ssm.SsmError) as ei:
        ssm.conv_selective_scan_fwd(g["u"], w.cuda(), cb.cuda(), g["delta"], g["A"], g["B"], g["C"], workspace=small)
    assert ei.value.code == ssm.SSM_ERR_WORKSPACE


# ---- exact zero-order hold (jsqmd.com section 2.3), on the channel-pair kernel ----------
ZOH_CASES = [
    # Bt, D, L, N, io, gate, dskip, forced chunks (0 = planner)
    (1, 4, 64, 4, "f32", False, "ones", 0),
    (2, 37, 1000, 16, "f32", True, "normal", 0),
    (3, 20, 520, 32, "f32", True, "ones", 3),
    (1, 40, 2000, 64, "bf16", False, "ones", 5),
    (2, 33, 136, 128, "bf16", True, "normal", 0),
]


def _zoh_inputs(cfg):
    inp = gen.scan_inputs(cfg)
    # a zero and a tiny A column: the polynomial branch of (e^x - 1)/x and the A -> 0 limit;
    # with a per-channel recipe, the zero and the tiny value sit in different columns of
    # different channels
    A = inp["A"]
    if cfg.a_kind == "s4d":
        A[:, 0] = 0.0
        if A.shape[1] > 1:
            A[:, 1] = -1e-4
    else:
        d = torch.arange(A.shape[0])
        A[d, d % A.shape[1]] = 0.0
        if A.shape[1] > 1:
            A[d, (d + 1) % A.shape[1]] = -1e-4 * (1.0 + d.float() / A.shape[0])
    return inp


@pytest.mark.parametrize("a_kind", ["s4d", "scaled"])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip,chunks", ZOH_CASES)
def test_zoh_shapes(Bt, D, L, N, io, gate, dskip, chunks, a_kind):
    cfg = gen.ScanConfig("zoh", Bt, D, L, N, io=io, gate=gate, dskip=dskip, seed=7 * L + N, a_kind=a_kind)
    inp = _zoh_inputs(cfg)
    with ssm.plan_override(chunks=chunks):
        y, h = gpu_scan(inp, discretization="zoh")
    compare_scan(inp, y, h, zoh=True)
    # the flag matters: Euler differs from the ZOH oracle on these inputs
    with ssm.plan_override(chunks=chunks):
        ye, he = gpu_scan(inp)
    with pytest.raises(AssertionError):
        compare_scan(inp, ye, he, zoh=True)


def test_zoh_long128k_sampled():
    inp = gen.scan_inputs(gen.LONG128K)
    y, h = gpu_scan(inp, discretization="zoh")
    compare_scan(inp, y, h, channels=sample_channels(1, 1536, 8, seed=5), zoh=True)


def test_zoh_ragged_rows():
    """Rows that are not 16-byte multiples take the channel-pair kernel on padded copies, so
    the zero-order hold covers them; with a workspace too small for the copies it returns
    SSM_ERR_UNSUPPORTED (the element-wise kernel has no zero-order hold)."""
    cfg = gen.ScanConfig("zr", 2, 8, 1001, 16, io="bf16", gate=True, seed=3, a_kind="scaled")
    inp = _zoh_inputs(cfg)
    y, h = gpu_scan(inp, discretization="zoh")
    compare_scan(inp, y, h, zoh=True)
    g = to_dev(inp)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ssm.SsmError) as ei:
        ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], discretization="zoh", workspace=small)
    assert ei.value.code == ssm.SSM_ERR_UNSUPPORTED


@pytest.mark.parametrize("N,io,a_kind", [(16, "bf16", "s4d"), (64, "bf16", "random"), (5, "f32", "scaled")])
def test_zoh_decode(N, io, a_kind):
    inp = gen.decode_inputs(gen.DECODE, Bt=3, D=50, N=N, gate=True, dskip="ones", steps=7, a_kind=a_kind)
    inp["A"][:, 0] = 0.0
    if io == "f32":
        for k in ("x", "dt", "B", "C", "z"):
            inp[k] = inp[k].float()
    g = to_dev(inp)
    st = g["state0"].clone()
    ys = [ssm.state_update(st, g["x"][s], g["dt"][s], g["A"], g["B"][s], g["C"][s], D=g["D"], z=g["z"][s],
                           discretization="zoh") for s in range(7)]
    torch.cuda.synchronize()
    f = gen.as_f64
    so = f(inp["state0"])
    sm = np.abs(so)
    for s in range(7):
        yo, so, ym, sm = oracle.state_update(so, f(inp["x"][s]), f(inp["dt"][s]), f(inp["A"]), f(inp["B"][s]),
                                             f(inp["C"][s]), D=f(inp["D"]), z=f(inp["z"][s]), smag=sm,
                                             with_mag=True, zoh=True)
        assert oracle.rel_err(ys[s].float().cpu().numpy(), yo, ym) <= TOL[io]
    assert oracle.rel_err(st.cpu().numpy(), so, sm) <= TOL[io]


@pytest.mark.parametrize("plan", ["16,4,5", "16,4,1", "4,4,3", "16,8,2", "8,1,7"])
def test_forced_plans(plan):
    N = {"16,4,5": 64, "16,4,1": 64, "4,4,3": 16, "16,8,2": 128, "8,1,7": 8}[plan]
    nper, g, nch = (int(v) for v in plan.split(","))
    cfg = gen.ScanConfig("plan", 2, 40, 1111, N, io="bf16", gate=True, dskip="normal", seed=5, a_kind="random")
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(seq_split=(nper, g), chunks=nch):
        y, h = gpu_scan(inp)
    compare_scan(inp, y, h)


@pytest.mark.parametrize("a_kind", ["s4d", "random"])
def test_chunked_fp32_long_decay(a_kind):
    # small steps keep the state alive across chunk boundaries
    cfg = gen.ScanConfig("chunks", 1, 16, 6000, 16, io="f32", gate=False, dskip="ones", seed=9, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    inp["delta_bias"] = torch.full_like(inp["delta_bias"], -6.0)
    y, h = gpu_scan(inp)
    assert ssm.workspace_bytes(1, 16, 6000, 16, ssm.SSM_F32) > 0
    compare_scan(inp, y, h)


def test_empty_inputs():
    d = "cuda"
    A = -torch.ones(4, 4, device=d)
    for (Bt, Dm, L) in [(0, 4, 8), (1, 0, 8)]:
        u = torch.empty(Bt, Dm, L, device=d)
        y, _ = ssm.selective_scan_fwd(u, u, A[:Dm], torch.empty(Bt, 4, L, device=d), torch.empty(Bt, 4, L, device=d))
        assert y.numel() == 0
    u = torch.empty(2, 4, 0, device=d)
    st = torch.full((2, 4, 4), 7.0, device=d)
    y, st2 = ssm.selective_scan_fwd(u, u, A, torch.empty(2, 4, 0, device=d), torch.empty(2, 4, 0, device=d),
                                    last_state=st)
    torch.cuda.synchronize()
    assert torch.equal(st, torch.zeros_like(st))


def test_misaligned_pointer_rejected():
    d = "cuda"
    buf = torch.zeros(1 * 4 * 64 + 1, device=d)
    u = buf[1:].view(1, 4, 64)
    good = torch.zeros(1, 4, 64, device=d)
    A = -torch.ones(4, 4, device=d)
    B = torch.zeros(1, 4, 64, device=d)
    with pytest.raises(ssm.SsmError) as e:
        ssm.selective_scan_fwd(u, good, A, B, B)
    assert e.value.code == ssm.SSM_ERR_ALIGN


def test_caller_workspace_and_stream():
    inp = gen.scan_inputs(gen.BLOCK512)
    need = ssm.workspace_bytes(1, 512, 1024, 16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    y, h = gpu_scan(inp, stream=s, workspace=ws)
    compare_scan(inp, y, h)
    small = torch.empty(max(need // 2, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(ssm.SsmError) as e:
        gpu_scan(inp, workspace=small)
    assert e.value.code == ssm.SSM_ERR_WORKSPACE
    assert ssm.stream_status(s) == ssm.SSM_OK


def test_registered_workspace():
    """ssm_set_workspace: with a workspace registered, the scans take their chunk carries
    from it (results match the oracle), a registration smaller than a call needs makes that
    call return SSM_ERR_WORKSPACE, and unregistering restores the library's allocation."""
    inp = gen.scan_inputs(gen.BLOCK512, a_kind="scaled")
    need = ssm.workspace_bytes(1, 512, 1024, 16)
    assert need > 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")   # stale bytes: must not matter
    try:
        ssm.set_workspace(ws)
        y, h = gpu_scan(inp)
        compare_scan(inp, y, h)
        ssm.set_workspace(ws[: need // 2])
        with pytest.raises(ssm.SsmError) as e:
            gpu_scan(inp)
        assert e.value.code == ssm.SSM_ERR_WORKSPACE
        # a shape that needs no workspace still runs with the small registration
        small = gen.scan_inputs(gen.ScanConfig("nows", 16, 2048, 64, 16, seed=2))
        assert ssm.workspace_bytes(16, 2048, 64, 16) == 0
        y2, h2 = gpu_scan(small)
        compare_scan(small, y2, h2, channels=sample_channels(16, 2048, 16))
    finally:
        ssm.set_workspace(None)
    y3, h3 = gpu_scan(inp)
    assert torch.equal(y3, y) and torch.equal(h3, h)


def test_registered_workspace_backward():
    """The backward with no workspace argument takes the registered one (time-split shape:
    checkpoints plus the split's arrays, over stale bytes), returns SSM_ERR_WORKSPACE when the
    registration is too small, and allocates again once it is removed."""
    import ctypes
    Bt, D, L, N = 1, 32, 2048, 16
    dm = ssm.dims(Bt, D, L, N, ssm.SSM_BF16)
    need = ssm.load().ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(dm))
    assert need > 4 * D * (L // 8) * N                    # the time split's arrays too
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    try:
        ssm.set_workspace(ws)
        _check_backward(Bt, D, L, N, "bf16", True, "ones", True, True, "random")
        ssm.set_workspace(ws[: need // 2])
        with pytest.raises(ssm.SsmError) as e:
            _check_backward(Bt, D, L, N, "bf16", True, "ones", True, True, "random")
        assert e.value.code == ssm.SSM_ERR_WORKSPACE
    finally:
        ssm.set_workspace(None)
    _check_backward(Bt, D, L, N, "bf16", True, "ones", True, True, "random")


@pytest.mark.parametrize("cfg", [gen.BLOCK512, gen.ScanConfig("h", 3, 70, 333, 16, io="f32", gate=True, seed=8)],
                         ids=["block512", "ragged_f32"])
def test_host_buffer_entry(cfg):
    inp = gen.scan_inputs(cfg)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    yh, hh = ssm.selective_scan_fwd_host(pin["u"], pin["delta"], pin["A"], pin["B"], pin["C"], D=pin["D"],
                                         z=pin["z"], delta_bias=pin["delta_bias"], return_last_state=True)
    assert yh.device.type == "cpu" and hh.device.type == "cpu"
    compare_scan(inp, yh, hh)


def test_host_buffer_entry_many_blocks():
    """Enough input bytes for several channel blocks per batch row (8 blocks through three
    rotating buffer sets): every block boundary and every buffer reuse is checked, on channels
    sampled at the block edges, against the oracle, and all of y against the device entry."""
    cfg = gen.ScanConfig("hb", 2, 256, 16384, 16, io="bf16", gate=True, dskip="normal", seed=21, a_kind="random")
    inp = gen.scan_inputs(cfg)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    yh, hh = ssm.selective_scan_fwd_host(pin["u"], pin["delta"], pin["A"], pin["B"], pin["C"], D=pin["D"],
                                         z=pin["z"], delta_bias=pin["delta_bias"], return_last_state=True)
    edges = [(b, d) for b in (0, 1) for d in (0, 63, 64, 127, 128, 191, 192, 255)]
    compare_scan(inp, yh, hh, channels=edges)
    yd, hd = gpu_scan(inp)
    ref = yd.float().cpu()
    assert float((yh.float() - ref).abs().max()) <= 2e-2 * max(float(ref.abs().max()), 1.0)
    assert torch.allclose(hh, hd.cpu(), rtol=1e-4, atol=1e-5)


def test_cuda_graph_capture_and_replay():
    """The device entry points queue only kernels (and, given a workspace, nothing else) on
    the caller's stream, so a CUDA graph can capture them: a chunked scan with a caller
    workspace followed by three recurrent steps from its final state, captured once (after
    one eager call has set the kernels' attributes) and replayed, gives the eager results
    bit for bit."""
    cfg = gen.ScanConfig("graph", 1, 96, 8192, 16, io="bf16", gate=True, dskip="normal", seed=31, a_kind="random")
    inp = gen.scan_inputs(cfg)
    dec = gen.decode_inputs(gen.DECODE, Bt=1, D=96, N=16, gate=True, dskip="ones", steps=3, a_kind="random")
    g = to_dev(inp)
    dg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in dec.items()}
    ws = torch.empty(max(ssm.workspace_bytes(1, 96, 8192, 16), 16), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(g["u"])
    h = torch.empty((1, 96, 16), dtype=torch.float32, device="cuda")
    ys = torch.empty((3, 1, 96), dtype=torch.bfloat16, device="cuda")

    def work(stream):
        ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                               delta_bias=g["delta_bias"], y=y, last_state=h, workspace=ws, stream=stream)
        for s in range(3):
            ssm.state_update(h, dg["x"][s], dg["dt"][s], g["A"], dg["B"][s], dg["C"][s], D=g["D"], z=dg["z"][s],
                             y=ys[s], stream=stream)

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        work(side)
    torch.cuda.synchronize()
    eager = (y.clone(), h.clone(), ys.clone())
    assert ssm.workspace_bytes(1, 96, 8192, 16) > 0        # the captured scan is chunked
    graph = torch.cuda.CUDAGraph()
    y.zero_(); h.zero_(); ys.zero_()
    with torch.cuda.graph(graph, stream=side):
        work(side)
    for _ in range(2):
        y.zero_(); h.zero_(); ys.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, eager[0]) and torch.equal(h, eager[1]) and torch.equal(ys, eager[2])
    assert ssm.stream_status() == ssm.SSM_OK


def test_backward_cuda_graph_capture_and_replay():
    """The backward with a caller workspace queues only memsets and kernels on the caller's
    stream: captured in a CUDA graph on a shape the planner splits in time (all four passes)
    and replayed, it reproduces the eager gradients (up to the order of fp32 atomic sums)."""
    import ctypes
    cfg = gen.ScanConfig("graphb", 1, 64, 4096, 16, io="bf16", gate=True, dskip="ones", seed=33, a_kind="random")
    inp = gen.scan_inputs(cfg)
    g = to_dev(inp)
    dy = torch.from_numpy(np.random.default_rng(34).standard_normal((1, 64, 4096)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    dm = ssm.dims(1, 64, 4096, 16, ssm.SSM_BF16)
    wsb = ssm.load().ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(dm))
    assert wsb > 4 * 64 * 512 * 16            # checkpoints plus the time split's arrays
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    def work():
        return ssm.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, D=g["D"], z=g["z"],
                                      delta_bias=g["delta_bias"], delta_softplus=True, workspace=ws, stream=side)

    with torch.cuda.stream(side):
        eager = {k: v.clone() for k, v in work().items() if v is not None}
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        out = work()
    for _ in range(2):
        for v in out.values():
            if v is not None:
                v.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for k, r in eager.items():
            err = float((out[k] - r).abs().max() / r.abs().max().clamp_min(1e-30))
            assert err <= 1e-5, f"d{k}: {err:.2e}"
    assert ssm.stream_status() == ssm.SSM_OK


# ---- decode ---------------------------------------------------------------------------------
def _decode_gpu(inp, steps):
    g = to_dev(inp)
    st = g["state0"].clone()
    ys = []
    for s in range(steps):
        ys.append(ssm.state_update(st, g["x"][s], g["dt"][s], g["A"], g["B"][s], g["C"][s], D=g["D"],
                                   z=None if g["z"] is None else g["z"][s]))
    torch.cuda.synchronize()
    return torch.stack(ys, -1), st


def _decode_oracle(inp, rows, steps):
    f = gen.as_f64
    st = f(inp["state0"])[rows]
    sm = np.abs(st)
    ys, yms = [], []
    for s in range(steps):
        y, st, ym, sm = oracle.state_update(st, f(inp["x"][s])[rows], f(inp["dt"][s])[rows], f(inp["A"]),
                                            f(inp["B"][s])[rows], f(inp["C"][s])[rows], D=f(inp["D"]),
                                            z=None if inp["z"] is None else f(inp["z"][s])[rows],
                                            smag=sm, with_mag=True)
        ys.append(y)
        yms.append(ym)
    return np.stack(ys, -1), st, np.stack(yms, -1), sm


@pytest.mark.parametrize("a_kind", ["s4d", "random"])
def test_decode_full_size_sampled_rows(a_kind):
    inp = gen.decode_inputs(gen.DECODE, a_kind=a_kind)
    y, st = _decode_gpu(inp, 64)
    rows = [0, 97, 255]
    yo, so, ym, sm = _decode_oracle(inp, rows, 64)
    assert oracle.rel_err(y[rows].float().cpu().numpy(), yo, ym) <= TOL["bf16"]
    assert oracle.rel_err(st[rows].cpu().numpy(), so, sm) <= TOL["bf16"]


@pytest.mark.parametrize("a_kind", ["s4d", "random"])
@pytest.mark.parametrize("N,gate,dskip,io", [(16, True, "ones", "bf16"), (5, False, None, "bf16"),
                                            (64, True, "normal", "bf16"), (128, False, "ones", "bf16"),
                                            (4, True, "ones", "f32"), (7, True, "normal", "f32")])
def test_decode_shapes(N, gate, dskip, io, a_kind):
    inp = gen.decode_inputs(gen.DECODE, Bt=3, D=50, N=N, gate=gate, dskip=dskip, steps=9, a_kind=a_kind)
    if io == "f32":
        for k in ("x", "dt", "B", "C", "z"):
            if inp[k] is not None:
                inp[k] = inp[k].float()
    y, st = _decode_gpu(inp, 9)
    rows = [0, 1, 2]
    yo, so, ym, sm = _decode_oracle(inp, rows, 9)
    tol = TOL[io]
    assert oracle.rel_err(y.float().cpu().numpy(), yo, ym) <= tol
    assert oracle.rel_err(st.cpu().numpy(), so, sm) <= tol


@pytest.mark.parametrize("N", [16, 64])
def test_decode_unaligned_bc_rows(N):
    """B and C rows at an odd element offset (allowed: per-token vectors need only element
    alignment) take the path that reads them element by element; results match the oracle."""
    inp = gen.decode_inputs(gen.DECODE, Bt=3, D=50, N=N, gate=True, dskip="ones", steps=5, a_kind="scaled")
    g = to_dev(inp)
    st = g["state0"].clone()
    ys = []
    for s in range(5):
        bc = []
        for k in ("B", "C"):
            big = torch.empty(g[k][s].numel() + 1, dtype=g[k].dtype, device="cuda")
            view = big[1:].view_as(g[k][s])
            view.copy_(g[k][s])
            bc.append(view)
        assert bc[0].data_ptr() % 8 != 0
        ys.append(ssm.state_update(st, g["x"][s], g["dt"][s], g["A"], bc[0], bc[1], D=g["D"], z=g["z"][s]))
    torch.cuda.synchronize()
    y = torch.stack(ys, -1)
    yo, so, ym, sm = _decode_oracle(inp, [0, 1, 2], 5)
    assert oracle.rel_err(y.float().cpu().numpy(), yo, ym) <= TOL["bf16"]
    assert oracle.rel_err(st.cpu().numpy(), so, sm) <= TOL["bf16"]


def test_scan_then_decode_equals_longer_scan():
    """A scan of L steps then k recurrent steps from its final state equals the oracle's
    scan of L+k steps (softplus folded: the decode step takes the final dt)."""
    cfg = gen.ScanConfig("sd", 2, 24, 300, 16, io="f32", gate=True, dskip="ones", softplus=False, bias=False, seed=21)
    inp = gen.scan_inputs(cfg)
    inp["delta"] = inp["delta"].abs() * 0.1
    L, k = 280, 20
    first = {kk: (v[..., :L].contiguous() if isinstance(v, torch.Tensor) and v.dim() == 3 else v) for kk, v in inp.items()}
    y1, h1 = gpu_scan(first)
    g = to_dev(inp)
    st = h1.clone()
    ys = []
    for t in range(L, L + k):
        ys.append(ssm.state_update(st, g["u"][..., t].contiguous(), g["delta"][..., t].contiguous(), g["A"],
                                   g["B"][..., t].contiguous(), g["C"][..., t].contiguous(), D=g["D"],
                                   z=g["z"][..., t].contiguous()))
    torch.cuda.synchronize()
    y_all = torch.cat([y1, torch.stack(ys, -1)], -1)
    compare_scan(inp, y_all, st)


# ---- persistent tensor-memory path, forced on small shapes -------------------------------------
TC_CASES = [
    # Bt, D, L, N, io, gate, dskip
    (1, 8, 128, 64, "bf16", False, "ones"),
    (2, 37, 1000, 16, "bf16", True, "normal"),
    (1, 20, 4096, 64, "f32", True, "ones"),
    (3, 9, 520, 128, "bf16", False, None),
    (1, 50, 2048, 32, "bf16", True, "ones"),
    (2, 33, 64, 5, "f32", False, "normal"),
    (1, 64, 8192, 64, "bf16", False, "ones"),
]


@pytest.mark.parametrize("kernel", ["tp", "tc"])
@pytest.mark.parametrize("Bt,D,L,N,io,gate,dskip", TC_CASES)
def test_tc_forced_shapes(Bt, D, L, N, io, gate, dskip, kernel):
    # alternate the A recipe over the cases so that both kernels see per-channel rows
    a_kind = A_KINDS[(D + L) % 3]
    cfg = gen.ScanConfig("tc", Bt, D, L, N, io=io, gate=gate, dskip=dskip, seed=D + L, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(kernel=kernel):
        y, h = gpu_scan(inp)
    assert ssm.stream_status() == ssm.SSM_OK
    compare_scan(inp, y, h)


@pytest.mark.parametrize("kernel", ["tp", "tc"])
def test_tc_bounded_wait_reports_timeout(kernel):
    """The carry wait between segments gives up after a bounded spin on a flag that is never
    set (test hook of the plan override), records SSM_ERR_TIMEOUT, and the next call runs
    normally."""
    cfg = gen.ScanConfig("to", 1, 16, 2048, 16, io="bf16", gate=False, seed=4)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(kernel=kernel, force_timeout=True):
        gpu_scan(inp)
    assert ssm.stream_status() == ssm.SSM_ERR_TIMEOUT
    assert ssm.stream_status() == ssm.SSM_OK          # reading clears it
    with ssm.plan_override(kernel=kernel):
        y, h = gpu_scan(inp)
    assert ssm.stream_status() == ssm.SSM_OK
    compare_scan(inp, y, h)


@pytest.mark.parametrize("a_kind", ["s4d", "scaled"])
def test_seq_forced_long(a_kind):
    cfg = gen.ScanConfig("seqlong", 1, 40, 20000, 64, io="bf16", gate=True, seed=6, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(kernel="seq"):
        y, h = gpu_scan(inp)
    compare_scan(inp, y, h)
