"""The checked build (-DSSM_CHECK) on edge-case shapes: every global and shared-memory access
of the scan and state-update kernels is bounds-checked (a failure records SSM_ERR_CHECK and
skips the access), shared memory starts as NaN (a read of a word no thread wrote spoils the
result), and y and the final state sit between guard words that must come back untouched.
Each case must finish with status OK, intact guards and results equal to the fp64 oracle.

These stand in for a memory checker, which this machine does not offer."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import TOL, compare_scan
from selective_state_space_153_b300 import build, gen, ssm

pytestmark = pytest.mark.gpu

GUARD = 64                       # guard elements on each side (keeps 16-byte alignment)
PATTERN = {torch.float32: 0x5A5A5A5A, torch.bfloat16: 0x5A5A}


@pytest.fixture(scope="module")
def checked():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ssm.load()
    lib = ssm.load_library(build.build_checked())
    with ssm.using(lib):
        yield lib


def _guarded(shape, dtype):
    """A device tensor of `shape` in the middle of a buffer whose every element, guards and
    interior alike, holds the sentinel bit pattern."""
    n = math.prod(shape)
    big = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    ib = big.view(torch.int32 if dtype == torch.float32 else torch.int16)
    ib.fill_(PATTERN[dtype] if dtype == torch.float32 else np.int16(PATTERN[dtype]).item())
    return big, big[GUARD:GUARD + n].view(*shape)


def _guards_intact(big):
    ib = big.view(torch.int32 if big.dtype == torch.float32 else torch.int16)
    want = PATTERN[big.dtype] if big.dtype == torch.float32 else np.int16(PATTERN[big.dtype]).item()
    return bool((ib[:GUARD] == want).all() and (ib[-GUARD:] == want).all())


def _scan_checked(inp, disc="euler", conv=None):
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    Bt, Dm, L = g["u"].shape
    N = g["A"].shape[1]
    ybig, y = _guarded((Bt, Dm, L), g["u"].dtype)
    hbig, h = _guarded((Bt, Dm, N), torch.float32)
    if conv is None:
        ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                               delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"], y=y, last_state=h,
                               discretization=disc)
    else:
        w, cb = conv
        ssm.conv_selective_scan_fwd(g["u"], w.cuda(), cb.cuda(), g["delta"], g["A"], g["B"], g["C"], D=g["D"],
                                    z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True, y=y, last_state=h)
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_OK, "a bounds check failed"
    assert _guards_intact(ybig), "write outside y"
    assert _guards_intact(hbig), "write outside last_state"
    return y, h


SCAN_CASES = [
    # Bt, D, L, N, io, gate, plan override (dict), A recipe -- channel-pair kernel unless the
    # row length is not a multiple of 16 bytes (then the sequential-lane kernel)
    (1, 3, 16, 1, "f32", False, {}, "s4d"),               # one tile, one state
    (1, 5, 8, 3, "f32", True, {}, "random"),              # half a tile
    (2, 37, 48, 16, "bf16", True, {}, "scaled"),          # partial channel block
    (1, 40, 1000, 64, "bf16", False, {"chunks": 5}, "random"),   # chunks with a ragged last tile
    (1, 40, 2000, 48, "bf16", True, {"pair_states_per_lane": 16, "chunks": 3}, "scaled"),
    (2, 33, 40, 128, "f32", False, {"pair_states_per_lane": 8, "chunks": 1}, "random"),
    (1, 1, 1, 1, "f32", False, {}, "s4d"),                # sequential lanes: L = 1
    (2, 37, 33, 16, "bf16", True, {}, "random"),          # sequential lanes: odd L
    (1, 9, 129, 64, "bf16", True, {}, "scaled"),
    (1, 10, 1000, 20, "f32", True, {"kernel": "seq", "chunks": 4}, "random"),
]


@pytest.mark.parametrize("Bt,D,L,N,io,gate,ov,a_kind", SCAN_CASES)
def test_scan_checked(checked, Bt, D, L, N, io, gate, ov, a_kind):
    cfg = gen.ScanConfig("chk", Bt, D, L, N, io=io, gate=gate, dskip="normal", seed=L + N, a_kind=a_kind)
    inp = gen.scan_inputs(cfg)
    with ssm.plan_override(**ov):
        y, h = _scan_checked(inp)
    compare_scan(inp, y, h)


def test_zoh_checked(checked):
    cfg = gen.ScanConfig("chkz", 2, 33, 136, 16, io="f32", gate=True, dskip="ones", seed=5, a_kind="scaled")
    inp = gen.scan_inputs(cfg)
    inp["A"][:, 0] = 0.0
    with ssm.plan_override(chunks=3):
        y, h = _scan_checked(inp, disc="zoh")
    compare_scan(inp, y, h, zoh=True)


def test_conv_front_checked(checked):
    cfg = gen.ScanConfig("chkc", 1, 20, 520, 32, io="f32", gate=True, dskip="ones", seed=6, a_kind="random")
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(7)
    w = torch.from_numpy(rng.standard_normal((20, 3)).astype(np.float32) * 0.5)
    cb = torch.from_numpy(rng.standard_normal(20).astype(np.float32) * 0.2)
    with ssm.plan_override(chunks=3):
        y, h = _scan_checked(inp, conv=(w, cb))
    u = oracle.conv_silu(gen.as_f64(inp["u"]), np.broadcast_to(w.double().numpy(), (1, 20, 3)),
                         np.broadcast_to(cb.double().numpy(), (1, 20)))
    ref = dict(inp)
    ref["u"] = torch.from_numpy(u)
    compare_scan(ref, y, h)


@pytest.mark.parametrize("N,io,unaligned,Dm", [(16, "bf16", False, 50), (5, "f32", False, 50), (64, "bf16", True, 50),
                                               (16, "bf16", False, 264), (64, "f32", False, 76)])
def test_decode_checked(checked, N, io, unaligned, Dm):
    """Wide (16-byte B/C), element-wise (B/C rows at an odd offset) and scalar (N % 4 != 0)
    state-update kernels, with guard words around the state and y, on channel counts that
    leave a partial last block."""
    inp = gen.decode_inputs(gen.DECODE, Bt=3, D=Dm, N=N, gate=True, dskip="ones", steps=3, a_kind="random")
    if io == "f32":
        for k in ("x", "dt", "B", "C", "z"):
            inp[k] = inp[k].float()
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sbig, st = _guarded((3, Dm, N), torch.float32)
    st.copy_(g["state0"])
    f = gen.as_f64
    so = f(inp["state0"])
    sm = np.abs(so)
    for s in range(3):
        ybig, y = _guarded((3, Dm), g["x"].dtype)
        Bv, Cv = g["B"][s], g["C"][s]
        if unaligned:
            bufs = []
            for t in (Bv, Cv):
                big = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
                view = big[1:].view_as(t)
                view.copy_(t)
                bufs.append(view)
            Bv, Cv = bufs
        ssm.state_update(st, g["x"][s], g["dt"][s], g["A"], Bv, Cv, D=g["D"], z=g["z"][s], y=y)
        torch.cuda.synchronize()
        assert ssm.stream_status() == ssm.SSM_OK, "a bounds check failed"
        assert _guards_intact(ybig) and _guards_intact(sbig)
        yo, so, ym, sm = oracle.state_update(so, f(inp["x"][s]), f(inp["dt"][s]), f(inp["A"]), f(inp["B"][s]),
                                             f(inp["C"][s]), D=f(inp["D"]), z=f(inp["z"][s]), smag=sm, with_mag=True)
        assert oracle.rel_err(y.float().cpu().numpy(), yo, ym) <= TOL[io]
    assert oracle.rel_err(st.cpu().numpy(), so, sm) <= TOL[io]


def test_check_records_a_caught_access(checked):
    """Positive control: with the plan override's check probe on, one thread of each
    channel-pair launch issues a checked load one element past the end of A. The check must
    catch it (the load is skipped, nothing is read out of range) and record SSM_ERR_CHECK; the
    scan's results are unaffected, and the next call without the probe reports OK."""
    cfg = gen.ScanConfig("chkp", 1, 8, 64, 4, io="f32", seed=2)
    inp = gen.scan_inputs(cfg)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with ssm.plan_override(check_probe=True):
        y, h = ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"],
                                      delta_bias=g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_ERR_CHECK
    compare_scan(inp, y, h)
    _scan_checked(inp)      # asserts status OK again


def _bwd_checked(inp, dy, dl, odd=False):
    """ssm_selective_scan_bwd through the checked library with every output and the workspace
    between guard words; returns the gradients (fp32 device tensors)."""
    import ctypes
    lib = ssm.load()
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dyd = dy.cuda()
    if odd:      # every io input one element off a 2-element boundary
        def off(t):
            if t is None:
                return None
            big = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
            v = big[1:].view(t.shape)
            v.copy_(t)
            return v
        for k in ("u", "delta", "B", "C", "z"):
            g[k] = off(g[k])
        dyd = off(dyd)
    Bt, Dm, L = g["u"].shape
    N = g["A"].shape[1]
    shapes = {"u": (Bt, Dm, L), "delta": (Bt, Dm, L), "A": (Dm, N), "B": (Bt, N, L), "C": (Bt, N, L),
              "D": (Dm,), "z": (Bt, Dm, L), "delta_bias": (Dm,)}
    outs = {k: _guarded(s, torch.float32) for k, s in shapes.items()}
    dm = ssm.dims(Bt, Dm, L, N, ssm._io_code(g["u"]))
    wsb = lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(dm))
    wbig, ws = _guarded((max(wsb, 4) // 4,), torch.float32)
    p = ssm._p
    rc = lib.ssm_selective_scan_bwd(ctypes.byref(dm), p(g["u"]), p(g["delta"]), p(g["A"]), p(g["B"]), p(g["C"]),
                                    p(g["D"]), p(g["z"]), p(g["delta_bias"]), 1, p(dyd),
                                    None if dl is None else p(dl.cuda()),
                                    *[p(outs[k][1]) for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")],
                                    p(ws), wsb, None)
    assert rc == ssm.SSM_OK, ssm.status_string(rc)
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_OK, "a bounds check failed"
    for k, (big, _) in outs.items():
        assert _guards_intact(big), f"write outside d{k}"
    assert _guards_intact(wbig), "write outside the workspace"
    return {k: v for k, (_, v) in outs.items()}


BWD_CHECK_CASES = [
    # Bt, D, L, N, io, chunks, lanes split (states per lane), odd offset -- every input path
    # (copy ring, two-step register loads, single steps) with and without the time split
    (2, 37, 96, 16, "bf16", 3, 0, False),    # ring, split, partial channel block
    (1, 9, 100, 16, "f32", 2, 2, False),     # ring with a half last segment, split, two states per lane
    (2, 7, 33, 8, "f32", 2, 0, False),       # single steps (odd L), split
    (1, 20, 70, 32, "bf16", 1, 0, False),    # two-step loads, unsplit
    (2, 9, 70, 16, "bf16", 3, 0, True),      # inputs off alignment: single steps, split
    (1, 5, 40, 100, "f32", 1, 0, False),     # N = 100: 32 lanes per channel
    (1, 9, 560, 16, "bf16", 40, 0, False),   # 35 chunks: the combine's warp scan
]


@pytest.mark.parametrize("Bt,D,L,N,io,chunks,q,odd", BWD_CHECK_CASES)
def test_backward_checked(checked, Bt, D, L, N, io, chunks, q, odd):
    """The backward through the checked build: status OK, guards intact, and gradients equal
    to the normal build's within fp32 summation-order noise (shared memory starts as NaN, so
    a read of an unwritten word would show)."""
    cfg = gen.ScanConfig("chkb", Bt, D, L, N, io=io, gate=True, dskip="normal", bias=True, seed=L + N,
                         a_kind="random")
    inp = gen.scan_inputs(cfg)
    rng = np.random.default_rng(L)
    dy = torch.from_numpy(rng.standard_normal((Bt, D, L)).astype(np.float32)).to(inp["u"].dtype)
    dl = torch.from_numpy(rng.standard_normal((Bt, D, N)).astype(np.float32))
    with ssm.plan_override(bwd_chunks=chunks, bwd_states_per_lane=q):
        got = _bwd_checked(inp, dy, dl, odd)
        with ssm.using(ssm.load_library(ssm.LIB_PATH)):
            ref = _bwd_checked(inp, dy, dl, odd)
    for k in got:
        r, v = ref[k].double(), got[k].double()
        assert torch.isfinite(v).all(), f"d{k}: non-finite"
        err = float((v - r).abs().max() / r.abs().max().clamp_min(1e-30))
        assert err <= 1e-5, f"d{k}: {err:.2e} against the normal build"
