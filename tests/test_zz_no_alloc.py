"""ssm_selective_scan_fwd_noalloc: the scan with the library's fixed per-device scratch
instead of an allocated workspace. It runs the same kernels as ssm_selective_scan_fwd, so
its outputs must equal that entry point's bit for bit, on every call in a row (the control
words at the head of the scratch are cleared by each call; stale carries or tickets from the
previous call would show as a mismatch or a timeout status).

Kept in the last-collected file so that it also runs after every other GPU test in one
process (the scratch address is resolved once per device and then reused)."""
import ctypes
import os
import re

import pytest
import torch

from selective_state_space_153_b300 import build, gen, ssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")

FAKE = ctypes.c_void_p(0x1000)   # aligned, never dereferenced: rejected before any CUDA work


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ssm.load()


def test_scratch_size_matches_header():
    m = re.search(r"#define\s+SSM_SCRATCH_MAX_BYTES\s+\(\(size_t\)([0-9 *]+)\)", open(HEADER).read())
    assert m is not None
    val = 1
    for f in m.group(1).split("*"):
        val *= int(f)
    assert val == ssm.SCRATCH_MAX_BYTES == 48 * 1024 * 1024


@pytest.fixture
def time_split_plan(lib):
    """The persistent time-split kernel keeps fp32 B/C for the whole sequence in its workspace:
    on the long-sequence shape that exceeds the fixed size, which the default plan (chunk
    carries only, about 41 MiB there) fits."""
    with ssm.plan_override(kernel="tc"):
        yield


def test_default_long_sequence_plan_fits_scratch(lib):
    """The default plan of the long-sequence shape keeps its chunk carries within the fixed
    scratch: a planner change that outgrew it would make that shape fail here first."""
    need = ssm.workspace_bytes(1, 1536, 131072, 64, ssm.SSM_BF16)
    assert 0 < need <= ssm.SCRATCH_MAX_BYTES
    for shape in ((8, 1536, 2048, 16), (1, 512, 1024, 16), (1, 2560, 65536, 64), (2, 1536, 65536, 64)):
        assert ssm.workspace_bytes(*shape, ssm.SSM_BF16) <= ssm.SCRATCH_MAX_BYTES, shape


def test_oversize_shape_rejected_on_host(lib, time_split_plan):
    # 1 x 1536 x 131072 x 64 on the time-split plan needs ~65 MiB of scratch: SSM_ERR_WORKSPACE
    d = ssm.dims(1, 1536, 131072, 64, ssm.SSM_BF16)
    assert ssm.workspace_bytes(1, 1536, 131072, 64) > ssm.SCRATCH_MAX_BYTES
    rc = lib.ssm_selective_scan_fwd_noalloc(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                                            None, 1, FAKE, None, None)
    assert rc == ssm.SSM_ERR_WORKSPACE
    # ordinary argument checks come first, as in ssm_selective_scan_fwd
    rc = lib.ssm_selective_scan_fwd_noalloc(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE, None, None,
                                            None, 1, FAKE, None, None)
    assert rc == ssm.SSM_ERR_NULL
    assert lib.ssm_selective_scan_fwd_noalloc(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1,
                                              FAKE, None, None) == ssm.SSM_ERR_NULL


def test_empty_problem_needs_no_gpu(lib):
    d = ssm.dims(0, 1536, 2048, 16, ssm.SSM_BF16)
    assert lib.ssm_selective_scan_fwd_noalloc(ctypes.byref(d), None, None, None, None, None, None, None,
                                              None, 1, None, None, None) == ssm.SSM_OK


# default plans: the chunked channel-pair kernel at 16 and 64 states (whose scratch holds the
# chunk carries), and shapes that need no scratch at all
CASES = [
    gen.M130,
    gen.ScanConfig("n64_l16k", 1, 1536, 16384, 64, gate=False, dskip="ones", u_kind="ar1", seed=11),
    gen.BLOCK512,
    gen.TINY,
]


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _existing(g):
    return ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                  delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                                  return_last_state=True)


def _noalloc(g):
    # outputs pre-filled with NaN so that an element the call fails to write cannot match
    y = torch.full_like(g["u"], float("nan"))
    Bt, Dm, _ = g["u"].shape
    h = torch.full((Bt, Dm, g["A"].shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    return ssm.selective_scan_fwd_noalloc(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                          delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                                          y=y, last_state=h)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_equals_existing_entry_two_calls_in_a_row(lib, cfg):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g = _dev(gen.scan_inputs(cfg))
    need = ssm.workspace_bytes(cfg.Bt, cfg.D, cfg.L, cfg.N, ssm.SSM_F32 if cfg.io == "f32" else ssm.SSM_BF16)
    assert need <= ssm.SCRATCH_MAX_BYTES
    y_ref, h_ref = _existing(g)
    first = _noalloc(g)
    second = _noalloc(g)
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_OK
    for y, h in (first, second):
        assert torch.equal(y, y_ref)
        assert torch.equal(h, h_ref)


@pytest.mark.gpu
def test_noalloc_back_to_back_different_shapes(lib):
    """Consecutive calls of different shapes on one stream reuse the scratch: each result
    still equals the existing entry point's."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gs = [_dev(gen.scan_inputs(c)) for c in (gen.M130, gen.BLOCK512)]
    refs = [_existing(g) for g in gs]
    outs = [_noalloc(g) for g in (gs[0], gs[1], gs[0])]
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_OK
    for (y, h), (yr, hr) in zip(outs, (refs[0], refs[1], refs[0])):
        assert torch.equal(y, yr)
        assert torch.equal(h, hr)


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", ["tp", "tc"])
def test_noalloc_persistent_kernels_clear_their_control_words(lib, kernel):
    """The persistent time-split kernels keep a work ticket and per-segment carry flags at the
    head of the scratch. Each call clears them: two calls in a row, then a call of another
    shape, then the first shape again, all equal the allocating entry point bit for bit (stale
    tickets or flags would show as a mismatch or as a timeout in the status word)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    small = gen.ScanConfig("tcs", 2, 40, 1000, 16, gate=True, dskip="normal", seed=7, a_kind="random")
    gs = [_dev(gen.scan_inputs(c)) for c in (gen.M130, small)]
    with ssm.plan_override(kernel=kernel):
        for c in (gen.M130, small):
            need = ssm.workspace_bytes(c.Bt, c.D, c.L, c.N, ssm.SSM_BF16)
            assert 0 < need <= ssm.SCRATCH_MAX_BYTES
        refs = [_existing(g) for g in gs]
        outs = [_noalloc(g) for g in (gs[0], gs[0], gs[1], gs[0])]
        torch.cuda.synchronize()
        assert ssm.stream_status() == ssm.SSM_OK
    for (y, h), (yr, hr) in zip(outs, (refs[0], refs[0], refs[1], refs[0])):
        assert torch.equal(y, yr)
        assert torch.equal(h, hr)


@pytest.mark.gpu
def test_noalloc_oversize_raises_clear_error(lib, time_split_plan):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    L, N, Dm = 131072, 64, 1536
    u = torch.zeros((1, Dm, L), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((Dm, N), dtype=torch.float32, device="cuda")
    Bm = torch.zeros((1, N, L), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ssm.SsmError, match="SSM_ERR_WORKSPACE.*|fixed size") as ei:
        ssm.selective_scan_fwd_noalloc(u, u, A, Bm, Bm)
    assert ei.value.code == ssm.SSM_ERR_WORKSPACE
    assert str(ssm.SCRATCH_MAX_BYTES) in str(ei.value)


@pytest.mark.gpu
@pytest.mark.parametrize("Bt,D,L,N", [(2, 48, 1001, 16), (1, 1536, 16383, 64)], ids=["copies_fit", "copies_too_big"])
def test_noalloc_ragged_rows(lib, Bt, D, L, N):
    """Rows that are not 16-byte multiples: the padded copies of the default kernel go into the
    scratch when they fit there; when they do not, the call takes the element-wise kernel
    (it needs only its chunk carries) instead of failing. Both match the fp64 oracle."""
    from parity import compare_scan, sample_channels
    cfg = gen.ScanConfig("nr", Bt, D, L, N, io="bf16", gate=True, dskip="ones", seed=L, a_kind="random")
    inp = gen.scan_inputs(cfg)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, h = ssm.selective_scan_fwd_noalloc(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                          delta_bias=g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    assert ssm.stream_status() == ssm.SSM_OK
    compare_scan(inp, y, h, channels=sample_channels(Bt, D, 6, seed=3))
