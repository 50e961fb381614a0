"""The C-ABI library loads, exports every symbol include/ssm_scan.h declares, and rejects bad
arguments on the host with the documented status codes (no GPU needed: nothing is
launched on an argument error)."""
import ctypes
import os
import re

import pytest

from selective_state_space_153_b300 import build, ssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ssm.load()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_]+)\s*\(", txt)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(ssm.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_nothing_else_and_no_shared_statics():
    """Only the header's functions (and the device-link registration hooks) are exported, and
    no symbol is a GNU "unique" object: two builds of the library in one process (the normal
    and the checked build) must not share, say, a kernel's attributes-already-set flag."""
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("nm not installed")
    out = subprocess.run(["nm", "-D", "--defined-only", ssm.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout.split("\n")
    syms = [ln.split() for ln in out if ln.strip()]
    assert not [x for x in syms if x[1] == "u"], "GNU unique symbols exported"
    names = {x[2] for x in syms}
    extra = {n for n in names if not n.startswith("__cudaRegisterLinkedBinary_")} - set(declared_functions())
    assert not extra, sorted(extra)[:10]


def test_status_strings_and_version(lib):
    for code in range(10):
        s = ssm.status_string(code)
        assert s.startswith("SSM_")
    assert ssm.status_string(99) == "SSM_ERR_UNKNOWN"
    assert ssm.version() == (1, 3)   # 1.1: workspace, plan override; 1.2: last CUDA error;
    # 1.3: the backward time split (plan override field bwd_chunks)


def test_last_cuda_error_query(lib):
    # nothing has failed on this thread: 0; the text comes from the runtime, with no GPU
    assert lib.ssm_last_cuda_error() == 0
    assert lib.ssm_cuda_error_string(0).decode() == "no error"
    assert len(lib.ssm_cuda_error_string(2).decode()) > 0      # cudaErrorMemoryAllocation
    assert len(lib.ssm_cuda_error_string(123456).decode()) > 0


A = ctypes.c_void_p(0x1000)      # fake, 16-byte aligned "device" pointers: never dereferenced
MIS = ctypes.c_void_p(0x1002)    # misaligned


def call_scan(lib, d, u=A, delta=A, Am=A, B=A, C=A, D=None, z=None, bias=None, y=A, last=None):
    return lib.ssm_selective_scan_fwd(ctypes.byref(d) if d is not None else None, u, delta, Am, B, C, D, z,
                                      bias, 1, y, last, None)


def test_scan_argument_errors(lib):
    d = ssm.dims(1, 4, 64, 4, ssm.SSM_F32)
    assert call_scan(lib, None) == ssm.SSM_ERR_NULL
    assert call_scan(lib, d, u=None) == ssm.SSM_ERR_NULL
    assert call_scan(lib, d, C=None) == ssm.SSM_ERR_NULL
    assert call_scan(lib, d, y=None) == ssm.SSM_ERR_NULL
    assert call_scan(lib, d, u=MIS) == ssm.SSM_ERR_ALIGN
    assert call_scan(lib, d, z=MIS) == ssm.SSM_ERR_ALIGN
    assert call_scan(lib, d, last=MIS) == ssm.SSM_ERR_ALIGN
    assert call_scan(lib, ssm.dims(-1, 4, 64, 4, 0)) == ssm.SSM_ERR_SHAPE
    assert call_scan(lib, ssm.dims(1, 4, -3, 4, 0)) == ssm.SSM_ERR_SHAPE
    assert call_scan(lib, ssm.dims(1, 4, 64, 0, 0)) == ssm.SSM_ERR_SHAPE
    assert call_scan(lib, ssm.dims(1, 4, 64, 4, 7)) == ssm.SSM_ERR_DTYPE
    assert call_scan(lib, ssm.dims(1, 4, 64, ssm.MAX_DSTATE + 1, 0)) == ssm.SSM_ERR_UNSUPPORTED
    assert call_scan(lib, ssm.dims(1 << 40, 1 << 20, 1 << 20, 4, 0)) == ssm.SSM_ERR_SHAPE
    # empty batch/dim: nothing to do, OK without touching the GPU
    assert call_scan(lib, ssm.dims(0, 4, 64, 4, 0), u=None, delta=None, y=None) == ssm.SSM_OK
    assert call_scan(lib, ssm.dims(2, 0, 64, 4, 0), u=None, delta=None, y=None) == ssm.SSM_OK


def test_state_update_argument_errors(lib):
    d = ssm.dims(2, 8, 1, 16, ssm.SSM_BF16)
    f = lib.ssm_state_update
    assert f(None, A, A, A, A, A, A, None, None, A, None) == ssm.SSM_ERR_NULL
    assert f(ctypes.byref(d), None, A, A, A, A, A, None, None, A, None) == ssm.SSM_ERR_NULL
    assert f(ctypes.byref(d), A, A, A, A, A, A, None, None, None, None) == ssm.SSM_ERR_NULL
    assert f(ctypes.byref(d), MIS, A, A, A, A, A, None, None, A, None) == ssm.SSM_ERR_ALIGN
    assert f(ctypes.byref(ssm.dims(2, 8, 1, 0, 1)), A, A, A, A, A, A, None, None, A, None) == ssm.SSM_ERR_SHAPE
    assert f(ctypes.byref(ssm.dims(0, 8, 1, 16, 1)), None, None, None, None, None, None, None, None, None, None) == ssm.SSM_OK


def test_backward_argument_errors(lib):
    """ssm_selective_scan_bwd rejects bad arguments on the host, before any CUDA call (a caller
    workspace is passed, so no default workspace is looked up)."""
    f = lib.ssm_selective_scan_bwd
    d = ssm.dims(1, 4, 64, 4, ssm.SSM_F32)

    def call(dims=d, u=A, delta=A, Am=A, B=A, C=A, dy=A, du=A, ddelta=A, dA=A, dB=A, dC=A, ws=A, wsb=1 << 20):
        return f(ctypes.byref(dims) if dims is not None else None, u, delta, Am, B, C, None, None, None, 1, dy,
                 None, du, ddelta, dA, dB, dC, None, None, None, ws, wsb, None)
    assert call(dims=None) == ssm.SSM_ERR_NULL
    assert call(u=None) == ssm.SSM_ERR_NULL
    assert call(dy=None) == ssm.SSM_ERR_NULL
    assert call(dA=None) == ssm.SSM_ERR_NULL
    assert call(dC=None) == ssm.SSM_ERR_NULL
    assert call(u=MIS) == ssm.SSM_ERR_ALIGN
    assert call(dB=MIS) == ssm.SSM_ERR_ALIGN
    assert call(ws=MIS) == ssm.SSM_ERR_ALIGN
    assert call(dims=ssm.dims(1, 4, 64, 4, 7)) == ssm.SSM_ERR_DTYPE
    assert call(dims=ssm.dims(1, 4, -64, 4, 0)) == ssm.SSM_ERR_SHAPE
    assert call(dims=ssm.dims(70000, 4, 64, 4, 0)) == ssm.SSM_ERR_UNSUPPORTED    # batch rows on grid.y
    need = lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d))
    assert need > 0
    assert call(wsb=need - 16) == ssm.SSM_ERR_WORKSPACE
    # nothing to do for an empty batch or channel count: OK without touching the GPU
    assert call(dims=ssm.dims(0, 4, 64, 4, 0), u=None, dy=None) == ssm.SSM_OK


def test_workspace_query(lib):
    # a sequence over too few channels to give every SM sub-partition two warps is cut into
    # chunks whose carries pass through the workspace; a batch wide enough needs none
    assert ssm.workspace_bytes(1, 1536, 131072, 64) > 0
    assert ssm.workspace_bytes(8, 1536, 2048, 16) > 0
    assert ssm.workspace_bytes(16, 2048, 2048, 16) == 0
    # rows that are not 16-byte multiples (2047 bf16 steps): padded copies of u, delta, z, y at
    # 2048 steps per row and of B, C, then the chunk carries
    pad = 8 * 1536 * 2048 * 2
    assert ssm.workspace_bytes(8, 1536, 2047, 16) >= 4 * pad + 2 * 8 * 16 * 2048 * 2
    with ssm.plan_override(kernel="seq"):   # the element-wise kernel needs no copies
        assert ssm.workspace_bytes(8, 1536, 2047, 16) < pad
    assert ssm.workspace_bytes(0, 1536, 2048, 16) == 0
    assert lib.ssm_selective_scan_workspace_bytes(None) == 0


def _chunks_from_workspace(Bt, Dm, L, N):
    """Chunk count of the pair kernel's plan, read back from its workspace size: two
    [chunks][Bt*Dm][64] fp32 carry arrays and one [chunks][Bt*Dm] fp32 dt-sum array, each
    rounded up to 256 bytes (64 padded states at N = 64)."""
    ws = ssm.workspace_bytes(Bt, Dm, L, N)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for nc in range(1, 4097):
        bd = Bt * Dm
        if 2 * up(nc * bd * 64 * 4) + up(nc * bd * 4) == ws:
            return nc
    raise AssertionError(f"workspace {ws} matches no chunk count")


@pytest.mark.parametrize("shape,chunks", [
    # sixteen states per lane, 3 CTAs per SM: 18 CTAs of 64 channels per wave, three waves
    # of chunks while a chunk keeps >= 2048 steps
    ((1, 1536, 131072, 64), 54),
    ((1, 768, 131072, 64), 37),
    # shorter sequences keep eight states per lane (8-warp full-pass CTAs, 2 per SM)
    ((1, 1536, 16384, 64), 12),
    ((4, 1536, 16384, 64), 6),
])
def test_planner_chunk_counts(lib, shape, chunks):
    """The long-sequence plans the bench and the parity tests run (148 SMs, the B300 count,
    is also the planner's fallback when no GPU is present)."""
    assert _chunks_from_workspace(*shape) == chunks


def test_ws_entry_rejects_small_workspace(lib):
    d = ssm.dims(1, 1536, 131072, 64, ssm.SSM_BF16)
    need = ssm.workspace_bytes(1, 1536, 131072, 64)
    assert need > 0
    rc = lib.ssm_selective_scan_fwd_ws(ctypes.byref(d), A, A, A, A, A, None, None, None, 1, A, None,
                                       MIS, need, None)
    assert rc == ssm.SSM_ERR_ALIGN


def test_set_workspace_argument_errors(lib):
    """ssm_set_workspace rejects bad arguments on the host (these checks run before any CUDA
    call); without a GPU, a valid registration fails only at the device query."""
    assert lib.ssm_set_workspace(None, 64) == ssm.SSM_ERR_NULL
    assert lib.ssm_set_workspace(ctypes.c_void_p(0x1000), 0) == ssm.SSM_ERR_WORKSPACE
    assert lib.ssm_set_workspace(ctypes.c_void_p(0x1001), 4096) == ssm.SSM_ERR_ALIGN
    rc = lib.ssm_set_workspace(None, 0)   # unregister: needs the current device only
    assert rc in (ssm.SSM_OK, ssm.SSM_ERR_CUDA)


def test_plan_override_roundtrip_and_errors(lib):
    """The override is read back as set, bad values leave the previous one in force, NULL
    clears it, and it changes what the planner reports (the workspace a shape needs)."""
    base = ssm.workspace_bytes(1, 1536, 131072, 64)
    assert ssm.get_plan_override().kernel == ssm.SSM_KERNEL_AUTO
    with ssm.plan_override(chunks=7) as ov:
        got = ssm.get_plan_override()
        assert got.chunks == 7 and got.kernel == 0
        assert _chunks_from_workspace(1, 1536, 131072, 64) == 7
        bad = ssm.PlanOverride(9, 0, 0, 0, 0, 0, 0, 0, 0)
        assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_UNSUPPORTED
        bad = ssm.PlanOverride(0, 5, 0, 0, 0, 0, 0, 0, 0)
        assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_UNSUPPORTED
        bad = ssm.PlanOverride(0, 0, -1, 0, 0, 0, 0, 0, 0)
        assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_SHAPE
        bad = ssm.PlanOverride(0, 0, 0, 16, 3, 0, 0, 0, 0)   # a lane split that is not built
        assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_UNSUPPORTED
        bad = ssm.PlanOverride(0, 0, 0, 0, 0, 0, 0, 0, 3)    # backward: 2 or 4 states per lane
        assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_UNSUPPORTED
        assert ssm.get_plan_override().chunks == 7
        assert ov.chunks == 7
    assert ssm.get_plan_override().chunks == 0
    assert ssm.workspace_bytes(1, 1536, 131072, 64) == base
    assert lib.ssm_get_plan_override(None) == ssm.SSM_ERR_NULL
    # two states per lane in the backward: twice the lanes, the same checkpoint bytes per state
    d = ssm.dims(8, 1536, 2048, 16, ssm.SSM_BF16)
    b4 = lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d))
    with ssm.plan_override(bwd_states_per_lane=2):
        assert lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d)) == b4
        d64 = ssm.dims(1, 8, 64, 64, ssm.SSM_F32)    # N > 32 keeps four states per lane
        with ssm.plan_override(bwd_states_per_lane=4):
            b64 = lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d64))
        assert lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d64)) == b64
    # backward time split: checkpoints [BD][nseg][np], then per-segment dt sums [BD][nseg] and
    # per-chunk hloc, cloc, cin [BD][K][np] and sdt [BD][K], the two per-row arrays padded to
    # 4 floats (2 x 7 x 100 x 16: np = 16, 13 segments, 3 chunks of 5 segments)
    d7 = ssm.dims(2, 7, 100, 16, ssm.SSM_F32)
    with ssm.plan_override(bwd_states_per_lane=2):
        assert lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d7)) == 4 * 14 * 13 * 16
        with ssm.plan_override(bwd_states_per_lane=2, bwd_chunks=3):
            assert lib.ssm_selective_scan_bwd_workspace_bytes(ctypes.byref(d7)) == \
                4 * (14 * 13 * 16 + 184 + 44 + 3 * 14 * 3 * 16)    # 14*13, 14*3 padded to 4
    bad = ssm.PlanOverride(0, 0, 0, 0, 0, 0, 0, 0, 0, -1)     # negative chunk count
    assert lib.ssm_set_plan_override(ctypes.byref(bad)) == ssm.SSM_ERR_SHAPE
    with ssm.plan_override(kernel="tc"):
        # the time-split plan keeps fp32 B/C of the whole sequence in its workspace
        assert ssm.workspace_bytes(1, 1536, 131072, 64) > 2 * 64 * 131072 * 4
    assert lib.ssm_set_plan_override(None) == ssm.SSM_OK


def test_library_reads_no_environment(lib, monkeypatch):
    """The experiment switches of earlier builds are gone: an environment variable of that
    name changes nothing the planner reports."""
    base = ssm.workspace_bytes(1, 1536, 131072, 64)
    for k, v in (("SSM_KERNEL", "tc"), ("SSM_PAIR_CHUNKS", "3"), ("SSM_PAIR_KS", "8"), ("SSM_PLAN", "4,4,3")):
        monkeypatch.setenv(k, v)
    assert ssm.workspace_bytes(1, 1536, 131072, 64) == base
