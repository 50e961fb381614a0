"""Plain fp64 CPU oracle for the selective scan (Mamba S6) and its recurrent state update.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package. The CUDA library never calls it and
the two share no code: the oracle is ``ssm_oracle.c`` (sequential loops in double, written
from the per-timestep loop in section 3.2 of "From RNN to Mamba: state-space model
principles and long-sequence modelling in practice") compiled with the host C compiler,
plus this ctypes wrapper, which only marshals numpy float64 arrays.

Parity status: pinned. Every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, invariants, a hand-computed case and brute force, and
``tests/test_oracle_mutants.py`` shows that planted mistakes in the C source fail a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssm_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle into a shared library with gcc (-O2, IEEE double, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", *extra_flags,
           "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _bind(lib):
    lib.oracle_scan_channels.restype = ctypes.c_int
    lib.oracle_scan_channels.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _dp, _dp, _dp, _dp, _dp, _ip, _dp, _dp, _dp, ctypes.c_int, _dp,
        _dp, _dp, _dp, _dp, ctypes.c_int]
    lib.oracle_state_update.restype = ctypes.c_int
    lib.oracle_state_update.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _dp, _dp,
        _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_conv_silu.restype = ctypes.c_int
    lib.oracle_conv_silu.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _dp, _dp, _dp, _dp]
    lib.oracle_scan_channels_disc.restype = ctypes.c_int
    lib.oracle_scan_channels_disc.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _dp, _dp, _dp, _dp, _dp, _ip, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, _dp,
        _dp, _dp, _dp, _dp, ctypes.c_int]
    lib.oracle_state_update_disc.restype = ctypes.c_int
    lib.oracle_state_update_disc.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _dp, _dp,
        _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, _dp, _dp]
    return lib


def load(path: Optional[str] = None):
    """Load (compiling first if needed) the oracle library. ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_oracle()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _c(a: Optional[np.ndarray]):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def scan_rows(u, delta, A, B, C, bidx, D=None, z=None, delta_bias=None,
              delta_softplus=False, h0=None, with_mag=False, nthreads=1, lib=None, zoh=False):
    """Scan channels given as packed rows (``zoh``: zero-order-hold B_bar instead of dt*B).

    u, delta, z: [nchan, L]; A, h0: [nchan, N]; D, delta_bias: [nchan];
    B, C: [nbatch, N, L]; bidx: [nchan] batch row of each channel.
    Returns (y [nchan, L], last_state [nchan, N]) or, with ``with_mag``,
    (y, last_state, ymag, hmag) where ymag/hmag are the magnitude companions.
    """
    lib = lib or load()
    u, delta, A, B, C = _c(u), _c(delta), _c(A), _c(B), _c(C)
    z, D, delta_bias, h0 = _c(z), _c(D), _c(delta_bias), _c(h0)
    nchan, L = u.shape
    N = A.shape[1]
    bidx = np.ascontiguousarray(bidx, dtype=np.int64)
    assert delta.shape == (nchan, L) and A.shape == (nchan, N)
    assert B.ndim == 3 and B.shape[1:] == (N, L) and C.shape == B.shape
    assert bidx.shape == (nchan,) and (nchan == 0 or (bidx.min() >= 0 and bidx.max() < B.shape[0]))
    y = np.zeros((nchan, L))
    hl = np.zeros((nchan, N))
    ym = np.zeros((nchan, L)) if with_mag else None
    hm = np.zeros((nchan, N)) if with_mag else None
    rc = lib.oracle_scan_channels_disc(
        nchan, L, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        bidx.ctypes.data_as(_ip), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
        int(bool(zoh)), _ptr(h0), _ptr(y), _ptr(ym), _ptr(hl), _ptr(hm), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_channels failed ({rc})")
    return (y, hl, ym, hm) if with_mag else (y, hl)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                   h0=None, with_mag=False, nthreads=1, channels=None, lib=None, zoh=False):
    """Scan full tensors: u, delta, z [Bt, D, L]; A [D, N]; B, C [Bt, N, L]; D, bias [D];
    h0 [Bt, D, N]. ``channels``: optional list of (b, d) pairs; then only those channels are
    computed and the results are packed [len(channels), ...] in that order."""
    Bt, Dm, L = np.shape(u)
    N = np.shape(A)[1]
    if channels is None:
        bs = np.repeat(np.arange(Bt), Dm)
        ds = np.tile(np.arange(Dm), Bt)
    else:
        ch = np.asarray(channels, dtype=np.int64).reshape(-1, 2)
        bs, ds = ch[:, 0], ch[:, 1]

    def rows3(x):
        return None if x is None else np.asarray(x)[bs, ds, :]

    out = scan_rows(rows3(u), rows3(delta), np.asarray(A)[ds, :], B, C, bs,
                    None if D is None else np.asarray(D)[ds],
                    rows3(z), None if delta_bias is None else np.asarray(delta_bias)[ds],
                    delta_softplus, None if h0 is None else np.asarray(h0)[bs, ds, :],
                    with_mag, nthreads, lib, zoh)
    if channels is not None:
        return out
    shp_y, shp_h = (Bt, Dm, L), (Bt, Dm, N)
    res = [out[0].reshape(shp_y), out[1].reshape(shp_h)]
    if with_mag:
        res += [out[2].reshape(shp_y), out[3].reshape(shp_h)]
    return tuple(res)


def state_update(state, x, dt, A, B, C, D=None, z=None, smag=None, with_mag=False, lib=None,
                 zoh=False):
    """One recurrent step. state [Bt, D, N] (a new array is returned; the input is not
    modified); x, dt, z [Bt, D]; A [D, N]; B, C [Bt, N]; D [D].
    Returns (y [Bt, D], new_state) or, with ``with_mag``, (y, new_state, ymag, new_smag);
    ``smag`` is the incoming magnitude companion (defaults to |state|)."""
    lib = lib or load()
    st = np.array(state, dtype=np.float64, order="C", copy=True)
    Bt, Dm, N = st.shape
    x, dt, A, B, C, D, z = _c(x), _c(dt), _c(A), _c(B), _c(C), _c(D), _c(z)
    sm = None
    if with_mag:
        sm = np.abs(st) if smag is None else np.array(smag, dtype=np.float64, order="C", copy=True)
    y = np.zeros((Bt, Dm))
    ym = np.zeros((Bt, Dm)) if with_mag else None
    rc = lib.oracle_state_update_disc(Bt, Dm, N, _ptr(st), _ptr(sm), _ptr(x), _ptr(dt), _ptr(A),
                                      _ptr(B), _ptr(C), _ptr(D), _ptr(z), int(bool(zoh)), _ptr(y), _ptr(ym))
    if rc != 0:
        raise RuntimeError(f"oracle_state_update failed ({rc})")
    return (y, st, ym, sm) if with_mag else (y, st)


def rel_err(got, ref, mag):
    """Parity error: max_i |got_i - ref_i| / max(|ref_i|, mag_i), with ``mag`` the oracle's
    magnitude companion (the same recurrence on absolute values), so that outputs that
    cancel to ~0 are judged against the size of the terms that produced them."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    den = np.maximum(np.maximum(np.abs(ref), mag), 1e-300)
    if got.size == 0:
        return 0.0
    e = np.abs(got - ref) / den
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(e.max())


def conv_silu(x, w, cb=None, lib=None):
    """Causal depthwise conv + bias + SiLU in front of the scan: x [..., L] rows with
    w [..., K] and cb [...] per row (leading dims flattened alike). Returns u like x."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    L = shp[-1]
    xr = np.ascontiguousarray(x.reshape(-1, L))
    wr = np.ascontiguousarray(np.asarray(w, dtype=np.float64).reshape(xr.shape[0], -1))
    cr = None if cb is None else np.ascontiguousarray(np.asarray(cb, dtype=np.float64).reshape(-1))
    u = np.zeros_like(xr)
    rc = lib.oracle_conv_silu(xr.shape[0], L, wr.shape[1], _ptr(xr), _ptr(wr), _ptr(cr), _ptr(u))
    if rc != 0:
        raise RuntimeError(f"oracle_conv_silu failed ({rc})")
    return u.reshape(shp)
