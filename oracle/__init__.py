"""fp64 CPU oracle for the single-token gated delta-rule decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library and is never on the product
path. The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, loops in the order the sources state
the method); this module only builds that file with gcc, moves dense fp64 numpy arrays in and out
and splits packed inputs into their named parts.

Readings of points the sources leave open:
  * packed ``mixed_qkv`` row = [q (H*K) | k (H*K) | v (HV*V)], each head-major;
  * q/k head of value head hv is hv // (HV // H);
  * L2 norm is x / sqrt(sum x^2 + 1e-6); the K^-1/2 scale multiplies the normalised q;
  * the state tile is S[V, K] (key index contiguous) and u = S k, o = S q.

The Mamba-1 selective-scan decode ("Triton decode kernel + MBU analysis", Kernel design) is a
second recurrence through the same kind of boundary.

Parity status: every routine is pinned by tests/test_oracle_pins.py. The KDA gate's two readings
are pinned to closed values of their own formulas (points where exp(A_log[h]), the head index and
the per-key dt_bias change the value), and mutants that drop or misindex those terms fail
(tests/test_oracle_mutants.py). Which formula the KDA page means is a reading, since it names the
inputs and the -5 lower bound but prints no formula.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIBPATH = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

L2_EPS = 1e-6

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_lib/liboracle.so (gcc, no fused multiply-add)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC)):
        return _LIBPATH
    tmp = f"{_LIBPATH}.{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _load(path: str):
    """Load an oracle shared library and declare its signatures."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


class using_library:
    """Context manager that points this module at another build of the oracle (used by the tests
    that check the pins catch a deliberately broken copy)."""

    def __init__(self, path: str):
        self._path = path
        self._saved = None

    def __enter__(self):
        global _lib
        with _lock:
            self._saved = _lib
            _lib = _load(self._path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


def _declare(L):
    c_int, c_dbl, c_size = ctypes.c_int, ctypes.c_double, ctypes.c_size_t
    L.oracle_round_bf16.restype = c_dbl
    L.oracle_round_bf16.argtypes = [c_dbl]
    L.oracle_gdn_gates.restype = None
    L.oracle_gdn_gates.argtypes = [c_int, c_int, _D, _D, _D, _D, _D, _D]
    L.oracle_kda_gate.restype = None
    L.oracle_kda_gate.argtypes = [c_int, c_int, c_int, _D, _D, _D, c_dbl, c_int, _D]
    L.oracle_sigmoid.restype = None
    L.oracle_sigmoid.argtypes = [c_size, _D, _D]
    L.oracle_delta_step.restype = c_int
    L.oracle_delta_step.argtypes = [c_int] * 6 + [_D, _D, _D, _D, c_int, _D, c_dbl, c_int,
                                                  c_dbl, _I32, ctypes.c_int32, c_int, _D, _D]
    L.oracle_gdn_buffered.restype = c_int
    L.oracle_gdn_buffered.argtypes = ([c_int] * 6 + [_D, _D, _D, _D, _D, c_dbl, c_int, c_dbl,
                                       _I32, ctypes.c_int32, c_int, c_int, _D, _D, _D, _I32,
                                       _D, _D])
    L.oracle_conv_update.restype = c_int
    L.oracle_conv_update.argtypes = [c_int, c_int, _D, _D, _D, _D, c_int, _I32,
                                      ctypes.c_int32, _D]
    L.oracle_mamba_decode.restype = None
    L.oracle_mamba_decode.argtypes = [c_int, c_int, c_int, _D, _D, _D, _D, _D, _D, _D, _D, _D]
    L.oracle_gemv.restype = None
    L.oracle_gemv.argtypes = [c_int, c_int, c_int, _D, _D, _D]
    L.oracle_gated_rmsnorm.restype = None
    L.oracle_gated_rmsnorm.argtypes = [c_int, c_int, _D, _D, _D, c_dbl, c_int, _D]


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _pi(a):
    return None if a is None else a.ctypes.data_as(_I32)


def _i32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.int32)


def _check_inplace(state: np.ndarray):
    if state.dtype != np.float64 or not state.flags.c_contiguous:
        raise TypeError("state must be a C-contiguous float64 array (it is updated in place)")


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even) of each fp64 element."""
    f = np.vectorize(lib().oracle_round_bf16, otypes=[np.float64])
    return f(_f64(x))


def gdn_gates(a, b, A_log, dt_bias):
    """g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b); a, b: [B, HV]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    B, HV = a.shape
    g = np.empty((B, HV)); beta = np.empty((B, HV))
    lib().oracle_gdn_gates(B, HV, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(g), _p(beta))
    return g, beta


def kda_gate(raw_g, A_log, dt_bias, lower_bound=-5.0, form=0):
    """Per-key-channel log-decay; raw_g: [T, heads, D]; form 0 = clamped GDN gate, form 1 =
    lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias))."""
    raw_g, A_log, dt_bias = _f64(raw_g), _f64(A_log), _f64(dt_bias)
    T, heads, D = raw_g.shape
    g = np.empty_like(raw_g)
    lib().oracle_kda_gate(T, heads, D, _p(raw_g), _p(A_log), _p(dt_bias), float(lower_bound),
                          int(form), _p(g))
    return g


def sigmoid(x):
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_sigmoid(x.size, _p(x), _p(out))
    return out


def delta_step(q, k, v, g, beta, state, *, scale, use_qk_l2norm=True, idx=None, pad_slot=-1,
               l2_eps=L2_EPS, state_bf16=False):
    """One decode step. q, k: [B, H, K]; v: [B, HV, V]; g: [B, HV] or [B, HV, K] (per key);
    beta: [B, HV]; state: [num_slots, HV, V, K] float64, updated in place (and rounded to bf16
    after the update when state_bf16). Returns (out [B, HV, V], number of out-of-range rows)."""
    _check_inplace(state)
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    num_slots = state.shape[0]
    if state.shape != (num_slots, HV, V, K):
        raise ValueError(f"state shape {state.shape} != (num_slots, {HV}, {V}, {K})")
    per_key = int(g.ndim == 3)
    idx = _i32(idx)
    out = np.empty((B, HV, V))
    bad = lib().oracle_delta_step(B, H, HV, K, V, num_slots, _p(q), _p(k), _p(v), _p(g), per_key,
                                  _p(beta), float(scale), int(bool(use_qk_l2norm)), float(l2_eps),
                                  _pi(idx), int(pad_slot), int(bool(state_bf16)), _p(state), _p(out))
    return out, bad


def split_packed(mixed_qkv, H, HV, K, V):
    """[B, 2HK + HV V] -> q [B, H, K], k [B, H, K], v [B, HV, V]."""
    x = _f64(mixed_qkv)
    B = x.shape[0]
    q = x[:, : H * K].reshape(B, H, K)
    k = x[:, H * K: 2 * H * K].reshape(B, H, K)
    v = x[:, 2 * H * K: 2 * H * K + HV * V].reshape(B, HV, V)
    return q, k, v


def gdn_step_packed(mixed_qkv, a, b, A_log, dt_bias, state, *, H, HV, K, V, scale=None,
                    use_qk_l2norm=True, idx=None, pad_slot=-1, state_bf16=False):
    """The packed GDN decode step with the raw gate inputs; returns (out, bad)."""
    q, k, v = split_packed(mixed_qkv, H, HV, K, V)
    g, beta = gdn_gates(a, b, A_log, dt_bias)
    scale = K ** -0.5 if scale is None else scale
    return delta_step(q, k, v, g, beta, state, scale=scale, use_qk_l2norm=use_qk_l2norm, idx=idx,
                      pad_slot=pad_slot, state_bf16=state_bf16)


def gdn_buffered(q, k, v, g, beta, state, d_cache, k_cache, g_cache, write_pos, *, L,
                 ring_bf16=True, scale, use_qk_l2norm=True, idx=None, pad_slot=-1, l2_eps=L2_EPS):
    """One buffered decode step; state (checkpoint) and the three rings are float64 arrays
    updated in place. Returns (out, bad)."""
    for arr in (state, d_cache, k_cache, g_cache):
        _check_inplace(arr)
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    num_slots = state.shape[0]
    assert d_cache.shape == (num_slots, HV, L, V)
    assert k_cache.shape == (num_slots, H, L, K)
    assert g_cache.shape == (num_slots, HV, L)
    idx = _i32(idx)
    wp = _i32(write_pos)
    out = np.empty((B, HV, V))
    bad = lib().oracle_gdn_buffered(B, H, HV, K, V, num_slots, _p(q), _p(k), _p(v), _p(g),
                                    _p(beta), float(scale), int(bool(use_qk_l2norm)), float(l2_eps),
                                    _pi(idx), int(pad_slot), int(L), int(bool(ring_bf16)),
                                    _p(d_cache), _p(k_cache), _p(g_cache), _pi(wp), _p(state),
                                    _p(out))
    return out, bad


def conv_update(x, w, conv_state, *, idx=None, pad_slot=-1, bias=None):
    """Width-4 causal conv update with SiLU. x: [T, C]; w: [C, 4]; conv_state: [num_slots, C, 3]
    float64 (tap 0 oldest), updated in place. Returns (y [T, C], bad)."""
    _check_inplace(conv_state)
    x, w = _f64(x), _f64(w)
    T, C = x.shape
    bias = None if bias is None else _f64(bias)
    y = np.empty((T, C))
    idx = _i32(idx)
    bad = lib().oracle_conv_update(T, C, _p(x), _p(w), None if bias is None else _p(bias),
                                   _p(conv_state), conv_state.shape[0], _pi(idx), int(pad_slot),
                                   _p(y))
    return y, bad


def gated_rmsnorm(x, gate, w, eps=1e-5, act="silu"):
    """x / sqrt(mean(x^2) + eps) * w * act(gate) over the last axis."""
    x, gate, w = _f64(x), _f64(gate), _f64(w)
    shape = x.shape
    D = shape[-1]
    rows = x.size // D
    out = np.empty_like(x)
    lib().oracle_gated_rmsnorm(rows, D, _p(x), _p(gate), _p(w), float(eps),
                               {"silu": 0, "sigmoid": 1}[act], _p(out))
    return out.reshape(shape)


def fused_kda(x, conv_w, conv_state, raw_g, raw_beta, A_log, dt_bias, state, out_gate, norm_w, *,
              idx, pad_slot=0, lower_bound=-5.0, gate_form=0, gate_kind="kda", norm_eps=1e-5,
              act="silu", scale=None, use_qk_l2norm=True):
    """Fused decode: conv update -> q/k/v split per head -> gate and beta -> delta step (per-key
    decay for KDA, one decay per head for the GDN gate) -> gated RMSNorm.
    x: [T, 3*dim]; conv_state [num_slots, 3*dim, 3] and state [num_slots, heads, D, D] are float64,
    updated in place. raw_g: [T, heads, D] (kda) or [T, heads] (gdn). Returns (out, bad)."""
    x = _f64(x)
    T = x.shape[0]
    heads, D = out_gate.shape[1], out_gate.shape[2]
    dim = heads * D
    y, bad = conv_update(x, conv_w, conv_state, idx=idx, pad_slot=pad_slot)
    q = y[:, :dim].reshape(T, heads, D)
    k = y[:, dim:2 * dim].reshape(T, heads, D)
    v = y[:, 2 * dim:].reshape(T, heads, D)
    if gate_kind == "kda":
        g = kda_gate(raw_g, A_log, dt_bias, lower_bound, gate_form)
    else:
        g, _ = gdn_gates(_f64(raw_g), np.zeros((T, heads)), A_log, dt_bias)
    beta = sigmoid(_f64(raw_beta).reshape(T, heads))
    scale = D ** -0.5 if scale is None else scale
    o, _ = delta_step(q, k, v, g, beta, state, scale=scale, use_qk_l2norm=use_qk_l2norm, idx=idx,
                      pad_slot=pad_slot)
    out = gated_rmsnorm(o, out_gate, norm_w, norm_eps, act)
    return out, bad


def mamba_decode(x, dt, A, Bm, Cm, h, *, Dskip=None, z=None):
    """Mamba-1 selective-scan decode step. x, dt, z: [B, D]; A: [D, N]; Bm, Cm: [B, N];
    Dskip: [D]; h: [B, D, N] float64, updated in place. Returns y [B, D]."""
    _check_inplace(h)
    x, dt, A, Bm, Cm = _f64(x), _f64(dt), _f64(A), _f64(Bm), _f64(Cm)
    B, D = x.shape
    N = A.shape[1]
    assert h.shape == (B, D, N)
    Dskip = None if Dskip is None else _f64(Dskip)
    z = None if z is None else _f64(z)
    y = np.empty((B, D))
    lib().oracle_mamba_decode(B, D, N, _p(x), _p(dt), _p(A), _p(Bm), _p(Cm),
                              None if Dskip is None else _p(Dskip), None if z is None else _p(z),
                              _p(h), _p(y))
    return y


def gemv(x, W):
    """y [T, N] = x [T, Kd] . W[N, Kd]^T in fp64 (the decode projection)."""
    x, W = _f64(x), _f64(W)
    T, Kd = x.shape
    N = W.shape[0]
    assert W.shape[1] == Kd
    y = np.empty((T, N))
    lib().oracle_gemv(T, N, Kd, _p(x), _p(W), _p(y))
    return y


def front_columns(heads, D, gate_kind="gdn"):
    """Column ranges of the front's projection output z: q|k|v (3*dim), out_gate (dim), raw_g
    (dim for the KDA gate, heads for the GDN gate), raw_beta (heads)."""
    dim = heads * D
    G = dim if gate_kind == "kda" else heads
    return {"qkv": (0, 3 * dim), "out_gate": (3 * dim, 4 * dim), "raw_g": (4 * dim, 4 * dim + G),
            "raw_beta": (4 * dim + G, 4 * dim + G + heads)}


def decode_front(x, W_in, W_out, conv_w, conv_state, A_log, dt_bias, state, norm_w, *, heads, D,
                 idx, pad_slot=0, gate_kind="gdn", gate_form=0, lower_bound=-5.0, act="silu",
                 norm_eps=1e-5):
    """One DeltaNet layer's decode forward ("Optimization Log", Integration: proj + conv1d +
    recurrent + norm_gated + output): z = x W_in^T, then the fused decode on the columns of z,
    then y = o W_out^T. z and o are rounded to bf16, the dtype the front stores them in; conv_state
    and state (float64) are updated in place. Returns (y, bad)."""
    x = _f64(x)
    T = x.shape[0]
    z = round_bf16(gemv(x, W_in))
    col = front_columns(heads, D, gate_kind)
    part = lambda name: z[:, col[name][0]:col[name][1]]
    raw_g = part("raw_g").reshape(T, heads, D) if gate_kind == "kda" else part("raw_g")
    o, bad = fused_kda(part("qkv"), conv_w, conv_state, raw_g, part("raw_beta"), A_log, dt_bias,
                       state, part("out_gate").reshape(T, heads, D), norm_w, idx=idx,
                       pad_slot=pad_slot, lower_bound=lower_bound, gate_form=gate_form,
                       gate_kind=gate_kind, norm_eps=norm_eps, act=act)
    o = round_bf16(o.reshape(T, heads * D))
    return gemv(o, W_out), bad
