"""Python binding of libgdn_decode.so, the GB300 (sm_103a) single-token gated delta-rule decode.

Argument marshalling only: every function here takes torch tensors that already live on the GPU,
passes their device pointers, sizes and strides through the C ABI declared in
``include/gdn_decode.h``, and launches on the current torch stream. Every step of the decode runs
in the library's CUDA kernels; there is no Python, PyTorch or CPU fallback, and a missing or
unbuildable library raises.

Entry points (same names as the C ABI):
  gdn_decode_step          row b on state slot b
  gdn_decode_step_indexed  row b on state slot cache_indices[b] (the packed decode over a pool)
  gdn_decode_buffered      output-only decode that writes the state back once every L steps
  gdn_decode_fused         conv1d update -> delta step (per-key or per-head decay) -> gated RMSNorm
  mamba_selective_scan_decode  the Mamba-1 selective-scan decode step (a diagonal recurrence)
plus ``fused_recurrent_gated_delta_rule_packed_decode``, the packed call with the keyword names
of "Microbenchmark: buffered output-only GDN decode (ReplaySSM Part A)" (_bench_cfg, run_packed).
"""
from __future__ import annotations

import contextlib
import ctypes
import threading

from . import _build

__all__ = [
    "lib", "build", "GdnError", "GdnStepArgs", "GdnRingArgs", "GdnFusedArgs",
    "gdn_decode_step", "gdn_decode_step_indexed", "gdn_decode_buffered", "gdn_decode_fused",
    "gdn_strerror", "split_mixed_qkv", "fused_recurrent_gated_delta_rule_packed_decode", "PreparedCall",
    "MambaArgs", "mamba_selective_scan_decode", "gdn_selftest_bounded_wait",
    "GemvArgs", "gdn_gemv_bf16", "gemv_workspace",
    "GDN_F32", "GDN_BF16", "GDN_DEVERR_BAD_INDEX", "GDN_DEVERR_BAD_WRITE_POS", "GDN_DEVERR_TIMEOUT",
    "GDN_DEVERR_RANGE", "debug_lib", "using_debug_build",
    "EXPORTS",
]

GDN_F32, GDN_BF16 = 0, 1
GDN_GATE_RAW, GDN_GATE_DIRECT = 0, 1
GDN_FUSED_GATE_KDA, GDN_FUSED_GATE_GDN = 0, 1
GDN_ACT_SILU, GDN_ACT_SIGMOID = 0, 1
GDN_DEVERR_BAD_INDEX, GDN_DEVERR_BAD_WRITE_POS, GDN_DEVERR_TIMEOUT = 0x1, 0x2, 0x4
GDN_DEVERR_RANGE = 0x8
GDN_KERNEL = {"auto": 0, "tile": 1, "pipe": 2, "stage": 3}
ABI_VERSION = 7

# every function the header declares
EXPORTS = ("gdn_decode_step", "gdn_decode_step_indexed", "gdn_decode_buffered", "gdn_decode_fused",
           "gdn_strerror", "gdn_abi_struct_size", "gdn_abi_version", "mamba_selective_scan_decode",
           "gdn_selftest_bounded_wait", "gdn_gemv_bf16", "gdn_gemv_default_splits",
           "gdn_gemv_workspace_bytes", "gdn_gemv_bf16_noalloc", "gdn_decode_front",
           "gdn_front_proj_width", "gdn_gemv_set_wait_limit", "gdn_decode_step_indexed_chained")

_i32, _i64, _f32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class GdnStepArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("H", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
                ("num_slots", _i32), ("in_dtype", _i32), ("out_dtype", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp),
                ("q_stride", _i64), ("k_stride", _i64), ("v_stride", _i64),
                ("gate_mode", _i32), ("a", _vp), ("b", _vp), ("A_log", _vp), ("dt_bias", _vp),
                ("g", _vp), ("beta", _vp), ("scale", _f32), ("use_qk_l2norm", _i32),
                ("state", _vp), ("out", _vp), ("err_flags", _vp), ("state_dtype", _i32)]


class GdnRingArgs(ctypes.Structure):
    _fields_ = [("L", _i32), ("ring_dtype", _i32), ("d_cache", _vp), ("k_cache", _vp),
                ("g_cache", _vp), ("write_pos", _vp), ("kernel", _i32)]


class GdnFusedArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("heads", _i32), ("head_dim", _i32), ("num_slots", _i32),
                ("x", _vp), ("x_stride", _i64), ("conv_w", _vp), ("conv_b", _vp),
                ("conv_state", _vp), ("cs_stride_slot", _i64), ("cs_stride_chan", _i64),
                ("cs_stride_tap", _i64), ("gate_kind", _i32), ("kda_gate_form", _i32),
                ("raw_g", _vp), ("raw_beta", _vp), ("A_log", _vp), ("dt_bias", _vp),
                ("lower_bound", _f32), ("scale", _f32), ("use_qk_l2norm", _i32),
                ("state", _vp), ("state_indices", _vp), ("pad_slot_id", _i32),
                ("out_gate", _vp), ("norm_w", _vp), ("norm_eps", _f32), ("gate_act", _i32),
                ("out", _vp), ("err_flags", _vp), ("kernel", _i32), ("raw_g_stride", _i64),
                ("raw_beta_stride", _i64), ("out_gate_stride", _i64)]


class GdnFrontArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("hidden", _i32), ("x", _vp), ("x_stride", _i64), ("W_in", _vp),
                ("W_out", _vp), ("z", _vp), ("o", _vp), ("y", _vp), ("y_dtype", _i32),
                ("y_stride", _i64), ("in_splits", _i32), ("out_splits", _i32), ("core", GdnFusedArgs)]


class MambaArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("D", _i32), ("N", _i32), ("in_dtype", _i32), ("out_dtype", _i32),
                ("x", _vp), ("dt", _vp), ("A", _vp), ("Bm", _vp), ("Cm", _vp), ("Dskip", _vp),
                ("z", _vp), ("h", _vp), ("h_out", _vp), ("y", _vp), ("err_flags", _vp)]


class GemvArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("N", _i32), ("Kd", _i32), ("out_dtype", _i32), ("x", _vp),
                ("x_stride", _i64), ("W", _vp), ("y", _vp), ("y_stride", _i64), ("splits", _i32),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("err_flags", _vp)]


class GdnError(RuntimeError):
    """A non-zero status from the library (the message is gdn_strerror's)."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {gdn_strerror(status)} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libgdn_decode.so in-tree (nvcc, sm_103a); returns its path."""
    return _build.build(force=force)


def _load(path: str):
    """Open one build of the library and declare its entry points' signatures."""
    L = ctypes.CDLL(path)
    for name in ("gdn_decode_step",):
        getattr(L, name).argtypes = [ctypes.POINTER(GdnStepArgs), _vp]
    L.gdn_decode_step_indexed.argtypes = [ctypes.POINTER(GdnStepArgs), _vp, _i32, _vp]
    L.gdn_decode_step_indexed_chained.argtypes = [ctypes.POINTER(GdnStepArgs), _vp, _i32, _vp]
    L.gdn_decode_buffered.argtypes = [ctypes.POINTER(GdnStepArgs), _vp, _i32,
                                      ctypes.POINTER(GdnRingArgs), _vp]
    L.gdn_decode_fused.argtypes = [ctypes.POINTER(GdnFusedArgs), _vp]
    L.mamba_selective_scan_decode.argtypes = [ctypes.POINTER(MambaArgs), _vp]
    L.mamba_selective_scan_decode.restype = ctypes.c_int
    L.gdn_selftest_bounded_wait.argtypes = [_vp, _i64, _i32, _vp]
    L.gdn_decode_front.argtypes = [ctypes.POINTER(GdnFrontArgs), _vp]
    L.gdn_decode_front.restype = ctypes.c_int
    L.gdn_front_proj_width.argtypes = [_i32, _i32, _i32]
    L.gdn_front_proj_width.restype = _i64
    L.gdn_gemv_bf16.argtypes = [ctypes.POINTER(GemvArgs), _vp]
    L.gdn_gemv_bf16.restype = ctypes.c_int
    L.gdn_gemv_default_splits.argtypes = [_i32, _i32, _i32]
    L.gdn_gemv_default_splits.restype = _i32
    L.gdn_gemv_workspace_bytes.argtypes = [_i32, _i32, _i32]
    L.gdn_gemv_workspace_bytes.restype = ctypes.c_size_t
    L.gdn_gemv_bf16_noalloc.argtypes = [ctypes.POINTER(GemvArgs), _vp]
    L.gdn_gemv_bf16_noalloc.restype = ctypes.c_int
    L.gdn_gemv_set_wait_limit.argtypes = [_i64]
    L.gdn_gemv_set_wait_limit.restype = _i64
    L.gdn_selftest_bounded_wait.restype = ctypes.c_int
    for name in ("gdn_decode_step", "gdn_decode_step_indexed", "gdn_decode_buffered",
                 "gdn_decode_fused", "gdn_abi_version", "gdn_decode_step_indexed_chained"):
        getattr(L, name).restype = ctypes.c_int
    L.gdn_strerror.argtypes = [ctypes.c_int]
    L.gdn_strerror.restype = ctypes.c_char_p
    L.gdn_abi_struct_size.argtypes = [ctypes.c_int]
    L.gdn_abi_struct_size.restype = ctypes.c_size_t
    sizes = [L.gdn_abi_struct_size(i) for i in range(6)]
    want = [ctypes.sizeof(GdnStepArgs), ctypes.sizeof(GdnRingArgs), ctypes.sizeof(GdnFusedArgs),
            ctypes.sizeof(GemvArgs), ctypes.sizeof(GdnFrontArgs), ctypes.sizeof(MambaArgs)]
    if sizes != want or L.gdn_abi_version() != ABI_VERSION:
        raise RuntimeError(f"libgdn_decode.so ABI mismatch: struct sizes {sizes} vs {want}")
    return L


def lib():
    """The loaded library (built first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(_build.build())
    return _lib


_debug_lib = None


@contextlib.contextmanager
def using_debug_build():
    """Inside the with-block every entry point of this module calls the index-checking debug
    build (debug_lib) instead of the release library; prepared calls keep the library they were
    made with. For tests."""
    global _lib
    L = debug_lib()
    prev = lib()
    with _lock:
        _lib = L
    try:
        yield L
    finally:
        with _lock:
            _lib = prev


def debug_lib():
    """The index-checking debug build, libgdn_decode_debug.so (built first if needed): the same
    entry points, whose kernels report an out-of-range computed index through the error word
    (GDN_DEVERR_RANGE) instead of making the access. For tests; not for timing."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _load(_build.build(debug=True))
    return _debug_lib


def gdn_strerror(status: int) -> str:
    return lib().gdn_strerror(int(status)).decode()


# ------------------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return GDN_F32
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _ptr(t, name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dense(t, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _rows(t, name: str, width: int):
    """A [B, width] or [B, heads, dim] view whose rows are dense: returns the row stride."""
    if t.dim() == 3:
        if t.stride(2) != 1 or t.stride(1) != t.shape[2] or t.shape[1] * t.shape[2] != width:
            raise ValueError(f"{name}: rows must be dense [heads, dim] of width {width}")
    elif t.dim() == 2:
        if t.stride(1) != 1 or t.shape[1] != width:
            raise ValueError(f"{name}: expected [B, {width}] with unit inner stride")
    else:
        raise ValueError(f"{name}: expected a 2-D or 3-D tensor")
    return t.stride(0)


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def split_mixed_qkv(mixed_qkv, H: int, HV: int, K: int, V: int):
    """Views q [B, H*K], k [B, H*K], v [B, HV*V] of a packed row [q | k | v] (no copy)."""
    hk = H * K
    return mixed_qkv[:, :hk], mixed_qkv[:, hk:2 * hk], mixed_qkv[:, 2 * hk:2 * hk + HV * V]


def _step_args(q, k, v, state, out, *, H, a, b, A_log, dt_bias, g, beta, scale, use_qk_l2norm,
               err_flags) -> GdnStepArgs:
    torch = _torch()
    if state.dim() != 4:
        raise ValueError("state must be [num_slots, HV, V, K]")
    _dense(state, "state")
    num_slots, HV, V, K = state.shape
    B = q.shape[0]
    if H is None:
        H = (q.shape[1] if q.dim() == 3 else q.shape[1] // K)
    _dense(out, "out")
    if out.numel() != B * HV * V:
        raise ValueError(f"out must hold B*HV*V = {B * HV * V} elements")
    s = GdnStepArgs()
    s.B, s.H, s.HV, s.K, s.V, s.num_slots = B, H, HV, K, V, num_slots
    s.in_dtype, s.out_dtype = _dtype_code(q), _dtype_code(out)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    s.q, s.k, s.v = _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v")
    s.q_stride, s.k_stride, s.v_stride = _rows(q, "q", H * K), _rows(k, "k", H * K), _rows(v, "v", HV * V)
    if g is not None or beta is not None:
        s.gate_mode = GDN_GATE_DIRECT
        s.g = _ptr(_dense(g, "g"), "g", torch.float32)
        s.beta = _ptr(_dense(beta, "beta"), "beta", torch.float32)
    else:
        s.gate_mode = GDN_GATE_RAW
        for t, n in ((a, "a"), (b, "b")):
            if t is None or t.dtype != q.dtype:
                raise TypeError(f"{n} must be given with the dtype of q")
        s.a, s.b = _ptr(_dense(a, "a"), "a"), _ptr(_dense(b, "b"), "b")
        s.A_log = _ptr(_dense(A_log, "A_log"), "A_log", torch.float32)
        s.dt_bias = _ptr(_dense(dt_bias, "dt_bias"), "dt_bias", torch.float32)
    s.scale = 0.0 if scale is None else float(scale)
    s.use_qk_l2norm = int(bool(use_qk_l2norm))
    s.state = _ptr(state, "state")
    s.state_dtype = _dtype_code(state)
    s.out = _ptr(out, "out")
    s.err_flags = _ptr(err_flags, "err_flags", torch.int32)
    return s


def _check(fn: str, rc: int):
    if rc != 0:
        raise GdnError(fn, rc)


class PreparedCall:
    """A library call whose argument structs were built once (``prepare=True`` on an entry
    point). Calling it only launches, which takes a few microseconds of host time instead of
    re-marshalling every tensor; that matters for small batches, where the kernels take a few
    microseconds themselves. The tensors it was built from must stay alive with the same storage;
    each launch reads their current contents."""

    __slots__ = ("_name", "_fn", "_args", "_keep")

    def __init__(self, name, fn, args, keep):
        self._name, self._fn, self._args, self._keep = name, fn, args, keep

    def __call__(self, stream=None):
        _check(self._name, self._fn(*self._args, _stream(stream)))


def _run_or_prepare(name, args, keep, stream, prepare, result):
    fn = getattr(lib(), name)
    if prepare:
        return PreparedCall(name, fn, args, keep)
    _check(name, fn(*args, _stream(stream)))
    return result


# ------------------------------------------------------------------------------------------------
# entry points
# ------------------------------------------------------------------------------------------------
def gdn_decode_step(q, k, v, state, out, *, H=None, a=None, b=None, A_log=None, dt_bias=None,
                    g=None, beta=None, scale=None, use_qk_l2norm=True, err_flags=None, stream=None,
                    prepare=False):
    """One decode step, row b on slot b. q, k: [B, H*K] (or [B, H, K]) row views; v: [B, HV*V];
    gates either raw (a, b [B, HV] in the dtype of q; A_log, dt_bias [HV] fp32) or direct
    (g, beta [B, HV] fp32); state [num_slots, HV, V, K] fp32 (or bf16: stored in bf16, computed in
    fp32) updated in place; out [B, HV, V] (or [B, 1, HV, V]) fp32 or bf16.
    prepare=True returns a PreparedCall instead of launching (every entry point takes it)."""
    s = _step_args(q, k, v, state, out, H=H, a=a, b=b, A_log=A_log, dt_bias=dt_bias, g=g,
                   beta=beta, scale=scale, use_qk_l2norm=use_qk_l2norm, err_flags=err_flags)
    return _run_or_prepare("gdn_decode_step", (ctypes.byref(s),), (s,), stream, prepare, out)


def gdn_decode_step_indexed(q, k, v, state, out, cache_indices, *, pad_slot_id=-1, H=None, a=None,
                            b=None, A_log=None, dt_bias=None, g=None, beta=None, scale=None,
                            use_qk_l2norm=True, err_flags=None, chained=False, stream=None,
                            prepare=False):
    """As gdn_decode_step, with row b on slot cache_indices[b] (int32 [B] on the device); rows
    whose index is pad_slot_id are skipped (state untouched, out zeroed). chained=True calls
    gdn_decode_step_indexed_chained (a layer of a multi-layer decode: the launch may overlap the
    kernel before it on the stream, which must not write this call's state or cache_indices)."""
    torch = _torch()
    s = _step_args(q, k, v, state, out, H=H, a=a, b=b, A_log=A_log, dt_bias=dt_bias, g=g,
                   beta=beta, scale=scale, use_qk_l2norm=use_qk_l2norm, err_flags=err_flags)
    idx = _ptr(_dense(cache_indices, "cache_indices"), "cache_indices", torch.int32)
    return _run_or_prepare("gdn_decode_step_indexed_chained" if chained else "gdn_decode_step_indexed",
                           (ctypes.byref(s), ctypes.c_void_p(idx), ctypes.c_int32(int(pad_slot_id))),
                           (s,), stream, prepare, out)


def gdn_decode_buffered(q, k, v, state, out, d_cache, k_cache, g_cache, write_pos, *,
                        cache_indices=None, pad_slot_id=-1, H=None, a=None, b=None, A_log=None,
                        dt_bias=None, g=None, beta=None, scale=None, use_qk_l2norm=True,
                        err_flags=None, kernel="auto", stream=None, prepare=False):
    """Buffered output-only decode. state holds the checkpoints; d_cache [num_slots, HV, L, V],
    k_cache [num_slots, H, L, K] (both fp32 or both bf16), g_cache [num_slots, HV, L] fp32;
    write_pos int32 [B] is read, never advanced (the caller moves it to (p+1) % L).
    kernel: "auto" (the persistent pipelined kernel when K == V == 128, rows are 16-byte aligned
    and L > 1, else the per-tile kernel), "tile", "pipe" or "stage" (one CTA per tile staged in
    shared memory) to force one."""
    torch = _torch()
    s = _step_args(q, k, v, state, out, H=H, a=a, b=b, A_log=A_log, dt_bias=dt_bias, g=g,
                   beta=beta, scale=scale, use_qk_l2norm=use_qk_l2norm, err_flags=err_flags)
    r = GdnRingArgs()
    r.L = d_cache.shape[2]
    if k_cache.dtype != d_cache.dtype:
        raise TypeError("d_cache and k_cache must share one dtype")
    r.ring_dtype = _dtype_code(d_cache)
    expect = {"d_cache": (s.num_slots, s.HV, r.L, s.V), "k_cache": (s.num_slots, s.H, r.L, s.K),
              "g_cache": (s.num_slots, s.HV, r.L)}
    for name, t in (("d_cache", d_cache), ("k_cache", k_cache), ("g_cache", g_cache)):
        if tuple(t.shape) != expect[name]:
            raise ValueError(f"{name} must be {expect[name]}, got {tuple(t.shape)}")
        _dense(t, name)
    r.d_cache, r.k_cache = _ptr(d_cache, "d_cache"), _ptr(k_cache, "k_cache")
    r.g_cache = _ptr(g_cache, "g_cache", torch.float32)
    r.write_pos = _ptr(_dense(write_pos, "write_pos"), "write_pos", torch.int32)
    r.kernel = GDN_KERNEL[kernel]
    idx = None if cache_indices is None else _ptr(_dense(cache_indices, "cache_indices"),
                                                  "cache_indices", torch.int32)
    return _run_or_prepare("gdn_decode_buffered",
                           (ctypes.byref(s), ctypes.c_void_p(idx), ctypes.c_int32(int(pad_slot_id)),
                            ctypes.byref(r)), (s, r), stream, prepare, out)


def _fused_core(conv_w, conv_state, A_log, dt_bias, state, state_indices, norm_w, *, conv_b,
                pad_slot_id, gate_kind, kda_gate_form, lower_bound, scale, use_qk_l2norm, norm_eps,
                gate_act, err_flags, kernel):
    """The arguments of gdn_decode_fused that do not depend on the per-token inputs."""
    torch = _torch()
    _dense(state, "state")
    num_slots, heads, D, _ = state.shape
    f = GdnFusedArgs()
    f.heads, f.head_dim, f.num_slots = heads, D, num_slots
    f.conv_w = _ptr(_dense(conv_w, "conv_w"), "conv_w", torch.float32)
    f.conv_b = _ptr(conv_b, "conv_b", torch.float32)
    if tuple(conv_state.shape) != (num_slots, 3 * heads * D, 3):
        raise ValueError("conv_state must have logical shape [num_slots, 3*dim, 3]")
    f.conv_state = _ptr(conv_state, "conv_state", torch.bfloat16)
    f.cs_stride_slot, f.cs_stride_chan, f.cs_stride_tap = conv_state.stride()
    f.gate_kind = {"kda": GDN_FUSED_GATE_KDA, "gdn": GDN_FUSED_GATE_GDN}[gate_kind]
    f.kda_gate_form = int(kda_gate_form)
    f.A_log = _ptr(_dense(A_log, "A_log"), "A_log", torch.float32)
    f.dt_bias = _ptr(_dense(dt_bias, "dt_bias"), "dt_bias", torch.float32)
    f.lower_bound = float(lower_bound)
    f.scale = 0.0 if scale is None else float(scale)
    f.use_qk_l2norm = int(bool(use_qk_l2norm))
    f.state = _ptr(state, "state", torch.float32)
    f.state_indices = _ptr(_dense(state_indices, "state_indices"), "state_indices", torch.int32)
    f.pad_slot_id = int(pad_slot_id)
    f.norm_w = _ptr(_dense(norm_w, "norm_w"), "norm_w", torch.float32)
    f.norm_eps = float(norm_eps)
    f.gate_act = {"silu": GDN_ACT_SILU, "sigmoid": GDN_ACT_SIGMOID}[gate_act]
    f.err_flags = _ptr(err_flags, "err_flags", torch.int32)
    f.kernel = GDN_KERNEL[kernel]
    return f


def front_proj_width(heads, head_dim, gate_kind="gdn"):
    """P, the width of the front's input projection output z (see gdn_decode_front)."""
    code = {"kda": GDN_FUSED_GATE_KDA, "gdn": GDN_FUSED_GATE_GDN}[gate_kind]
    return int(lib().gdn_front_proj_width(int(heads), int(head_dim), code))


def gdn_decode_front(x, W_in, W_out, z, o, y, conv_w, conv_state, A_log, dt_bias, state,
                     state_indices, norm_w, *, conv_b=None, pad_slot_id=0, gate_kind="gdn",
                     kda_gate_form=0, lower_bound=-5.0, scale=None, use_qk_l2norm=True,
                     norm_eps=1e-5, gate_act="silu", in_splits=0, out_splits=0, err_flags=None,
                     kernel="auto", stream=None, prepare=False):
    """One DeltaNet layer's decode forward (declared in include/gdn_front.h): z = x W_in^T (bf16
    z [T, P], columns q|k|v, out_gate, raw_g, raw_beta), o = conv -> step -> gated RMSNorm on views
    of z, y = o W_out^T. x bf16 [T, hidden] (row view allowed); W_in bf16 [P, hidden]; W_out bf16
    [hidden, dim]; z, o dense bf16 scratch [T, P], [T, dim]; y fp32 or bf16 [T, hidden]; the rest
    as for gdn_decode_fused."""
    torch = _torch()
    T, hidden = x.shape
    c = _fused_core(conv_w, conv_state, A_log, dt_bias, state, state_indices, norm_w,
                    conv_b=conv_b, pad_slot_id=pad_slot_id, gate_kind=gate_kind,
                    kda_gate_form=kda_gate_form, lower_bound=lower_bound, scale=scale,
                    use_qk_l2norm=use_qk_l2norm, norm_eps=norm_eps, gate_act=gate_act,
                    err_flags=err_flags, kernel=kernel)
    P = front_proj_width(c.heads, c.head_dim, gate_kind)
    dim = c.heads * c.head_dim
    if tuple(W_in.shape) != (P, hidden) or tuple(W_out.shape) != (hidden, dim):
        raise ValueError(f"expected W_in [{P}, {hidden}] and W_out [{hidden}, {dim}]")
    if tuple(z.shape) != (T, P) or tuple(o.shape) != (T, dim) or tuple(y.shape) != (T, hidden):
        raise ValueError(f"expected z [{T}, {P}], o [{T}, {dim}], y [{T}, {hidden}]")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y need unit inner stride")
    a = GdnFrontArgs()
    a.T, a.hidden = T, hidden
    a.x, a.x_stride = _ptr(x, "x", torch.bfloat16), x.stride(0)
    a.W_in = _ptr(_dense(W_in, "W_in"), "W_in", torch.bfloat16)
    a.W_out = _ptr(_dense(W_out, "W_out"), "W_out", torch.bfloat16)
    a.z = _ptr(_dense(z, "z"), "z", torch.bfloat16)
    a.o = _ptr(_dense(o, "o"), "o", torch.bfloat16)
    a.y, a.y_dtype, a.y_stride = _ptr(y, "y"), _dtype_code(y), y.stride(0)
    a.in_splits, a.out_splits = int(in_splits), int(out_splits)
    a.core = c
    return _run_or_prepare("gdn_decode_front", (ctypes.byref(a),), (a,), stream, prepare, y)


def gdn_decode_fused(x, conv_w, conv_state, raw_g, raw_beta, A_log, dt_bias, state, state_indices,
                     out_gate, norm_w, out, *, conv_b=None, pad_slot_id=0, gate_kind="kda",
                     kda_gate_form=0, lower_bound=-5.0, scale=None, use_qk_l2norm=True,
                     norm_eps=1e-5, gate_act="silu", err_flags=None, kernel="auto", stream=None,
                     prepare=False):
    """Fused decode: conv update -> delta step -> gated RMSNorm, one launch.
    kernel: "auto" (when head_dim is 128, the conv state is in the DS or SD layout, rows are
    16-byte aligned and there are more than two (token, head) tiles per SM: one CTA per tile
    staged in shared memory from sixteen tiles per SM, the persistent pipelined kernel below that;
    else the per-tile kernel), "tile", "pipe" or "stage" to force one.
    x bf16 [T, 3*dim]; conv_w fp32 [3*dim, 4]; conv_state bf16 with logical shape
    [num_slots, 3*dim, 3] (any strides: the "DS" layout is the plain tensor, the "SD" layout a
    transposed view of [num_slots, 3, 3*dim]); raw_g bf16 [T, heads, D] (kda) or [T, heads] (gdn);
    raw_beta bf16 [T, heads]; A_log fp32 [heads]; dt_bias fp32 [heads*D] (kda) or [heads] (gdn);
    state fp32 [num_slots, heads, D, D]; state_indices int32 [T]; out_gate bf16 [T, heads, D];
    norm_w fp32 [D]; out bf16 [T, heads, D]. raw_g, raw_beta and out_gate may be row views (any
    token stride, dense within a row), e.g. slices of one projection output."""
    torch = _torch()
    T = x.shape[0]
    f = _fused_core(conv_w, conv_state, A_log, dt_bias, state, state_indices, norm_w,
                    conv_b=conv_b, pad_slot_id=pad_slot_id, gate_kind=gate_kind,
                    kda_gate_form=kda_gate_form, lower_bound=lower_bound, scale=scale,
                    use_qk_l2norm=use_qk_l2norm, norm_eps=norm_eps, gate_act=gate_act,
                    err_flags=err_flags, kernel=kernel)
    heads, D = f.heads, f.head_dim
    f.T = T
    if x.stride(1) != 1:
        raise ValueError("x must have unit inner stride")
    f.x, f.x_stride = _ptr(x, "x", torch.bfloat16), x.stride(0)
    f.raw_g_stride = _rows(raw_g, "raw_g", heads * D if gate_kind == "kda" else heads)
    f.raw_g = _ptr(raw_g, "raw_g", torch.bfloat16)
    f.raw_beta_stride = _rows(raw_beta, "raw_beta", heads)
    f.raw_beta = _ptr(raw_beta, "raw_beta", torch.bfloat16)
    f.out_gate_stride = _rows(out_gate, "out_gate", heads * D)
    f.out_gate = _ptr(out_gate, "out_gate", torch.bfloat16)
    f.out = _ptr(_dense(out, "out"), "out", torch.bfloat16)
    return _run_or_prepare("gdn_decode_fused", (ctypes.byref(f),), (f,), stream, prepare, out)


def fused_recurrent_gated_delta_rule_packed_decode(mixed_qkv, a, b, A_log, dt_bias, scale,
                                                   initial_state, out, ssm_state_indices,
                                                   use_qk_l2norm_in_kernel=True, pad_slot_id=-1,
                                                   err_flags=None, stream=None):
    """The packed decode with the keyword names of the sglang microbenchmark's run_packed:
    mixed_qkv [B, 2*H*K + HV*V], a, b [B, HV], A_log, dt_bias [HV], initial_state
    [num_slots, HV, V, K] fp32 (updated in place), out [B, 1, HV, V], ssm_state_indices int32 [B].
    H is recovered from the row width."""
    _, HV, V, K = initial_state.shape
    H = _heads_from_width(mixed_qkv, HV, V, K)
    q, k, v = split_mixed_qkv(mixed_qkv, H, HV, K, V)
    return gdn_decode_step_indexed(q, k, v, initial_state, out, ssm_state_indices,
                                   pad_slot_id=pad_slot_id, H=H, a=a, b=b, A_log=A_log,
                                   dt_bias=dt_bias, scale=scale,
                                   use_qk_l2norm=use_qk_l2norm_in_kernel, err_flags=err_flags,
                                   stream=stream)


def _heads_from_width(mixed_qkv, HV, V, K):
    width = mixed_qkv.shape[1]
    if (width - HV * V) <= 0 or (width - HV * V) % (2 * K):
        raise ValueError("mixed_qkv width does not match 2*H*K + HV*V")
    return (width - HV * V) // (2 * K)


def fused_recurrent_gdn_replayssm_decode(mixed_qkv, a, b, A_log, dt_bias, scale, initial_state,
                                         d_cache, k_cache, g_cache, out, ssm_state_indices,
                                         write_pos, use_qk_l2norm_in_kernel=True, nk=2,
                                         pad_slot_id=-1, err_flags=None, stream=None):
    """The buffered output-only decode with the keyword names of the sglang microbenchmark's
    run_replay: initial_state [num_slots, HV, V, K] fp32 holds the checkpoints; d_cache
    [num_slots, HV, L, V], k_cache [num_slots, H, L, K], g_cache [num_slots, HV, L]; write_pos
    int32 [B] is read, not advanced. nk (the number of key chunks that page's kernel walks while
    replaying its ring) is accepted and has no effect: this library's replay is low-rank and
    never re-forms the state outside the flush step."""
    del nk
    _, HV, V, K = initial_state.shape
    H = _heads_from_width(mixed_qkv, HV, V, K)
    q, k, v = split_mixed_qkv(mixed_qkv, H, HV, K, V)
    return gdn_decode_buffered(q, k, v, initial_state, out, d_cache, k_cache, g_cache, write_pos,
                               cache_indices=ssm_state_indices, pad_slot_id=pad_slot_id, H=H, a=a,
                               b=b, A_log=A_log, dt_bias=dt_bias, scale=scale,
                               use_qk_l2norm=use_qk_l2norm_in_kernel, err_flags=err_flags,
                               stream=stream)


def conv_weight_from_stacked(weight):
    """Converts conv weights stacked per q/k/v part as [3, width, dim] (the layout the KDA
    microbenchmark passes to its fused op) to this library's [3*dim, width], channel-major. A
    one-time parameter conversion, not part of the decode step."""
    parts, width, dim = weight.shape
    return weight.permute(0, 2, 1).reshape(parts * dim, width).contiguous()


def fused_kda_decode(x, weight, bias, conv_state, raw_g, raw_beta, A_log, dt_bias, state_indices,
                     state, out, lower_bound, output_gate, norm_weight, norm_eps, *,
                     pad_slot_id=0, gate_act="silu", err_flags=None, stream=None):
    """The fused KDA decode with the keyword names of the KDA microbenchmark's `fused` call: x
    [T, 3*dim], weight [3*dim, 4] (conv_weight_from_stacked converts the stacked layout), bias or
    None, conv_state logical [num_slots, 3*dim, 3] (DS tensor or SD transposed view), raw_g
    [1, T, heads, D] or [T, heads, D], raw_beta [1, T, heads] or [T, heads], state [num_slots,
    heads, D, D], out [1, T, heads, D] or [T, heads, D], output_gate [T, heads, D], norm_weight
    [D] fp32. Slot 0 is the NULL (pad) slot, as on that page."""
    T = x.shape[0]
    heads, D = state.shape[1], state.shape[2]
    return gdn_decode_fused(x, weight, conv_state, raw_g.view(T, heads, D), raw_beta.view(T, heads),
                            A_log, dt_bias, state, state_indices, output_gate, norm_weight,
                            out.view(T, heads, D), conv_b=bias, pad_slot_id=pad_slot_id,
                            gate_kind="kda", lower_bound=lower_bound, norm_eps=norm_eps,
                            gate_act=gate_act, err_flags=err_flags, stream=stream)


def mamba_selective_scan_decode(x, dt, A, Bm, Cm, h, y, *, Dskip=None, z=None, h_out=None,
                                err_flags=None, stream=None, prepare=False):
    """Mamba-1 selective-scan decode step (declared in include/mamba_decode.h).
    x, dt: [B, D] and Bm, Cm: [B, N] (fp32 or bf16, one dtype); A: [D, N] fp32; Dskip: [D] fp32 or
    None; z: [B, D] or None; h: [B, D, N] fp32 state, updated in place unless h_out (same shape)
    is given; y: [B, D] fp32 or bf16; err_flags: an int32 CUDA tensor of one element or None."""
    torch = _torch()
    B, D = x.shape
    N = A.shape[1]
    m = MambaArgs()
    m.B, m.D, m.N = B, D, N
    m.in_dtype, m.out_dtype = _dtype_code(x), _dtype_code(y)
    for t, name in ((dt, "dt"), (Bm, "Bm"), (Cm, "Cm"), (z, "z")):
        if t is not None and t.dtype != x.dtype:
            raise TypeError(f"{name} must have the dtype of x")
    if tuple(h.shape) != (B, D, N) or (h_out is not None and tuple(h_out.shape) != (B, D, N)):
        raise ValueError(f"h (and h_out) must be [{B}, {D}, {N}]")
    m.x, m.dt = _ptr(_dense(x, "x"), "x"), _ptr(_dense(dt, "dt"), "dt")
    m.A = _ptr(_dense(A, "A"), "A", torch.float32)
    m.Bm, m.Cm = _ptr(_dense(Bm, "Bm"), "Bm"), _ptr(_dense(Cm, "Cm"), "Cm")
    m.Dskip = _ptr(None if Dskip is None else _dense(Dskip, "Dskip"), "Dskip", torch.float32)
    m.z = _ptr(None if z is None else _dense(z, "z"), "z")
    m.h = _ptr(_dense(h, "h"), "h", torch.float32)
    m.h_out = _ptr(None if h_out is None else _dense(h_out, "h_out"), "h_out", torch.float32)
    m.y = _ptr(_dense(y, "y"), "y")
    m.err_flags = _ptr(err_flags, "err_flags", torch.int32)
    return _run_or_prepare("mamba_selective_scan_decode", (ctypes.byref(m),), (m,), stream, prepare, y)


def gdn_selftest_bounded_wait(err_flags, limit_cycles, arrive, stream=None):
    """Run the bounded-wait self-test kernel (see include/gdn_decode.h); err_flags is a CUDA int32
    tensor of one element that receives GDN_DEVERR_TIMEOUT when the wait gives up."""
    torch = _torch()
    _check("gdn_selftest_bounded_wait",
           lib().gdn_selftest_bounded_wait(_ptr(err_flags, "err_flags", torch.int32), int(limit_cycles),
                                           int(bool(arrive)), _stream(stream)))


def gemv_workspace(T, N, Kd, splits=0, device=None):
    """A workspace tensor for gdn_gemv_bf16 with this split count (0: the library's choice), or
    None when the call needs none."""
    torch = _torch()
    L = lib()
    s = splits or L.gdn_gemv_default_splits(int(T), int(N), int(Kd))
    nbytes = L.gdn_gemv_workspace_bytes(int(T), int(N), int(s))
    if nbytes == 0:
        return None
    return torch.empty(nbytes // 4, dtype=torch.float32, device=device or "cuda")


def gdn_gemv_bf16(x, W, y, *, splits=0, workspace=None, err_flags=None, stream=None, prepare=False):
    """Decode projection y [T, N] = x [T, Kd] W[N, Kd]^T (declared in include/gdn_gemv.h). x and W
    bf16 with dense rows (x may be a row view), y fp32 or bf16. With more than one K split (splits
    = 0 lets the library choose) a workspace is needed: see gemv_workspace. err_flags: optional
    int32 CUDA tensor of one element that a kernel giving up a bounded wait ORs a bit into."""
    torch = _torch()
    T, Kd = x.shape
    N = W.shape[0]
    if W.shape[1] != Kd or tuple(y.shape) != (T, N):
        raise ValueError(f"expected W [{N}, {Kd}] and y [{T}, {N}]")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y need unit inner stride")
    g = GemvArgs()
    g.T, g.N, g.Kd = T, N, Kd
    g.out_dtype = _dtype_code(y)
    g.x, g.x_stride = _ptr(x, "x", torch.bfloat16), x.stride(0)
    g.W = _ptr(_dense(W, "W"), "W", torch.bfloat16)
    g.y, g.y_stride = _ptr(y, "y"), y.stride(0)
    g.splits = int(splits)
    if workspace is not None:
        g.workspace = _ptr(_dense(workspace, "workspace"), "workspace", torch.float32)
        g.workspace_bytes = workspace.numel() * 4
    if err_flags is not None:
        g.err_flags = _ptr(err_flags, "err_flags", torch.int32)
    return _run_or_prepare("gdn_gemv_bf16", (ctypes.byref(g),), (g, workspace, err_flags), stream, prepare, y)
