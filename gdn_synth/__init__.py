"""Seeded synthetic inputs for the gated delta-rule decode step.

This module is the one piece shared by the fp64 oracle's tests, the GPU parity tests and the
benchmark. It holds no arithmetic of the decode method itself: only a counter-based random
number generator and the recipes that shape its output into the workloads' tensors.

Generator
---------
Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
SC 2011): a 128-bit counter and a 64-bit key go through ten rounds of two 32x32->64-bit
multiplies with the published multipliers and Weyl key increments. Every element of every
tensor has its own counter, so any element can be generated on its own, in any order, on the
host (numpy, here) or on the device (``gdn_synth/csrc/synth.cu``), with bit-identical results.
That lets a multi-gigabyte state pool be generated on the GPU while the oracle regenerates only
the tiles it checks.

Counter layout: ``(index_lo, index_hi, step, stream)`` with ``stream = tag | layer << 16``,
key ``(seed_lo, seed_hi)``. ``index`` is the row-major element index inside the tensor.

Normal values
-------------
An Irwin-Hall sum of four 22-bit uniforms (the four Philox output words shifted right by 10)
is centred and scaled to unit variance: ``x = float32(s - 2**23) * c`` with
``c = float32(std * sqrt(3) / 2**22)``. The integer part is exact in fp32 and the single fp32
multiply rounds to nearest-even on both host and device, so the result is bit-identical.
The distribution has the stated mean and variance and is bounded by about 3.46 standard
deviations. bf16 tensors are the fp32 values rounded to nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "philox4x32_10", "normal_f32", "normal_at", "scale_constant",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "Tag", "stream_id",
    "packed_inputs", "fused_inputs", "state_tile_values", "permutation", "mamba_inputs",
]

_MASK32 = np.uint64(0xFFFFFFFF)
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds. Inputs are broadcastable uint32 arrays or ints.

    Returns the four output words as uint32 arrays.
    """
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    key0 = np.uint64(int(k0) & 0xFFFFFFFF)
    key1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            key0 = (key0 + PHILOX_W0) & _MASK32
            key1 = (key1 + PHILOX_W1) & _MASK32
        p0 = PHILOX_M0 * c[0]
        p1 = PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ key0, lo1, hi0 ^ c[3] ^ key1, lo0]
    return [x.astype(np.uint32) for x in c]


class Tag:
    """Stream tags: one per synthetic tensor kind."""
    QKV = 1          # packed mixed_qkv [B, 2*H*K + HV*V] (or q, k, v for the tiny fp32 case)
    A = 2            # raw gate input a [B, HV]
    B = 3            # raw beta input b [B, HV]
    A_LOG = 4        # A_log [HV] (or [heads])
    DT_BIAS = 5      # dt_bias [HV] (or [heads*head_dim])
    STATE = 6        # recurrent state pool [num_slots, HV, V, K]
    X = 7            # fused: pre-conv mixed_qkv [T, 3*dim]
    CONV_W = 8       # fused: conv weights [3*dim, 4]
    CONV_STATE = 9   # fused: conv state, logical [num_slots, 3*dim, 3]
    RAW_G = 10       # fused: raw per-key-channel gate [T, heads, head_dim]
    RAW_BETA = 11    # fused: raw beta [T, heads]
    OUT_GATE = 12    # fused: output gate [T, heads, head_dim]
    G_DIRECT = 13    # direct-gate mode: g [B, HV]
    BETA_DIRECT = 14  # direct-gate mode: beta logits [B, HV]
    M_X = 15         # Mamba decode: x [B, D]
    M_DT = 16        # Mamba decode: dt [B, D]
    M_A = 17         # Mamba decode: A [D, N]
    M_B = 18         # Mamba decode: B rows [B, N]
    M_C = 19         # Mamba decode: C rows [B, N]
    M_D = 20         # Mamba decode: skip D [D]
    M_Z = 21         # Mamba decode: gate z [B, D]
    M_H = 22         # Mamba decode: state h [B, D, N]


def stream_id(tag: int, layer: int = 0) -> int:
    return (int(tag) & 0xFFFF) | ((int(layer) & 0xFFFF) << 16)


def scale_constant(std: float) -> np.float32:
    """The fp32 constant that maps the centred Irwin-Hall integer to N(0, std^2)."""
    return np.float32(std * math.sqrt(3.0) / float(1 << 22))


def normal_at(seed: int, tag: int, step: int, index, std: float, layer: int = 0) -> np.ndarray:
    """fp32 normal values at the given element indices of one tensor."""
    idx = np.asarray(index, dtype=np.uint64)
    r = philox4x32_10(idx & _MASK32, idx >> np.uint64(32), np.uint64(step),
                      np.uint64(stream_id(tag, layer)), seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    s = sum((w >> np.uint32(10)).astype(np.int64) for w in r) - (1 << 23)
    return s.astype(np.float32) * scale_constant(std)


def normal_f32(seed: int, tag: int, step: int, shape, std: float, layer: int = 0,
               start: int = 0) -> np.ndarray:
    """A whole tensor (row-major element indices start .. start+numel) of fp32 normals."""
    n = int(np.prod(shape, dtype=np.int64))
    idx = np.arange(start, start + n, dtype=np.uint64)
    return normal_at(seed, tag, step, idx, std, layer).reshape(shape)


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); finite inputs. Returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _maybe_bf16(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> the storage form for `dtype`: float32 array, or uint16 bf16 bits."""
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of arange(n) as int32 (used for cache indices)."""
    return np.random.Generator(np.random.PCG64(seed)).permutation(n).astype(np.int32)


@dataclass(frozen=True)
class GdnRecipe:
    """Value distributions of the GDN packed workload, as (std) of N(0, std^2)."""
    qkv_std: float = 1.0
    a_std: float = 0.5        # N(0, 0.25)
    b_std: float = 0.5        # N(0, 0.25)
    A_log_std: float = 0.3    # N(0, 0.09)
    dt_bias_std: float = 0.1  # N(0, 0.01)
    state_std: float = 1.0


def packed_inputs(B: int, H: int, HV: int, K: int, V: int, dtype: str, seed: int, step: int,
                  layer: int = 0, recipe: GdnRecipe = GdnRecipe()) -> dict:
    """Per-step inputs of the packed GDN decode: mixed_qkv [B, 2HK+HV*V], a, b [B, HV]
    in `dtype` ("f32" arrays or "bf16" uint16 bit arrays), and the per-layer parameters
    A_log, dt_bias [HV] fp32 (drawn at step 0 so they are the same on every step)."""
    width = 2 * H * K + HV * V
    qkv = normal_f32(seed, Tag.QKV, step, (B, width), recipe.qkv_std, layer)
    a = normal_f32(seed, Tag.A, step, (B, HV), recipe.a_std, layer)
    b = normal_f32(seed, Tag.B, step, (B, HV), recipe.b_std, layer)
    return {
        "mixed_qkv": _maybe_bf16(qkv, dtype),
        "a": _maybe_bf16(a, dtype),
        "b": _maybe_bf16(b, dtype),
        "A_log": normal_f32(seed, Tag.A_LOG, 0, (HV,), recipe.A_log_std, layer),
        "dt_bias": normal_f32(seed, Tag.DT_BIAS, 0, (HV,), recipe.dt_bias_std, layer),
    }


def state_tile_values(seed: int, HV: int, V: int, K: int, slot: int, hv: int,
                      std: float = 1.0, layer: int = 0) -> np.ndarray:
    """Initial fp32 values of one state tile [V, K] of a pool [num_slots, HV, V, K]."""
    start = ((slot * HV) + hv) * V * K
    return normal_f32(seed, Tag.STATE, 0, (V, K), std, layer, start=start)


def fused_inputs(T: int, heads: int, head_dim: int, num_slots: int, seed: int, step: int = 0,
                 layer: int = 0) -> dict:
    """Per-step and parameter inputs of the fused KDA decode (all N(0,1) as in the workload;
    norm weight is ones). bf16 tensors come back as uint16 bit arrays; conv_state is logical
    [num_slots, 3*dim, 3] with tap 0 the oldest input."""
    dim = heads * head_dim
    return {
        "x": f32_to_bf16_bits(normal_f32(seed, Tag.X, step, (T, 3 * dim), 1.0, layer)),
        "conv_w": normal_f32(seed, Tag.CONV_W, 0, (3 * dim, 4), 1.0, layer),
        "conv_state": f32_to_bf16_bits(
            normal_f32(seed, Tag.CONV_STATE, 0, (num_slots, 3 * dim, 3), 1.0, layer)),
        "raw_g": f32_to_bf16_bits(normal_f32(seed, Tag.RAW_G, step, (T, heads, head_dim), 1.0, layer)),
        "raw_beta": f32_to_bf16_bits(normal_f32(seed, Tag.RAW_BETA, step, (T, heads), 1.0, layer)),
        "A_log": normal_f32(seed, Tag.A_LOG, 0, (heads,), 1.0, layer),
        "dt_bias": normal_f32(seed, Tag.DT_BIAS, 0, (dim,), 1.0, layer),
        "out_gate": f32_to_bf16_bits(normal_f32(seed, Tag.OUT_GATE, step, (T, heads, head_dim), 1.0, layer)),
        "norm_w": np.ones(head_dim, dtype=np.float32),
    }


def mamba_inputs(B: int, D: int, N: int, dtype: str, seed: int, step: int = 0) -> dict:
    """Inputs of one Mamba-1 decode step: x, z ~ N(0,1), dt positive (0.01 + |N(0, 0.1)|),
    B and C rows ~ N(0,1) (in `dtype`); parameters A negative (-(0.5 + |N(0,1)|)) and skip
    D ~ N(0,1) in fp32; the fp32 state h ~ N(0,1) (drawn at step 0)."""
    dt = np.float32(0.01) + np.abs(normal_f32(seed, Tag.M_DT, step, (B, D), 0.1))
    return {
        "x": _maybe_bf16(normal_f32(seed, Tag.M_X, step, (B, D), 1.0), dtype),
        "dt": _maybe_bf16(dt, dtype),
        "Bm": _maybe_bf16(normal_f32(seed, Tag.M_B, step, (B, N), 1.0), dtype),
        "Cm": _maybe_bf16(normal_f32(seed, Tag.M_C, step, (B, N), 1.0), dtype),
        "z": _maybe_bf16(normal_f32(seed, Tag.M_Z, step, (B, D), 1.0), dtype),
        "A": -(np.float32(0.5) + np.abs(normal_f32(seed, Tag.M_A, 0, (D, N), 1.0))),
        "Dskip": normal_f32(seed, Tag.M_D, 0, (D,), 1.0),
        "h": normal_f32(seed, Tag.M_H, 0, (B, D, N), 1.0),
    }


# ------------------------------------------------------------------------------------------------
# device twin (gdn_synth/csrc/synth.cu): fills CUDA tensors with the same values, bit for bit
# ------------------------------------------------------------------------------------------------
import ctypes as _ct
import os as _os
import subprocess as _sp
import threading as _th

_HERE = _os.path.dirname(_os.path.abspath(__file__))
_SYNTH_SRC = _os.path.join(_HERE, "csrc", "synth.cu")
_SYNTH_LIB = _os.path.join(_HERE, "_lib", "libgdn_synth.so")
_synth_lock = _th.Lock()
_synth = None


def build_device(force: bool = False) -> str:
    """Compile synth.cu for sm_103a into gdn_synth/_lib/libgdn_synth.so (nvcc)."""
    _os.makedirs(_os.path.dirname(_SYNTH_LIB), exist_ok=True)
    if (not force and _os.path.exists(_SYNTH_LIB)
            and _os.path.getmtime(_SYNTH_LIB) >= _os.path.getmtime(_SYNTH_SRC)):
        return _SYNTH_LIB
    tmp = f"{_SYNTH_LIB}.{_os.getpid()}.tmp"
    _sp.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
             "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SYNTH_SRC], check=True)
    _os.replace(tmp, _SYNTH_LIB)
    return _SYNTH_LIB


def _device_lib():
    global _synth
    with _synth_lock:
        if _synth is None:
            L = _ct.CDLL(build_device())
            L.synth_fill_normal.restype = _ct.c_int
            L.synth_fill_normal.argtypes = [_ct.c_void_p, _ct.c_int64, _ct.c_uint64, _ct.c_uint32,
                                            _ct.c_uint32, _ct.c_uint32, _ct.c_void_p, _ct.c_int64,
                                            _ct.c_float, _ct.c_int, _ct.c_void_p]
            L.synth_add_i32.restype = _ct.c_int
            L.synth_add_i32.argtypes = [_ct.c_void_p, _ct.c_int32, _ct.c_void_p]
            _synth = L
    return _synth


def fill_normal_(t, seed: int, tag: int, step: int, std: float, layer: int = 0, start: int = 0,
                 step_ptr=None, stream=None):
    """Fill a contiguous CUDA tensor (float32 or bfloat16) in place with the normals that
    normal_f32(seed, tag, step, t.shape, std, layer, start) gives on the host (bf16: rounded to
    nearest even). With step_ptr (a CUDA int32 tensor of one element) the step is
    step + step_ptr[0], read on the device."""
    import torch
    if not t.is_cuda or not t.is_contiguous() or t.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("fill_normal_ needs a contiguous CUDA float32 or bfloat16 tensor")
    s = torch.cuda.current_stream(t.device).cuda_stream if stream is None else stream
    rc = _device_lib().synth_fill_normal(
        t.data_ptr(), t.numel(), seed & 0xFFFFFFFFFFFFFFFF, tag, layer, step,
        None if step_ptr is None else step_ptr.data_ptr(), start, float(scale_constant(std)),
        int(t.dtype == torch.bfloat16), s)
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal failed with CUDA error {rc}")
    return t


def add_i32_(p, d: int, stream=None):
    """p[0] += d on the device (p: CUDA int32 tensor)."""
    import torch
    s = torch.cuda.current_stream(p.device).cuda_stream if stream is None else stream
    rc = _device_lib().synth_add_i32(p.data_ptr(), int(d), s)
    if rc != 0:
        raise RuntimeError(f"synth_add_i32 failed with CUDA error {rc}")
