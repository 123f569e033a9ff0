"""Workload builders shared by the GPU parity tests: the same seeded inputs as device tensors (for
the CUDA library) and as fp64 numpy arrays (for the oracle). Inputs come from gdn_synth only; no
expected value comes from the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import gdn_synth as syn

RECIPE = syn.GdnRecipe()


def bits_to_torch_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host_value(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values of a storage array from gdn_synth ("f32" float32, "bf16" uint16 bits)."""
    if dtype == "bf16":
        return syn.bf16_bits_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return bits_to_torch_bf16(x, device)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


class PackedCase:
    """Packed GDN decode inputs for one step: mixed_qkv, a, b (dtype), A_log, dt_bias (fp32)."""

    def __init__(self, B, H, HV, K, V, dtype, seed, step, layer=0):
        self.B, self.H, self.HV, self.K, self.V, self.dtype = B, H, HV, K, V, dtype
        self.host = syn.packed_inputs(B, H, HV, K, V, dtype, seed, step, layer)
        d = self.host
        self.mixed_qkv = to_device(d["mixed_qkv"], dtype)
        self.a = to_device(d["a"], dtype)
        self.b = to_device(d["b"], dtype)
        self.A_log = torch.from_numpy(d["A_log"]).cuda()
        self.dt_bias = torch.from_numpy(d["dt_bias"]).cuda()

    def views(self):
        hk = self.H * self.K
        x = self.mixed_qkv
        return x[:, :hk], x[:, hk:2 * hk], x[:, 2 * hk:]

    def oracle_args(self, rows=None):
        """fp64 (mixed_qkv, a, b, A_log, dt_bias) for the oracle, optionally only some rows."""
        d = self.host
        sel = slice(None) if rows is None else rows
        return (host_value(d["mixed_qkv"], self.dtype)[sel], host_value(d["a"], self.dtype)[sel],
                host_value(d["b"], self.dtype)[sel], d["A_log"].astype(np.float64),
                d["dt_bias"].astype(np.float64))


def device_state(num_slots, HV, V, K, seed, layer=0, std=1.0) -> torch.Tensor:
    """State pool [num_slots, HV, V, K] fp32 generated on the device (bit-identical to
    host_state_tile)."""
    s = torch.empty((num_slots, HV, V, K), dtype=torch.float32, device="cuda")
    syn.fill_normal_(s, seed, syn.Tag.STATE, 0, std, layer)
    return s


def host_state_tile(seed, HV, V, K, slot, hv, layer=0) -> np.ndarray:
    return syn.state_tile_values(seed, HV, V, K, slot, hv, 1.0, layer).astype(np.float64)


def host_state(num_slots, HV, V, K, seed, layer=0) -> np.ndarray:
    return syn.normal_f32(seed, syn.Tag.STATE, 0, (num_slots, HV, V, K), 1.0, layer).astype(np.float64)
