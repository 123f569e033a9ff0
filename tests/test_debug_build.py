"""The index-checking debug build (libgdn_decode_debug.so, compiled with -DGDN_DEBUG).

Its kernels check every global-memory index they compute from their arguments (state tiles, q/k/v
rows, gate inputs, outputs, ring records, conv state, projection outputs and workspaces) against
the extents those arguments describe; an index outside its range would raise GDN_DEVERR_RANGE in
the error word and the access would be skipped. On the library's own cases, including the ragged
ones, no check may fire, and the debug build must give bit-identical results to the release
build (the checks change nothing else). The checks fire only on a wrong index computation inside
a kernel, which these tests cannot plant on the GPU; the guard-band tests watch the same accesses
from outside."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import ssm_recurrent_decode_gb300 as gdn
from gdn_cases import bits_to_torch_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _both(run):
    """run(err) -> list of output tensors, on fresh inputs each time; release, then debug."""
    err_r = torch.zeros(1, dtype=torch.int32, device="cuda")
    rel = run(err_r)
    err_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    with gdn.using_debug_build():
        dbg = run(err_d)
    torch.cuda.synchronize()
    assert int(err_d.item()) & gdn.GDN_DEVERR_RANGE == 0, "a debug index check fired"
    assert int(err_d.item()) == int(err_r.item())
    for a, b in zip(rel, dbg):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("B,K,V,sdt,chained", [
    (1, 128, 200, "f32", False), (8, 128, 200, "f32", False), (16, 128, 128, "f32", True),
    (32, 64, 200, "f32", False), (32, 128, 128, "bf16", False), (2, 128, 128, "bf16", False),
])
def test_step(B, K, V, sdt, chained):
    H, HV = 16, 32
    seed = 800 + B + K

    def run(err):
        x = torch.empty((B, 2 * H * K + HV * V), dtype=torch.bfloat16, device="cuda")
        a = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
        b = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(x, seed, syn.Tag.QKV, 0, 1.0)
        syn.fill_normal_(a, seed, syn.Tag.A, 0, 0.5)
        syn.fill_normal_(b, seed, syn.Tag.B, 0, 0.5)
        state = torch.empty((B + 3, HV, V, K), device="cuda")
        syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
        if sdt == "bf16":
            state = state.to(torch.bfloat16)
        idx = torch.from_numpy(syn.permutation(seed, B + 3)[:B].copy()).cuda()
        if B > 1:
            idx[0] = -1
        out = torch.full((B, 1, HV, V), 3.0, dtype=torch.bfloat16, device="cuda")
        q, k, v = gdn.split_mixed_qkv(x, H, HV, K, V)
        gdn.gdn_decode_step_indexed(q, k, v, state, out, idx, H=H, a=a, b=b,
                                    A_log=torch.full((HV,), 0.1, device="cuda"),
                                    dt_bias=torch.zeros(HV, device="cuda"), err_flags=err, chained=chained)
        return [state, out]

    _both(run)


@pytest.mark.parametrize("kernel,L", [("pipe", 8), ("stage", 8), ("stage", 16), ("tile", 8), ("tile", 3)])
def test_buffered(kernel, L):
    B, H, HV, K, V = 8, 16, 32, 128, 128
    seed = 820 + L

    def run(err):
        x = torch.empty((B, 2 * H * K + HV * V), dtype=torch.bfloat16, device="cuda")
        a = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
        b = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(x, seed, syn.Tag.QKV, 0, 1.0)
        syn.fill_normal_(a, seed, syn.Tag.A, 0, 0.5)
        syn.fill_normal_(b, seed, syn.Tag.B, 0, 0.5)
        state = torch.empty((B, HV, V, K), device="cuda")
        syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
        d = torch.zeros((B, HV, L, V), dtype=torch.bfloat16, device="cuda")
        kc = torch.zeros((B, H, L, K), dtype=torch.bfloat16, device="cuda")
        g = torch.zeros((B, HV, L), device="cuda")
        q, k, v = gdn.split_mixed_qkv(x, H, HV, K, V)
        outs = []
        for p in range(L):
            wp = torch.tensor([(p + r) % L for r in range(B)], dtype=torch.int32, device="cuda")
            out = torch.full((B, 1, HV, V), 3.0, dtype=torch.bfloat16, device="cuda")
            gdn.gdn_decode_buffered(q, k, v, state, out, d, kc, g, wp, H=H, a=a, b=b,
                                    A_log=torch.full((HV,), 0.1, device="cuda"),
                                    dt_bias=torch.zeros(HV, device="cuda"), err_flags=err, kernel=kernel)
            outs.append(out)
        return [state, d, kc, g] + outs

    _both(run)


@pytest.mark.parametrize("T,layout,kernel", [(4, "DS", "pipe"), (4, "SD", "pipe"), (4, "DS", "stage"),
                                             (4, "SD", "stage"), (2, "DS", "tile"), (3, "SD", "tile")])
def test_fused(T, layout, kernel):
    heads, D = 96, 128
    seed = 840 + T
    num_slots = T + 8

    def run(err):
        ins = syn.fused_inputs(T, heads, D, num_slots, seed)
        state = torch.empty((num_slots, heads, D, D), device="cuda")
        syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
        cs_ds = bits_to_torch_bf16(ins["conv_state"])
        cs = cs_ds.clone() if layout == "DS" else cs_ds.transpose(1, 2).contiguous()
        view = cs if layout == "DS" else cs.transpose(1, 2)
        x = torch.empty((T, 3 * heads * D), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
        gate = torch.empty((T, heads, D), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(gate, seed, syn.Tag.OUT_GATE, 0, 1.0)
        idx = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
        idx[1] = 0
        out = torch.full((T, heads, D), 3.0, dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_fused(x, torch.from_numpy(ins["conv_w"]).cuda(), view, bits_to_torch_bf16(ins["raw_g"]),
                             bits_to_torch_bf16(ins["raw_beta"]), torch.from_numpy(ins["A_log"]).cuda(),
                             torch.from_numpy(ins["dt_bias"]).cuda(), state, idx, gate,
                             torch.from_numpy(ins["norm_w"]).cuda(), out, pad_slot_id=0, err_flags=err,
                             kernel=kernel)
        return [state, cs, out]

    _both(run)


@pytest.mark.parametrize("T,N,Kd,splits", [(3, 1000, 1000, 0), (17, 5120, 1000, 12), (1, 1000, 1000, 3),
                                           (16, 1000, 5128, 4)])
def test_projection(T, N, Kd, splits):
    seed = 860 + T

    def run(err):
        x = torch.empty((T, Kd), dtype=torch.bfloat16, device="cuda")
        W = torch.empty((N, Kd), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
        syn.fill_normal_(W, seed, syn.Tag.CONV_W, 0, 0.02)
        y = torch.full((T, N), 3.0, device="cuda")
        gdn.gdn_gemv_bf16(x, W, y, splits=splits, workspace=gdn.gemv_workspace(T, N, Kd, splits), err_flags=err)
        return [y]

    _both(run)


def test_front():
    T, hidden, heads, D = 3, 512, 4, 64
    dim = heads * D
    seed = 880
    num_slots = T + 4

    def run(err):
        P = gdn.front_proj_width(heads, D, "gdn")
        ins = syn.fused_inputs(T, heads, D, num_slots, seed)
        W_in = torch.empty((P, hidden), dtype=torch.bfloat16, device="cuda")
        W_out = torch.empty((hidden, dim), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(W_in, seed, syn.Tag.CONV_W, 1, hidden ** -0.5)
        syn.fill_normal_(W_out, seed, syn.Tag.CONV_W, 2, dim ** -0.5)
        x = torch.empty((T, hidden), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
        state = torch.empty((num_slots, heads, D, D), device="cuda")
        syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
        cs = bits_to_torch_bf16(ins["conv_state"]).clone()
        z = torch.zeros((T, P), dtype=torch.bfloat16, device="cuda")
        o = torch.zeros((T, dim), dtype=torch.bfloat16, device="cuda")
        y = torch.full((T, hidden), 3.0, device="cuda")
        gdn.gdn_decode_front(x, W_in, W_out, z, o, y, torch.from_numpy(ins["conv_w"]).cuda(), cs,
                             torch.from_numpy(ins["A_log"]).cuda(),
                             torch.from_numpy(np.ascontiguousarray(ins["dt_bias"][:heads])).cuda(), state,
                             torch.arange(1, T + 1, dtype=torch.int32, device="cuda"),
                             torch.from_numpy(ins["norm_w"]).cuda(), pad_slot_id=0, gate_kind="gdn",
                             err_flags=err)
        return [z, o, y, cs, state]

    _both(run)
