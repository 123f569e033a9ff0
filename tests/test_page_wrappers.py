"""The wrappers that carry the source pages' keyword names (the ReplaySSM microbenchmark's
run_replay, the KDA microbenchmark's fused call) marshal to the same kernels as the library's own
entry points: on identical inputs they give identical bits. The conv-weight layout conversion is
checked on the CPU against the stacking the KDA microbenchmark builds."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import ssm_recurrent_decode_gb300 as gdn
from gdn_cases import PackedCase, bits_to_torch_bf16, host_state


def test_conv_weight_from_stacked_inverts_the_page_stacking():
    dim, width = 12, 4
    conv_weights = torch.randn(3 * dim, width, generator=torch.Generator().manual_seed(5))
    # the stacking of the KDA microbenchmark's Inputs: per part, the [dim, width] block transposed
    stacked = torch.stack([conv_weights[i * dim:(i + 1) * dim].transpose(0, 1).contiguous()
                           for i in range(3)])
    assert tuple(stacked.shape) == (3, width, dim)
    assert torch.equal(gdn.conv_weight_from_stacked(stacked), conv_weights)


@pytest.mark.gpu
def test_replay_wrapper_matches_the_buffered_entry_point():
    B, H, HV, K, V, L = 3, 2, 4, 64, 64, 4
    c = PackedCase(B, H, HV, K, V, "bf16", 71, 0)
    S = torch.from_numpy(host_state(B + 1, HV, V, K, 71).astype(np.float32)).cuda()
    idx = torch.tensor([2, 0, 3], dtype=torch.int32, device="cuda")
    wp = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")
    runs = []
    for wrapper in (False, True):
        state = S.clone()
        ring = [torch.zeros((B + 1, HV, L, V), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((B + 1, H, L, K), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((B + 1, HV, L), device="cuda")]
        out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device="cuda")
        if wrapper:
            gdn.fused_recurrent_gdn_replayssm_decode(
                mixed_qkv=c.mixed_qkv, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias,
                scale=K ** -0.5, initial_state=state, d_cache=ring[0], k_cache=ring[1], g_cache=ring[2], out=out,
                ssm_state_indices=idx, write_pos=wp, use_qk_l2norm_in_kernel=True, nk=2)
        else:
            q, k, v = c.views()
            gdn.gdn_decode_buffered(q, k, v, state, out, *ring, wp, cache_indices=idx, H=H, a=c.a,
                                    b=c.b, A_log=c.A_log, dt_bias=c.dt_bias, scale=K ** -0.5)
        torch.cuda.synchronize()
        runs.append([out, state] + ring)
    for x, y in zip(*runs):
        assert torch.equal(x, y)


@pytest.mark.gpu
def test_fused_kda_wrapper_matches_the_fused_entry_point():
    T, heads, D = 3, 4, 64
    dim, num_slots = heads * D, T + 8
    ins = syn.fused_inputs(T, heads, D, num_slots, 72)
    x = bits_to_torch_bf16(ins["x"])
    conv_w = torch.from_numpy(ins["conv_w"]).cuda()
    stacked = torch.stack([conv_w[i * dim:(i + 1) * dim].transpose(0, 1).contiguous() for i in range(3)])
    g1 = bits_to_torch_bf16(ins["raw_g"]).view(1, T, heads, D)
    beta = bits_to_torch_bf16(ins["raw_beta"]).view(1, T, heads)
    g2 = bits_to_torch_bf16(ins["out_gate"])
    A_log = torch.from_numpy(ins["A_log"]).cuda()
    dt_bias = torch.from_numpy(ins["dt_bias"]).cuda()
    norm_w = torch.from_numpy(ins["norm_w"]).cuda()
    idx = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
    S0 = torch.empty((num_slots, heads, D, D), device="cuda")
    syn.fill_normal_(S0, 72, syn.Tag.STATE, 0, 1.0)
    # the page's SD layout: [num_slots, 3, 3*dim] seen through a transpose
    cs0 = bits_to_torch_bf16(ins["conv_state"]).transpose(1, 2).contiguous().transpose(1, 2)
    runs = []
    for wrapper in (False, True):
        state, cs = S0.clone(), cs0.clone().transpose(1, 2).contiguous().transpose(1, 2)
        if wrapper:
            out = torch.empty((1, T, heads, D), dtype=torch.bfloat16, device="cuda")
            gdn.fused_kda_decode(x=x, weight=gdn.conv_weight_from_stacked(stacked), bias=None,
                                 conv_state=cs, raw_g=g1, raw_beta=beta, A_log=A_log,
                                 dt_bias=dt_bias, state_indices=idx, state=state, out=out,
                                 lower_bound=-5.0, output_gate=g2, norm_weight=norm_w,
                                 norm_eps=1e-5)
            out = out.view(T, heads, D)
        else:
            out = torch.empty((T, heads, D), dtype=torch.bfloat16, device="cuda")
            gdn.gdn_decode_fused(x, conv_w, cs, g1.view(T, heads, D), beta.view(T, heads), A_log,
                                 dt_bias, state, idx, g2, norm_w, out, pad_slot_id=0,
                                 gate_kind="kda", lower_bound=-5.0, norm_eps=1e-5)
        torch.cuda.synchronize()
        runs.append((out, state, cs))
    for x_, y_ in zip(*runs):
        assert torch.equal(x_, y_)
