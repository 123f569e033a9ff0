"""GPU parity of gdn_decode_fused (conv1d update -> delta step -> gated RMSNorm in one launch)
against the fp64 oracle. Tolerances: bf16 output within 2e-2, fp32 state within 1e-5, conv state
bit-exact (it only moves bf16 values)."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import bits_to_torch_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def _run_fused(T, heads, D, *, layout="DS", gate_kind="kda", form=0, act="silu", seed=0,
               pad_rows=(), steps=1, sample_rows=None, kernel="auto"):
    dim = heads * D
    num_slots = T + 8
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    if gate_kind == "gdn":
        raw_g_bits = syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.RAW_G, 0, (T, heads), 1.0))
        dt_bias = syn.normal_f32(seed, syn.Tag.DT_BIAS, 0, (heads,), 1.0)
    else:
        raw_g_bits, dt_bias = ins["raw_g"], ins["dt_bias"]
    state = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device="cuda")
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
    S64 = state.cpu().numpy().astype(np.float64)
    cs_ds = bits_to_torch_bf16(ins["conv_state"])          # logical [slots, 3*dim, 3]
    if layout == "DS":
        conv_state = cs_ds.clone()
    else:                                                  # physical [slots, 3, 3*dim]
        conv_state = cs_ds.transpose(1, 2).contiguous().transpose(1, 2)
    cs64 = f64(ins["conv_state"]).reshape(num_slots, 3 * dim, 3).copy()
    idx_np = np.arange(1, T + 1, dtype=np.int32)           # slot 0 is the NULL (pad) slot
    for r in pad_rows:
        idx_np[r] = 0
    idx = torch.from_numpy(idx_np).cuda()
    conv_w = torch.from_numpy(ins["conv_w"]).cuda()
    A_log = torch.from_numpy(ins["A_log"]).cuda()
    dtb = torch.from_numpy(np.ascontiguousarray(dt_bias)).cuda()
    norm_w = torch.from_numpy(ins["norm_w"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst = {"out": 0.0, "state": 0.0}
    for step in range(steps):
        x_bits = syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.X, step, (T, 3 * dim), 1.0))
        gate_bits = syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.OUT_GATE, step, (T, heads, D), 1.0))
        out = torch.full((T, heads, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_fused(bits_to_torch_bf16(x_bits), conv_w, conv_state,
                             bits_to_torch_bf16(raw_g_bits), bits_to_torch_bf16(ins["raw_beta"]),
                             A_log, dtb, state, idx, bits_to_torch_bf16(gate_bits), norm_w, out,
                             pad_slot_id=0, gate_kind=gate_kind, kda_gate_form=form, gate_act=act,
                             err_flags=err, kernel=kernel)
        rows = np.arange(T) if sample_rows is None else np.asarray(sample_rows)
        if sample_rows is not None:
            # only the sampled rows' slots are followed by the oracle
            sl = idx_np[rows]
            S_sub = np.ascontiguousarray(S64[sl]); cs_sub = np.ascontiguousarray(cs64[sl])
            o_ref, _ = oracle.fused_kda(f64(x_bits)[rows], ins["conv_w"], cs_sub,
                                        f64(raw_g_bits)[rows], f64(ins["raw_beta"])[rows],
                                        ins["A_log"], dt_bias, S_sub, f64(gate_bits)[rows],
                                        ins["norm_w"], idx=np.arange(len(rows), dtype=np.int32),
                                        pad_slot=-1, gate_form=form, gate_kind=gate_kind, act=act)
            S64[sl], cs64[sl] = S_sub, cs_sub
        else:
            o_ref, _ = oracle.fused_kda(f64(x_bits), ins["conv_w"], cs64, f64(raw_g_bits),
                                        f64(ins["raw_beta"]), ins["A_log"], dt_bias, S64,
                                        f64(gate_bits), ins["norm_w"], idx=idx_np, pad_slot=0,
                                        gate_form=form, gate_kind=gate_kind, act=act)
        got = out.float().cpu().numpy()[rows]
        assert np.all(np.isfinite(got))
        worst["out"] = max(worst["out"], rel_err(got, o_ref))
    torch.cuda.synchronize()
    slots = idx_np if sample_rows is None else idx_np[np.asarray(sample_rows)]
    worst["state"] = rel_err(state.cpu().numpy()[slots], S64[slots])
    got_cs = conv_state.float().cpu().numpy()
    np.testing.assert_array_equal(got_cs[slots], cs64[slots])
    assert int(err.item()) == 0
    return worst


@pytest.mark.parametrize("kernel", ["tile", "pipe", "stage"])
@pytest.mark.parametrize("layout", ["DS", "SD"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_kda_config_shapes(layout, T, kernel):
    """The fused KDA decode shapes: 96 heads x 128, conv width 4, lower bound -5, silu gate, at
    the token counts where the library picks the per-tile kernel (one CTA per (token, head)); the
    per-tile, pipelined and staged kernels forced."""
    w = _run_fused(T, 96, 128, layout=layout, seed=T, kernel=kernel)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


@pytest.mark.parametrize("kernel", ["tile", "pipe", "stage", "auto"])
def test_kda_32_tokens_sampled_rows(kernel):
    """3072 tiles: the pipelined kernel walks about twenty per CTA through its stages; the library's
    own choice at this size is one CTA per tile staged in shared memory."""
    w = _run_fused(32, 96, 128, seed=32, sample_rows=[0, 7, 19, 31], kernel=kernel, steps=2)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


def test_kda_full_size_sampled_rows():
    """The benchmark's launch: 128 tokens x 96 heads (12288 tiles; the library's choice is one CTA
    per tile staged in shared memory), sampled token rows against the oracle."""
    w = _run_fused(128, 96, 128, seed=128, sample_rows=[0, 41, 90, 127])
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("act", ["silu", "sigmoid"])
def test_gate_readings_and_activations(form, act):
    w = _run_fused(4, 6, 64, form=form, act=act, seed=3 + form, steps=3)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w
    w = _run_fused(4, 6, 128, form=form, act=act, seed=13 + form, steps=3, kernel="pipe")
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


@pytest.mark.parametrize("D,kernel", [(16, "auto"), (32, "auto"), (128, "auto"), (128, "tile")])
def test_gdn_gate_and_small_heads(D, kernel):
    """The GDN gate (one decay per head) at several head sizes; 20 (token, head) tiles."""
    w = _run_fused(5, 4, D, gate_kind="gdn", seed=D, steps=2, layout="SD", kernel=kernel)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


@pytest.mark.parametrize("D,kernel", [(64, "auto"), (128, "pipe"), (128, "tile"), (128, "stage")])
def test_null_slot_rows_are_skipped(D, kernel):
    w = _run_fused(6, 4, D, seed=9, pad_rows=(0, 4), steps=2, kernel=kernel)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w


@pytest.mark.parametrize("T", [20, 24])
def test_kda_auto_choice_near_the_staged_threshold(T):
    """Token counts just past the staged kernel's threshold (about twelve tiles per SM) under the
    library's own choice, on sampled rows over two steps."""
    w = _run_fused(T, 96, 128, seed=40 + T, sample_rows=[0, T // 2, T - 1], kernel="auto", steps=2)
    assert w["out"] <= 2e-2 and w["state"] <= 1e-5, w
