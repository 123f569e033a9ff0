"""GPU parity of gdn_decode_step / gdn_decode_step_indexed against the fp64 oracle.

Tolerances (max |gpu - oracle| / max(1, |oracle|)): 1e-5 for fp32 outputs and for the fp32 state;
2e-2 for bf16 outputs. Both sides get the same seeded inputs from gdn_synth; each keeps its own
state across sequential steps."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import PackedCase, device_state, host_state, host_state_tile

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 2e-2


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _out_tensor(B, HV, V, out_dtype):
    dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    return torch.full((B, 1, HV, V), float("nan"), dtype=dt, device="cuda")


def _tol(out_dtype):
    return TOL_BF16 if out_dtype == "bf16" else TOL_F32


def _run(B, H, HV, K, V, dtype, out_dtype, seed, *, steps=1, indexed=True, num_slots=None,
         pad_rows=(), bad_rows=(), use_l2=True, scale=None, state_dtype="f32", first_out=None,
         chained=False):
    """Run `steps` sequential steps on both sides; compare out every step and the state at the
    end. Returns the worst errors (first_out, if a list, receives the first step's error)."""
    num_slots = num_slots or (B + len(pad_rows) + 2 if indexed else B)
    state = torch.from_numpy(host_state(num_slots, HV, V, K, seed).astype(np.float32)).cuda()
    if state_dtype == "bf16":
        state = state.to(torch.bfloat16)
    S64 = state.float().cpu().numpy().astype(np.float64)
    idx_np = None
    if indexed:
        idx_np = syn.permutation(seed + 1, num_slots)[:B].copy()
        for r in pad_rows:
            idx_np[r] = -1
        for r in bad_rows:
            idx_np[r] = num_slots + 3 + r
        idx = torch.from_numpy(idx_np).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst_out = 0.0
    for step in range(steps):
        c = PackedCase(B, H, HV, K, V, dtype, seed, step)
        out = _out_tensor(B, HV, V, out_dtype)
        q, k, v = c.views()
        kw = dict(H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias, scale=scale,
                  use_qk_l2norm=use_l2, err_flags=err)
        if indexed:
            gdn.gdn_decode_step_indexed(q, k, v, state, out, idx, pad_slot_id=-1, chained=chained, **kw)
        else:
            gdn.gdn_decode_step(q, k, v, state, out, **kw)
        o_ref, bad = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V,
                                            scale=scale, use_qk_l2norm=use_l2, idx=idx_np,
                                            pad_slot=-1, state_bf16=(state_dtype == "bf16"))
        got = out.float().cpu().numpy().reshape(B, HV, V)
        assert np.all(np.isfinite(got))
        worst_out = max(worst_out, rel_err(got, o_ref))
        if first_out is not None and step == 0:
            first_out.append(rel_err(got, o_ref))
        assert bad == len(bad_rows)
    torch.cuda.synchronize()
    worst_state = rel_err(state.float().cpu().numpy(), S64)
    flags = int(err.item())
    return worst_out, worst_state, flags


def test_tiny_fp32_eight_sequential_steps():
    """The tiny decode: B=2, H=2, HV=4, K=V=16, fp32 everything, 8 sequential steps."""
    for indexed in (False, True):
        wo, ws, flags = _run(2, 2, 4, 16, 16, "f32", "f32", seed=0, steps=8, indexed=indexed)
        assert wo <= TOL_F32 and ws <= TOL_F32 and flags == 0, (indexed, wo, ws)


@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("G", [1, 2, 3])
def test_shapes_fp32(K, G):
    H = 2
    for V in (K, 40):
        wo, ws, flags = _run(3, H, H * G, K, V, "f32", "f32", seed=K + G, steps=2)
        assert wo <= TOL_F32 and ws <= TOL_F32 and flags == 0, (V, wo, ws)


def test_ragged_multi_pass_rows():
    """V = 200 at K = 128 with few tiles: the rows are split over 13 CTAs per tile, the last ragged."""
    wo, ws, _ = _run(2, 1, 2, 128, 200, "f32", "f32", seed=5, steps=2)
    assert wo <= TOL_F32 and ws <= TOL_F32


def test_ragged_multi_pass_rows_whole_tiles():
    """V = 200 at K = 128 with 640 tiles: one CTA per tile, two row passes, the second ragged."""
    wo, ws, _ = _run(160, 2, 4, 128, 200, "f32", "f32", seed=6, steps=1)
    assert wo <= TOL_F32 and ws <= TOL_F32


@pytest.mark.parametrize("B", [1, 4, 16, 64])
def test_row_split_batches(B):
    """Small batches split each tile's rows over several CTAs (8 at B = 1, 2 at B = 16); the
    results do not depend on the split."""
    wo, ws, flags = _run(B, 16, 32, 128, 128, "bf16", "f32", seed=300 + B, steps=2)
    assert wo <= TOL_F32 and ws <= TOL_F32 and flags == 0, (B, wo, ws)


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_packed_bf16_small_batches(out_dtype):
    """The packed decode shapes (H=16, HV=32, K=V=128, bf16 in) at B = 1 and 16, every output."""
    for B in (1, 16):
        wo, ws, flags = _run(B, 16, 32, 128, 128, "bf16", out_dtype, seed=10 + B)
        assert wo <= _tol(out_dtype) and ws <= TOL_F32 and flags == 0, (B, wo, ws)


def test_pad_and_bad_indices():
    B, H, HV, K, V = 6, 2, 4, 32, 32
    wo, ws, flags = _run(B, H, HV, K, V, "bf16", "bf16", seed=3, pad_rows=(1,), bad_rows=(4,))
    assert wo <= TOL_BF16 and ws <= TOL_F32
    assert flags == gdn.GDN_DEVERR_BAD_INDEX


def test_no_l2norm_and_explicit_scale():
    wo, ws, _ = _run(3, 2, 4, 64, 64, "f32", "f32", seed=4, use_l2=False, scale=0.05, steps=1)
    assert wo <= TOL_F32 and ws <= TOL_F32


def test_direct_gates():
    B, H, HV, K, V = 4, 2, 4, 64, 32
    c = PackedCase(B, H, HV, K, V, "f32", 7, 0)
    g = syn.normal_f32(7, syn.Tag.G_DIRECT, 0, (B, HV), 0.5) - 0.3
    beta = 1.0 / (1.0 + np.exp(-syn.normal_f32(7, syn.Tag.BETA_DIRECT, 0, (B, HV), 1.0).astype(np.float64)))
    beta32 = beta.astype(np.float32)
    state = device_state(B, HV, V, K, 7)
    S64 = host_state(B, HV, V, K, 7)
    out = torch.empty((B, HV, V), device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_step(q, k, v, state, out, H=H, g=torch.from_numpy(g).cuda(),
                        beta=torch.from_numpy(beta32).cuda())
    qo, ko, vo = oracle.split_packed(c.oracle_args()[0], H, HV, K, V)
    o_ref, _ = oracle.delta_step(qo, ko, vo, g.astype(np.float64), beta32.astype(np.float64), S64,
                                 scale=K ** -0.5)
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL_F32
    assert rel_err(state.cpu().numpy(), S64) <= TOL_F32


def test_packed_call_with_page_keywords():
    """fused_recurrent_gated_delta_rule_packed_decode recovers H from the row width."""
    B, H, HV, K, V = 4, 16, 32, 128, 128
    c = PackedCase(B, H, HV, K, V, "bf16", 9, 0)
    state = device_state(B, HV, V, K, 9)
    S64 = host_state(B, HV, V, K, 9)
    idx = torch.arange(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device="cuda")
    gdn.fused_recurrent_gated_delta_rule_packed_decode(
        mixed_qkv=c.mixed_qkv, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias, scale=K ** -0.5,
        initial_state=state, out=out, ssm_state_indices=idx, use_qk_l2norm_in_kernel=True)
    o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V,
                                      idx=np.arange(B, dtype=np.int32))
    assert rel_err(out.float().cpu().numpy().reshape(B, HV, V), o_ref) <= TOL_BF16
    assert rel_err(state.cpu().numpy(), S64) <= TOL_F32


def test_empty_batch_is_a_no_op():
    state = torch.zeros((2, 4, 16, 16), device="cuda")
    x = torch.zeros((0, 2 * 2 * 16 + 4 * 16), device="cuda")
    q, k, v = gdn.split_mixed_qkv(x, 2, 4, 16, 16)
    out = torch.zeros((0, 4, 16), device="cuda")
    ab = torch.zeros((0, 4), device="cuda")
    gdn.gdn_decode_step(q, k, v, state, out, H=2, a=ab, b=ab, A_log=torch.zeros(4, device="cuda"),
                        dt_bias=torch.zeros(4, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(state == 0)


def test_side_stream():
    B, H, HV, K, V = 8, 2, 4, 128, 128
    c = PackedCase(B, H, HV, K, V, "bf16", 12, 0)
    state = device_state(B, HV, V, K, 12)
    S64 = host_state(B, HV, V, K, 12)
    out = torch.empty((B, HV, V), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        q, k, v = c.views()
        gdn.gdn_decode_step(q, k, v, state, out, H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias)
    s.synchronize()
    o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V)
    assert rel_err(out.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_device_generator_matches_host():
    """The device twin of the input generator gives the host generator's bits."""
    t = torch.empty((3, 5, 7, 16), dtype=torch.float32, device="cuda")
    syn.fill_normal_(t, 123, syn.Tag.STATE, 0, 1.0, layer=4)
    ref = syn.normal_f32(123, syn.Tag.STATE, 0, (3, 5, 7, 16), 1.0, layer=4)
    np.testing.assert_array_equal(t.cpu().numpy(), ref)
    tb = torch.empty((9, 33), dtype=torch.bfloat16, device="cuda")
    step = torch.tensor([5], dtype=torch.int32, device="cuda")
    syn.fill_normal_(tb, 77, syn.Tag.QKV, 2, 0.5, step_ptr=step)
    refb = syn.f32_to_bf16_bits(syn.normal_f32(77, syn.Tag.QKV, 7, (9, 33), 0.5))
    np.testing.assert_array_equal(tb.cpu().view(torch.int16).numpy().view(np.uint16), refb)


@pytest.mark.parametrize("B", [64, 256])
def test_packed_full_size_sampled_rows(B):
    """The packed decode at full batch sizes in the launch configuration the benchmark times:
    every row runs on the GPU; the oracle recomputes a sample of rows (first, last and seeded
    others) from their own state tiles."""
    H, HV, K, V = 16, 32, 128, 128
    seed = 100 + B
    c = PackedCase(B, H, HV, K, V, "bf16", seed, 0)
    idx_np = syn.permutation(seed, B)
    idx = torch.from_numpy(idx_np).cuda()
    state = device_state(B, HV, V, K, seed)
    out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_step_indexed(q, k, v, state, out, idx, H=H, a=c.a, b=c.b, A_log=c.A_log,
                                dt_bias=c.dt_bias)
    rows = sorted({0, B - 1, *np.random.default_rng(seed).choice(B, 6, replace=False).tolist()})
    mixed, a, b, A_log, dt_bias = c.oracle_args(rows)
    slots = idx_np[rows]
    S64 = np.stack([[host_state_tile(seed, HV, V, K, int(s), hv) for hv in range(HV)] for s in slots])
    o_ref, _ = oracle.gdn_step_packed(mixed, a, b, A_log, dt_bias, S64, H=H, HV=HV, K=K, V=V)
    got = out.float().cpu().numpy().reshape(B, HV, V)[rows]
    assert rel_err(got, o_ref) <= TOL_BF16
    got_state = state[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy()
    assert rel_err(got_state, S64) <= TOL_F32


# ------------------------------------------------------------------------------------------------
# bf16 state storage: fp32 arithmetic, the state rounded to bf16 as it is stored. Both sides round
# their own updated state, so a value next to a rounding midpoint may land one bf16 ulp apart (about
# 0.4% of that element); states and later outputs are held to the bf16 bar, 2e-2. The first step,
# which starts from identical bf16 values, is held to the fp32 bar when the output is fp32.
# ------------------------------------------------------------------------------------------------
def test_bf16_state_tiny_fp32_io():
    first = []
    wo, ws, flags = _run(2, 2, 4, 16, 16, "f32", "f32", seed=0, steps=8, state_dtype="bf16",
                         first_out=first)
    assert first[0] <= TOL_F32, first
    assert wo <= TOL_BF16 and ws <= TOL_BF16 and flags == 0, (wo, ws)


@pytest.mark.parametrize("K,G", [(32, 2), (64, 3), (128, 1)])
def test_bf16_state_shapes(K, G):
    wo, ws, flags = _run(3, 2, 2 * G, K, 40, "f32", "f32", seed=200 + K, steps=3, state_dtype="bf16")
    assert wo <= TOL_BF16 and ws <= TOL_BF16 and flags == 0, (wo, ws)


def test_bf16_state_packed_B16():
    first = []
    wo, ws, flags = _run(16, 16, 32, 128, 128, "bf16", "f32", seed=210, steps=2, state_dtype="bf16",
                         first_out=first, pad_rows=(3,))
    assert first[0] <= TOL_F32, first
    assert wo <= TOL_BF16 and ws <= TOL_BF16 and flags == 0, (wo, ws)


def test_bf16_state_packed_full_size_sampled_rows():
    B, H, HV, K, V = 256, 16, 32, 128, 128
    seed = 333
    c = PackedCase(B, H, HV, K, V, "bf16", seed, 0)
    idx_np = syn.permutation(seed, B)
    idx = torch.from_numpy(idx_np).cuda()
    state = device_state(B, HV, V, K, seed).to(torch.bfloat16)
    rows = sorted({0, B - 1, *np.random.default_rng(seed).choice(B, 6, replace=False).tolist()})
    slots = idx_np[rows]
    S64 = state[torch.from_numpy(slots.astype(np.int64)).cuda()].float().cpu().numpy().astype(np.float64)
    out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_step_indexed(q, k, v, state, out, idx, H=H, a=c.a, b=c.b, A_log=c.A_log,
                                dt_bias=c.dt_bias)
    mixed, a, b, A_log, dt_bias = c.oracle_args(rows)
    o_ref, _ = oracle.gdn_step_packed(mixed, a, b, A_log, dt_bias, S64, H=H, HV=HV, K=K, V=V,
                                      state_bf16=True)
    got = out.float().cpu().numpy().reshape(B, HV, V)[rows]
    assert rel_err(got, o_ref) <= TOL_BF16
    got_state = state[torch.from_numpy(slots.astype(np.int64)).cuda()].float().cpu().numpy()
    assert rel_err(got_state, S64) <= TOL_BF16


def test_bf16_state_rejected_by_the_buffered_decode():
    B, H, HV, K, V, L = 2, 1, 2, 32, 32, 4
    c = PackedCase(B, H, HV, K, V, "f32", 5, 0)
    state = torch.zeros((B, HV, V, K), dtype=torch.bfloat16, device="cuda")
    ring = [torch.zeros((B, HV, L, V), device="cuda"), torch.zeros((B, H, L, K), device="cuda"),
            torch.zeros((B, HV, L), device="cuda")]
    q, k, v = c.views()
    with pytest.raises(gdn.GdnError, match="dtype"):
        gdn.gdn_decode_buffered(q, k, v, state, torch.zeros((B, HV, V), device="cuda"), *ring,
                                torch.zeros(B, dtype=torch.int32, device="cuda"), H=H, a=c.a, b=c.b,
                                A_log=c.A_log, dt_bias=c.dt_bias)


@pytest.mark.parametrize("B,K", [(16, 128), (4, 128), (1, 128), (32, 64)])
def test_chained_layers_wait_for_the_previous_layer_output(B, K):
    """Two layers, the second taking the first one's output as its v (a data dependence between
    layers), in every order of ordinary and chained calls: a chained kernel may start early and
    load its state, but must read v only after the kernel before it has finished; an ordinary one
    (launched programmatically) waits before it touches memory. Repeated with fresh inputs; the
    results must equal, bit for bit, the two layers as ordinary calls, and match the oracle. Covers
    8, 4 and 2 rows per thread at K = 128 and whole tiles at K = 64."""
    H, HV, V = 4, 16, K
    G = HV // H
    num_slots = B + 2
    idx_np = syn.permutation(91, num_slots)[:B].copy()
    idx = torch.from_numpy(idx_np).cuda()
    results = {}
    # (first layer chained, second layer chained): an ordinary call waits before it touches memory
    # and only then lets the next kernel start, so every order must give the ordinary results. The
    # pools are reused every iteration, so a chained first layer follows a plain torch kernel (which
    # lets nothing start early): no run of chained calls then holds two calls on one pool.
    orders = [(False, False), (True, True), (False, True), (True, False)]
    fence = torch.zeros(1, device="cuda")
    for order in orders:
        pools = [torch.from_numpy(host_state(num_slots, HV, V, K, 90 + l).astype(np.float32)).cuda()
                 for l in range(2)]
        outs = []
        for it in range(6):
            q0 = torch.from_numpy(syn.normal_f32(92, syn.Tag.QKV, it, (B, H * K), 1.0)).cuda()
            k0 = torch.from_numpy(syn.normal_f32(93, syn.Tag.QKV, it, (B, H * K), 1.0)).cuda()
            v0 = torch.from_numpy(syn.normal_f32(94, syn.Tag.QKV, it, (B, HV * V), 1.0)).cuda()
            g = torch.full((B, HV), -0.1, device="cuda")
            beta = torch.full((B, HV), 0.5, device="cuda")
            out0 = torch.empty((B, HV * V), device="cuda")
            out1 = torch.empty((B, HV * V), device="cuda")
            if order[0]:
                fence.add_(1.0)
            gdn.gdn_decode_step_indexed(q0, k0, v0, pools[0], out0, idx, H=H, g=g, beta=beta,
                                        chained=order[0])
            gdn.gdn_decode_step_indexed(q0, k0, out0, pools[1], out1, idx, H=H, g=g, beta=beta,
                                        chained=order[1])
            outs.append((out0, out1))
        torch.cuda.synchronize()
        results[order] = ([o.cpu().numpy() for pair in outs for o in pair], [p.cpu().numpy() for p in pools])
    for order in orders[1:]:
        for a, b in zip(results[orders[0]][0] + results[orders[0]][1], results[order][0] + results[order][1]):
            np.testing.assert_array_equal(a, b)
    # the last iteration against the oracle, from the layers' states before it
    S = [host_state(num_slots, HV, V, K, 90 + l) for l in range(2)]
    for it in range(6):
        q0 = syn.normal_f32(92, syn.Tag.QKV, it, (B, H, K), 1.0).astype(np.float64)
        k0 = syn.normal_f32(93, syn.Tag.QKV, it, (B, H, K), 1.0).astype(np.float64)
        v0 = syn.normal_f32(94, syn.Tag.QKV, it, (B, HV, V), 1.0).astype(np.float64)
        g = np.full((B, HV), np.float32(-0.1), dtype=np.float64)
        beta = np.full((B, HV), 0.5)
        o0, _ = oracle.delta_step(q0, k0, v0, g, beta, S[0], scale=K ** -0.5, idx=idx_np)
        v1 = results[(True, True)][0][2 * it].reshape(B, HV, V).astype(np.float64)   # the GPU's layer-0 output
        o1, _ = oracle.delta_step(q0, k0, v1, g, beta, S[1], scale=K ** -0.5, idx=idx_np)
        assert rel_err(results[(True, True)][0][2 * it].reshape(B, HV, V), o0) <= TOL_F32
        assert rel_err(results[(True, True)][0][2 * it + 1].reshape(B, HV, V), o1) <= TOL_F32
    for l in range(2):
        assert rel_err(results[(True, True)][1][l], S[l]) <= TOL_F32


@pytest.mark.parametrize("B,H,HV,dtype,out_dtype,pad_rows,bad_rows,steps", [
    (3, 16, 32, "bf16", "bf16", (1,), (), 3),      # 96 tiles: eight CTAs per tile
    (16, 16, 32, "bf16", "bf16", (2,), (5,), 2),   # a pad row and a bad slot index
    (75, 16, 32, "bf16", "bf16", (), (), 1),       # 2400 tiles: two CTAs per tile
    (8, 4, 16, "f32", "f32", (), (), 4),           # fp32 inputs, four value heads per q/k head
    (1, 16, 32, "bf16", "f32", (), (), 2),         # 32 tiles: eight CTAs per tile
])
def test_chained_calls_against_the_oracle(B, H, HV, dtype, out_dtype, pad_rows, bad_rows, steps):
    """gdn_decode_step_indexed_chained on packed bf16 (and fp32) inputs with raw gates: sequential
    steps against the oracle, with pad rows and a bad index (flagged, its output zero), across the
    row splits the chained instance runs at these batch sizes."""
    wo, ws, flags = _run(B, H, HV, 128, 128, dtype, out_dtype, 960 + B, steps=steps, pad_rows=pad_rows,
                         bad_rows=bad_rows, chained=True)
    assert wo <= _tol(out_dtype)
    assert ws <= TOL_F32
    assert flags == (gdn.GDN_DEVERR_BAD_INDEX if bad_rows else 0)
