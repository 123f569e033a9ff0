"""The delta rule's invariants and the method's edge cases, run through the CUDA kernels.

The invariants are the ones the delta rule itself fixes ("Optimization Log: Qwen3.5-27B Dense on
B200", Kernel 4 Math block: decay, u = S k, delta = beta (v - u), S += delta k^T, o = S q):
  (i)   g = 0, beta = 0 leaves S bit-identical and gives o = S q_hat;
  (ii)  beta = 1, g = 0 and a unit key recall v exactly: S' k_hat = v;
  (iii) g -> -inf (g = -1e30 given directly) forgets S: S' = beta v k_hat^T;
and the edge cases: rows whose k or q is all zero (the epsilon of the L2 norm) and saturating gate
inputs (a + dt_bias = +-40, b = +-40: softplus and sigmoid at their overflow ends). Every case is
also compared element by element with the fp64 oracle on the same inputs (1e-5 for fp32 outputs
and the fp32 state, 2e-2 for bf16 outputs and a bf16 state), on these kernels:
  - gdn_decode_step_indexed with 8 rows per thread (two CTAs per tile, K = 128), 16 rows per
    thread (one CTA per tile, K = 64), 2 rows per thread (one request row), and the bf16-state
    kernel;
  - gdn_decode_buffered on the pipelined kernel, L = 8, one whole cycle (7 replay steps and the
    flush), fp32 ring so that the checkpoint is held to 1e-5;
  - gdn_decode_fused on the pipelined kernel (head_dim 128, 384 (token, head) tiles), where g and
    beta come from the gate inputs (A_log = -inf gives g = 0, raw_beta = -inf / +inf gives
    beta = 0 / 1, A_log = 80 gives exp(g) = 0) and k, q come out of the conv update.
NaN and Inf inputs: a NaN in one state tile, in one q head or an Inf in one k head must stay in
the tiles that read it, with the oracle's NaN pattern there and the oracle's values everywhere
else."""
import math

import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import bits_to_torch_bf16, host_state

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16 = 1e-5, 2e-2


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _normal(seed, tag, step, shape, std=1.0):
    return syn.normal_f32(seed, tag, step, shape, std).astype(np.float64)


def _gates(case, B, HV, seed, step):
    """Direct gates (g, beta) [B, HV] for a case, or None for the raw-gate cases."""
    if case == "keep":                   # (i)
        return np.zeros((B, HV)), np.zeros((B, HV))
    if case == "recall":                 # (ii)
        return np.zeros((B, HV)), np.ones((B, HV))
    if case == "forget":                 # (iii)
        beta = 1.0 / (1.0 + np.exp(-_normal(seed, syn.Tag.B, step, (B, HV))))
        return np.full((B, HV), -1e30), beta.astype(np.float32).astype(np.float64)
    return None


def _qkv(case, B, H, HV, K, V, seed, step):
    q = _normal(seed, syn.Tag.QKV, step, (B, H, K))
    k = _normal(seed, syn.Tag.QKV, step + 1000, (B, H, K))
    v = _normal(seed, syn.Tag.QKV, step + 2000, (B, HV, V))
    if case == "recall":                 # unit keys, exact in fp32 after the cast
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    if case == "zero_k":                 # every other row: k all zero
        k[::2] = 0.0
    if case == "zero_q":
        q[1::2] = 0.0
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    return f32(q), f32(k), f32(v)


def _raw_gates(B, HV, seed, step):
    """a + dt_bias and b at the saturating ends +-40, in every combination across heads."""
    a = np.where((np.arange(HV) % 2) == 0, 40.0, -40.0)[None].repeat(B, 0)
    b = np.where((np.arange(HV) // 2) % 2 == 0, 40.0, -40.0)[None].repeat(B, 0)
    A_log = syn.normal_f32(seed, syn.Tag.A_LOG, 0, (HV,), 0.3).astype(np.float64)
    return a, b, A_log, np.zeros(HV)


CASES = ["keep", "recall", "forget", "zero_k", "zero_q", "saturating"]


def _step_config(path):
    # (B, H, HV, K, V, state dtype): the kernel the library picks for each on 152 SMs
    return {"rows8": (16, 16, 32, 128, 128, "f32"),      # 512 tiles -> two CTAs per tile
            "rows16": (32, 16, 32, 64, 64, "f32"),       # K = 64, 1024 tiles -> one CTA per tile
            "rows2": (1, 16, 32, 128, 128, "f32"),       # 32 tiles -> eight CTAs per tile
            "bf16state": (32, 16, 32, 128, 128, "bf16")}[path]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("path", ["rows8", "rows16", "rows2", "bf16state"])
def test_step_invariants_and_edge_cases(path, case):
    B, H, HV, K, V, sdt = _step_config(path)
    seed = 300 + CASES.index(case)
    num_slots = B + 3
    S64 = host_state(num_slots, HV, V, K, seed)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    if sdt == "bf16":
        state = state.to(torch.bfloat16)
        S64 = state.float().cpu().numpy().astype(np.float64)
    S0 = state.clone()
    idx_np = syn.permutation(seed, num_slots)[:B].copy()
    idx = torch.from_numpy(idx_np).cuda()
    q, k, v = _qkv(case, B, H, HV, K, V, seed, 0)
    l2 = case != "recall"                # (ii) with the unit key used as it is
    t = lambda x: torch.from_numpy(x.astype(np.float32)).cuda()
    qt, kt, vt = t(q.reshape(B, H * K)), t(k.reshape(B, H * K)), t(v.reshape(B, HV * V))
    out = torch.full((B, 1, HV, V), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gates = _gates(case, B, HV, seed, 0)
    if gates is None and case == "saturating":
        a, b, A_log, dt_bias = _raw_gates(B, HV, seed, 0)
        gdn.gdn_decode_step_indexed(qt, kt, vt, state, out, idx, H=H, a=t(a), b=t(b), A_log=t(A_log),
                                    dt_bias=t(dt_bias), err_flags=err)
        g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
    else:
        if gates is None:                # zero_k / zero_q: ordinary gates
            g = -np.exp(0.1) * np.log1p(np.exp(_normal(seed, syn.Tag.A, 0, (B, HV), 0.5)))
            beta = 1.0 / (1.0 + np.exp(-_normal(seed, syn.Tag.B, 0, (B, HV), 0.5)))
            g, beta = (x.astype(np.float32).astype(np.float64) for x in (g, beta))
        else:
            g, beta = gates
        gdn.gdn_decode_step_indexed(qt, kt, vt, state, out, idx, H=H, g=t(g), beta=t(beta),
                                    use_qk_l2norm=l2, err_flags=err)
    S_before = S64.copy()
    o_ref, bad = oracle.delta_step(q, k, v, g, beta, S64, scale=K ** -0.5, use_qk_l2norm=l2,
                                   idx=idx_np, state_bf16=(sdt == "bf16"))
    torch.cuda.synchronize()
    assert bad == 0 and int(err.item()) == 0
    got_o = out.cpu().numpy().reshape(B, HV, V)
    got_S = state.float().cpu().numpy().astype(np.float64)
    tol_s = TOL_BF16 if sdt == "bf16" else TOL_F32
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_S))
    assert rel_err(got_o, o_ref) <= TOL_F32         # fp32 out, from the update before storage
    assert rel_err(got_S, S64) <= tol_s
    G = HV // H
    Sg = got_S[idx_np]                                            # [B, HV, V, K], row order
    if case == "keep":
        assert torch.equal(state, S0)                             # bit-identical
    if case == "recall" and sdt == "f32":
        kh = np.repeat(k, G, axis=1)                              # [B, HV, K], unit keys
        recalled = np.einsum("bhvk,bhk->bhv", Sg, kh)
        assert rel_err(recalled, v) <= TOL_F32
    if case == "forget" and sdt == "f32":
        kh = np.repeat(k / np.sqrt(np.sum(k * k, -1, keepdims=True) + 1e-6), G, axis=1)
        want = beta[:, :, None, None] * v[:, :, :, None] * kh[:, :, None, :]
        assert rel_err(Sg, want) <= TOL_F32
    if case == "zero_q":
        assert np.all(got_o[1::2] == 0.0)
    if case == "zero_k":                                          # k_hat = 0: S' = exp(g) S
        want = np.exp(g[::2])[:, :, None, None] * S_before[idx_np[::2]]
        assert rel_err(Sg[::2], want) <= tol_s


# ------------------------------------------------------------------------------------------------
# buffered decode (pipelined kernel, L = 8, fp32 ring): one whole cycle
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", CASES)
def test_buffered_pipe_invariants_and_edge_cases(case):
    B, H, HV, K, V, L = 8, 16, 32, 128, 128, 8
    seed = 400 + CASES.index(case)
    S64 = host_state(B, HV, V, K, seed)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    S0 = state.clone()
    d_cache = torch.zeros((B, HV, L, V), device="cuda")
    k_cache = torch.zeros((B, H, L, K), device="cuda")
    g_cache = torch.zeros((B, HV, L), device="cuda")
    d64, k64, g64 = np.zeros((B, HV, L, V)), np.zeros((B, H, L, K)), np.zeros((B, HV, L))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    l2 = case != "recall"
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    last = None
    for p in range(L):
        wp = np.full(B, p, np.int32)
        q, k, v = _qkv(case, B, H, HV, K, V, seed, p)
        out = torch.full((B, 1, HV, V), float("nan"), device="cuda")
        gates = _gates(case, B, HV, seed, p)
        qt, kt, vt = t(q.reshape(B, H * K)), t(k.reshape(B, H * K)), t(v.reshape(B, HV * V))
        if case == "saturating":
            a, b, A_log, dt_bias = _raw_gates(B, HV, seed, p)
            gdn.gdn_decode_buffered(qt, kt, vt, state, out, d_cache, k_cache, g_cache, torch.from_numpy(wp).cuda(),
                                    H=H, a=t(a), b=t(b), A_log=t(A_log), dt_bias=t(dt_bias),
                                    err_flags=err, kernel="pipe")
            g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
        else:
            if gates is None:
                g = -np.exp(0.1) * np.log1p(np.exp(_normal(seed, syn.Tag.A, p, (B, HV), 0.5)))
                beta = 1.0 / (1.0 + np.exp(-_normal(seed, syn.Tag.B, p, (B, HV), 0.5)))
                g, beta = (x.astype(np.float32).astype(np.float64) for x in (g, beta))
            else:
                g, beta = gates
            gdn.gdn_decode_buffered(qt, kt, vt, state, out, d_cache, k_cache, g_cache,
                                    torch.from_numpy(wp).cuda(), H=H, g=t(g), beta=t(beta),
                                    use_qk_l2norm=l2, err_flags=err, kernel="pipe")
        o_ref, bad = oracle.gdn_buffered(q, k, v, g, beta, S64, d64, k64, g64, wp, L=L,
                                         ring_bf16=False, scale=K ** -0.5, use_qk_l2norm=l2)
        assert bad == 0
        got_o = out.cpu().numpy().reshape(B, HV, V)
        assert np.all(np.isfinite(got_o))
        assert rel_err(got_o, o_ref) <= TOL_F32, p
        if case == "zero_q":
            assert np.all(got_o[1::2] == 0.0)
        last = (k, v, beta)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_S = state.cpu().numpy().astype(np.float64)
    assert rel_err(got_S, S64) <= TOL_F32
    assert rel_err(d_cache.cpu().numpy(), d64) <= TOL_F32
    assert rel_err(k_cache.cpu().numpy(), k64) <= TOL_F32
    k, v, beta = last
    G = HV // H
    if case == "keep":                   # nothing learned in a whole cycle: the flush writes S back
        assert torch.equal(state, S0)
        assert np.all(d_cache.cpu().numpy()[:, :, :L - 1] == 0.0)
    if case == "recall":                 # the flushed checkpoint recalls the last step's value
        recalled = np.einsum("bhvk,bhk->bhv", got_S, np.repeat(k, G, axis=1))
        assert rel_err(recalled, v) <= TOL_F32
    if case == "forget":                 # only the last step survives the flush
        kh = np.repeat(k / np.sqrt(np.sum(k * k, -1, keepdims=True) + 1e-6), G, axis=1)
        want = beta[:, :, None, None] * v[:, :, :, None] * kh[:, :, None, :]
        assert rel_err(got_S, want) <= TOL_F32


# ------------------------------------------------------------------------------------------------
# fused decode (pipelined kernel): gates from the gate inputs, q/k/v from the conv update
# ------------------------------------------------------------------------------------------------
FUSED_CASES = ["keep", "recall", "forget", "zero_k", "zero_q", "saturating"]


@pytest.mark.parametrize("case", FUSED_CASES)
def test_fused_pipe_invariants_and_edge_cases(case):
    T, heads, D = 4, 96, 128
    dim = heads * D
    seed = 500 + FUSED_CASES.index(case)
    num_slots = T + 8
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    f64 = lambda bits: syn.bf16_bits_to_f32(bits).astype(np.float64)
    gate_kind = "gdn"
    raw_g = f64(syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.RAW_G, 0, (T, heads), 1.0)))
    raw_beta = f64(ins["raw_beta"])
    A_log = ins["A_log"].astype(np.float64).copy()
    dt_bias = syn.normal_f32(seed, syn.Tag.DT_BIAS, 0, (heads,), 1.0).astype(np.float64)
    conv_w = ins["conv_w"].astype(np.float64).copy()
    if case in ("keep", "recall"):
        A_log[:] = -np.inf               # g = -0: exp(g) = 1
    if case == "keep":
        raw_beta[:] = -np.inf            # beta = 0
    if case == "recall":
        raw_beta[:] = np.inf             # beta = 1
    if case == "forget":
        A_log[:] = 80.0                  # exp(g) = exp(-exp(80) softplus(.)) = 0
    if case == "zero_k":
        conv_w[dim:2 * dim] = 0.0        # k = silu(0) = 0 for every head
    if case == "zero_q":
        conv_w[:dim] = 0.0
    if case == "saturating":
        raw_g = np.where((np.arange(heads) % 2) == 0, 40.0, -40.0)[None].repeat(T, 0)
        raw_beta = np.where((np.arange(heads) // 2) % 2 == 0, 40.0, -40.0)[None].repeat(T, 0)
        dt_bias[:] = 0.0
    bf = lambda x: bits_to_torch_bf16(syn.f32_to_bf16_bits(np.asarray(x, np.float32)))
    state = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device="cuda")
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
    S0 = state.clone()
    S64 = state.cpu().numpy().astype(np.float64)
    conv_state = bits_to_torch_bf16(ins["conv_state"]).clone()
    cs64 = f64(ins["conv_state"]).reshape(num_slots, 3 * dim, 3).copy()
    idx_np = np.arange(1, T + 1, dtype=np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    x_bits = syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.X, 0, (T, 3 * dim), 1.0))
    gate_bits = syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.OUT_GATE, 0, (T, heads, D), 1.0))
    out = torch.full((T, heads, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tf = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    gdn.gdn_decode_fused(bits_to_torch_bf16(x_bits), tf(conv_w), conv_state, bf(raw_g), bf(raw_beta),
                         tf(A_log), tf(dt_bias), state, idx, bits_to_torch_bf16(gate_bits),
                         torch.from_numpy(ins["norm_w"]).cuda(), out, pad_slot_id=0,
                         gate_kind=gate_kind, err_flags=err, kernel="pipe")
    # the conv output the step sees (the oracle's, fp64), before the oracle updates conv state
    y_conv, _ = oracle.conv_update(f64(x_bits), conv_w, cs64.copy(), idx=idx_np, pad_slot=0)
    o_ref, bad = oracle.fused_kda(f64(x_bits), conv_w, cs64, raw_g, raw_beta, A_log, dt_bias, S64,
                                  f64(gate_bits), ins["norm_w"], idx=idx_np, pad_slot=0,
                                  gate_kind=gate_kind)
    torch.cuda.synchronize()
    assert bad == 0 and int(err.item()) == 0
    got_o = out.float().cpu().numpy()
    got_S = state.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_S))
    assert rel_err(got_o, o_ref) <= TOL_BF16
    assert rel_err(got_S[idx_np], S64[idx_np]) <= TOL_F32
    np.testing.assert_array_equal(conv_state.float().cpu().numpy()[idx_np], cs64[idx_np])
    k = y_conv[:, dim:2 * dim].reshape(T, heads, D)
    v = y_conv[:, 2 * dim:].reshape(T, heads, D)
    kh = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + 1e-6)
    Sg = got_S[idx_np]
    if case == "keep":
        assert torch.equal(state, S0)
    if case == "recall":
        assert rel_err(np.einsum("thvk,thk->thv", Sg, kh), v) <= TOL_F32
    if case == "forget":
        beta = 1.0 / (1.0 + np.exp(-raw_beta))
        want = beta[:, :, None, None] * v[:, :, :, None] * kh[:, :, None, :]
        assert rel_err(Sg, want) <= TOL_F32
    if case == "zero_q":
        assert np.all(got_o == 0.0)


# ------------------------------------------------------------------------------------------------
# NaN and Inf inputs stay in the tiles that read them
# ------------------------------------------------------------------------------------------------
def _same_nan_pattern(got, ref, tol):
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), (int(gn.sum()), int(rn.sum()))
    fin = ~rn
    assert rel_err(got[fin], ref[fin]) <= tol


@pytest.mark.parametrize("where", ["state", "q", "k_inf"])
@pytest.mark.parametrize("path", ["rows8", "bf16state"])
def test_step_nan_and_inf_stay_in_their_tiles(path, where):
    B, H, HV, K, V, sdt = _step_config(path)
    G = HV // H
    seed = 600
    S64 = host_state(B, HV, V, K, seed)
    b0, h0 = 3, 5                                  # the row and q/k head that get the bad value
    if where == "state":
        S64[b0, h0 * G, 17, 33] = np.nan
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    if sdt == "bf16":
        state = state.to(torch.bfloat16)
        S64 = state.float().cpu().numpy().astype(np.float64)
    idx_np = np.arange(B, dtype=np.int32)
    q, k, v = _qkv("plain", B, H, HV, K, V, seed, 0)
    if where == "q":
        q[b0, h0, 7] = np.nan
    if where == "k_inf":
        k[b0, h0, 9] = np.inf
    g = -np.exp(0.1) * np.log1p(np.exp(_normal(seed, syn.Tag.A, 0, (B, HV), 0.5)))
    beta = 1.0 / (1.0 + np.exp(-_normal(seed, syn.Tag.B, 0, (B, HV), 0.5)))
    g, beta = (x.astype(np.float32).astype(np.float64) for x in (g, beta))
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    out = torch.full((B, 1, HV, V), 7.0, device="cuda")
    gdn.gdn_decode_step_indexed(t(q.reshape(B, -1)), t(k.reshape(B, -1)), t(v.reshape(B, -1)), state,
                                out, torch.from_numpy(idx_np).cuda(), H=H, g=t(g), beta=t(beta))
    o_ref, _ = oracle.delta_step(q, k, v, g, beta, S64, scale=K ** -0.5, idx=idx_np,
                                 state_bf16=(sdt == "bf16"))
    torch.cuda.synchronize()
    got_o = out.cpu().numpy().reshape(B, HV, V)
    got_S = state.float().cpu().numpy().astype(np.float64)
    tol = TOL_BF16 if sdt == "bf16" else TOL_F32
    _same_nan_pattern(got_o, o_ref, tol)
    _same_nan_pattern(got_S, S64, tol)
    bad_tiles = np.zeros((B, HV), bool)
    bad_tiles[b0, h0 * G:(h0 + 1) * G] = True
    assert np.isnan(got_o).any()
    assert not np.isnan(got_o[~bad_tiles]).any()
    assert not np.isnan(got_S[~bad_tiles]).any()


def test_buffered_pipe_nan_in_a_checkpoint_stays_in_its_tile():
    B, H, HV, K, V, L = 8, 16, 32, 128, 128, 8
    seed = 601
    S64 = host_state(B, HV, V, K, seed)
    S64[2, 11, 40, 3] = np.nan
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    d_cache = torch.zeros((B, HV, L, V), device="cuda")
    k_cache = torch.zeros((B, H, L, K), device="cuda")
    g_cache = torch.zeros((B, HV, L), device="cuda")
    d64, k64, g64 = np.zeros((B, HV, L, V)), np.zeros((B, H, L, K)), np.zeros((B, HV, L))
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    for p in range(L):
        wp = np.full(B, p, np.int32)
        q, k, v = _qkv("plain", B, H, HV, K, V, seed, p)
        g = -np.exp(0.1) * np.log1p(np.exp(_normal(seed, syn.Tag.A, p, (B, HV), 0.5)))
        beta = 1.0 / (1.0 + np.exp(-_normal(seed, syn.Tag.B, p, (B, HV), 0.5)))
        g, beta = (x.astype(np.float32).astype(np.float64) for x in (g, beta))
        out = torch.full((B, 1, HV, V), 7.0, device="cuda")
        gdn.gdn_decode_buffered(t(q.reshape(B, -1)), t(k.reshape(B, -1)), t(v.reshape(B, -1)), state,
                                out, d_cache, k_cache, g_cache, torch.from_numpy(wp).cuda(), H=H,
                                g=t(g), beta=t(beta), kernel="pipe")
        o_ref, _ = oracle.gdn_buffered(q, k, v, g, beta, S64, d64, k64, g64, wp, L=L, ring_bf16=False,
                                       scale=K ** -0.5)
        got_o = out.cpu().numpy().reshape(B, HV, V)
        _same_nan_pattern(got_o, o_ref, TOL_F32)
        assert not np.isnan(np.delete(got_o.reshape(B * HV, V), 2 * HV + 11, axis=0)).any()
    torch.cuda.synchronize()
    got_S = state.cpu().numpy().astype(np.float64)
    _same_nan_pattern(got_S, S64, TOL_F32)
    _same_nan_pattern(d_cache.cpu().numpy(), d64, TOL_F32)
    assert not np.isnan(np.delete(got_S.reshape(B * HV, V, K), 2 * HV + 11, axis=0)).any()


def test_inputs_plain_case_is_defined():
    # "plain" draws ordinary inputs (no case applies): used by the NaN tests above
    q, k, v = _qkv("plain", 2, 2, 4, 16, 16, 1, 0)
    assert np.all(np.isfinite(q)) and math.isfinite(float(np.sum(k * k)))
