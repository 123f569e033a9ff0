"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

The sources print no worked numeric example of the gated delta-rule step, so the oracle is pinned
by: the invariants the delta rule fixes; the closed matrix form of one step; hand-derived exact
results on tiny inputs; special cases that reduce to library routines (softplus, sigmoid, bf16
rounding, convolution, RMSNorm); structural identities (GQA duplication, slot permutation, the
buffered replay against looped single steps, the low-rank form of the replay); and contraction
over many steps. Each check_* function raises AssertionError on a mismatch; the tests below call
them, and tests/test_oracle_mutants.py runs them against deliberately broken builds of the oracle
to show that each plausible mistake fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
from conftest import rel_err

TINY = dict(B=2, H=2, HV=4, K=16, V=16)


# --------------------------------------------------------------------------------------------
# input helpers (tiny GDN decode: fp32 q/k/v ~ N(0,1), a,b ~ N(0,0.25), A_log ~ N(0,0.09),
# dt_bias ~ N(0,0.01), state ~ N(0,1))
# --------------------------------------------------------------------------------------------
def tiny_step_inputs(seed=0, step=0, B=2, H=2, HV=4, K=16, V=16):
    d = syn.packed_inputs(B, H, HV, K, V, "f32", seed, step)
    q, k, v = oracle.split_packed(d["mixed_qkv"], H, HV, K, V)
    g, beta = oracle.gdn_gates(d["a"], d["b"], d["A_log"], d["dt_bias"])
    return q, k, v, g, beta


def tiny_state(seed=0, num_slots=2, HV=4, V=16, K=16):
    return syn.normal_f32(seed, syn.Tag.STATE, 0, (num_slots, HV, V, K), 1.0).astype(np.float64)


def l2n(x, eps=oracle.L2_EPS):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


# --------------------------------------------------------------------------------------------
# generator and rounding
# --------------------------------------------------------------------------------------------
def check_philox_known_answers():
    # Published Philox4x32-10 known-answer vectors (Random123 distribution of Salmon et al.).
    kat = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in kat:
        got = syn.philox4x32_10(*ctr, *key)
        assert tuple(int(x) for x in got) == want


def test_philox_known_answers():
    check_philox_known_answers()


def test_normal_generator_moments_and_bounds():
    x = syn.normal_f32(7, syn.Tag.QKV, 3, (1 << 20,), 0.5).astype(np.float64)
    assert abs(x.mean()) < 2e-3
    assert abs(x.std() - 0.5) < 2e-3
    assert np.max(np.abs(x)) <= 0.5 * 2 * math.sqrt(3) + 1e-6
    # random access: any slice regenerates the same values
    idx = np.array([5, 99, 1 << 19], dtype=np.uint64)
    np.testing.assert_array_equal(syn.normal_at(7, syn.Tag.QKV, 3, idx, 0.5), x[idx.astype(int)])


def check_bf16_rounding():
    rng = np.random.default_rng(1)
    y = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(y)), ref)
    np.testing.assert_array_equal(oracle.round_bf16(y.astype(np.float64)), ref)
    # ties go to the even neighbour (8 significant bits)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), (1.5 + 2 ** -8) * 2 ** -9,
                     (1.5 + 3 * 2 ** -8) * 2 ** 9])
    want = np.array([1.0, 1 + 2 ** -6, -1.0, 1.5 * 2 ** -9, (1.5 + 2 ** -6) * 2 ** 9])
    np.testing.assert_array_equal(oracle.round_bf16(ties), want)


def test_bf16_rounding():
    check_bf16_rounding()


# --------------------------------------------------------------------------------------------
# gates
# --------------------------------------------------------------------------------------------
def check_gdn_gates():
    B, HV = 3, 5
    rng = np.random.default_rng(2)
    a = rng.normal(0, 2, (B, HV)); b = rng.normal(0, 2, (B, HV))
    A_log = rng.normal(0, 1, HV); dt_bias = rng.normal(0, 1, HV)
    g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
    sp = torch.nn.functional.softplus(torch.from_numpy(a + dt_bias)).numpy()
    assert rel_err(g, -np.exp(A_log) * sp) < 1e-14
    assert rel_err(beta, torch.sigmoid(torch.from_numpy(b)).numpy()) < 1e-15
    # special values
    z = np.zeros((1, 2))
    g0, b0 = oracle.gdn_gates(z, z, np.array([-np.inf, 0.3]), np.zeros(2))
    assert g0[0, 0] == 0.0 and b0[0, 0] == 0.5
    assert abs(g0[0, 1] - (-math.exp(0.3) * math.log(2.0))) < 1e-15
    _, bb = oracle.gdn_gates(z, np.array([[800.0, -800.0]]), np.zeros(2), np.zeros(2))
    assert bb[0, 0] == 1.0 and bb[0, 1] == 0.0


def test_gdn_gates():
    check_gdn_gates()


def check_kda_gate_reading():
    """The KDA microbenchmark page ("Microbenchmark for the fused Kimi-K3 KDA decode kernel on
    ROCm", `Inputs`) names raw_g, A_log [heads], dt_bias [heads * D] and lower_bound = -5 but
    prints no formula; the oracle implements two readings, each pinned here to its own formula:
      form 0: g[t,h,d] = max(lb, -exp(A_log[h]) * softplus(raw_g[t,h,d] + dt_bias[h*D + d]))
      form 1: g[t,h,d] = lb * sigmoid(exp(A_log[h]) * (raw_g[t,h,d] + dt_bias[h*D + d]))
    Pins: both forms lie in [lb, 0] and do not increase with raw_g; form 1 at x = 0 is lb/2;
    form 0 saturates at lb; form 0 with the bound inactive equals the GDN gate; closed values
    where exp(A_log[h]) differs between heads and dt_bias between channels (below)."""
    T, heads, D = 2, 3, 8
    rng = np.random.default_rng(3)
    raw = rng.normal(0, 2, (T, heads, D)); A_log = rng.normal(0, 1, heads)
    dtb = rng.normal(0, 1, heads * D)
    for form in (0, 1):
        g = oracle.kda_gate(raw, A_log, dtb, -5.0, form)
        assert np.all(g >= -5.0) and np.all(g <= 0.0)
        # monotone non-increasing in raw_g
        g2 = oracle.kda_gate(raw + 0.25, A_log, dtb, -5.0, form)
        assert np.all(g2 <= g + 1e-15)
    # form 1 at raw + dt_bias = 0 is lower_bound / 2; form 0 saturates at the bound
    zero = np.zeros((1, 1, 2))
    assert np.allclose(oracle.kda_gate(zero, np.array([0.7]), np.zeros(2), -5.0, 1), -2.5, atol=0)
    big = np.full((1, 1, 2), 50.0)
    assert np.all(oracle.kda_gate(big, np.zeros(1), np.zeros(2), -5.0, 0) == -5.0)
    # form 0 where the bound is inactive is the GDN gate with a per-channel bias
    small = rng.normal(-3, 0.1, (1, 1, 4))
    gk = oracle.kda_gate(small, np.array([0.1]), np.zeros(4), -5.0, 0)
    gg, _ = oracle.gdn_gates(small.reshape(4, 1), np.zeros((4, 1)), np.array([0.1]), np.zeros(1))
    assert rel_err(gk.reshape(4), gg.reshape(4)) < 1e-15
    # Closed values with exp(A_log[h]) = 2 and 4 on two heads, so the scale on x matters and a
    # head-0 lookup is visible. Form 1: x = ln(3)/2 split between raw_g and dt_bias gives
    # sigmoid(2 x) = sigmoid(ln 3) = 3/4 and sigmoid(4 x) = sigmoid(2 ln 3) = 9/10.
    A2 = np.array([math.log(2.0), math.log(4.0)])
    x1 = math.log(3.0) / 2
    raw1 = np.full((1, 2, 2), x1 / 4)
    dtb1 = np.full(4, 3 * x1 / 4)
    g1 = oracle.kda_gate(raw1, A2, dtb1, -5.0, 1)
    assert np.max(np.abs(g1[0, 0] - (-5.0 * 0.75))) < 1e-14
    assert np.max(np.abs(g1[0, 1] - (-5.0 * 0.9))) < 1e-14
    # Form 0: dt_bias[h*D + d] = ln(e^c - 1) with a different c per channel makes
    # softplus(0 + dt_bias) = c, so g = -exp(A_log[h]) * c (all above the bound).
    c = 0.05 * np.arange(1, 5, dtype=np.float64)
    dtb0 = np.log(np.expm1(c))
    g0 = oracle.kda_gate(np.zeros((1, 2, 2)), A2, dtb0, -5.0, 0)
    want0 = -np.array([[2.0 * c[0], 2.0 * c[1]], [4.0 * c[2], 4.0 * c[3]]])
    assert np.max(np.abs(g0[0] - want0)) < 1e-14


def test_kda_gate_reading():
    check_kda_gate_reading()


# --------------------------------------------------------------------------------------------
# the step
# --------------------------------------------------------------------------------------------
def check_hand_worked_step():
    """K = V = 2, every quantity dyadic; derived by hand from the Math block of 'Kernel 4: Fused
    DeltaNet Recurrent': decay, u = S k, delta, rank-1 update, o from the updated state.
      S = [[1,2],[3,4]], k = (1,0), q = (1,1), v = (5,6), beta = 1/2, exp(g) = 1/2, no L2 norm,
      scale 1:  S <- [[.5,1],[1.5,2]];  u = (.5,1.5);  delta = (2.25,2.25);
      S' = [[2.75,1],[3.75,2]];  o = S' q = (3.75,5.75)."""
    S = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    q = np.array([[[1.0, 1.0]]]); k = np.array([[[1.0, 0.0]]]); v = np.array([[[5.0, 6.0]]])
    out, bad = oracle.delta_step(q, k, v, np.array([[-math.log(2.0)]]), np.array([[0.5]]), S,
                                 scale=1.0, use_qk_l2norm=False)
    assert bad == 0
    assert np.max(np.abs(S[0, 0] - np.array([[2.75, 1.0], [3.75, 2.0]]))) < 1e-15
    assert np.max(np.abs(out[0, 0] - np.array([3.75, 5.75]))) < 1e-15


def test_hand_worked_step():
    check_hand_worked_step()


def check_invariant_no_decay_no_write():
    """g = 0 and beta = 0 leave S unchanged, and o = S q_hat."""
    q, k, v, _, _ = tiny_step_inputs(seed=11)
    S0 = tiny_state(seed=11)
    S = S0.copy()
    B, HV = 2, 4
    out, _ = oracle.delta_step(q, k, v, np.zeros((B, HV)), np.zeros((B, HV)), S, scale=0.25)
    np.testing.assert_array_equal(S, S0)
    qh = 0.25 * l2n(q)
    for b in range(B):
        for hv in range(HV):
            assert rel_err(out[b, hv], S0[b, hv] @ qh[b, hv // 2]) < 1e-13


def test_invariant_no_decay_no_write():
    check_invariant_no_decay_no_write()


def check_invariant_exact_recall():
    """beta = 1, g = 0, unit k: after the update S k = v exactly (the delta rule's recall)."""
    q, k, v, _, _ = tiny_step_inputs(seed=12)
    ku = k / np.linalg.norm(k, axis=-1, keepdims=True)
    S = tiny_state(seed=12)
    B, HV = 2, 4
    oracle.delta_step(q, ku, v, np.zeros((B, HV)), np.ones((B, HV)), S, scale=0.25,
                      use_qk_l2norm=False)
    for b in range(B):
        for hv in range(HV):
            assert rel_err(S[b, hv] @ ku[b, hv // 2], v[b, hv]) < 1e-13
    # with the in-kernel L2 norm the recall is off only by the norm's epsilon
    S = tiny_state(seed=12)
    oracle.delta_step(q, k, v, np.zeros((B, HV)), np.ones((B, HV)), S, scale=0.25)
    kh = l2n(k)
    for b in range(B):
        for hv in range(HV):
            assert rel_err(S[b, hv] @ kh[b, hv // 2], v[b, hv]) < 1e-6


def test_invariant_exact_recall():
    check_invariant_exact_recall()


def check_invariant_full_decay():
    """g -> -inf: the old state is forgotten and S' = delta k_hat^T = beta v k_hat^T."""
    q, k, v, _, beta = tiny_step_inputs(seed=13)
    S = tiny_state(seed=13)
    B, HV = 2, 4
    out, _ = oracle.delta_step(q, k, v, np.full((B, HV), -np.inf), beta, S, scale=0.25)
    kh = l2n(k); qh = 0.25 * l2n(q)
    for b in range(B):
        for hv in range(HV):
            want = beta[b, hv] * np.outer(v[b, hv], kh[b, hv // 2])
            assert rel_err(S[b, hv], want) < 1e-14
            assert rel_err(out[b, hv], want @ qh[b, hv // 2]) < 1e-13


def test_invariant_full_decay():
    check_invariant_full_decay()


@pytest.mark.parametrize("shape", [dict(B=2, H=2, HV=4, K=16, V=16),
                                   dict(B=3, H=1, HV=3, K=8, V=12),
                                   dict(B=2, H=3, HV=3, K=32, V=8)])
def test_closed_matrix_form(shape):
    check_closed_matrix_form(**shape)


def check_closed_matrix_form(B=2, H=2, HV=4, K=16, V=16):
    """S' = exp(g) S (I - beta k k^T) + beta v k^T, o = S' q (scalar decay), and with a per-key
    decay D = diag(exp(g_k)): S' = S D (I - beta k k^T) + beta v k^T."""
    q, k, v, g, beta = tiny_step_inputs(seed=14, B=B, H=H, HV=HV, K=K, V=V)
    G = HV // H
    kh = l2n(k); qh = K ** -0.5 * l2n(q)
    S0 = tiny_state(seed=14, num_slots=B, HV=HV, V=V, K=K)
    S = S0.copy()
    out, _ = oracle.delta_step(q, k, v, g, beta, S, scale=K ** -0.5)
    gk = syn.normal_f32(15, syn.Tag.G_DIRECT, 0, (B, HV, K), 0.5).astype(np.float64) - 0.5
    S2 = S0.copy()
    out2, _ = oracle.delta_step(q, k, v, gk, beta, S2, scale=K ** -0.5)
    I = np.eye(K)
    for b in range(B):
        for hv in range(HV):
            kk, qq = kh[b, hv // G], qh[b, hv // G]
            P = I - beta[b, hv] * np.outer(kk, kk)
            want = math.exp(g[b, hv]) * S0[b, hv] @ P + beta[b, hv] * np.outer(v[b, hv], kk)
            assert rel_err(S[b, hv], want) < 1e-13
            assert rel_err(out[b, hv], want @ qq) < 1e-13
            want2 = S0[b, hv] @ np.diag(np.exp(gk[b, hv])) @ P + beta[b, hv] * np.outer(v[b, hv], kk)
            assert rel_err(S2[b, hv], want2) < 1e-13
            assert rel_err(out2[b, hv], want2 @ qq) < 1e-13


def check_bf16_state_storage():
    """bf16 state storage: the step runs on the stored values, out comes from the updated state
    before storage, and the stored state is the update rounded to bf16 -- checked against the
    closed matrix form (numpy) rounded with torch's own bf16 conversion."""
    B, H, HV, K, V = 2, 2, 4, 16, 16
    q, k, v, g, beta = tiny_step_inputs(seed=19, B=B, H=H, HV=HV, K=K, V=V)
    S0 = torch.from_numpy(tiny_state(seed=19)).to(torch.bfloat16).to(torch.float64).numpy()
    S = S0.copy()
    out, _ = oracle.delta_step(q, k, v, g, beta, S, scale=0.25, state_bf16=True)
    kh = l2n(k); qh = 0.25 * l2n(q)
    I = np.eye(K)
    for b in range(B):
        for hv in range(HV):
            kk = kh[b, hv // 2]
            want = math.exp(g[b, hv]) * S0[b, hv] @ (I - beta[b, hv] * np.outer(kk, kk)) \
                + beta[b, hv] * np.outer(v[b, hv], kk)
            assert rel_err(out[b, hv], want @ qh[b, hv // 2]) < 1e-13
            stored = torch.from_numpy(want).to(torch.bfloat16).to(torch.float64).numpy()
            # the fp64 update and the closed form agree to ~1e-15, so only values within that of a
            # bf16 rounding midpoint could round apart; none is expected at these inputs
            assert np.array_equal(S[b, hv], stored)


def test_bf16_state_storage():
    check_bf16_state_storage()


def check_gqa_duplication():
    """G > 1 equals G = 1 with each q/k head repeated for its G value heads."""
    B, H, HV, K, V = 2, 2, 6, 16, 16
    q, k, v, g, beta = tiny_step_inputs(seed=16, B=B, H=H, HV=HV, K=K, V=V)
    S = tiny_state(seed=16, num_slots=B, HV=HV, V=V, K=K)
    S1 = S.copy()
    out, _ = oracle.delta_step(q, k, v, g, beta, S, scale=0.25)
    qr = np.repeat(q, HV // H, axis=1); kr = np.repeat(k, HV // H, axis=1)
    out1, _ = oracle.delta_step(qr, kr, v, g, beta, S1, scale=0.25)
    np.testing.assert_array_equal(out, out1)
    np.testing.assert_array_equal(S, S1)


def test_gqa_duplication():
    check_gqa_duplication()


def check_indices_permute_and_pad():
    """Permuting cache indices permutes the slots and nothing else; a pad row leaves every slot
    bit-identical and gets out = 0; an out-of-range slot is counted and skipped."""
    B, H, HV, K, V = 4, 2, 4, 16, 16
    q, k, v, g, beta = tiny_step_inputs(seed=17, B=B, H=H, HV=HV, K=K, V=V)
    S0 = tiny_state(seed=17, num_slots=6, HV=HV, V=V, K=K)
    ref = S0.copy()
    out_ref, _ = oracle.delta_step(q, k, v, g, beta, ref[:B].copy(order="C"), scale=0.25)
    ref_slots = ref[:B].copy(order="C")
    oracle.delta_step(q, k, v, g, beta, ref_slots, scale=0.25)
    perm = np.array([5, 2, 0, 3], dtype=np.int32)
    S = np.ascontiguousarray(S0[[0, 1, 2, 3, 4, 5]])
    S[perm] = S0[:B]
    Sp = S.copy()
    out, bad = oracle.delta_step(q, k, v, g, beta, Sp, scale=0.25, idx=perm, pad_slot=-1)
    assert bad == 0
    np.testing.assert_array_equal(out, out_ref)
    np.testing.assert_array_equal(Sp[perm], ref_slots)
    np.testing.assert_array_equal(Sp[[1, 4]], S[[1, 4]])
    idx = np.array([5, -1, 9, 3], dtype=np.int32)
    Sq = S.copy()
    out, bad = oracle.delta_step(q, k, v, g, beta, Sq, scale=0.25, idx=idx, pad_slot=-1)
    assert bad == 1
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    np.testing.assert_array_equal(Sq[[0, 1, 2, 4]], S[[0, 1, 2, 4]])


def test_indices_permute_and_pad():
    check_indices_permute_and_pad()


def check_contraction():
    """|I - beta k k^T| <= 1 for beta in [0,1] and exp(g) < 1: a perturbation of the state
    shrinks step by step, and the state stays bounded over 1000 steps."""
    S = tiny_state(seed=18)
    P = S.copy()
    P[0, 0, 0, 0] += 1e-3
    for step in range(1000):
        q, k, v, g, beta = tiny_step_inputs(seed=18, step=step)
        oracle.delta_step(q, k, v, g, beta, S, scale=0.25)
        oracle.delta_step(q, k, v, g, beta, P, scale=0.25)
        if step == 0:
            first = np.max(np.abs(P - S))
    assert first <= 1e-3 * (1 + 1e-12)
    assert np.max(np.abs(P - S)) < 1e-12
    assert np.max(np.abs(S)) < 50


def test_contraction():
    check_contraction()


# --------------------------------------------------------------------------------------------
# buffered (output-only) decode
# --------------------------------------------------------------------------------------------
def _buffered_vs_looped(L, ring_bf16, cycles=2, seed=20, B=2, H=2, HV=4, K=16, V=16):
    S_loop = tiny_state(seed=seed, num_slots=B, HV=HV, V=V, K=K)
    S_ckpt = S_loop.copy()
    d_cache = np.zeros((B, HV, L, V)); k_cache = np.zeros((B, H, L, K)); g_cache = np.zeros((B, HV, L))
    worst = 0.0
    for step in range(cycles * L):
        p = step % L
        q, k, v, g, beta = tiny_step_inputs(seed=seed, step=step, B=B, H=H, HV=HV, K=K, V=V)
        o_loop, _ = oracle.delta_step(q, k, v, g, beta, S_loop, scale=K ** -0.5)
        o_buf, bad = oracle.gdn_buffered(q, k, v, g, beta, S_ckpt, d_cache, k_cache, g_cache,
                                         np.full(B, p, np.int32), L=L, ring_bf16=ring_bf16,
                                         scale=K ** -0.5)
        assert bad == 0
        worst = max(worst, rel_err(o_buf, o_loop))
        if p == L - 1:
            worst = max(worst, rel_err(S_ckpt, S_loop))
            if not ring_bf16:
                S_ckpt[...] = S_loop   # keep the two paths on the same state in exact mode
    return worst


def check_buffered_equals_looped():
    for L in (1, 3, 8):
        assert _buffered_vs_looped(L, ring_bf16=False) < 1e-13
    assert _buffered_vs_looped(16, ring_bf16=True) < 2e-2


@pytest.mark.parametrize("L", [1, 3, 8])
def test_buffered_equals_looped_exact_ring(L):
    assert _buffered_vs_looped(L, ring_bf16=False) < 1e-13


def test_buffered_bf16_ring_within_tolerance():
    assert _buffered_vs_looped(16, ring_bf16=True) < 2e-2


def test_buffered_L1_is_the_packed_step():
    q, k, v, g, beta = tiny_step_inputs(seed=21)
    S = tiny_state(seed=21); S1 = S.copy()
    out, _ = oracle.delta_step(q, k, v, g, beta, S, scale=0.25)
    z = lambda *s: np.zeros(s)
    out1, _ = oracle.gdn_buffered(q, k, v, g, beta, S1, z(2, 4, 1, 16), z(2, 2, 1, 16), z(2, 4, 1),
                                  np.zeros(2, np.int32), L=1, scale=0.25)
    np.testing.assert_array_equal(out, out1)
    np.testing.assert_array_equal(S, S1)


def check_buffered_ring_records_and_lowrank():
    """The ring holds (delta, k_hat, g) of each step, and u and o of step p follow from the
    checkpoint and the records alone (the low-rank form the CUDA kernel uses):
      Gamma = exp(sum_{i<=p} g_i), c_j = exp(sum_{j<i<=p} g_i),
      u = Gamma S_c k + sum_{j<p} c_j d_j (k_j . k),  delta = beta (v - u),
      o = Gamma S_c q + sum_{j<p} c_j d_j (k_j . q) + delta (k . q)."""
    B, H, HV, K, V, L = 2, 2, 4, 16, 16, 6
    S_c = tiny_state(seed=22, num_slots=B, HV=HV, V=V, K=K)
    S0 = S_c.copy()
    d_cache = np.zeros((B, HV, L, V)); k_cache = np.zeros((B, H, L, K)); g_cache = np.zeros((B, HV, L))
    for p in range(L):
        q, k, v, g, beta = tiny_step_inputs(seed=22, step=p, B=B, H=H, HV=HV, K=K, V=V)
        kh = l2n(k); qh = K ** -0.5 * l2n(q)
        o, _ = oracle.gdn_buffered(q, k, v, g, beta, S_c, d_cache, k_cache, g_cache,
                                   np.full(B, p, np.int32), L=L, ring_bf16=False, scale=K ** -0.5)
        for b in range(B):
            for hv in range(HV):
                h = hv // (HV // H)
                gs = np.concatenate([g_cache[b, hv, :p], [g[b, hv]]])
                Gam = math.exp(gs.sum())
                c = np.array([math.exp(gs[j + 1:].sum()) for j in range(p)])
                dj = d_cache[b, hv, :p]; kj = k_cache[b, h, :p]
                u = Gam * S0[b, hv] @ kh[b, h] + (c[:, None] * dj).T @ (kj @ kh[b, h]) if p else \
                    Gam * S0[b, hv] @ kh[b, h]
                delta = beta[b, hv] * (v[b, hv] - u)
                o_lr = Gam * S0[b, hv] @ qh[b, h] + delta * (kh[b, h] @ qh[b, h])
                if p:
                    o_lr = o_lr + (c[:, None] * dj).T @ (kj @ qh[b, h])
                assert rel_err(o[b, hv], o_lr) < 1e-12
                assert rel_err(d_cache[b, hv, p], delta) < 1e-12
                assert rel_err(k_cache[b, h, p], kh[b, h]) < 1e-15
                assert g_cache[b, hv, p] == g[b, hv]
    # the flush at p = L-1 wrote the checkpoint; it equals L looped single steps
    S_loop = S0.copy()
    for p in range(L):
        q, k, v, g, beta = tiny_step_inputs(seed=22, step=p, B=B, H=H, HV=HV, K=K, V=V)
        oracle.delta_step(q, k, v, g, beta, S_loop, scale=K ** -0.5)
    assert rel_err(S_c, S_loop) < 1e-13


def test_buffered_ring_records_and_lowrank():
    check_buffered_ring_records_and_lowrank()


def test_buffered_bad_rows():
    q, k, v, g, beta = tiny_step_inputs(seed=23)
    S = tiny_state(seed=23); S0 = S.copy()
    L = 4
    rings = [np.zeros((2, 4, L, 16)), np.zeros((2, 2, L, 16)), np.zeros((2, 4, L))]
    out, bad = oracle.gdn_buffered(q, k, v, g, beta, S, *rings, np.array([L, -1], np.int32), L=L,
                                   scale=0.25)
    assert bad == 2 and np.all(out == 0)
    np.testing.assert_array_equal(S, S0)
    assert all(np.all(r == 0) for r in rings)


# --------------------------------------------------------------------------------------------
# fused KDA decode parts
# --------------------------------------------------------------------------------------------
def check_conv_update_is_causal_convolution():
    """T successive updates of one slot equal the causal convolution of the whole input stream
    (numpy.convolve), with the initial conv state as the three inputs before it, and the state
    ends holding the last three inputs."""
    C, steps = 5, 9
    rng = np.random.default_rng(30)
    w = rng.normal(size=(C, 4)); hist = rng.normal(size=(C, 3)); xs = rng.normal(size=(steps, C))
    cs = np.ascontiguousarray(hist[None].copy())
    ys = []
    for t in range(steps):
        y, _ = oracle.conv_update(xs[t:t + 1], w, cs, idx=np.array([0], np.int32), pad_slot=-1)
        ys.append(y[0])
    ys = np.array(ys)
    for c in range(C):
        stream = np.concatenate([hist[c], xs[:, c]])
        pre = np.convolve(stream, w[c, ::-1], mode="valid")      # y_t = sum_j w[j] x_{t-3+j}
        want = pre * (1.0 / (1.0 + np.exp(-pre)))
        assert rel_err(ys[:, c], want) < 1e-13
    np.testing.assert_array_equal(cs[0], xs[-3:].T)


def test_conv_update_is_causal_convolution():
    check_conv_update_is_causal_convolution()


def test_conv_update_pad_and_bad_rows():
    rng = np.random.default_rng(31)
    cs = rng.normal(size=(3, 4, 3)); cs0 = cs.copy()
    y, bad = oracle.conv_update(rng.normal(size=(2, 4)), rng.normal(size=(4, 4)), cs,
                                idx=np.array([0, 7], np.int32), pad_slot=0)
    assert bad == 1 and np.all(y == 0)
    np.testing.assert_array_equal(cs, cs0)


def check_gated_rmsnorm():
    rng = np.random.default_rng(32)
    x = rng.normal(size=(6, 128)); gate = rng.normal(size=(6, 128)); w = rng.normal(size=128)
    tx, tg, tw = (torch.from_numpy(a) for a in (x, gate, w))
    base = torch.nn.functional.rms_norm(tx, (128,), tw, eps=1e-5)
    assert rel_err(oracle.gated_rmsnorm(x, gate, w, 1e-5, "silu"),
                   (base * torch.nn.functional.silu(tg)).numpy()) < 1e-13
    assert rel_err(oracle.gated_rmsnorm(x, gate, w, 1e-5, "sigmoid"),
                   (base * torch.sigmoid(tg)).numpy()) < 1e-13
    # with gate -> +inf (sigmoid = 1), unit weight and eps = 0 the output has unit RMS
    out = oracle.gated_rmsnorm(x, np.full_like(x, 800.0), np.ones(128), 0.0, "sigmoid")
    assert np.allclose(np.mean(out ** 2, axis=-1), 1.0, atol=1e-13)


def test_gated_rmsnorm():
    check_gated_rmsnorm()


def check_fused_per_key_gate_reduces_to_scalar():
    """With raw_g and dt_bias constant over the key channels of a head and the bound inactive,
    the per-key-channel (KDA) decay equals the one-decay-per-head (GDN) path."""
    T, heads, D = 2, 2, 16
    dim = heads * D
    ins = syn.fused_inputs(T, heads, D, T + 2, seed=33)
    f = lambda bits: syn.bf16_bits_to_f32(bits).astype(np.float64)
    raw_head = -2.0 + 0.1 * f(ins["raw_g"])[:, :, 0]
    raw_kda = np.repeat(raw_head[:, :, None], D, axis=2)
    dtb_head = 0.1 * ins["dt_bias"][:heads].astype(np.float64)
    dtb_kda = np.repeat(dtb_head, D)
    idx = np.arange(1, T + 1, dtype=np.int32)
    st = syn.normal_f32(33, syn.Tag.STATE, 0, (T + 2, heads, D, D), 1.0).astype(np.float64)
    cs = f(ins["conv_state"]).reshape(T + 2, 3 * dim, 3)
    args = (f(ins["x"]), ins["conv_w"], )
    outs = []
    for kind, raw, dtb in (("kda", raw_kda, dtb_kda), ("gdn", raw_head, dtb_head)):
        s, c = st.copy(), cs.copy()
        o, _ = oracle.fused_kda(*args, c, raw, f(ins["raw_beta"]), ins["A_log"] * 0.1, dtb, s,
                                f(ins["out_gate"]), ins["norm_w"], idx=idx, pad_slot=0,
                                gate_kind=kind)
        outs.append((o, s))
    assert rel_err(outs[0][0], outs[1][0]) < 1e-13
    assert rel_err(outs[0][1], outs[1][1]) < 1e-13


def test_fused_per_key_gate_reduces_to_scalar():
    check_fused_per_key_gate_reduces_to_scalar()


# --------------------------------------------------------------------------------------------
# Mamba-1 selective-scan decode
# --------------------------------------------------------------------------------------------
def _mamba_inputs(B, D, N, seed):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(B, D)), dt=np.log1p(np.exp(rng.normal(size=(B, D)))),
                A=-np.exp(rng.normal(size=(D, N))), Bm=rng.normal(size=(B, N)),
                Cm=rng.normal(size=(B, N)), Dskip=rng.normal(size=D), z=rng.normal(size=(B, D)),
                h=rng.normal(size=(B, D, N)))


def check_mamba_constant_input_geometric_series():
    """With dt, A, B, x fixed over T steps the recurrence is h_T = a^T h_0 + b x (1 - a^T)/(1 - a)
    per state element (a = exp(dt A), b = dt B): a closed form of the linear recurrence."""
    B, D, N, T = 2, 3, 5, 7
    m = _mamba_inputs(B, D, N, 40)
    h = m["h"].copy()
    for _ in range(T):
        oracle.mamba_decode(m["x"], m["dt"], m["A"], m["Bm"], m["Cm"], h)
    a = np.exp(m["dt"][:, :, None] * m["A"][None])
    bx = m["dt"][:, :, None] * m["Bm"][:, None, :] * m["x"][:, :, None]
    want = a ** T * m["h"] + bx * (1 - a ** T) / (1 - a)
    assert rel_err(h, want) < 1e-12


def check_mamba_output_and_gates():
    """y = C . h_new, plus D x, times silu(z); with dt = 0 the state is unchanged; A = 0 makes the
    state accumulate dt B x; z = 0 zeroes y and a large z multiplies it by z (silu(z) -> z)."""
    B, D, N = 2, 4, 6
    m = _mamba_inputs(B, D, N, 41)
    h = m["h"].copy()
    y = oracle.mamba_decode(m["x"], m["dt"], m["A"], m["Bm"], m["Cm"], h, Dskip=m["Dskip"], z=m["z"])
    plain = np.einsum("bn,bdn->bd", m["Cm"], h) + m["Dskip"][None] * m["x"]
    silu = torch.nn.functional.silu(torch.from_numpy(m["z"])).numpy()
    assert rel_err(y, plain * silu) < 1e-13
    h0 = m["h"].copy()
    y0 = oracle.mamba_decode(m["x"], np.zeros((B, D)), m["A"], m["Bm"], m["Cm"], h0)
    np.testing.assert_array_equal(h0, m["h"])
    assert rel_err(y0, np.einsum("bn,bdn->bd", m["Cm"], m["h"])) < 1e-13
    ha = m["h"].copy()
    oracle.mamba_decode(m["x"], m["dt"], np.zeros((D, N)), m["Bm"], m["Cm"], ha)
    assert rel_err(ha, m["h"] + m["dt"][:, :, None] * m["Bm"][:, None, :] * m["x"][:, :, None]) < 1e-14
    hz = m["h"].copy()
    yz = oracle.mamba_decode(m["x"], m["dt"], m["A"], m["Bm"], m["Cm"], hz, z=np.zeros((B, D)))
    assert np.all(yz == 0)
    hb = m["h"].copy()
    yb = oracle.mamba_decode(m["x"], m["dt"], m["A"], m["Bm"], m["Cm"], hb, z=np.full((B, D), 800.0))
    assert rel_err(yb, 800.0 * np.einsum("bn,bdn->bd", m["Cm"], hb)) < 1e-13


def test_mamba_constant_input_geometric_series():
    check_mamba_constant_input_geometric_series()


def test_mamba_output_and_gates():
    check_mamba_output_and_gates()


# --------------------------------------------------------------------------------------------
# decode projection (GEMV)
# --------------------------------------------------------------------------------------------
def check_gemv():
    """Against numpy's matmul (a different implementation), and two closed forms: identity
    weights return x, and a rank-1 W = u w^T gives y = (x . w) u."""
    rng = np.random.default_rng(50)
    x = rng.normal(size=(3, 37)); W = rng.normal(size=(11, 37))
    assert rel_err(oracle.gemv(x, W), x @ W.T) < 1e-13
    np.testing.assert_array_equal(oracle.gemv(x, np.eye(37)), x)
    u, w = rng.normal(size=5), rng.normal(size=37)
    assert rel_err(oracle.gemv(x, np.outer(u, w)), np.outer(x @ w, u)) < 1e-13


def test_gemv():
    check_gemv()


# --------------------------------------------------------------------------------------------
# decode layer front (projection -> fused decode -> projection)
# --------------------------------------------------------------------------------------------
def check_decode_front_selects_columns():
    """With an identity input projection (x carries z itself) and an output projection that copies
    the first dim columns, the front is the fused decode on z's column blocks, its output rounded
    to bf16: exactly, for both gate kinds. Each block holds different random values, so a block
    read from the wrong columns fails."""
    T, heads, D = 3, 2, 16
    dim = heads * D
    f = lambda bits: syn.bf16_bits_to_f32(bits).astype(np.float64)
    for kind in ("gdn", "kda"):
        ins = syn.fused_inputs(T, heads, D, T + 2, seed=61)
        raw_g = f(ins["raw_g"]) if kind == "kda" else f(ins["raw_g"])[:, :, 0]
        dt_bias = ins["dt_bias"] if kind == "kda" else ins["dt_bias"][:heads]
        z = np.concatenate([f(ins["x"]), f(ins["out_gate"]).reshape(T, dim), raw_g.reshape(T, -1),
                            f(ins["raw_beta"]).reshape(T, heads)], axis=1)
        P = z.shape[1]
        col = oracle.front_columns(heads, D, kind)
        assert col["raw_beta"][1] == P
        W_out = np.zeros((P, dim))
        W_out[np.arange(dim), np.arange(dim)] = 1.0
        idx = np.array([2, 0, 1], dtype=np.int32)          # row 1 is the pad (slot 0) row
        st = syn.normal_f32(61, syn.Tag.STATE, 0, (T + 2, heads, D, D), 1.0).astype(np.float64)
        cs = f(ins["conv_state"]).reshape(T + 2, 3 * dim, 3)
        s1, c1, s2, c2 = st.copy(), cs.copy(), st.copy(), cs.copy()
        y, _ = oracle.decode_front(z, np.eye(P), W_out, ins["conv_w"], c1, ins["A_log"], dt_bias,
                                   s1, ins["norm_w"], heads=heads, D=D, idx=idx, pad_slot=0,
                                   gate_kind=kind)
        o, _ = oracle.fused_kda(f(ins["x"]), ins["conv_w"], c2, raw_g, f(ins["raw_beta"]),
                                ins["A_log"], dt_bias, s2, f(ins["out_gate"]), ins["norm_w"],
                                idx=idx, pad_slot=0, gate_kind=kind)
        np.testing.assert_array_equal(y[:, :dim], oracle.round_bf16(o.reshape(T, dim)))
        np.testing.assert_array_equal(y[:, dim:], 0.0)
        np.testing.assert_array_equal(s1, s2)
        np.testing.assert_array_equal(c1, c2)


def test_decode_front_selects_columns():
    check_decode_front_selects_columns()


# --------------------------------------------------------------------------------------------
# scalar closed form and an independent restatement of the packed step
# --------------------------------------------------------------------------------------------
def check_scalar_closed_form():
    """K = V = 1 with |k|, |q| so large that x / sqrt(x^2 + 1e-6) rounds to sign(x) in fp64: one
    step is S' = e^g S (1 - beta) + beta v sign(k) and o = S' sign(q) (the scale 1^-1/2 is 1)."""
    gs = [0.0, -0.7, -3.0, 0.0, -0.2, -1.5]
    betas = [0.0, 0.3, 1.0, 1.0, 0.55, 0.9]
    ks = [1e5, -2e5, 3e4, -1e6, 5e4, -7e4]
    qs = [-4e4, 1e5, 2e5, 3e4, -6e5, 1e4]
    vs = [0.25, -1.5, 2.0, 0.75, -0.3, 1.1]
    S0 = [1.0, -0.5, 3.0, -2.0, 0.125, 0.7]
    B = len(gs)
    q = np.array(qs).reshape(B, 1, 1); k = np.array(ks).reshape(B, 1, 1)
    v = np.array(vs).reshape(B, 1, 1)
    S = np.array(S0).reshape(B, 1, 1, 1)
    out, _ = oracle.delta_step(q, k, v, np.array(gs).reshape(B, 1), np.array(betas).reshape(B, 1), S,
                               scale=1.0)
    for i in range(B):
        want = math.exp(gs[i]) * S0[i] * (1.0 - betas[i]) + betas[i] * vs[i] * math.copysign(1.0, ks[i])
        assert abs(S[i, 0, 0, 0] - want) <= 1e-14 * max(1.0, abs(want)), (i, S[i, 0, 0, 0], want)
        assert abs(out[i, 0, 0] - want * math.copysign(1.0, qs[i])) <= 1e-14 * max(1.0, abs(want)), i


def _twin_packed_step(mixed, a, b, A_log, dt_bias, S, H, HV, K, V):
    """One packed GDN decode step restated with Python floats and loops, row b on slot b, written
    from the sources independently of the oracle: the gates g = -exp(A_log) softplus(a + dt_bias)
    and beta = sigmoid(b), q/k L2-normalised with eps 1e-6 and q scaled by K^-1/2, q/k head
    hv // (HV / H), then decay, u = S k, delta = beta (v - u), S += delta k^T, o = S q
    ("Optimization Log: Qwen3.5-27B Dense on B200", Kernel 4 Math block). S is nested lists
    [slot][hv][v][k], updated in place; returns o as nested lists [b][hv][v]."""
    G = HV // H
    out = []
    for bb in range(len(mixed)):
        row = [float(x) for x in mixed[bb]]
        o_row = []
        for hv in range(HV):
            h = hv // G
            q = row[h * K:(h + 1) * K]
            k = row[H * K + h * K:H * K + (h + 1) * K]
            v = row[2 * H * K + hv * V:2 * H * K + (hv + 1) * V]
            g = -math.exp(float(A_log[hv])) * math.log1p(math.exp(float(a[bb][hv]) + float(dt_bias[hv])))
            beta = 1.0 / (1.0 + math.exp(-float(b[bb][hv])))
            nk = math.sqrt(sum(t * t for t in k) + 1e-6)
            nq = math.sqrt(sum(t * t for t in q) + 1e-6)
            kh = [t / nk for t in k]
            qh = [t / nq * K ** -0.5 for t in q]
            M = S[bb][hv]
            e = math.exp(g)
            for i in range(V):
                for j in range(K):
                    M[i][j] *= e
            u = [sum(M[i][j] * kh[j] for j in range(K)) for i in range(V)]
            d = [beta * (v[i] - u[i]) for i in range(V)]
            for i in range(V):
                for j in range(K):
                    M[i][j] += d[i] * kh[j]
            o_row.append([sum(M[i][j] * qh[j] for j in range(K)) for i in range(V)])
        out.append(o_row)
    return out


def check_python_twin_tiny():
    """The tiny decode (B=2, H=2, HV=4, K=V=16, fp32 inputs, 8 sequential steps): the C oracle
    and its pure-Python restatement agree to 1e-12 on every output and on the final state."""
    B, H, HV, K, V = TINY["B"], TINY["H"], TINY["HV"], TINY["K"], TINY["V"]
    S64 = tiny_state(seed=31, num_slots=B, HV=HV, V=V, K=K)
    S_twin = S64.tolist()
    for step in range(8):
        d = syn.packed_inputs(B, H, HV, K, V, "f32", 31, step)
        mixed, a, b = (d[n].astype(np.float64) for n in ("mixed_qkv", "a", "b"))
        A_log, dt_bias = d["A_log"].astype(np.float64), d["dt_bias"].astype(np.float64)
        o, _ = oracle.gdn_step_packed(mixed, a, b, A_log, dt_bias, S64, H=H, HV=HV, K=K, V=V)
        o_twin = _twin_packed_step(mixed.tolist(), a.tolist(), b.tolist(), A_log.tolist(),
                                   dt_bias.tolist(), S_twin, H, HV, K, V)
        assert rel_err(o, np.array(o_twin)) <= 1e-12, step
    assert rel_err(S64, np.array(S_twin)) <= 1e-12


def test_scalar_closed_form():
    check_scalar_closed_form()


def test_python_twin_tiny():
    check_python_twin_tiny()


ALL_CHECKS = [
    check_hand_worked_step, check_invariant_no_decay_no_write, check_invariant_exact_recall,
    check_invariant_full_decay, check_closed_matrix_form, check_gqa_duplication,
    check_indices_permute_and_pad, check_buffered_equals_looped,
    check_buffered_ring_records_and_lowrank, check_gdn_gates, check_kda_gate_reading,
    check_conv_update_is_causal_convolution, check_gated_rmsnorm, check_bf16_rounding,
    check_fused_per_key_gate_reduces_to_scalar, check_bf16_state_storage,
    check_mamba_constant_input_geometric_series, check_mamba_output_and_gates, check_gemv,
    check_decode_front_selects_columns, check_scalar_closed_form, check_python_twin_tiny,
]
