"""GPU parity of gdn_decode_buffered (the output-only decode that writes the state back once every
L steps) against the fp64 oracle, which replays the ring records element by element.

Exact-ring mode (fp32 records, fp32 inputs): outputs, checkpoints and records within 1e-5.
bf16-ring mode at the packed shapes: outputs within 2e-2; the checkpoint state and the records
within 2e-2 as well, since both sides round their own delta to bf16 and a value next to a rounding
midpoint can land on either neighbour (a one-ulp bf16 difference, about 0.4% of that record)."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import PackedCase, host_state

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_buffered(B, H, HV, K, V, L, dtype, ring, seed, steps, *, start_pos=None, indexed=False,
                  out_dtype=None, pad_rows=(), kernel="auto"):
    out_dtype = out_dtype or dtype
    num_slots = B + 2 if indexed else B
    S64 = host_state(num_slots, HV, V, K, seed)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    rdt = torch.bfloat16 if ring == "bf16" else torch.float32
    d_cache = torch.zeros((num_slots, HV, L, V), dtype=rdt, device="cuda")
    k_cache = torch.zeros((num_slots, H, L, K), dtype=rdt, device="cuda")
    g_cache = torch.zeros((num_slots, HV, L), dtype=torch.float32, device="cuda")
    d64, k64, g64 = np.zeros((num_slots, HV, L, V)), np.zeros((num_slots, H, L, K)), np.zeros((num_slots, HV, L))
    wp = np.zeros(B, np.int32) if start_pos is None else np.array(start_pos, np.int32) % L
    idx_np, idx = None, None
    if indexed:
        idx_np = syn.permutation(seed + 5, num_slots)[:B].copy()
        for r in pad_rows:
            idx_np[r] = -1
        idx = torch.from_numpy(idx_np).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst = {"out": 0.0, "state": 0.0, "ring": 0.0}
    odt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    for step in range(steps):
        c = PackedCase(B, H, HV, K, V, dtype, seed, step)
        out = torch.full((B, 1, HV, V), float("nan"), dtype=odt, device="cuda")
        q, k, v = c.views()
        gdn.gdn_decode_buffered(q, k, v, state, out, d_cache, k_cache, g_cache,
                                torch.from_numpy(wp).cuda(), cache_indices=idx, pad_slot_id=-1,
                                H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias, err_flags=err,
                                kernel=kernel)
        mixed, a, b, A_log, dt_bias = c.oracle_args()
        qo, ko, vo = oracle.split_packed(mixed, H, HV, K, V)
        g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
        o_ref, bad = oracle.gdn_buffered(qo, ko, vo, g, beta, S64, d64, k64, g64, wp, L=L,
                                         ring_bf16=(ring == "bf16"), scale=K ** -0.5, idx=idx_np,
                                         pad_slot=-1)
        assert bad == 0
        got = out.float().cpu().numpy().reshape(B, HV, V)
        assert np.all(np.isfinite(got))
        worst["out"] = max(worst["out"], rel_err(got, o_ref))
        worst["state"] = max(worst["state"], rel_err(state.cpu().numpy(), S64))
        for dev_r, host_r in ((d_cache, d64), (k_cache, k64), (g_cache, g64)):
            worst["ring"] = max(worst["ring"], rel_err(dev_r.float().cpu().numpy(), host_r))
        wp = (wp + 1) % L
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return worst


@pytest.mark.parametrize("L", [1, 3, 8])
def test_exact_ring_tiny_two_cycles(L):
    """The tiny decode shapes with fp32 records: two full cycles, every phase."""
    w = _run_buffered(2, 2, 4, 16, 16, L, "f32", "f32", seed=40 + L, steps=2 * L)
    assert max(w.values()) <= 1e-5, w


@pytest.mark.parametrize("K,G,kernel", [(32, 1, "auto"), (64, 3, "auto"), (128, 2, "tile"),
                                        (128, 2, "pipe"), (128, 3, "pipe"), (128, 2, "stage"),
                                        (128, 3, "stage")])
def test_exact_ring_shapes_mixed_phases(K, G, kernel):
    """Rows at different cursors in one call (each row's own phase), records of one q/k head
    shared by G value heads; at K = V = 128 the per-tile, the pipelined and the staged kernel."""
    H = 2
    w = _run_buffered(3, H, H * G, K, K, 4, "f32", "f32", seed=K + G, steps=7, start_pos=[0, 1, 3],
                      indexed=True, kernel=kernel)
    assert max(w.values()) <= 1e-5, w


@pytest.mark.parametrize("kernel", ["auto", "tile", "pipe", "stage"])
@pytest.mark.parametrize("L", [1, 8, 16])
def test_bf16_ring_packed_shapes(L, kernel):
    """The packed decode shapes (H=16, HV=32, K=V=128) with bf16 inputs, outputs and records over
    one full cycle plus one step."""
    w = _run_buffered(4, 16, 32, 128, 128, L, "bf16", "bf16", seed=50 + L, steps=L + 1, indexed=True,
                      kernel=kernel)
    assert w["out"] <= 2e-2 and w["state"] <= 2e-2 and w["ring"] <= 2e-2, w


def test_pipelined_kernel_many_tiles_per_cta():
    """1536 tiles: every CTA of the persistent kernel walks about ten tiles through its
    shared-memory stages, with rows at mixed cursors and a pad row."""
    B = 48
    w = _run_buffered(B, 16, 32, 128, 128, 8, "bf16", "bf16", seed=91, steps=9, indexed=True,
                      start_pos=[(3 * r) % 8 for r in range(B)], pad_rows=(5,), kernel="pipe")
    assert w["out"] <= 2e-2 and w["state"] <= 2e-2 and w["ring"] <= 2e-2, w


@pytest.mark.parametrize("kernel", ["pipe", "stage"])
def test_pipelined_kernel_exact_ring_fp32_inputs(kernel):
    w = _run_buffered(6, 4, 8, 128, 128, 4, "f32", "f32", seed=92, steps=9, indexed=True,
                      start_pos=[0, 1, 2, 3, 0, 1], kernel=kernel)
    assert max(w.values()) <= 1e-5, w


def test_staged_kernel_many_tiles():
    """1536 tiles, one CTA per tile staged in shared memory; rows at mixed cursors and a pad row,
    two cycles of L = 8."""
    B = 48
    w = _run_buffered(B, 16, 32, 128, 128, 8, "bf16", "bf16", seed=93, steps=17, indexed=True,
                      start_pos=[(5 * r) % 8 for r in range(B)], pad_rows=(7,), kernel="stage")
    assert w["out"] <= 2e-2 and w["state"] <= 2e-2 and w["ring"] <= 2e-2, w


def test_pad_rows_are_skipped():
    w = _run_buffered(4, 2, 4, 32, 32, 4, "f32", "f32", seed=61, steps=5, indexed=True, pad_rows=(2,))
    assert max(w.values()) <= 1e-5, w


def test_L1_equals_the_packed_step():
    B, H, HV, K, V = 4, 2, 4, 64, 64
    c = PackedCase(B, H, HV, K, V, "bf16", 70, 0)
    S = torch.from_numpy(host_state(B, HV, V, K, 70).astype(np.float32)).cuda()
    S1 = S.clone()
    out = torch.empty((B, HV, V), dtype=torch.float32, device="cuda")
    out1 = torch.empty_like(out)
    q, k, v = c.views()
    kw = dict(H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias)
    gdn.gdn_decode_step(q, k, v, S, out, **kw)
    ring = [torch.zeros((B, HV, 1, V), device="cuda"), torch.zeros((B, H, 1, K), device="cuda"),
            torch.zeros((B, HV, 1), device="cuda")]
    gdn.gdn_decode_buffered(q, k, v, S1, out1, *ring, torch.zeros(B, dtype=torch.int32, device="cuda"), **kw)
    torch.cuda.synchronize()
    assert rel_err(out1.cpu().numpy(), out.cpu().numpy()) <= 1e-6
    assert rel_err(S1.cpu().numpy(), S.cpu().numpy()) <= 1e-6


def test_bad_cursor_sets_the_flag_and_skips_the_row():
    B, H, HV, K, V, L = 3, 1, 2, 32, 32, 4
    c = PackedCase(B, H, HV, K, V, "f32", 80, 0)
    S = torch.from_numpy(host_state(B, HV, V, K, 80).astype(np.float32)).cuda()
    S0 = S.clone()
    out = torch.full((B, HV, V), 7.0, device="cuda")
    ring = [torch.zeros((B, HV, L, V), device="cuda"), torch.zeros((B, H, L, K), device="cuda"),
            torch.zeros((B, HV, L), device="cuda")]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    wp = torch.tensor([L - 1, L, -1], dtype=torch.int32, device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_buffered(q, k, v, S, out, *ring, wp, H=H, a=c.a, b=c.b, A_log=c.A_log,
                            dt_bias=c.dt_bias, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.GDN_DEVERR_BAD_WRITE_POS
    assert torch.all(out[1:] == 0)
    assert torch.equal(S[1:], S0[1:])
    assert not torch.equal(S[0], S0[0])   # row 0 flushed at L-1
