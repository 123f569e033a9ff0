"""Edge cases at the documented limits and the degenerate inputs, against the fp64 oracle:
the largest value dim (V = 1024, eight row passes), the longest ring (L = 64, where the pipelined
kernel fits only two stages), single rows, and empty batches on every entry point."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import PackedCase, host_state, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("B,HV", [(2, 2), (400, 2)])
def test_largest_value_dim(B, HV):
    """V = 1024 at K = 128: split over CTAs for the small batch, eight passes in one CTA for the
    large one."""
    H, K, V = 1, 128, 1024
    c = PackedCase(B, H, HV, K, V, "bf16", 500 + B, 0)
    S64 = host_state(B, HV, V, K, 500 + B)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    out = torch.empty((B, HV, V), device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_step(q, k, v, state, out, H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias)
    o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V)
    assert rel_err(out.cpu().numpy(), o_ref) <= 1e-5
    assert rel_err(state.cpu().numpy(), S64) <= 1e-5


@pytest.mark.parametrize("kernel", ["tile", "pipe"])
def test_longest_ring(kernel):
    """L = 64 over a full cycle plus one step (the ring's last record is read by the flush)."""
    B, H, HV, K, V, L = 2, 1, 2, 128, 128, 64
    S64 = host_state(B, HV, V, K, 510)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    d_cache = torch.zeros((B, HV, L, V), dtype=torch.bfloat16, device="cuda")
    k_cache = torch.zeros((B, H, L, K), dtype=torch.bfloat16, device="cuda")
    g_cache = torch.zeros((B, HV, L), device="cuda")
    d64, k64, g64 = np.zeros((B, HV, L, V)), np.zeros((B, H, L, K)), np.zeros((B, HV, L))
    worst = 0.0
    for step in range(L + 1):
        p = step % L
        c = PackedCase(B, H, HV, K, V, "bf16", 510, step)
        out = torch.empty((B, HV, V), device="cuda")
        q, k, v = c.views()
        wp = np.full(B, p, np.int32)
        gdn.gdn_decode_buffered(q, k, v, state, out, d_cache, k_cache, g_cache, torch.from_numpy(wp).cuda(),
                                H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias, kernel=kernel)
        mixed, a, b, A_log, dt_bias = c.oracle_args()
        qo, ko, vo = oracle.split_packed(mixed, H, HV, K, V)
        g, beta = oracle.gdn_gates(a, b, A_log, dt_bias)
        o_ref, _ = oracle.gdn_buffered(qo, ko, vo, g, beta, S64, d64, k64, g64, wp, L=L, ring_bf16=True,
                                       scale=K ** -0.5)
        worst = max(worst, rel_err(out.cpu().numpy(), o_ref))
    assert worst <= 2e-2
    assert rel_err(state.cpu().numpy(), S64) <= 2e-2


def test_single_row_every_entry_point():
    """B = 1 through the step, the indexed step (slot 5 of 8) and the buffered decode (L = 1)."""
    H, HV, K, V = 2, 4, 64, 64
    c = PackedCase(1, H, HV, K, V, "f32", 520, 0)
    q, k, v = c.views()
    kw = dict(H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias)
    S64 = host_state(8, HV, V, K, 520)
    for mode in ("step", "indexed", "buffered"):
        S = S64.copy()
        state = torch.from_numpy(S.astype(np.float32)).cuda()
        out = torch.empty((1, HV, V), device="cuda")
        idx_np = np.array([5], np.int32)
        if mode == "step":
            gdn.gdn_decode_step(q, k, v, state, out, **kw)
            idx_np = None
        elif mode == "indexed":
            gdn.gdn_decode_step_indexed(q, k, v, state, out, torch.from_numpy(idx_np).cuda(), **kw)
        else:
            ring = [torch.zeros((8, HV, 1, V), device="cuda"), torch.zeros((8, H, 1, K), device="cuda"),
                    torch.zeros((8, HV, 1), device="cuda")]
            gdn.gdn_decode_buffered(q, k, v, state, out, *ring, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                    cache_indices=torch.from_numpy(idx_np).cuda(), **kw)
        o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S, H=H, HV=HV, K=K, V=V, idx=idx_np)
        assert rel_err(out.cpu().numpy(), o_ref) <= 1e-5, mode
        assert rel_err(state.cpu().numpy(), S) <= 1e-5, mode


def test_empty_inputs_launch_nothing():
    """B = 0 / T = 0 are valid and touch nothing."""
    dev = "cuda"
    state = torch.ones((2, 4, 16, 16), device=dev)
    x = torch.zeros((0, 2 * 2 * 16 + 4 * 16), device=dev)
    q, k, v = gdn.split_mixed_qkv(x, 2, 4, 16, 16)
    ab = torch.zeros((0, 4), device=dev)
    kw = dict(H=2, a=ab, b=ab, A_log=torch.zeros(4, device=dev), dt_bias=torch.zeros(4, device=dev))
    ring = [torch.zeros((2, 4, 4, 16), device=dev), torch.zeros((2, 2, 4, 16), device=dev),
            torch.zeros((2, 4, 4), device=dev)]
    gdn.gdn_decode_buffered(q, k, v, state, torch.zeros((0, 4, 16), device=dev), *ring,
                            torch.zeros(0, dtype=torch.int32, device=dev), **kw)
    gdn.gdn_decode_step_indexed(q, k, v, state, torch.zeros((0, 4, 16), device=dev),
                                torch.zeros(0, dtype=torch.int32, device=dev), **kw)
    ins = syn.fused_inputs(1, 2, 16, 4, seed=3)
    bf = lambda bits: to_device(bits, "bf16")
    fstate = torch.ones((4, 2, 16, 16), device=dev)
    gdn.gdn_decode_fused(bf(ins["x"])[:0], torch.from_numpy(ins["conv_w"]).cuda(), bf(ins["conv_state"]),
                         bf(ins["raw_g"])[:0], bf(ins["raw_beta"])[:0], torch.from_numpy(ins["A_log"]).cuda(),
                         torch.from_numpy(ins["dt_bias"]).cuda(), fstate, torch.zeros(0, dtype=torch.int32, device=dev),
                         bf(ins["out_gate"])[:0], torch.from_numpy(ins["norm_w"]).cuda(),
                         torch.zeros((0, 2, 16), dtype=torch.bfloat16, device=dev))
    h = torch.ones((0, 8, 16), device=dev)
    z0 = torch.zeros((0, 8), device=dev)
    gdn.mamba_selective_scan_decode(z0, z0, torch.zeros((8, 16), device=dev), torch.zeros((0, 16), device=dev),
                                    torch.zeros((0, 16), device=dev), h, torch.zeros((0, 8), device=dev))
    torch.cuda.synchronize()
    assert torch.all(state == 1) and torch.all(fstate == 1)
