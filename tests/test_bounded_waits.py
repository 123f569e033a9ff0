"""The pipelined kernels bound every wait. The self-test kernel waits on an mbarrier that nothing
arrives at: the wait must give up after its limit (about a millisecond here), report
GDN_DEVERR_TIMEOUT through the error word, and leave the CUDA context usable (a decode step
afterwards still matches the oracle). No GPU fault is caused: the kernel returns normally."""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import PackedCase, host_state

pytestmark = pytest.mark.gpu


def test_wait_that_completes_sets_no_flag():
    assert torch.cuda.is_available()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_selftest_bounded_wait(err, 2_000_000, arrive=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_wait_that_never_completes_times_out_and_the_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_selftest_bounded_wait(err, 2_000_000, arrive=False)   # about 1 ms at 2 GHz
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.GDN_DEVERR_TIMEOUT
    # the context is still usable: a decode step runs and matches the oracle
    B, H, HV, K, V = 2, 2, 4, 32, 32
    c = PackedCase(B, H, HV, K, V, "f32", 3, 0)
    S64 = host_state(B, HV, V, K, 3)
    state = torch.from_numpy(S64.astype(np.float32)).cuda()
    out = torch.empty((B, HV, V), device="cuda")
    q, k, v = c.views()
    gdn.gdn_decode_step(q, k, v, state, out, H=H, a=c.a, b=c.b, A_log=c.A_log, dt_bias=c.dt_bias)
    o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V)
    assert rel_err(out.cpu().numpy(), o_ref) <= 1e-5


def _gemv_inputs(T, N, Kd, seed):
    import gdn_synth as syn
    x = torch.empty((T, Kd), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((N, Kd), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    syn.fill_normal_(W, seed, syn.Tag.CONV_W, 0, 0.02)
    return x, W


@pytest.mark.parametrize("splits", [16, 4, 1])
def test_projection_waits_that_run_out_leave_y_unwritten_or_nan(splits):
    """The tensor-core projection (two or more token rows) with its give-up limit cut to 64 SM
    cycles, far below one copy's latency: the call returns normally, raises GDN_DEVERR_TIMEOUT,
    and every output is either the correct sum (a CTA whose waits all succeeded) or untouched
    (one or up to 8 K ranges) or NaN (more than 8 ranges: the ranges that gave up write NaN
    partial sums, never sums of stale workspace contents). With the default limit restored the
    same call is exact again, so the context stays usable."""
    T, N, Kd = 2, 5120, 17408
    x, W = _gemv_inputs(T, N, Kd, 41)
    ws = gdn.gemv_workspace(T, N, Kd, splits)
    want = torch.empty((T, N), device="cuda")
    gdn.gdn_gemv_bf16(x, W, want, splits=splits, workspace=ws)
    if ws is not None:
        ws.fill_(3.0)    # stale partial sums that must not reach y
    L = gdn.lib()
    y = torch.full((T, N), 7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = L.gdn_gemv_set_wait_limit(64)
    try:
        gdn.gdn_gemv_bf16(x, W, y, splits=splits, workspace=ws, err_flags=err)
        torch.cuda.synchronize()
    finally:
        L.gdn_gemv_set_wait_limit(old)
    assert int(err.item()) & gdn.GDN_DEVERR_TIMEOUT
    got, ref = y.cpu().numpy(), want.cpu().numpy()
    correct = np.abs(got - ref) <= 1e-5 * np.maximum(1.0, np.abs(ref))
    if splits > 8:
        missing = np.isnan(got)
    else:
        missing = got == 7.0
    assert np.all(correct | missing)
    assert np.any(missing)
    # default limit again: the same call is exact and raises nothing
    err.zero_()
    y.fill_(7.0)
    gdn.gdn_gemv_bf16(x, W, y, splits=splits, workspace=ws, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert rel_err(y.cpu().numpy(), ref) <= 1e-5
