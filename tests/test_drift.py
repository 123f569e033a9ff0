"""Long-run drift: 1000 sequential decode steps on the GPU and in the fp64 oracle, each side on its
own state, with fresh seeded inputs every step. The fp32 state must stay within 1e-4 of the
oracle's (max |gpu - oracle| / max(1, |oracle|)) and every step's output within the per-step
tolerance; a state stored in bf16 is held to the bf16 bar, 2e-2."""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import PackedCase, host_state

pytestmark = pytest.mark.gpu

STEPS = 1000


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("shape,dtype,out_tol,state_dtype,drift_tol", [
    ((2, 2, 4, 16, 16), "f32", 1e-5, "f32", 1e-4),          # the tiny decode, fp32 everywhere
    ((2, 16, 32, 128, 128), "bf16", 2e-2, "f32", 1e-4),     # the packed shapes, bf16 in and out
    ((2, 16, 32, 128, 128), "bf16", 2e-2, "bf16", 2e-2),    # ... with the state stored in bf16
])
def test_thousand_step_drift(shape, dtype, out_tol, state_dtype, drift_tol):
    B, H, HV, K, V = shape
    seed = 900 + K
    state = torch.from_numpy(host_state(B, HV, V, K, seed).astype(np.float32)).cuda()
    if state_dtype == "bf16":
        state = state.to(torch.bfloat16)
    S64 = state.float().cpu().numpy().astype(np.float64)
    idx_np = np.arange(B, dtype=np.int32)[::-1].copy()
    idx = torch.from_numpy(idx_np).cuda()
    odt = torch.bfloat16 if dtype == "bf16" else torch.float32
    worst_out, drift_curve = 0.0, []
    for step in range(STEPS):
        c = PackedCase(B, H, HV, K, V, dtype, seed, step)
        out = torch.empty((B, 1, HV, V), dtype=odt, device="cuda")
        q, k, v = c.views()
        gdn.gdn_decode_step_indexed(q, k, v, state, out, idx, H=H, a=c.a, b=c.b, A_log=c.A_log,
                                    dt_bias=c.dt_bias)
        o_ref, _ = oracle.gdn_step_packed(*c.oracle_args(), S64, H=H, HV=HV, K=K, V=V, idx=idx_np,
                                          state_bf16=(state_dtype == "bf16"))
        worst_out = max(worst_out, rel_err(out.float().cpu().numpy().reshape(B, HV, V), o_ref))
        if step % 100 == 99:
            drift_curve.append(rel_err(state.float().cpu().numpy(), S64))
    assert worst_out <= out_tol, worst_out
    assert drift_curve[-1] <= drift_tol, drift_curve
    # the delta rule contracts: the error does not grow without bound over the run
    assert max(drift_curve) <= drift_tol, drift_curve
