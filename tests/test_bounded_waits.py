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
