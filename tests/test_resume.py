"""Checkpoint and resume of the buffered decode: the checkpoint tiles, the three rings and the
cursors are the whole resumable state ("Microbenchmark: buffered output-only GDN decode", module
docstring: the ring folds into the checkpoint). A snapshot taken mid-cycle and restored into fresh
buffers continues bit for bit like the uninterrupted run (the kernels are deterministic)."""
import numpy as np
import pytest
import torch

import ssm_recurrent_decode_gb300 as gdn
from gdn_cases import PackedCase, host_state

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["tile", "pipe"])
def test_snapshot_mid_cycle_resumes_bit_identically(kernel):
    assert torch.cuda.is_available()
    B, H, HV, K, V, L = 8, 4, 8, 128, 128, 8
    state = torch.from_numpy(host_state(B, HV, V, K, 600).astype(np.float32)).cuda()
    rings = [torch.zeros((B, HV, L, V), dtype=torch.bfloat16, device="cuda"),
             torch.zeros((B, H, L, K), dtype=torch.bfloat16, device="cuda"),
             torch.zeros((B, HV, L), device="cuda")]
    cases = [PackedCase(B, H, HV, K, V, "bf16", 600, s) for s in range(2 * L)]

    def run(st, rg, steps, start):
        outs = []
        for s in steps:
            c = cases[s]
            q, k, v = c.views()
            out = torch.empty((B, HV, V), dtype=torch.bfloat16, device="cuda")
            wp = torch.full((B,), (start + s) % L, dtype=torch.int32, device="cuda")
            gdn.gdn_decode_buffered(q, k, v, st, out, *rg, wp, H=H, a=c.a, b=c.b, A_log=c.A_log,
                                    dt_bias=c.dt_bias, kernel=kernel)
            outs.append(out.clone())
        return outs

    run(state, rings, range(5), 0)                        # five steps: cursor now at 5 of 8
    snap = (state.clone(), [r.clone() for r in rings])
    cont = run(state, rings, range(5, 2 * L), 0)          # through a flush and into the next cycle
    state2, rings2 = snap[0].clone(), [r.clone() for r in snap[1]]
    resumed = run(state2, rings2, range(5, 2 * L), 0)
    torch.cuda.synchronize()
    for a, b in zip(cont, resumed):
        assert torch.equal(a, b)
    assert torch.equal(state, state2)
    for a, b in zip(rings, rings2):
        assert torch.equal(a, b)
