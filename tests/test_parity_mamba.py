"""GPU parity of mamba_selective_scan_decode (the Mamba-1 selective-scan decode step) against the
fp64 oracle. Tolerances: 1e-5 for fp32 outputs and the fp32 state; 2e-2 for bf16 outputs."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import host_value, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run(B, D, N, dtype="f32", out_dtype="f32", seed=0, steps=1, skip=True, gate=True, functional=False):
    first = syn.mamba_inputs(B, D, N, dtype, seed, 0)
    h = torch.from_numpy(first["h"]).cuda()
    h64 = first["h"].astype(np.float64)
    A = torch.from_numpy(first["A"]).cuda()
    Dskip = torch.from_numpy(first["Dskip"]).cuda() if skip else None
    odt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    worst_y = 0.0
    for step in range(steps):
        m = syn.mamba_inputs(B, D, N, dtype, seed, step)
        dev = {k: to_device(m[k], dtype) for k in ("x", "dt", "Bm", "Cm", "z")}
        y = torch.full((B, D), float("nan"), dtype=odt, device="cuda")
        h_out = torch.full_like(h, float("nan")) if functional else None
        gdn.mamba_selective_scan_decode(dev["x"], dev["dt"], A, dev["Bm"], dev["Cm"], h, y, Dskip=Dskip,
                                        z=dev["z"] if gate else None, h_out=h_out)
        y_ref = oracle.mamba_decode(*(host_value(m[k], dtype) for k in ("x", "dt")), first["A"],
                                    host_value(m["Bm"], dtype), host_value(m["Cm"], dtype), h64,
                                    Dskip=first["Dskip"] if skip else None,
                                    z=host_value(m["z"], dtype) if gate else None)
        got = y.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        worst_y = max(worst_y, rel_err(got, y_ref))
        if functional:
            torch.cuda.synchronize()
            np.testing.assert_array_equal(h.cpu().numpy(), first["h"] if step == 0 else h.cpu().numpy())
            h = h_out
    torch.cuda.synchronize()
    return worst_y, rel_err(h.cpu().numpy(), h64)


@pytest.mark.parametrize("B", [1, 4, 8])
@pytest.mark.parametrize("skip,gate", [(True, True), (False, False), (True, False)])
def test_page_shapes_fp32(B, skip, gate):
    """The decode shapes the Mamba page benchmarks: D = 1536, N = 16, fp32."""
    wy, wh = _run(B, 1536, 16, seed=B, skip=skip, gate=gate)
    assert wy <= 1e-5 and wh <= 1e-5, (wy, wh)


@pytest.mark.parametrize("N", [1, 3, 5, 16, 24, 64, 128])
def test_state_sizes_and_ragged_channels(N):
    """Powers of two use 16-byte accesses; other sizes are masked element by element."""
    wy, wh = _run(3, 37, N, seed=N, steps=3)
    assert wy <= 1e-5 and wh <= 1e-5, (N, wy, wh)


def test_bf16_inputs_and_output():
    wy, wh = _run(8, 1536, 16, dtype="bf16", out_dtype="bf16", seed=11, steps=2)
    assert wy <= 2e-2 and wh <= 1e-5, (wy, wh)


def test_bf16_inputs_fp32_output_many_steps():
    wy, wh = _run(4, 256, 16, dtype="bf16", out_dtype="f32", seed=12, steps=64)
    assert wy <= 1e-5 and wh <= 1e-5, (wy, wh)


def test_new_state_buffer_leaves_the_old_one():
    """With h_out the old state is read only, as in the page's functional API (a fresh new_state
    buffer each call)."""
    wy, wh = _run(2, 64, 16, seed=13, steps=3, functional=True)
    assert wy <= 1e-5 and wh <= 1e-5, (wy, wh)


def test_large_batch():
    wy, wh = _run(256, 1536, 16, seed=14)
    assert wy <= 1e-5 and wh <= 1e-5, (wy, wh)


@pytest.mark.parametrize("B,D,N,dtype,out_dtype,functional", [
    (128, 1536, 64, "f32", "f32", False),    # 3072 blocks of 2 rows x 32 channels: the staged form
    (64, 1536, 128, "bf16", "bf16", False),  # 3072 blocks of 2 rows x 16 channels, bf16 in and out
    (403, 1000, 32, "f32", "f32", True),     # ragged channel and row blocks (1000 / 64, 403 / 2); h_out
    (512, 1536, 16, "f32", "f32", False),    # 3072 blocks of 2 rows x 128 channels
    (514, 1000, 64, "f32", "f32", False),    # 4128 blocks of 4 rows x 32 channels, both edges ragged
    (512, 1536, 64, "bf16", "f32", False),   # 6144 blocks of 4 rows x 32 channels, bf16 inputs
    (48, 1536, 64, "f32", "f32", False),     # 576 blocks: below the staged form, the grid-stride one
])
def test_staged_and_grid_stride_forms(B, D, N, dtype, out_dtype, functional):
    """Batches large enough for the staged form (each block of 2 or 4 batch rows' state bulk-copied
    into shared memory) and for the grid-stride form, over two sequential steps."""
    wy, wh = _run(B, D, N, dtype=dtype, out_dtype=out_dtype, seed=20 + N, steps=2, functional=functional)
    tol = 2e-2 if out_dtype == "bf16" else 1e-5
    assert wy <= tol and wh <= 1e-5, (wy, wh)
