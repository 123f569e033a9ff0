"""GPU parity of gdn_gemv_bf16 (the decode projection) against the fp64 oracle, at the shapes the
Optimization Log lists for decode ([5120, 17408] and [17408, 5120]). Both sides see the same bf16
values; the GPU accumulates in fp32: fp32 outputs within 1e-5, bf16 outputs within 2e-2."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _inputs(T, N, Kd, seed):
    x = torch.empty((T, Kd), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((N, Kd), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    syn.fill_normal_(W, seed, syn.Tag.CONV_W, 0, 0.02)
    return x, W


def _check(T, N, Kd, seed, out_dtype=torch.float32, splits=0):
    x, W = _inputs(T, N, Kd, seed)
    y = torch.full((T, N), float("nan"), dtype=out_dtype, device="cuda")
    ws = gdn.gemv_workspace(T, N, Kd, splits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_gemv_bf16(x, W, y, splits=splits, workspace=ws, err_flags=err)
    ref = oracle.gemv(x.float().cpu().numpy(), W.float().cpu().numpy())
    got = y.float().cpu().numpy()
    assert int(err.item()) == 0
    assert np.all(np.isfinite(got))
    return rel_err(got, ref)


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("N,Kd", [(17408, 5120), (5120, 17408)])
def test_page_shapes(T, N, Kd):
    assert _check(T, N, Kd, seed=T) <= 1e-5


def test_bf16_output():
    assert _check(2, 17408, 5120, seed=3, out_dtype=torch.bfloat16) <= 2e-2


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("splits", [1, 2, 5, 8, 16])
def test_explicit_splits_and_ragged_inputs(splits, T):
    """N = 300 and Kd = 1000 are not multiples of the row and input tiles. 2, 5 and 8 ranges are
    added inside a thread-block cluster, 16 in a workspace (some of them empty: zeros); T = 1 runs
    the CUDA-core form, T = 3 the tensor-core one."""
    assert _check(T, 300, 1000, seed=10 + splits + T, splits=splits) <= 1e-5


@pytest.mark.parametrize("T", [2, 3, 5, 16, 17])
def test_token_counts_of_the_tensor_core_form(T):
    """From 2 token rows on, the tensor-core form with 16 token columns per pass: partly filled
    (2, 3, 5), full (16), and a second pass of one token row (17)."""
    assert _check(T, 17408 if T < 16 else 1000, 5120 if T < 16 else 2048, seed=30 + T) <= 1e-5


@pytest.mark.parametrize("T,splits", [(8, 1), (1, 1), (6, 2)])
def test_long_k_ranges(T, splits):
    """K ranges of 17408 and 8704 inputs: the tensor-core form cycles its shared-memory ring about
    70 and 35 times; at one token row the x slice (34 KB) is too large to stage and is read through
    L1."""
    assert _check(T, 640, 17408, seed=40 + T, splits=splits) <= 1e-5


def test_twelve_token_rows():
    """T = 12: one pass of the tensor-core form with 12 of its 16 token columns."""
    assert _check(12, 1000, 2048, seed=21) <= 1e-5


def test_row_views_and_missing_workspace():
    T, N, Kd = 4, 256, 512
    x, W = _inputs(T, N, 2 * Kd, 22)
    xv = x[:, Kd:]                                  # a row view with stride 2 * Kd
    Wd = W[:, :Kd].contiguous()
    y = torch.empty((T, N), device="cuda")
    gdn.gdn_gemv_bf16(xv, Wd, y, splits=1)
    ref = oracle.gemv(xv.float().cpu().numpy(), Wd.float().cpu().numpy())
    assert rel_err(y.cpu().numpy(), ref) <= 1e-5
    with pytest.raises(gdn.GdnError):
        gdn.gdn_gemv_bf16(xv, Wd, y, splits=12)     # more than 8 ranges need a workspace
