"""gdn_gemv_bf16_noalloc: the decode projection for callers that cannot allocate device memory
(code that only receives raw pointers from a framework owning every allocation, serving loops that
must never call cudaMalloc, fixed memory budgets). With more K ranges than one thread-block
cluster holds (8), its split-K partial sums live in a buffer the library holds itself. Called through the C ABI twice in a row, on two different shapes, it must
give what gdn_gemv_bf16 with a caller workspace gives, within the fp32 tolerance of the other
tests; a request larger than its buffer is refused before anything runs.

This file is collected last on purpose: it runs after every other GPU test, and also passes on its
own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import gdn_synth as syn
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err

pytestmark = pytest.mark.gpu

GDN_ERR_SCRATCH = -7
MAX_FLOATS = 1 << 20


def _args(x, W, y, splits=0):
    g = gdn.GemvArgs()
    g.T, g.N, g.Kd = x.shape[0], W.shape[0], x.shape[1]
    g.out_dtype = gdn.GDN_F32 if y.dtype == torch.float32 else gdn.GDN_BF16
    g.x, g.x_stride = x.data_ptr(), x.stride(0)
    g.W = W.data_ptr()
    g.y, g.y_stride = y.data_ptr(), y.stride(0)
    g.splits = splits
    return g


def _noalloc(x, W, y, splits=0):
    L = gdn.lib()
    fn = L.gdn_gemv_bf16_noalloc
    fn.argtypes = [ctypes.POINTER(gdn.GemvArgs), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    g = _args(x, W, y, splits)
    return fn(ctypes.byref(g), torch.cuda.current_stream().cuda_stream)


def _inputs(T, N, Kd, seed):
    x = torch.empty((T, Kd), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((N, Kd), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    syn.fill_normal_(W, seed, syn.Tag.CONV_W, 0, 0.02)
    return x, W


def test_no_alloc_gemv_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    # [N, Kd] of the projections listed for decode: two calls with more than 8 K ranges (the
    # buffer is used), then one with the library's choice (ranges added inside a cluster)
    shapes = [(4, 17408, 5120, 31, 12), (3, 5120, 17408, 32, 16), (2, 5120, 17408, 34, 0)]
    for T, N, Kd, seed, splits in shapes:
        x, W = _inputs(T, N, Kd, seed)
        uses_buffer = gdn.lib().gdn_gemv_workspace_bytes(T, N, splits) > 0
        assert uses_buffer == (splits > 8)
        want = torch.empty((T, N), device="cuda")
        gdn.gdn_gemv_bf16(x, W, want, splits=splits, workspace=gdn.gemv_workspace(T, N, Kd, splits))
        got = torch.full((T, N), float("nan"), device="cuda")
        assert _noalloc(x, W, got, splits) == 0
        torch.cuda.synchronize()
        assert np.all(np.isfinite(got.cpu().numpy()))
        assert rel_err(got.cpu().numpy(), want.cpu().numpy()) <= 1e-5


def test_no_alloc_gemv_refuses_more_than_its_buffer():
    T, N, Kd, splits = 8, 65536, 1024, 16         # 16 * 8 * 65536 fp32 partial sums > 1 Mi
    assert splits * T * N > MAX_FLOATS
    x, W = _inputs(T, N, Kd, 33)
    y = torch.full((T, N), 7.0, device="cuda")
    assert _noalloc(x, W, y, splits=splits) == GDN_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert "scratch" in gdn.gdn_strerror(GDN_ERR_SCRATCH)
    # with one K range the call needs no buffer and runs
    assert _noalloc(x[:1], W[:1024], y[:1, :1024], splits=1) == 0


def test_no_alloc_gemv_reserves_no_device_memory_after_its_first_call():
    """The first call in a process may make the driver load this library's device code (with
    lazy module loading) and so place the fixed buffer; a later call changes no device memory
    reservation: the free bytes cudaMemGetInfo reports stay the same across it."""
    T, N, Kd, splits = 4, 17408, 5120, 12
    x, W = _inputs(T, N, Kd, 35)
    y = torch.empty((T, N), device="cuda")
    assert _noalloc(x, W, y, splits) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _noalloc(x, W, y, splits) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_no_alloc_gemv_that_gives_up_a_wait_writes_nan_not_the_previous_sums():
    """The shared buffer keeps the previous call's partial sums. When the tensor-core kernel gives
    up a bounded wait (its limit cut to 64 cycles with the library's test hook), the affected
    outputs must come out NaN, not sums of that previous call's contents."""
    T, N, Kd, splits = 2, 5120, 17408, 16
    x, W = _inputs(T, N, Kd, 36)
    want = torch.empty((T, N), device="cuda")
    assert _noalloc(x, W, want, splits) == 0      # fills the buffer with this call's sums
    x2 = x * 2                                      # a different call: every sum doubles
    L = gdn.lib()
    y = torch.full((T, N), 7.0, device="cuda")
    old = L.gdn_gemv_set_wait_limit(64)
    try:
        assert _noalloc(x2, W, y, splits) == 0
        torch.cuda.synchronize()
    finally:
        L.gdn_gemv_set_wait_limit(old)
    got, ref = y.cpu().numpy(), 2 * want.cpu().numpy()
    done = np.abs(got - ref) <= 1e-5 * np.maximum(1.0, np.abs(ref))
    assert np.all(done | np.isnan(got))
    assert np.any(np.isnan(got))
    # default limit: exact again
    assert _noalloc(x2, W, y, splits) == 0
    torch.cuda.synchronize()
    assert rel_err(y.cpu().numpy(), ref) <= 1e-5
