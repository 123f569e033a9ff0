"""Guard bands around every buffer a kernel writes: the stand-in for an out-of-bounds checker.

Each written buffer (state, outputs, rings, conv state, projection outputs and workspaces) is
placed inside a larger allocation whose bytes before and after it hold a canary pattern. After the
call every canary byte must be untouched, and the results must equal, bit for bit, those of the
same call on plain buffers. The cases are the ones whose index arithmetic has ragged edges: the
step's row splits (2, 4, 8 and 16 rows per thread) with a value dimension of 200 (not a multiple
of any row pass), the bf16-state kernel, the pipelined buffered and fused kernels (bulk copies
into shared memory; the fused one in both conv-state layouts), the tensor-core projection (TMA
tiles) at 3, 16 and 17 token rows with ragged output and input counts, and the layer front."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import ssm_recurrent_decode_gb300 as gdn
from gdn_cases import bits_to_torch_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of canary on each side (keeps the buffer 1024-byte aligned)
CANARY = 0xA5


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


class Guarded:
    """A tensor of `shape` and `dtype` at byte offset GUARD inside a canary-filled allocation."""

    def __init__(self, src: torch.Tensor):
        nbytes = src.numel() * src.element_size()
        self.nbytes = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(src.dtype).view(src.shape)
        self.t.copy_(src)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool(torch.all(head == CANARY)) and bool(torch.all(tail == CANARY))


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b)


# ------------------------------------------------------------------------------------------------
# packed / indexed step
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,K,V,sdt,chained", [
    (1, 128, 200, "f32", False),      # 32 tiles: 2 rows per thread, ragged last row pass
    (8, 128, 200, "f32", False),      # 256 tiles: 4 rows per thread
    (16, 128, 200, "f32", False),     # 512 tiles: 8 rows per thread (two CTAs per tile)
    (32, 64, 200, "f32", False),      # K = 64, 1024 tiles: 16 rows per thread
    (32, 128, 128, "bf16", False),    # the bf16-state kernel
    (2, 128, 200, "bf16", False),     # bf16 state through the row split
    (16, 128, 128, "f32", True),      # the chained instance, two CTAs per tile
    (3, 128, 128, "f32", True),       # the chained instance, eight CTAs per tile
])
def test_step_writes_only_its_buffers(B, K, V, sdt, chained):
    H, HV = 16, 32
    seed = 700 + B + K
    num_slots = B + 3
    x = torch.empty((B, 2 * H * K + HV * V), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.QKV, 0, 1.0)
    syn.fill_normal_(a, seed, syn.Tag.A, 0, 0.5)
    syn.fill_normal_(b, seed, syn.Tag.B, 0, 0.5)
    A_log = torch.full((HV,), 0.1, device="cuda")
    dt_bias = torch.zeros(HV, device="cuda")
    state0 = torch.empty((num_slots, HV, V, K), device="cuda")
    syn.fill_normal_(state0, seed, syn.Tag.STATE, 0, 1.0)
    if sdt == "bf16":
        state0 = state0.to(torch.bfloat16)
    idx0 = torch.from_numpy(syn.permutation(seed, num_slots)[:B].copy()).cuda()
    if B > 1:
        idx0[0] = -1                               # a pad row
    out0 = torch.full((B, 1, HV, V), 3.0, dtype=torch.bfloat16, device="cuda")
    q, k, v = gdn.split_mixed_qkv(x, H, HV, K, V)

    plain_state, plain_out = state0.clone(), out0.clone()
    gdn.gdn_decode_step_indexed(q, k, v, plain_state, plain_out, idx0, H=H, a=a, b=b, A_log=A_log,
                                dt_bias=dt_bias)
    gs, go, ge = Guarded(state0), Guarded(out0), Guarded(torch.zeros(1, dtype=torch.int32, device="cuda"))
    gdn.gdn_decode_step_indexed(q, k, v, gs.t, go.t, idx0, H=H, a=a, b=b, A_log=A_log,
                                dt_bias=dt_bias, err_flags=ge.t, chained=chained)
    assert gs.intact() and go.intact() and ge.intact()
    assert _same(gs.t, plain_state) and _same(go.t, plain_out)
    assert int(ge.t.item()) == 0


# ------------------------------------------------------------------------------------------------
# buffered decode, pipelined kernel
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("kernel", ["pipe", "stage"])
@pytest.mark.parametrize("L,start", [(8, 0), (8, 7), (16, 5)])
def test_buffered_pipe_writes_only_its_buffers(L, start, kernel):
    B, H, HV, K, V = 8, 16, 32, 128, 128
    seed = 720 + L + start
    x = torch.empty((B, 2 * H * K + HV * V), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((B, HV), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.QKV, 0, 1.0)
    syn.fill_normal_(a, seed, syn.Tag.A, 0, 0.5)
    syn.fill_normal_(b, seed, syn.Tag.B, 0, 0.5)
    A_log = torch.full((HV,), 0.1, device="cuda")
    dt_bias = torch.zeros(HV, device="cuda")
    state0 = torch.empty((B, HV, V, K), device="cuda")
    syn.fill_normal_(state0, seed, syn.Tag.STATE, 0, 1.0)
    d0 = torch.empty((B, HV, L, V), dtype=torch.bfloat16, device="cuda")
    k0 = torch.empty((B, H, L, K), dtype=torch.bfloat16, device="cuda")
    g0 = torch.empty((B, HV, L), device="cuda")
    syn.fill_normal_(d0, seed, syn.Tag.QKV, 1, 0.1)
    syn.fill_normal_(k0, seed, syn.Tag.QKV, 2, 0.1)
    g0.fill_(-0.05)
    out0 = torch.full((B, 1, HV, V), 3.0, dtype=torch.bfloat16, device="cuda")
    wp = torch.tensor([(start + r) % L for r in range(B)], dtype=torch.int32, device="cuda")
    q, k, v = gdn.split_mixed_qkv(x, H, HV, K, V)
    plain = [t.clone() for t in (state0, out0, d0, k0, g0)]
    gdn.gdn_decode_buffered(q, k, v, plain[0], plain[1], plain[2], plain[3], plain[4], wp, H=H, a=a,
                            b=b, A_log=A_log, dt_bias=dt_bias, kernel=kernel)
    g = [Guarded(t) for t in (state0, out0, d0, k0, g0)]
    ge = Guarded(torch.zeros(1, dtype=torch.int32, device="cuda"))
    gdn.gdn_decode_buffered(q, k, v, g[0].t, g[1].t, g[2].t, g[3].t, g[4].t, wp, H=H, a=a, b=b,
                            A_log=A_log, dt_bias=dt_bias, err_flags=ge.t, kernel=kernel)
    assert all(x.intact() for x in g) and ge.intact()
    for x, p in zip(g, plain):
        assert _same(x.t, p)
    assert int(ge.t.item()) == 0


# ------------------------------------------------------------------------------------------------
# fused decode, pipelined kernel (DS and SD conv-state layouts)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T,kernel", [(4, "pipe"), (9, "pipe"), (4, "stage"), (9, "stage")])
@pytest.mark.parametrize("layout", ["DS", "SD"])
def test_fused_pipe_writes_only_its_buffers(layout, T, kernel):
    heads, D = 96, 128
    dim = heads * D
    seed = 740 + T
    num_slots = T + 8
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    state0 = torch.empty((num_slots, heads, D, D), device="cuda")
    syn.fill_normal_(state0, seed, syn.Tag.STATE, 0, 1.0)
    cs_ds = bits_to_torch_bf16(ins["conv_state"])                   # [slots, 3*dim, 3]
    cs_phys = cs_ds.clone() if layout == "DS" else cs_ds.transpose(1, 2).contiguous()
    view = (lambda t: t) if layout == "DS" else (lambda t: t.transpose(1, 2))
    x = torch.empty((T, 3 * dim), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    gate = torch.empty((T, heads, D), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(gate, seed, syn.Tag.OUT_GATE, 0, 1.0)
    idx = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
    if T > 1:
        idx[1] = 0                                                  # a pad row (NULL slot 0)
    common = dict(conv_w=torch.from_numpy(ins["conv_w"]).cuda(),
                  raw_g=bits_to_torch_bf16(ins["raw_g"]), raw_beta=bits_to_torch_bf16(ins["raw_beta"]),
                  A_log=torch.from_numpy(ins["A_log"]).cuda(), dt_bias=torch.from_numpy(ins["dt_bias"]).cuda(),
                  norm_w=torch.from_numpy(ins["norm_w"]).cuda())
    out0 = torch.full((T, heads, D), 3.0, dtype=torch.bfloat16, device="cuda")

    def call(state, cs, out, err=None):
        gdn.gdn_decode_fused(x, common["conv_w"], view(cs), common["raw_g"], common["raw_beta"],
                             common["A_log"], common["dt_bias"], state, idx, gate, common["norm_w"], out,
                             pad_slot_id=0, err_flags=err, kernel=kernel)

    plain = [state0.clone(), cs_phys.clone(), out0.clone()]
    call(*plain)
    g = [Guarded(t) for t in (state0, cs_phys, out0)]
    ge = Guarded(torch.zeros(1, dtype=torch.int32, device="cuda"))
    call(g[0].t, g[1].t, g[2].t, ge.t)
    assert all(x.intact() for x in g) and ge.intact()
    for x_, p in zip(g, plain):
        assert _same(x_.t, p)
    assert int(ge.t.item()) == 0


# ------------------------------------------------------------------------------------------------
# decode projection (tensor-core form from two token rows; CUDA-core form at one)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T,N,Kd,splits", [
    (3, 1000, 1000, 0),        # ragged outputs (not a multiple of 128) and inputs (of 128)
    (16, 1000, 5128, 4),       # ranges added inside a cluster
    (17, 5120, 1000, 12),      # two passes of token rows, partial sums in a workspace
    (1, 1000, 1000, 3),        # the CUDA-core form
])
def test_projection_writes_only_its_buffers(T, N, Kd, splits):
    seed = 760 + T
    x = torch.empty((T, Kd), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((N, Kd), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    syn.fill_normal_(W, seed, syn.Tag.CONV_W, 0, 0.02)
    y0 = torch.full((T, N), 3.0, device="cuda")
    ws0 = gdn.gemv_workspace(T, N, Kd, splits)
    plain_y = y0.clone()
    gdn.gdn_gemv_bf16(x, W, plain_y, splits=splits, workspace=None if ws0 is None else ws0.clone())
    gy = Guarded(y0)
    gw = None if ws0 is None else Guarded(ws0)
    ge = Guarded(torch.zeros(1, dtype=torch.int32, device="cuda"))
    gdn.gdn_gemv_bf16(x, W, gy.t, splits=splits, workspace=None if gw is None else gw.t, err_flags=ge.t)
    assert gy.intact() and ge.intact() and (gw is None or gw.intact())
    assert _same(gy.t, plain_y)
    assert int(ge.t.item()) == 0


# ------------------------------------------------------------------------------------------------
# layer front (projection -> fused decode -> projection)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 3])
def test_front_writes_only_its_buffers(T):
    hidden, heads, D = 512, 4, 64
    dim = heads * D
    seed = 780 + T
    P = gdn.front_proj_width(heads, D, "gdn")
    num_slots = T + 4
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    W_in = torch.empty((P, hidden), dtype=torch.bfloat16, device="cuda")
    W_out = torch.empty((hidden, dim), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(W_in, seed, syn.Tag.CONV_W, 1, hidden ** -0.5)
    syn.fill_normal_(W_out, seed, syn.Tag.CONV_W, 2, dim ** -0.5)
    x = torch.empty((T, hidden), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    state0 = torch.empty((num_slots, heads, D, D), device="cuda")
    syn.fill_normal_(state0, seed, syn.Tag.STATE, 0, 1.0)
    cs0 = bits_to_torch_bf16(ins["conv_state"]).clone()
    z0 = torch.zeros((T, P), dtype=torch.bfloat16, device="cuda")
    o0 = torch.zeros((T, dim), dtype=torch.bfloat16, device="cuda")
    y0 = torch.full((T, hidden), 3.0, device="cuda")
    idx = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
    conv_w = torch.from_numpy(ins["conv_w"]).cuda()
    A_log = torch.from_numpy(ins["A_log"]).cuda()
    dtb = torch.from_numpy(np.ascontiguousarray(ins["dt_bias"][:heads])).cuda()
    norm_w = torch.from_numpy(ins["norm_w"]).cuda()

    def call(z, o, y, cs, state, err=None):
        gdn.gdn_decode_front(x, W_in, W_out, z, o, y, conv_w, cs, A_log, dtb, state, idx, norm_w,
                             pad_slot_id=0, gate_kind="gdn", err_flags=err)

    plain = [t.clone() for t in (z0, o0, y0, cs0, state0)]
    call(*plain)
    g = [Guarded(t) for t in (z0, o0, y0, cs0, state0)]
    ge = Guarded(torch.zeros(1, dtype=torch.int32, device="cuda"))
    call(*(x_.t for x_ in g), err=ge.t)
    assert all(x_.intact() for x_ in g) and ge.intact()
    for x_, p in zip(g, plain):
        assert _same(x_.t, p)
    assert int(ge.t.item()) == 0


def test_guard_helper_detects_a_write_into_the_band():
    """The helper itself: a byte written just past the buffer is seen (a host-side write through
    the raw allocation, not a kernel)."""
    g = Guarded(torch.zeros(16, dtype=torch.float32, device="cuda"))
    assert g.intact()
    g.raw[GUARD + 64] = 0
    assert not g.intact()


# ------------------------------------------------------------------------------------------------
# Mamba-1 decode (the second recurrence)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,D,N,in_place", [(3, 96, 64, True), (5, 40, 16, False), (2, 33, 48, True),
                                            (4, 64, 128, False),
                                            (128, 1536, 64, True), (403, 1000, 32, False),  # staged, 2 rows
                                            (514, 1000, 64, True),                          # staged, 4 rows
                                            (48, 1536, 64, False)])                         # grid-stride
def test_mamba_writes_only_its_buffers(B, D, N, in_place):
    m = syn.mamba_inputs(B, D, N, "f32", 900 + N)
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in m.items()}
    y0 = torch.full((B, D), 3.0, device="cuda")
    h_out0 = torch.full((B, D, N), 3.0, device="cuda")

    def call(h, y, h_out):
        gdn.mamba_selective_scan_decode(t["x"], t["dt"], t["A"], t["Bm"], t["Cm"], h, y, Dskip=t["Dskip"],
                                        z=t["z"], h_out=None if in_place else h_out)

    plain = [t["h"].clone(), y0.clone(), h_out0.clone()]
    call(*plain)
    g = [Guarded(x_) for x_ in (t["h"], y0, h_out0)]
    call(*(x_.t for x_ in g))
    assert all(x_.intact() for x_ in g)
    for x_, p in zip(g, plain):
        assert _same(x_.t, p)
