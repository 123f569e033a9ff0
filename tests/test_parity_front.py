"""GPU parity of gdn_decode_front (input projection -> conv update, delta step, gated RMSNorm ->
output projection) against the fp64 oracle's composition of the same steps.

Both sides round the projection output z and the normalised output o to bf16, the dtype the front
stores them in. The GPU computes z in fp32 (error ~1e-6 relative), so an element of z or o next to
a bf16 rounding midpoint may land on the other neighbour than the oracle's: one bf16 ulp (2^-8
relative) of that element. Through the step and the output projection (weights of size
dim^-1/2) such a flip moves y and the state by at most ~1e-4 relative; the bars are 2e-3 for the
fp32 y and the state, and 1e-2 for the bf16 conv state (which holds z's rounded values). A value
read from the wrong column of z, or a dropped stage, is off by O(1)."""
import numpy as np
import pytest
import torch

import gdn_synth as syn
import oracle
import ssm_recurrent_decode_gb300 as gdn
from conftest import rel_err
from gdn_cases import bits_to_torch_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _weights(P, hidden, dim, seed):
    """Synthetic projection weights N(0, 1/fan_in), bf16."""
    W_in = torch.empty((P, hidden), dtype=torch.bfloat16, device="cuda")
    W_out = torch.empty((hidden, dim), dtype=torch.bfloat16, device="cuda")
    syn.fill_normal_(W_in, seed, syn.Tag.CONV_W, 1, hidden ** -0.5)
    syn.fill_normal_(W_out, seed, syn.Tag.CONV_W, 2, dim ** -0.5)
    return W_in, W_out


def _run_front(T, hidden, heads, D, *, gate_kind="gdn", seed=0, steps=1, pad_rows=(), kernel="auto",
               y_dtype=torch.float32, in_splits=0, out_splits=0, x_pitch=None):
    dim = heads * D
    P = gdn.front_proj_width(heads, D, gate_kind)
    num_slots = T + 4
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    dt_bias = np.ascontiguousarray(ins["dt_bias"] if gate_kind == "kda" else ins["dt_bias"][:heads])
    W_in, W_out = _weights(P, hidden, dim, seed)
    W_in64, W_out64 = W_in.float().cpu().numpy(), W_out.float().cpu().numpy()
    state = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device="cuda")
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
    S64 = state.cpu().numpy().astype(np.float64)
    conv_state = bits_to_torch_bf16(ins["conv_state"]).clone()
    cs64 = syn.bf16_bits_to_f32(ins["conv_state"]).astype(np.float64).reshape(num_slots, 3 * dim, 3)
    idx_np = np.arange(1, T + 1, dtype=np.int32)             # slot 0 is the NULL (pad) slot
    for r in pad_rows:
        idx_np[r] = 0
    idx = torch.from_numpy(idx_np).cuda()
    conv_w = torch.from_numpy(ins["conv_w"]).cuda()
    A_log = torch.from_numpy(ins["A_log"]).cuda()
    dtb = torch.from_numpy(dt_bias).cuda()
    norm_w = torch.from_numpy(ins["norm_w"]).cuda()
    z = torch.empty((T, P), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((T, dim), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst = {"y": 0.0}
    for step in range(steps):
        xb = torch.empty((T, x_pitch or hidden), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(xb, seed, syn.Tag.X, step, 1.0)
        x = xb[:, :hidden]
        y = torch.full((T, hidden), float("nan"), dtype=y_dtype, device="cuda")
        gdn.gdn_decode_front(x, W_in, W_out, z, o, y, conv_w, conv_state, A_log, dtb, state, idx,
                             norm_w, pad_slot_id=0, gate_kind=gate_kind, err_flags=err,
                             kernel=kernel, in_splits=in_splits, out_splits=out_splits)
        y_ref, bad = oracle.decode_front(x.float().cpu().numpy(), W_in64, W_out64, ins["conv_w"],
                                         cs64, ins["A_log"], dt_bias, S64, ins["norm_w"],
                                         heads=heads, D=D, idx=idx_np, pad_slot=0,
                                         gate_kind=gate_kind)
        assert bad == 0
        got = y.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        worst["y"] = max(worst["y"], rel_err(got, y_ref))
    torch.cuda.synchronize()
    slots = idx_np[idx_np != 0]
    worst["state"] = rel_err(state.cpu().numpy()[slots], S64[slots])
    worst["conv"] = rel_err(conv_state.float().cpu().numpy()[slots], cs64[slots])
    assert int(err.item()) == 0
    return worst


def _ok(w, y_bar=2e-3):
    return w["y"] <= y_bar and w["state"] <= 2e-3 and w["conv"] <= 1e-2


@pytest.mark.parametrize("kernel", ["auto", "tile"])
def test_layer_shapes_gdn(kernel):
    """hidden 5120 (the Optimization Log's model width), 32 heads x 128, two steps; "auto" takes
    the pipelined fused kernel."""
    w = _run_front(2, 5120, 32, 128, seed=1, steps=2, kernel=kernel)
    assert _ok(w), w


def test_layer_shapes_kda_gate():
    w = _run_front(3, 5120, 16, 128, gate_kind="kda", seed=2, steps=2)
    assert _ok(w), w


@pytest.mark.parametrize("heads,D", [(4, 32), (2, 64)])
@pytest.mark.parametrize("gate_kind", ["gdn", "kda"])
def test_small_shapes_with_a_pad_row(heads, D, gate_kind):
    w = _run_front(4, 256, heads, D, gate_kind=gate_kind, seed=3 + D, steps=3, pad_rows=(1,))
    assert _ok(w), w


@pytest.mark.parametrize("in_splits,out_splits", [(1, 1), (8, 3)])
def test_explicit_splits_bf16_output_and_row_view(in_splits, out_splits):
    w = _run_front(5, 512, 4, 64, seed=9, steps=2, in_splits=in_splits, out_splits=out_splits,
                   y_dtype=torch.bfloat16, x_pitch=640)
    assert _ok(w, y_bar=2e-2), w          # bf16 y: its own rounding, 2^-8 relative


@pytest.mark.parametrize("T", [1, 3, 12])
def test_graph_replay_matches_eager_calls(T):
    """The chained launches of one call (programmatic dependent launch) become graph edges under
    capture; replaying the captured call gives the same bits as eager calls, step after step, for
    the one-row projection (T = 1), the tensor-core projection (T = 3) and the pipelined fused
    kernel (T = 12: 384 (token, head) tiles)."""
    hidden, heads, D, steps = 512, 32, 128, 3
    dim = heads * D
    P = gdn.front_proj_width(heads, D, "gdn")
    num_slots = T + 4
    ins = syn.fused_inputs(T, heads, D, num_slots, 21)
    W_in, W_out = _weights(P, hidden, dim, 21)
    conv_w = torch.from_numpy(ins["conv_w"]).cuda()
    A_log = torch.from_numpy(ins["A_log"]).cuda()
    dtb = torch.from_numpy(np.ascontiguousarray(ins["dt_bias"][:heads])).cuda()
    norm_w = torch.from_numpy(ins["norm_w"]).cuda()
    idx = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
    S0 = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device="cuda")
    syn.fill_normal_(S0, 21, syn.Tag.STATE, 0, 1.0)
    cs0 = bits_to_torch_bf16(ins["conv_state"]).clone()
    xs = []
    for step in range(steps):
        xb = torch.empty((T, hidden), dtype=torch.bfloat16, device="cuda")
        syn.fill_normal_(xb, 21, syn.Tag.X, step, 1.0)
        xs.append(xb)
    runs = []
    for graphed in (False, True):
        state, cs = S0.clone(), cs0.clone()
        x = torch.empty((T, hidden), dtype=torch.bfloat16, device="cuda")
        z = torch.empty((T, P), dtype=torch.bfloat16, device="cuda")
        o = torch.empty((T, dim), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((T, hidden), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")

        def call():
            gdn.gdn_decode_front(x, W_in, W_out, z, o, y, conv_w, cs, A_log, dtb, state, idx,
                                 norm_w, pad_slot_id=0, gate_kind="gdn", err_flags=err)

        graph = None
        if graphed:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                call()
            torch.cuda.current_stream().wait_stream(side)
        ys = []
        for step in range(steps):
            x.copy_(xs[step])
            graph.replay() if graph is not None else call()
            ys.append(y.clone())
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        runs.append(ys + [state, cs])
    for a_, b_ in zip(*runs):
        assert torch.equal(a_, b_)
