"""The stacked decode under CUDA graphs (independent state pool per layer, inputs drawn on the
device every step from a step counter, all layers' decode calls in one graph), reduced in size:
drift of sampled (layer, slot) pairs against the fp64 oracle replaying every step."""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chained", [True, False])
def test_stacked_graph_decode_matches_the_oracle(chained):
    """Chained: layers after the first go through gdn_decode_step_indexed_chained (programmatic
    dependent launches that overlap the previous layer); unchained: ordinary launches."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    res = bench.stack_decode(layers=3, B=16, H=4, HV=12, K=128, V=128, steps=60, seed=77, pairs=3,
                             heads_per_pair=1, chained=chained)
    assert res["drift"] <= 1e-4, res
    assert res["last_out_err"] <= 2e-2, res
    assert res["dec_ms_per_step"] > 0


def test_full_size_stacked_graph_decode_1000_steps():
    """The full stacked workload: 48 layers x B = 256 x HV = 48 (K = V = 128, about 38.7 GB of
    fp32 state in independent pools), 1000 steps under CUDA graphs with fresh inputs every step,
    drift of 8 sampled (layer, slot) pairs (two q/k heads, six value heads each) against the fp64
    oracle replaying every step: at most 1e-4 on the state, 2e-2 on the last step's bf16 output."""
    res = bench.stack_decode(layers=48, B=256, H=16, HV=48, K=128, V=128, steps=1000, seed=2024,
                             pairs=8, heads_per_pair=2)
    assert res["drift"] <= 1e-4, res
    assert res["last_out_err"] <= 2e-2, res
