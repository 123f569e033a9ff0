"""The stacked decode under CUDA graphs (independent state pool per layer, inputs drawn on the
device every step from a step counter, all layers' decode calls in one graph), reduced in size:
drift of sampled (layer, slot) pairs against the fp64 oracle replaying every step."""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def test_stacked_graph_decode_matches_the_oracle():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    res = bench.stack_decode(layers=3, B=16, H=4, HV=12, K=128, V=128, steps=60, seed=77, pairs=3,
                             heads_per_pair=1)
    assert res["drift"] <= 1e-4, res
    assert res["last_out_err"] <= 2e-2, res
    assert res["dec_ms_per_step"] > 0
