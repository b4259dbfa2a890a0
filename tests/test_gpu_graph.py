"""The rollout layer's forward recorded in a CUDA graph (RolloutMoE.capture):
every replay gives the same bits as an eager forward on the same
inputs, also after new inputs are written into the captured buffers, for the
calibrated-channel layer and the online-selection layer (QUADS §3.3 Eq. 21,
Eq. 23-24) at the decode workload's full size (2048 tokens top-8 over 64
experts, hidden 2048, intermediate 768, k = 64)."""
import pytest
import torch

from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def decode():
    import nvfp4_precision_moe_gb300 as nv
    import bench

    nv.load(build=True)
    return bench.build_workload(torch.device(G.DEV), 3)


@pytest.mark.parametrize("online", [False, True])
def test_graph_replay_is_the_eager_forward(decode, online):
    import nvfp4_precision_moe_gb300 as nv

    c, layer, x, logits, w = decode
    if online:
        layer = nv.RolloutMoE(w[0], w[1], layer.S13, layer.Sd, layer.topk, c["T"], online=True)
    xs, ls = x.clone(), logits.clone()  # the captured input buffers
    graph, out = layer.capture(xs, ls)
    g = torch.Generator(device=G.DEV)
    g.manual_seed(3)
    for step in range(3):
        if step:  # new inputs in the captured buffers: other tokens, another routing
            xs.copy_((torch.randn(x.shape, device=G.DEV, generator=g) * (1 + step)).to(torch.bfloat16))
            ls.copy_(logits.roll(step, 1))
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        ref = layer.forward(xs.clone(), ls.clone()).clone()
        torch.cuda.synchronize()
        G.status_ok(layer.dev_status)
        assert torch.equal(got, ref), step
