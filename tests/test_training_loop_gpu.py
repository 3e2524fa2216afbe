"""The unit inside a training loop: autograd accumulates every emulated
rank's gradients straight into that rank's flat gradient buffer (the
parameters' .grad are views of it, as FlatParameter gradients are), the
step updates the shards and gathers them, and the model reads its
parameters as views of the gathered buffer. Two steps of a small two-layer
model, checked against plain torch autograd and the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import host

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sharded_fsdp_reduce_gb300 as F
    return F


def forward(params, x):
    h = torch.relu(x @ params["w1"] + params["b1"])
    return (h @ params["w2"] + params["b2"]).float().pow(2).mean()


def test_gradients_land_in_the_flat_buffers_and_the_model_reads_the_gather(F, orc):
    world = 2
    shapes = [("w1", (64, 96)), ("b1", (96,)), ("w2", (96, 32)), ("b2", (32,))]
    unit = F.FlatParamUnit(shapes, world, torch.bfloat16, torch.bfloat16, device=DEV)
    g = torch.Generator().manual_seed(3)
    init = [(torch.rand(s, generator=g) * 0.2 - 0.1) for _, s in shapes]
    unit.load_master([t.to(DEV) for t in init])
    unit.shard_out.copy_(unit.master.to(torch.bfloat16))
    unit.all_gather()  # the compute copy before the first forward
    model = unit.param_views(unit.full[0])  # the model's parameters: views of rank 0's gathered buffer
    p_o = host(unit.master).copy()
    m_o, v_o = np.zeros_like(p_o), np.zeros_like(p_o)
    for t in (1, 2):
        xs = [torch.randn(16, 64, generator=g).to(DEV, torch.bfloat16) for _ in range(world)]
        ref_grads = []
        for r in range(world):
            # rank r: leaves that read the gathered parameters, with .grad set
            # to views of rank r's flat gradient buffer (zeroed)
            unit.grads[r].zero_()
            gviews = unit.param_views(unit.grads[r])
            leaves = {n: model[n].detach().requires_grad_(True) for n, _ in shapes}
            for n, _ in shapes:
                leaves[n].grad = gviews[n]
            forward(leaves, xs[r]).backward()
            for n, _ in shapes:  # autograd accumulated into the flat buffer in place
                assert leaves[n].grad.data_ptr() == gviews[n].data_ptr()
            # the same gradients by plain autograd, for comparison
            fresh = {n: model[n].detach().clone().requires_grad_(True) for n, _ in shapes}
            forward(fresh, xs[r]).backward()
            ref_grads.append(torch.cat([fresh[n].grad.reshape(-1) for n, _ in shapes]))
            assert torch.equal(unit.grads[r][:unit.numel], ref_grads[r])
            assert not unit.grads[r][unit.numel:].any()  # the pad receives nothing
        before = model["w1"].clone()
        unit.step(F.AdamWHParams(1e-2, weight_decay=0.01, step=t), gathers=1)
        orc.fsdp_step([host(gr) for gr in unit.grads], "bf16", world, p_o, m_o, v_o, "bf16",
                      orc.hparams(1e-2, 0.9, 0.999, 1e-8, 0.01, t))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(unit.master).view(np.uint32), p_o.view(np.uint32))
        assert not torch.equal(model["w1"], before)  # the model sees the gathered update
        assert torch.equal(model["w1"].reshape(-1), unit.shard_out[:64 * 96])
