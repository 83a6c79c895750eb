"""The host-streamed layer (inputs and outputs in pinned host memory, transfers on their
own streams) gives exactly the outputs of the plain device-resident run."""
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from nvfp4_precision_transformer_gb300.linear import HostStreamedLayer, Layer
from synthetic import gaussian

pytestmark = pytest.mark.gpu


def _tensors(M, h, f, seed):
    shapes = [(h, 3 * h), (h, h), (h, f), (f, h)]
    out = []
    for i, (k_in, n_out) in enumerate(shapes):
        out.append((gaussian((M, k_in), 1.0, seed + 10 * i, dtype=torch.bfloat16),
                    gaussian((n_out, k_in), 0.02, seed + 10 * i + 1, dtype=torch.bfloat16),
                    gaussian((M, n_out), 1e-3, seed + 10 * i + 2, dtype=torch.bfloat16),
                    gaussian((n_out,), 0.02, seed + 10 * i + 3, dtype=torch.float32)))
    return out


@pytest.mark.parametrize("recipe", ["fp8_current", "nvfp4"])
def test_streamed_layer_matches_plain_run(recipe):
    M, h, f = 512, 256, 1024
    steps = [_tensors(M, h, f, 100), _tensors(M, h, f, 200)]
    dev_tensors = [tuple(t.to("cuda") for t in tup) for tup in steps[0]]
    layer = Layer(dev_tensors, recipes=(recipe,), rht_signs=0x1357, sr_seed=9)
    host_in = [tuple(torch.empty_like(t).pin_memory() for t in tup) for tup in steps[0]]
    host_out = [tuple(torch.empty_like(b, device="cpu").pin_memory() for b in (l.y, l.dx, l.dw)) for l in layer.linears]
    hs = HostStreamedLayer(layer, host_in, host_out)
    for step in steps:
        for dst, src in zip(host_in, step):
            for d, s in zip(dst, src):
                d.copy_(s)
        hs.step(recipe)
        torch.cuda.synchronize()
        got = [tuple(t.clone() for t in tup) for tup in host_out]
        # plain run on the same inputs
        for lin, (x, w, dy, b) in zip(layer.linears, step):
            lin.x.copy_(x)
            lin.w.copy_(w)
            lin.dy.copy_(dy)
            lin.bias.copy_(b)
        layer.run(recipe)
        torch.cuda.synchronize()
        for lin, (y, dx, dw) in zip(layer.linears, got):
            assert torch.equal(lin.y.cpu(), y) and torch.equal(lin.dx.cpu(), dx) and torch.equal(lin.dw.cpu(), dw)
    assert te.te_get_last_error() == 0
