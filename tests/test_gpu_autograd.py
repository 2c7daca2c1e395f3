"""layer.MoEFunction, the torch.autograd wrapper: its gradients are the ones a
direct moe_backward call gives (bitwise: the same kernels on the same inputs),
in the parameters' dtypes."""
import pytest
import torch

from moe_layer_gb300 import _abi, layer
from synth.inputs import MoEShape, make_inputs

from .helpers import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ensure_lib()


@pytest.mark.parametrize("n_shared", [1, 0])
def test_autograd_function_matches_the_direct_calls(n_shared):
    s = MoEShape(T=300, d=256, I=192, E=6, k=2, n_shared=n_shared, I_shared=128 if n_shared else 0,
                 w_std=0.05)
    inp = make_inputs(s, seed=4, device="cuda")
    cfg = _abi.make_config(s.T, s.d, s.I, s.E, s.k, s.n_shared, s.I_shared)

    bufs = layer.MoEBuffers(cfg)
    y_ref = layer.forward(cfg, inp, bufs)
    g_ref = layer.alloc_grads(cfg, with_topk=False)
    dx_ref = layer.backward(cfg, inp, inp["dy"], bufs, g_ref)

    names = ["x", "W_router", "W_gate", "W_up", "W_down"] + (["Ws_gate", "Ws_up", "Ws_down"] if n_shared else [])
    leaves = {n: inp[n].detach().clone().requires_grad_(True) for n in names}
    y = layer.MoEFunction.apply(cfg, layer.MoEBuffers(cfg), leaves["x"], leaves["W_router"], leaves["W_gate"],
                                leaves["W_up"], leaves["W_down"], leaves.get("Ws_gate"), leaves.get("Ws_up"),
                                leaves.get("Ws_down"), inp.get("router_bias"), None)
    y.backward(inp["dy"])
    torch.cuda.synchronize()

    assert torch.equal(y.detach(), y_ref)
    assert torch.equal(leaves["x"].grad, dx_ref)
    for n in names[1:]:
        ref = g_ref["d" + n]
        assert leaves[n].grad.dtype == leaves[n].dtype, n
        assert torch.equal(leaves[n].grad, ref.to(leaves[n].dtype)), n
