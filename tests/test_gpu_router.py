"""The router projection (logits = x . W_r, and its backward) through the C ABI
against the oracle: standalone on seeded inputs, and in front of the whole
layer (route, forward, backward) on inputs whose logits are exact in fp32, so
both sides route identically and the router's weight gradient and the layer
input's full gradient can be compared."""
import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape, f32_to_bf16_bits
from oracle import oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


SHAPES = [MoEShape(T=1000, H=256, I=64, E=64, k=2),   # several M tiles, E below one tile
          MoEShape(T=333, H=192, I=64, E=136, k=4),   # H with an odd count of 64-blocks, E % 64 != 0
          MoEShape(T=4096, H=2048, I=64, E=128, k=8),  # the 30B router's width and depth (dW_r in 4 segments)
          MoEShape(T=5000, H=256, I=64, E=64, k=2)]    # dW_r in 4 segments of 1250 tokens (ragged K tails)


@pytest.mark.parametrize("shape", SHAPES, ids=["t1000_e64", "t333_e136", "t4096_h2048", "t5000_split4"])
def test_router_projection_matches_oracle(shape):
    rng = np.random.default_rng(81)
    x = f32_to_bf16_bits(rng.standard_normal((shape.T, shape.H)).astype(np.float32))
    W_r = f32_to_bf16_bits((rng.standard_normal((shape.H, shape.E)) * 0.02).astype(np.float32))
    d_logits = (rng.standard_normal((shape.T, shape.E)) * 1e-2).astype(np.float32)
    dx0 = f32_to_bf16_bits(rng.standard_normal((shape.T, shape.H)).astype(np.float32) * 0.1)
    r = moe.Router(shape)
    lg = r.forward(dev16(x), dev16(W_r))
    dx = dev16(dx0)
    dW = r.backward(dev16(x), dev16(W_r), torch.from_numpy(d_logits).cuda(), dx)
    torch.cuda.synchronize()
    assert r.status() == {"forward": 0, "backward": 0}
    # dW_r does not read dx: a second backward gives the same bits (split
    # weight gradients are added in a fixed order)
    dW2 = r.backward(dev16(x), dev16(W_r), torch.from_numpy(d_logits).cuda(), dev16(dx0))
    torch.cuda.synchronize()
    assert torch.equal(dW2, dW)
    ref_lg = O.router_forward(x, W_r)
    G.close("logits", lg.cpu().numpy(), ref_lg, rel_l2=1e-5, max_rel=1e-4)
    ref_dW, ref_dx = O.router_backward(x, W_r, d_logits.astype(np.float64))
    G.close("dW_r", dW.cpu().numpy(), ref_dW)
    G.close("dx (in place)", G.bf(dx), synth.bf16_bits_to_f32(dx0).astype(np.float64) + ref_dx)


def test_router_in_front_of_the_layer():
    shape = MoEShape(T=512, H=256, I=128, E=16, k=4)
    inp = synth.make_inputs_shape(shape, 83)
    rng = np.random.default_rng(84)
    # x on a 1/64 grid, W_r on a 1/256 grid: every partial sum is exact in fp32, so the
    # GPU's logits equal the oracle's and both route the same way
    inp["x"] = f32_to_bf16_bits((rng.integers(-64, 65, (shape.T, shape.H)) / 64.0).astype(np.float32))
    W_r = f32_to_bf16_bits((rng.integers(-64, 65, (shape.H, shape.E)) / 256.0).astype(np.float32))
    ref_lg = O.router_forward(inp["x"], W_r)
    inp["logits"] = ref_lg.astype(np.float32)
    assert np.array_equal(inp["logits"].astype(np.float64), ref_lg)
    r = moe.Router(shape)
    xd = dev16(inp["x"])
    lg = r.forward(xd, dev16(W_r))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(lg.cpu().numpy(), inp["logits"])
    t = G.to_dev(inp)
    layer = moe.MoELayer(shape)
    layer.route(lg)
    out = layer.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"])
    grads = layer.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"])
    dW = r.backward(xd, dev16(W_r), grads["d_logits"], grads["dx"])
    torch.cuda.synchronize()
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w, *_ = G.check_routing(shape, inp, layer)
    dx_l, dl, _ = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                    inp["W_down"], inp["dy"])
    ref_dW, ref_dx_r = O.router_backward(inp["x"], W_r, dl)
    G.close("dW_r", dW.cpu().numpy(), ref_dW)
    G.close("dx (layer + router)", G.bf(grads["dx"]), dx_l + ref_dx_r)
