"""Activation checkpointing through the C ABI: moe_forward_nosave (out only),
then moe_forward_recompute (what the backward reads) and moe_backward, against
moe_forward + moe_backward on the same inputs.  Same kernels on the same
inputs, so out and every gradient must be bit-identical; `saved` is filled
with garbage between the two forward passes, so the recompute must rebuild
everything the backward reads.  The checkpointed results are also compared
with the oracle."""
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SHAPE = MoEShape(T=700, H=256, I=256, E=6, k=2)  # H, I multiples of 128 for the fp8 modes


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


@pytest.mark.parametrize("precision", ["bf16", "fp8_bwd", "mxfp8"])
def test_checkpointed_step_matches_saved_step(precision):
    inp = synth.make_inputs_shape(SHAPE, 71)
    layer, out, grads = G.run_layer(SHAPE, inp, precision=precision)
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}

    t = G.to_dev(inp)
    ck = moe.MoELayer(SHAPE, precision=precision)
    ck.route(t["logits"])
    out_ns = ck.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"], save=False)
    torch.cuda.synchronize()
    ck.saved.fill_(0xA5)  # anything the recompute does not rebuild is now garbage
    ck.recompute(t["x"], t["W_gate"], t["W_up"], t["W_down"])
    grads_ck = ck.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"])
    torch.cuda.synchronize()
    assert ck.status() == {"route": 0, "forward": 0, "backward": 0}

    assert torch.equal(out_ns, out)
    for n in grads:
        assert torch.equal(grads_ck[n], grads[n]), n
    G.check_full(SHAPE, inp, ck, out_ns, grads_ck, precision=precision, check_saved=False)
