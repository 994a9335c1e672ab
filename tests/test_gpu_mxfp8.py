"""The mxfp8 mode (both forward grouped GEMMs in MXFP8 too, the fp8_bwd backward)
through the C ABI against the oracle's mxfp8 mode.

Forward operands: the codes and scales the forward leaves in its scratch for
operands that come straight from the inputs (the permuted x along H; W_gate and
W_up along H, transposed and interleaved by 32 columns; W_down along I,
transposed) must equal the oracle quantiser's bit for bit, and A's codes
(quantised inside GEMM1's epilogue) must equal the oracle quantiser applied to
the bf16 A the same epilogue stored.  Outputs and gradients: every element on
small shapes (several tiles, ragged experts, 192-row tiles past I, empty and
hot experts)."""
import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape
from oracle import oracle as O
from tests import gpu_util as G
from tests.gpu_util import atoms_to_scales, padded_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


def _interleaved(gate_rows, up_rows, E, I):
    """[E*I, K] rows of W_gate^T and W_up^T -> the gate|up interleave [E*2I, K]:
    row e*2I + (i/32)*64 + i%32 is gate column i, the row 32 after it up column i."""
    K = gate_rows.shape[1]
    out = np.zeros((E * 2 * I, K), gate_rows.dtype)
    e = np.repeat(np.arange(E), I)
    i = np.tile(np.arange(I), E)
    r = e * 2 * I + (i // 32) * 64 + i % 32
    out[r] = gate_rows
    out[r + 32] = up_rows
    return out


SHAPES = [
    ("ragged", MoEShape(T=700, H=384, I=384, E=6, k=2)),   # 2I = 768: four 192-row gate|up tiles
    ("partial_tiles", MoEShape(T=300, H=256, I=128, E=8, k=2)),  # 2I = 256: a 192-row tile half past it
    ("wide", MoEShape(T=300, H=640, I=256, E=16, k=4)),
    ("E256_k16_max", MoEShape(T=300, H=256, I=128, E=256, k=16)),
]


@pytest.mark.parametrize("name,shape", SHAPES[:2], ids=[s[0] for s in SHAPES[:2]])
def test_forward_operands_bit_exact(name, shape):
    inp = synth.make_inputs_shape(shape, 61)
    inp["logits"][:, 3] -= 30.0  # an empty expert
    layer, out, grads = G.run_layer(shape, inp, precision="mxfp8")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w, counts, offsets, ros, sor = G.check_routing(shape, inp, layer)
    assert counts[3] == 0
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    lay = moe.mxfp8_forward_offsets(layer.cfg)
    Mp = lay["m_pad"]
    pad = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    P = int(pad[-1])
    np.testing.assert_array_equal(layer.fwd_fp8_tensor("pad_offsets").cpu().numpy(), pad)
    # x permuted, along H, in the padded row space
    codes, sc, _ = O.mx_quantize_rows(inp["x"][sor // k])
    np.testing.assert_array_equal(layer.fwd_fp8_tensor("x_q").cpu().numpy()[:P], padded_rows(codes, offsets, pad, Mp)[:P])
    np.testing.assert_array_equal(atoms_to_scales(layer.fwd_fp8_tensor("x_sf").cpu().numpy(), Mp, H)[:P],
                                  padded_rows(sc, offsets, pad, Mp)[:P])
    # W_gate | W_up along H, transposed, interleaved by 32
    qg = O.mx_quantize_rows(np.ascontiguousarray(inp["W_gate"].transpose(0, 2, 1)).reshape(E * I, H))
    qu = O.mx_quantize_rows(np.ascontiguousarray(inp["W_up"].transpose(0, 2, 1)).reshape(E * I, H))
    np.testing.assert_array_equal(layer.fwd_fp8_tensor("wgu_q").cpu().numpy(), _interleaved(qg[0], qu[0], E, I))
    seg, group = moe.sf_grouping("wgu_q", shape, Mp)
    got_sc = atoms_to_scales(layer.fwd_fp8_tensor("wgu_sf").cpu().numpy(), E * 2 * I, H, seg, group)
    np.testing.assert_array_equal(got_sc, _interleaved(qg[1], qu[1], E, I))
    # W_down along I, transposed
    qd = O.mx_quantize_rows(np.ascontiguousarray(inp["W_down"].transpose(0, 2, 1)).reshape(E * H, I))
    np.testing.assert_array_equal(layer.fwd_fp8_tensor("wdt_q").cpu().numpy(), qd[0])
    seg, group = moe.sf_grouping("wdt_q", shape, Mp)
    np.testing.assert_array_equal(
        atoms_to_scales(layer.fwd_fp8_tensor("wdt_sf").cpu().numpy(), E * H, I, seg, group), qd[1])
    # A along I, quantised in GEMM1's epilogue from the bf16 A it stored
    A = layer.saved_tensor("A").cpu().numpy().view(np.uint16)
    codes, sc, _ = O.mx_quantize_rows(A)
    np.testing.assert_array_equal(layer.fwd_fp8_tensor("a_q").cpu().numpy()[:P], padded_rows(codes, offsets, pad, Mp)[:P])
    np.testing.assert_array_equal(atoms_to_scales(layer.fwd_fp8_tensor("a_sf").cpu().numpy(), Mp, I)[:P],
                                  padded_rows(sc, offsets, pad, Mp)[:P])


@pytest.mark.parametrize("name,shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_mxfp8_layer_matches_oracle(name, shape):
    inp = synth.make_inputs_shape(shape, 63)
    layer, out, grads = G.run_layer(shape, inp, precision="mxfp8")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w = G.check_full(shape, inp, layer, out, grads, precision="mxfp8")
    # the result follows the quantised forward, not the exact one
    exact = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    quant = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], fwd_quant=True)
    got = G.bf(out)
    err_q = np.linalg.norm(got - quant) / np.linalg.norm(quant)
    err_exact = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert err_q < 0.5 * err_exact, (err_q, err_exact)


def test_mxfp8_empty_and_hot_experts():
    shape = MoEShape(T=640, H=256, I=256, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 65)
    inp["logits"][:, 1] -= 30.0
    inp["logits"][:, 6] -= 30.0
    inp["logits"][:, 2] += 12.0
    layer, out, grads = G.run_layer(shape, inp, precision="mxfp8")
    G.check_full(shape, inp, layer, out, grads, precision="mxfp8")


def test_mxfp8_rejects_unaligned_shape():
    with pytest.raises(moe.MoEError):
        moe.MoELayer(MoEShape(T=64, H=192, I=128, E=4, k=2), precision="mxfp8")


def test_backward_weight_codes_from_the_forward():
    """In this mode the forward's passes over the weights also write the
    backward GEMMs' weight operands (into `saved`): W_down along H, W_gate and
    W_up along I, bit-exact against the oracle's quantiser."""
    shape = MoEShape(T=300, H=256, I=384, E=4, k=2)
    inp = synth.make_inputs_shape(shape, 67)
    layer, out, grads = G.run_layer(shape, inp, precision="mxfp8")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    E, H, I = shape.E, shape.H, shape.I
    Mp = moe.mxfp8_forward_offsets(layer.cfg)["m_pad"]
    for name, W, R, K, seg in (("bwd_wd", inp["W_down"], E * I, H, I), ("bwd_wg", inp["W_gate"], E * H, I, H),
                               ("bwd_wu", inp["W_up"], E * H, I, H)):
        codes, sc, _ = O.mx_quantize_rows(W.reshape(R, K))
        np.testing.assert_array_equal(layer.fwd_fp8_tensor(name + "_q").cpu().numpy(), codes, err_msg=name)
        np.testing.assert_array_equal(
            atoms_to_scales(layer.fwd_fp8_tensor(name + "_sf").cpu().numpy(), R, K, seg, moe.MX_BN), sc,
            err_msg=name + "_sf")
