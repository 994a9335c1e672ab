"""The fp8_bwd backward (MXFP8 grouped GEMMs) through the C ABI against the
oracle's quantised backward.

Quantisers: the MXFP8 codes and scales the backward leaves in its scratch for
operands that come straight from the seeded inputs (weights, dy, x) must equal
the oracle quantiser's bit for bit, in the padded per-expert row space and the
scale-atom order the tensor core reads.  Gradients: every element on small
shapes (several tiles, ragged experts, half-filled 256-row operand boxes, empty
and hot experts), sampled elements at the 30B-shaped full size."""
import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape
from oracle import oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


def atoms_to_scales(sf, R, K):
    """[R, K/32] scale codes from the 512-byte atoms: byte l*16 + q*4 + j of atom
    (rb, kg) is row rb*128 + 32q + l, K-block kg*4 + j."""
    a = np.asarray(sf, np.uint8).reshape(R // 128, K // 128, 32, 4, 4)
    return a.transpose(0, 3, 2, 1, 4).reshape(R, K // 32)


def padded_rows(rows, offsets, pad, Mp):
    out = np.zeros((Mp,) + rows.shape[1:], rows.dtype)
    for e in range(len(offsets) - 1):
        n = offsets[e + 1] - offsets[e]
        out[pad[e]:pad[e] + n] = rows[offsets[e]:offsets[e + 1]]
    return out


def check_token_axis(layer, name, src_rows, offsets, pad, Mp):
    """Codes [C, Mp] and scales of an operand quantised along tokens, per expert."""
    C = src_rows.shape[1]
    got = layer.fp8_tensor(name).cpu().numpy()
    got_sc = atoms_to_scales(layer.fp8_tensor(name + "_sf").cpu().numpy(), C, Mp)
    exp = np.zeros((C, Mp), np.uint8)
    exp_sc = np.zeros((C, Mp // 32), np.uint8)
    for e in range(len(offsets) - 1):
        n = int(offsets[e + 1] - offsets[e])
        if n == 0:
            continue
        codes, sc = O.mx_quantize_cols(src_rows, int(offsets[e]), n)
        exp[:, pad[e]:pad[e] + codes.shape[0]] = codes.T
        exp_sc[:, pad[e] // 32:pad[e] // 32 + sc.shape[0]] = sc.T
    np.testing.assert_array_equal(got, exp, err_msg=name)
    np.testing.assert_array_equal(got_sc, exp_sc, err_msg=name + "_sf")


def test_quantised_operands_bit_exact():
    shape = MoEShape(T=700, H=384, I=384, E=6, k=2)
    inp = synth.make_inputs_shape(shape, 51)
    inp["logits"][:, 4] -= 30.0  # an empty expert
    layer, out, grads = G.run_layer(shape, inp, precision="fp8_bwd")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w, counts, offsets, ros, sor = G.check_routing(shape, inp, layer)
    assert counts[4] == 0
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    lay = moe.fp8_scratch_offsets(layer.cfg)
    Mp = lay["m_pad"]
    pad = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    np.testing.assert_array_equal(layer.fp8_tensor("pad_offsets").cpu().numpy(), pad)
    # weights, quantised along each backward GEMM's K
    for name, W, R, K in (("wd", inp["W_down"], E * I, H), ("wg", inp["W_gate"], E * H, I),
                          ("wu", inp["W_up"], E * H, I)):
        codes, sc, _ = O.mx_quantize_rows(W.reshape(R, K))
        np.testing.assert_array_equal(layer.fp8_tensor(name + "_q").cpu().numpy(), codes, err_msg=name)
        np.testing.assert_array_equal(atoms_to_scales(layer.fp8_tensor(name + "_sf").cpu().numpy(), R, K),
                                      sc, err_msg=name + "_sf")
    # dy in the padded row space (dA's A operand), along H
    dy_perm = inp["dy"][sor // k]
    codes, sc, _ = O.mx_quantize_rows(dy_perm)
    np.testing.assert_array_equal(layer.fp8_tensor("dy_q").cpu().numpy(), padded_rows(codes, offsets, pad, Mp))
    np.testing.assert_array_equal(atoms_to_scales(layer.fp8_tensor("dy_sf").cpu().numpy(), Mp, H),
                                  padded_rows(sc, offsets, pad, Mp))
    # token-axis operands of the weight gradients: dy and x, blocks of 32 from each expert's first row
    check_token_axis(layer, "dy_t", dy_perm, offsets, pad, Mp)
    check_token_axis(layer, "x_t", inp["x"][sor // k], offsets, pad, Mp)


FP8_SHAPES = [
    ("small", MoEShape(T=512, H=128, I=128, E=8, k=2)),
    ("ragged_half_boxes", MoEShape(T=700, H=384, I=384, E=6, k=2)),  # 256-row B boxes half past the operand
    ("wide", MoEShape(T=300, H=640, I=256, E=16, k=4)),
    ("single_expert", MoEShape(T=333, H=128, I=256, E=1, k=1)),
]


@pytest.mark.parametrize("name,shape", FP8_SHAPES, ids=[s[0] for s in FP8_SHAPES])
def test_fp8_layer_matches_quantised_oracle(name, shape):
    inp = synth.make_inputs_shape(shape, 53)
    layer, out, grads = G.run_layer(shape, inp, precision="fp8_bwd")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w = G.check_full(shape, inp, layer, out, grads, precision="fp8_bwd")
    # the result follows the quantised semantics, not the exact ones
    dx_exact, _, _ = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                       inp["W_down"], inp["dy"])
    dx_q, _, _ = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                   inp["W_down"], inp["dy"], quant=True)
    got = G.bf(grads["dx"])
    err_q = np.linalg.norm(got - dx_q) / np.linalg.norm(dx_q)
    err_exact = np.linalg.norm(got - dx_exact) / np.linalg.norm(dx_exact)
    assert err_q < 0.5 * err_exact, (err_q, err_exact)


def test_fp8_empty_and_hot_experts():
    shape = MoEShape(T=640, H=256, I=128, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 57)
    inp["logits"][:, 1] -= 30.0
    inp["logits"][:, 7] -= 30.0
    inp["logits"][:, 3] += 12.0
    layer, out, grads = G.run_layer(shape, inp, precision="fp8_bwd")
    G.check_full(shape, inp, layer, out, grads, precision="fp8_bwd")
    counts = layer.routing["counts"].cpu().numpy()
    assert counts[1] == 0 and counts[7] == 0 and counts[3] == shape.T


def test_fp8_rejects_unaligned_shape():
    with pytest.raises(moe.MoEError):
        moe.MoELayer(MoEShape(T=64, H=192, I=128, E=4, k=2), precision="fp8_bwd")
