"""The fp8_bwd backward (MXFP8 grouped GEMMs) through the C ABI against the
oracle's quantised backward.

Quantisers: the MXFP8 codes and scales of the operands that come straight
from the seeded inputs (the weights, which the forward's bf16 GEMMs quantise as
they pass through them, and dy and x, which the backward quantises) must equal
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
from tests.gpu_util import atoms_to_scales, padded_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


def check_weight_codes(layer, inp, counts):
    """The weights quantised along each backward GEMM's K by the forward GEMMs that
    read them: every expert with rows (an empty expert's weights pass through no
    GEMM, and no backward GEMM reads them)."""
    s = layer.shape
    E, H, I = s.E, s.H, s.I
    Mp = moe.fp8_scratch_offsets(layer.cfg)["m_pad"]
    for name, W, R, K in (("wd", inp["W_down"], E * I, H), ("wg", inp["W_gate"], E * H, I),
                          ("wu", inp["W_up"], E * H, I)):
        codes, sc, _ = O.mx_quantize_rows(W.reshape(R, K))
        got = layer.fp8_tensor(name + "_q").cpu().numpy()
        seg, group = moe.sf_grouping(name + "_q", s, Mp)
        got_sc = atoms_to_scales(layer.fp8_tensor(name + "_sf").cpu().numpy(), R, K, seg, group)
        rows = R // E
        for e in np.nonzero(counts)[0]:
            sl = slice(e * rows, (e + 1) * rows)
            np.testing.assert_array_equal(got[sl], codes[sl], err_msg=f"{name} expert {e}")
            np.testing.assert_array_equal(got_sc[sl], sc[sl], err_msg=f"{name}_sf expert {e}")


def check_token_axis(layer, name, src_rows, offsets, pad, Mp):
    """Codes [C, Mp] and scales of an operand quantised along tokens, per expert."""
    C = src_rows.shape[1]
    got = layer.fp8_tensor(name).cpu().numpy()
    seg, group = moe.sf_grouping(name, layer.shape, Mp)
    got_sc = atoms_to_scales(layer.fp8_tensor(name + "_sf").cpu().numpy(), C, Mp, seg, group)
    exp = np.zeros((C, Mp), np.uint8)
    exp_sc = np.zeros((C, Mp // 32), np.uint8)
    for e in range(len(offsets) - 1):
        n = int(offsets[e + 1] - offsets[e])
        if n == 0:
            continue
        codes, sc = O.mx_quantize_cols(src_rows, int(offsets[e]), n)
        exp[:, pad[e]:pad[e] + codes.shape[0]] = codes.T
        exp_sc[:, pad[e] // 32:pad[e] // 32 + sc.shape[0]] = sc.T
    P = int(pad[-1])  # padded rows past the total are never read and left unwritten
    np.testing.assert_array_equal(got[:, :P], exp[:, :P], err_msg=name)
    np.testing.assert_array_equal(got_sc[:, :P // 32], exp_sc[:, :P // 32], err_msg=name + "_sf")


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
    check_weight_codes(layer, inp, counts)
    # dy in the padded row space (dA's A operand), along H
    dy_perm = inp["dy"][sor // k]
    codes, sc, _ = O.mx_quantize_rows(dy_perm)
    P = int(pad[-1])
    np.testing.assert_array_equal(layer.fp8_tensor("dy_q").cpu().numpy()[:P],
                                  padded_rows(codes, offsets, pad, Mp)[:P])
    np.testing.assert_array_equal(atoms_to_scales(layer.fp8_tensor("dy_sf").cpu().numpy(), Mp, H)[:P],
                                  padded_rows(sc, offsets, pad, Mp)[:P])
    # token-axis operands of the weight gradients: dy and x, blocks of 32 from each expert's first row
    check_token_axis(layer, "dy_t", dy_perm, offsets, pad, Mp)
    check_token_axis(layer, "x_t", inp["x"][sor // k], offsets, pad, Mp)


FP8_SHAPES = [
    ("small", MoEShape(T=512, H=128, I=128, E=8, k=2)),
    ("ragged_half_boxes", MoEShape(T=700, H=384, I=384, E=6, k=2)),  # 256-row B boxes half past the operand
    ("wide", MoEShape(T=300, H=640, I=256, E=16, k=4)),
    ("single_expert", MoEShape(T=333, H=128, I=256, E=1, k=1)),
    ("E256_k16_max", MoEShape(T=300, H=256, I=128, E=256, k=16)),  # padded row space ~8x the rows
    # one expert of four 256-row tiles, six stages per tile in both forward GEMMs: each
    # tile's weight quantisers read one or two of its stages and pass over the rest
    ("deep_k_row_tiles", MoEShape(T=1024, H=768, I=768, E=1, k=1)),
]


@pytest.mark.parametrize("name,shape", FP8_SHAPES, ids=[s[0] for s in FP8_SHAPES])
def test_fp8_layer_matches_quantised_oracle(name, shape):
    inp = synth.make_inputs_shape(shape, 53)
    layer, out, grads = G.run_layer(shape, inp, precision="fp8_bwd")
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    idx, w = G.check_full(shape, inp, layer, out, grads, precision="fp8_bwd")
    check_weight_codes(layer, inp, layer.routing["counts"].cpu().numpy())
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


def test_quantiser_sweeps_every_bf16_value():
    """Every finite bf16 value through the GPU quantiser (CUDA's E4M3 conversion)
    against the oracle's: blocks of 32 neighbouring magnitudes (each block's own
    scale, so saturation, subnormals and ties all occur) plus blocks that mix
    extremes."""
    shape = MoEShape(T=64, H=256, I=512, E=2, k=1)
    E, H, I = shape.E, shape.H, shape.I
    rng = np.random.default_rng(61)
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = bits[(bits & 0x7F80) != 0x7F80]                       # drop Inf / NaN
    mag = synth.bf16_bits_to_f32(finite & 0x7FFF)
    order = np.argsort(mag, kind="stable")
    sweep = finite[order]                                          # neighbouring magnitudes together
    n = E * I * H
    assert len(sweep) <= n
    vals = np.concatenate([sweep, rng.choice(finite, n - len(sweep))])  # then random blocks
    W_down = vals.reshape(E, I, H)
    inp = synth.make_inputs_shape(shape, 63)
    inp["W_down"] = W_down
    inp["logits"][0::2, 0] += 50.0  # both experts receive tokens, so GEMM2 passes every weight row
    inp["logits"][1::2, 1] += 50.0
    layer, out, grads = G.run_layer(shape, inp, precision="fp8_bwd")  # outputs may overflow: not compared
    codes, sc, _ = O.mx_quantize_rows(W_down.reshape(E * I, H))
    Mp = moe.fp8_scratch_offsets(layer.cfg)["m_pad"]
    np.testing.assert_array_equal(layer.fp8_tensor("wd_q").cpu().numpy(), codes)
    seg, group = moe.sf_grouping("wd_q", shape, Mp)
    np.testing.assert_array_equal(atoms_to_scales(layer.fp8_tensor("wd_sf").cpu().numpy(), E * I, H, seg, group),
                                  sc)
