"""Helpers for the GPU parity tests: run the layer through the C ABI on seeded
inputs and compare with the fp64 oracle.

Tolerances (floating point): relative L2 <= 5e-3 and max |diff| <= 2e-2 *
max |ref| for bf16 outputs and gradients; 1e-2 and 5e-2 for the MXFP8 backward
(fp8_bwd) gradients dx, dW_*, against the oracle's quantised backward, and in
the mxfp8 mode for every output (its forward is quantised too); router
weights within 1e-6; integer routing and permutation bit-exact.
"""
import json
import os

import numpy as np
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import bf16_bits_to_f32
from oracle import oracle as O

REL_L2 = 5e-3
MAX_REL = 2e-2
W_ATOL = 1e-6
# fp8_bwd backward outputs against the oracle's quantised backward.  Both sides
# decide every E4M3 code on the same bf16 tensors, so what remains is the bf16
# rounding of the outputs and fp32 accumulation, as in the bf16 path, plus the
# rare code that lands one step apart (one E4M3 step is 6-12% of an element)
# where fp32 evaluation order moves a bf16 value across a rounding boundary.
FP8_REL_L2 = 1e-2
FP8_MAX_REL = 5e-2


def atoms_to_scales(sf, R, K, seg=None, group=128):
    """[R, K/32] scale codes from the 512-byte atoms: row w of atom row-block rb,
    K-block b at byte (rb*(K/128) + b/4)*512 + (w%32)*16 + (w/32)*4 + b%4; rows
    map to (rb, w) through segments of `seg` rows cut into groups of `group`."""
    seg = seg or R
    r = np.arange(R)
    s, j = r // seg, r % seg
    g, jj = j // group, j % group
    gps, apg = -(-seg // group), -(-group // 128)
    rb = (s * gps + g) * apg + jj // 128
    w = jj % 128
    b = np.arange(K // 32)
    idx = ((rb[:, None] * (K // 128) + b[None, :] // 4) * 512 + (w[:, None] % 32) * 16 + (w[:, None] // 32) * 4
           + b[None, :] % 4)
    return np.asarray(sf, np.uint8)[idx]


def padded_rows(rows, offsets, pad, Mp):
    out = np.zeros((Mp,) + rows.shape[1:], rows.dtype)
    for e in range(len(offsets) - 1):
        n = offsets[e + 1] - offsets[e]
        out[pad[e]:pad[e] + n] = rows[offsets[e]:offsets[e + 1]]
    return out


def to_dev(inp, dev="cuda"):
    t = {n: torch.from_numpy(np.ascontiguousarray(inp[n]).view(np.int16)).to(dev)
         for n in ("x", "W_gate", "W_up", "W_down", "dy") if n in inp}
    t["logits"] = torch.from_numpy(inp["logits"]).to(dev)
    return t


def bf(t):
    return bf16_bits_to_f32(t.cpu().numpy().view(np.uint16)).astype(np.float64)


def close(name, got, ref, rel_l2=REL_L2, max_rel=MAX_REL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    nref = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    rel = err / nref if nref > 0 else err
    mx = np.abs(got - ref).max() if got.size else 0.0
    amax = np.abs(ref).max() if ref.size else 0.0
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "tensor": name, "n": int(got.size), "rel_l2": float(rel),
                                "max_abs_over_max_ref": float(mx / amax) if amax else 0.0}) + "\n")
    assert rel <= rel_l2, f"{name}: rel L2 {rel:.3e} > {rel_l2}"
    assert mx <= max_rel * amax + 1e-30, f"{name}: max|diff| {mx:.3e} > {max_rel} * {amax:.3e}"
    return rel


def run_layer(shape, inp, precision="bf16", layer=None, stream=None):
    t = to_dev(inp)
    layer = layer or moe.MoELayer(shape, precision=precision)
    layer.route(t["logits"], stream)
    out = layer.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"], stream=stream)
    grads = layer.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"], stream=stream)
    torch.cuda.synchronize()
    return layer, out, grads


def check_routing(shape, inp, layer):
    idx, w = O.route(inp["logits"], shape.k)
    counts, offsets, ros, sor = O.dispatch(idx, shape.E)
    r = {n: v.cpu().numpy() for n, v in layer.routing.items()}
    np.testing.assert_array_equal(r["topk_idx"], idx)
    np.testing.assert_array_equal(r["counts"], counts)
    np.testing.assert_array_equal(r["offsets"], offsets)
    np.testing.assert_array_equal(r["row_of_slot"], ros)
    np.testing.assert_array_equal(r["slot_of_row"], sor)
    assert np.abs(r["topk_w"].astype(np.float64) - w).max() <= W_ATOL
    np.testing.assert_array_equal(r["w_row"], r["topk_w"].ravel()[sor])
    return idx, w, counts, offsets, ros, sor


_E4M3 = None


def e4m3_values():
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([O.e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3


def check_aw_t(shape, layer, aw, offsets):
    """w * A quantised along tokens [I, m_pad] (from its bf16 value, in the GPU's
    fp32 arithmetic, so not bit-comparable with the oracle): dequantised, within
    MXFP8 error of the oracle's w * a in every expert's tokens, and exactly zero
    in the padded tokens past each expert's count."""
    Mp = moe.fp8_scratch_offsets(layer.cfg)["m_pad"]
    I = shape.I
    codes = layer.fp8_tensor("aw_t").cpu().numpy()
    sc = atoms_to_scales(layer.fp8_tensor("aw_t_sf").cpu().numpy(), I, Mp, I, 128).astype(np.int64)
    deq = e4m3_values()[codes] * np.exp2(np.repeat(sc, 32, axis=1) - 127.0)
    counts = np.diff(offsets)
    pad = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int64)
    ref = np.zeros((I, Mp))
    for e in range(len(counts)):
        n = int(counts[e])
        ref[:, pad[e]:pad[e] + n] = aw[offsets[e]:offsets[e] + n].T
        assert np.all(codes[:, pad[e] + n:pad[e + 1]] == 0), e
    P = int(pad[-1])
    close("aw_t", deq[:, :P], ref[:, :P], rel_l2=5e-2, max_rel=8e-2)


def check_full(shape, inp, layer, out, grads, precision="bf16", check_saved=True):
    """Every output element against the oracle (small shapes)."""
    idx, w, counts, offsets, ros, sor = check_routing(shape, inp, layer)
    quant = precision in ("fp8_bwd", "mxfp8")
    fq = precision == "mxfp8"  # the forward GEMMs quantised too
    fW = O.quant_weights_fwd(inp["W_gate"], inp["W_up"], inp["W_down"]) if fq else None
    tol = dict(rel_l2=FP8_REL_L2, max_rel=FP8_MAX_REL) if quant else {}
    ftol = tol if fq else {}
    if check_saved:
        if not fq:  # the mxfp8 mode keeps x only quantised (its backward reads x itself)
            xp = layer.saved_tensor("x_perm").cpu().numpy().view(np.uint16)
            np.testing.assert_array_equal(xp, inp["x"][sor // shape.k])
        toks = sor // shape.k
        experts = idx.ravel()[sor]
        g, u, a, y = O.expert_rows(shape, inp["x"], inp["W_gate"], inp["W_up"], inp["W_down"], toks, experts,
                                   fwd_quant=fq, fW=fW)
        close("G", bf(layer.saved_tensor("G")), g, **ftol)
        close("U", bf(layer.saved_tensor("U")), u, **ftol)
        close("A", bf(layer.saved_tensor("A")), a, **ftol)
        close("Y", bf(layer.saved_tensor("Y")), y, **ftol)
        if quant:  # w * A exists only quantised along tokens, written by the forward's gate/up epilogue
            check_aw_t(shape, layer, a * w.ravel()[sor][:, None], offsets)
        else:
            close("A_w", bf(layer.saved_tensor("A_w")), a * w.ravel()[sor][:, None], **ftol)
    ref = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], fwd_quant=fq, fW=fW)
    close("out", bf(out), ref, **ftol)
    dx, dl, gd = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                   inp["W_down"], inp["dy"], quant=quant, fwd_quant=fq, fW=fW)
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"],
                              inp["dy"], quant=quant, fwd_quant=fq, fW=fW)
    close("d_logits", grads["d_logits"].cpu().numpy(), dl, **ftol)
    close("d_topk_w", grads["d_topk_w"].cpu().numpy(), gd, **ftol)
    close("dx", bf(grads["dx"]), dx, **tol)
    close("dW_gate", bf(grads["dW_gate"]), dWg, **tol)
    close("dW_up", bf(grads["dW_up"]), dWu, **tol)
    close("dW_down", bf(grads["dW_down"]), dWd, **tol)
    for e in np.flatnonzero(counts == 0):
        for n in ("dW_gate", "dW_up", "dW_down"):
            assert np.all(grads[n][e].cpu().numpy() == 0), (n, e)
    return idx, w
