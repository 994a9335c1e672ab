"""Pins for the fp64 oracle: each test checks it against something other than itself.

  * routing against a brute-force full sort and scipy's softmax;
  * dispatch against numpy's stable argsort;
  * forward and every gradient against torch autograd in fp64 (an independent
    derivation of the backward), and against a dense SwiGLU MLP for E=1, k=1;
  * gradients against Richardson-extrapolated central finite differences on
    inputs chosen so that every perturbed value is exactly representable;
  * invariants: weights sum to 1, d_logits rows sum to 0 with k non-zeros,
    empty experts get exactly zero weight gradients, linearity in W_up/W_down
    and dy, expert relabelling equivariance;
  * the MXFP8 quantiser against a brute-force nearest-value search over all
    E4M3 codes, and its scale rule against its defining inequality;
  * the bf16 rounding the fp8_bwd mode applies against torch's fp32 -> bf16
    conversion, and the fp8_bwd backward against a numpy composition of the
    pinned quantiser and rounding (which operands, along which axis, rounded
    where);
  * the mxfp8 mode's forward (both forward GEMMs in MXFP8) and its backward
    against the same kind of composition, with the weights quantised through
    the column quantiser (a different routine from the one the oracle uses).
"""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from dropless_mixture_experts_top_gb300 import synth
from dropless_mixture_experts_top_gb300.synth import MoEShape, bf16_bits_to_f32, f32_to_bf16_bits
from oracle import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def small_inputs(shape, c=11, routing="uniform", w_scale=0.3):
    return synth.make_inputs_shape(shape, c, routing=routing, w_scale=w_scale)


# ----------------------------------------------------------------------------- routing

@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (128, 8), (5, 5), (7, 1)])
def test_route_matches_full_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 257
    # coarse grid: many exact ties, so the tie rule (lower expert first) is exercised
    logits = (np.round(rng.standard_normal((T, E)) * 4) / 4).astype(np.float32)
    idx, w = O.route(logits, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))  # by -logit, then index
        assert list(idx[t]) == list(order[:k])
        p = scipy.special.softmax(logits[t].astype(np.float64))
        np.testing.assert_allclose(w[t], p[order[:k]] / p[order[:k]].sum(), rtol=1e-14, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-15 * k)


def test_route_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 6)).astype(np.float32)
    idx, w = O.route(logits, 6)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-14)
    assert np.all(np.sort(idx, 1) == np.arange(6))


def test_dispatch_is_stable_counting_sort():
    rng = np.random.default_rng(3)
    T, E, k = 300, 16, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 5] -= 50.0  # expert 5 never chosen: an empty group
    idx, _ = O.route(logits, k)
    counts, offsets, ros, sor = O.dispatch(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts[5] == 0 and counts.sum() == T * k
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    # slot order sorted by expert, stable in token (and choice) order
    np.testing.assert_array_equal(sor, np.argsort(idx.ravel(), kind="stable"))
    np.testing.assert_array_equal(ros.ravel()[sor], np.arange(T * k))
    # permute then un-permute-sum of x is k * x
    x = rng.standard_normal((T, 4))
    x_perm = x[sor // k]
    back = np.zeros_like(x)
    np.add.at(back, sor // k, x_perm)
    np.testing.assert_array_equal(back, k * x)


# ----------------------------------------------------------------------------- torch autograd

def torch_moe(shape, inp, idx):
    """Independent formulation: gathered per-(token, choice) weights, einsum, autograd."""
    f = lambda b: torch.from_numpy(bf16_bits_to_f32(b).astype(np.float64)).requires_grad_(True)
    x, Wg, Wu, Wd, dy = (f(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dy"))
    lg = torch.from_numpy(inp["logits"].astype(np.float64)).requires_grad_(True)
    sel = torch.from_numpy(idx.astype(np.int64))
    p = torch.softmax(lg, dim=1)
    ps = torch.gather(p, 1, sel)
    w = ps / ps.sum(1, keepdim=True)
    g = torch.einsum("th,tkhi->tki", x, Wg[sel])
    u = torch.einsum("th,tkhi->tki", x, Wu[sel])
    a = torch.nn.functional.silu(g) * u
    y = torch.einsum("tki,tkih->tkh", a, Wd[sel])
    out = (w.unsqueeze(-1) * y).sum(1)
    (out * dy).sum().backward()
    return out.detach().numpy(), {n: t.grad.numpy() for n, t in
                                  dict(x=x, W_gate=Wg, W_up=Wu, W_down=Wd, logits=lg).items()}


@pytest.mark.parametrize("shape", [MoEShape(T=48, H=32, I=16, E=4, k=2),
                                   MoEShape(T=33, H=64, I=32, E=6, k=3),
                                   MoEShape(T=20, H=32, I=32, E=3, k=3)])
def test_oracle_matches_torch_autograd(shape):
    inp = small_inputs(shape)
    idx, w = O.route(inp["logits"], shape.k)
    out = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    dx, dl, gd = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                   inp["W_down"], inp["dy"])
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    t_out, t_grad = torch_moe(shape, inp, idx)
    np.testing.assert_allclose(out, t_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dx, t_grad["x"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dl, t_grad["logits"], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dWg, t_grad["W_gate"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dWu, t_grad["W_up"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dWd, t_grad["W_down"], rtol=1e-10, atol=1e-12)
    # g_j = <dy_t, y_tj> is the gradient with respect to the renormalised weight
    _, y = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], want_y=True)
    dyf = bf16_bits_to_f32(inp["dy"]).astype(np.float64)
    np.testing.assert_allclose(gd, np.einsum("th,tkh->tk", dyf, y), rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu_mlp():
    shape = MoEShape(T=40, H=64, I=32, E=1, k=1)
    inp = small_inputs(shape)
    idx, w = O.route(inp["logits"], 1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    out = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    f = lambda b: torch.from_numpy(bf16_bits_to_f32(b).astype(np.float64))
    x, Wg, Wu, Wd = f(inp["x"]), f(inp["W_gate"][0]), f(inp["W_up"][0]), f(inp["W_down"][0])
    ref = (torch.nn.functional.silu(x @ Wg) * (x @ Wu)) @ Wd
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- finite differences

def fd_inputs(shape, seed):
    """Inputs whose values are +-(1 + m/16) * 2^s, m in [2, 13]: every value v +- j*ulp(v),
    j <= 4, stays in its binade and is exactly representable in bf16."""
    rng = np.random.default_rng(seed)

    def vals(n, s_lo, s_hi):
        m = rng.integers(2, 14, n)
        s = rng.integers(s_lo, s_hi + 1, n)
        sign = rng.choice([-1.0, 1.0], n)
        return (sign * (1 + m / 16.0) * 2.0 ** s).astype(np.float32)

    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    inp = {
        "x": f32_to_bf16_bits(vals(T * H, -2, 0)).reshape(T, H),
        "dy": f32_to_bf16_bits(vals(T * H, -2, 0)).reshape(T, H),
        "W_gate": f32_to_bf16_bits(vals(E * H * I, -4, -3)).reshape(E, H, I),
        "W_up": f32_to_bf16_bits(vals(E * H * I, -4, -3)).reshape(E, H, I),
        "W_down": f32_to_bf16_bits(vals(E * I * H, -4, -3)).reshape(E, I, H),
    }
    # logits on a well separated grid: no top-k flip for perturbations up to 4 * 2^-10
    lg = np.stack([rng.permutation(E) for _ in range(T)]).astype(np.float64) * 0.25
    lg += rng.uniform(-0.05, 0.05, lg.shape)
    inp["logits"] = (np.round(lg * 1024) / 1024).astype(np.float32)
    assert synth.topk_gap_ok(inp["logits"], k, 0.01)
    for n in ("x", "dy", "W_gate", "W_up", "W_down"):
        assert np.all(f32_to_bf16_bits(bf16_bits_to_f32(inp[n])) == inp[n])
    return inp


def loss(shape, inp):
    idx, w = O.route(inp["logits"], shape.k)
    out = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    return float(np.sum(out * bf16_bits_to_f32(inp["dy"]).astype(np.float64)))


def richardson(shape, inp, name, pos, step):
    """Central differences at steps d, 2d, 4d combined to cancel the d^2 and d^4 terms."""
    def D(h):
        vals = []
        for sgn in (1, -1):
            mod = dict(inp)
            arr = inp[name].copy()
            if name == "logits":
                arr[pos] = np.float32(float(arr[pos]) + sgn * h)
                assert float(arr[pos]) == float(inp[name][pos]) + sgn * h
            else:
                v = float(bf16_bits_to_f32(arr[pos][None])[0]) + sgn * h
                arr[pos] = f32_to_bf16_bits(np.array([v], np.float32))[0]
                assert float(bf16_bits_to_f32(arr[pos][None])[0]) == v
            mod[name] = arr
            vals.append(loss(shape, mod))
        return (vals[0] - vals[1]) / (2 * h)

    d1, d2, d4 = D(step), D(2 * step), D(4 * step)
    r1, r2 = (4 * d1 - d2) / 3, (4 * d2 - d4) / 3
    return (16 * r1 - r2) / 15


@pytest.mark.parametrize("seed", [0, 1])
def test_gradients_match_finite_differences(seed):
    shape = MoEShape(T=6, H=16, I=8, E=4, k=2)
    inp = fd_inputs(shape, seed)
    idx, w = O.route(inp["logits"], shape.k)
    dx, dl, _ = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                  inp["W_down"], inp["dy"])
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    grads = {"x": dx, "logits": dl, "W_gate": dWg, "W_up": dWu, "W_down": dWd}
    rng = np.random.default_rng(100 + seed)
    for name, g in grads.items():
        for _ in range(6):
            if name.startswith("W"):
                e = int(idx[rng.integers(shape.T), rng.integers(shape.k)])  # an expert in use
                pos = (e,) + tuple(int(rng.integers(n)) for n in inp[name].shape[1:])
            else:
                pos = tuple(int(rng.integers(n)) for n in inp[name].shape)
            if name == "logits":
                step = 2.0 ** -10
            else:
                v = abs(float(bf16_bits_to_f32(inp[name][pos][None])[0]))
                step = 2.0 ** (np.floor(np.log2(v)) - 7)  # one bf16 ulp
            fd = richardson(shape, inp, name, pos, step)
            scale = np.max(np.abs(g)) + 1e-300
            assert abs(fd - g[pos]) <= 1e-7 * scale, (name, pos, fd, g[pos])


# ----------------------------------------------------------------------------- invariants

def test_router_gradient_invariants_and_empty_experts():
    shape = MoEShape(T=64, H=32, I=16, E=8, k=2)
    inp = small_inputs(shape)
    inp["logits"][:, 3] = -1e4  # expert 3 receives no token
    idx, w = O.route(inp["logits"], shape.k)
    dx, dl, gd = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                   inp["W_down"], inp["dy"])
    np.testing.assert_allclose(dl.sum(1), 0.0, atol=1e-13 * np.abs(dl).max())
    nz = (dl != 0).sum(1)
    assert np.all(nz == shape.k)
    # d_logits is w_j (g_j - sum_i w_i g_i) at the chosen experts
    gbar = (w * gd).sum(1, keepdims=True)
    np.testing.assert_allclose(np.take_along_axis(dl, idx, 1), w * (gd - gbar), rtol=1e-11, atol=1e-14)
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    assert np.all(dWg[3] == 0) and np.all(dWu[3] == 0) and np.all(dWd[3] == 0)
    assert np.abs(dWg[0]).max() > 0


def test_linearity_and_sign():
    shape = MoEShape(T=32, H=32, I=16, E=4, k=2)
    inp = small_inputs(shape)
    idx, w = O.route(inp["logits"], shape.k)
    base = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    # exact power-of-two scalings and sign flips of bf16 weights are exact
    Wd2 = f32_to_bf16_bits(bf16_bits_to_f32(inp["W_down"]) * 2)
    np.testing.assert_allclose(O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], Wd2),
                               2 * base, rtol=1e-14, atol=0)
    Wun = inp["W_up"] ^ np.uint16(0x8000)
    np.testing.assert_allclose(O.forward(shape, inp["x"], idx, w, inp["W_gate"], Wun, inp["W_down"]),
                               -base, rtol=1e-14, atol=0)
    # gradients are linear in dy
    dy4 = f32_to_bf16_bits(bf16_bits_to_f32(inp["dy"]) * 4)
    a = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                          inp["W_down"], inp["dy"])
    b = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                          inp["W_down"], dy4)
    for u, v in zip(a, b):
        np.testing.assert_allclose(v, 4 * u, rtol=1e-13, atol=1e-300)


def test_expert_relabelling_equivariance():
    shape = MoEShape(T=40, H=32, I=16, E=5, k=2)
    inp = small_inputs(shape)
    perm = np.array([3, 0, 4, 1, 2])  # new expert perm[e] holds old expert e
    inv = np.argsort(perm)
    relab = dict(inp)
    relab["logits"] = np.ascontiguousarray(inp["logits"][:, inv])
    for n in ("W_gate", "W_up", "W_down"):
        relab[n] = np.ascontiguousarray(inp[n][inv])
    res = []
    for d in (inp, relab):
        idx, w = O.route(d["logits"], shape.k)
        out = O.forward(shape, d["x"], idx, w, d["W_gate"], d["W_up"], d["W_down"])
        dWs = O.dw_full(shape, d["x"], idx, w, d["W_gate"], d["W_up"], d["W_down"], d["dy"])
        res.append((idx, out, dWs))
    np.testing.assert_array_equal(perm[res[0][0]], res[1][0])
    np.testing.assert_allclose(res[0][1], res[1][1], rtol=1e-13, atol=1e-15)
    for a, b in zip(res[0][2], res[1][2]):
        np.testing.assert_allclose(a, b[perm], rtol=1e-13, atol=1e-15)


def test_sampled_entry_points_agree_with_full():
    shape = MoEShape(T=50, H=64, I=32, E=4, k=2)
    inp = small_inputs(shape)
    idx, w = O.route(inp["logits"], shape.k)
    args = (shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    full = O.dw_full(*args)
    rng = np.random.default_rng(0)
    n = 40
    which = rng.integers(0, 3, n)
    e = rng.integers(0, shape.E, n)
    r = np.where(which == 2, rng.integers(0, shape.I, n), rng.integers(0, shape.H, n))
    c = np.where(which == 2, rng.integers(0, shape.H, n), rng.integers(0, shape.I, n))
    vals = O.dw_elements(*args, which, e, r, c)
    ref = np.array([full[wh][ee, rr, cc] for wh, ee, rr, cc in zip(which, e, r, c)])
    np.testing.assert_allclose(vals, ref, rtol=1e-13, atol=1e-15)
    qvals = O.dw_elements(*args, which, e, r, c, quant=True)  # fp8_bwd: the same two code paths agree
    qfull = O.dw_full(*args, quant=True)
    np.testing.assert_allclose(qvals, np.array([qfull[wh][ee, rr, cc] for wh, ee, rr, cc in zip(which, e, r, c)]),
                               rtol=1e-13, atol=1e-15)
    toks = np.array([49, 0, 7])
    out_all = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    np.testing.assert_array_equal(
        O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], tokens=toks),
        out_all[toks])


# ----------------------------------------------------------------------------- MXFP8

def all_e4m3():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    return codes, np.array([O.e4m3_decode(c) for c in codes])


def test_e4m3_decode_table_and_roundtrip():
    codes, vals = all_e4m3()
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x01) == 2.0 ** -9 and O.e4m3_decode(0x38) == 1.0
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    for c, v in zip(codes, vals):
        if c == 0x80:
            continue  # -0 encodes back to the negative zero code, checked below
        assert O.e4m3_encode(v) == c
    assert O.e4m3_encode(-0.0) == 0x80


def test_e4m3_encode_is_nearest_even_brute_force():
    codes, vals = all_e4m3()
    pos = [(v, c) for v, c in zip(vals, codes) if c < 0x80]
    pv = np.array([v for v, _ in pos])
    pc = np.array([c for _, c in pos])
    rng = np.random.default_rng(0)
    samples = np.concatenate([
        rng.uniform(0, 480, 4000), rng.uniform(0, 0.02, 2000),
        (pv[1:] + pv[:-1]) / 2,  # exact midpoints: ties go to the even code
        [448.0, 449.0, 464.0, 1e9, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]])
    for s in samples:
        sign = 1 if rng.random() < 0.5 else -1
        d = np.abs(pv - s)
        best = np.flatnonzero(d == d.min())
        exp_code = pc[best[0]] if len(best) == 1 else [c for c in pc[best] if c % 2 == 0][0]
        if s > 448.0:
            exp_code = 0x7E  # saturating conversion
        got = O.e4m3_encode(sign * s)
        assert got == (exp_code | (0x80 if sign < 0 else 0)) or (exp_code == 0 and got in (0, 0x80)), (s, got)


def test_mx_scale_rule():
    rng = np.random.default_rng(1)
    amaxes = np.concatenate([rng.lognormal(0, 6, 3000), [448.0, 448.0 * 2 ** 5, 449.0, 224.0, 1.0]])
    for a in amaxes:
        X = O.mx_scale_exp(a)
        assert a / 2.0 ** X <= 448.0 and a / 2.0 ** (X - 1) > 448.0  # smallest such power
        assert 224.0 < a / 2.0 ** X <= 448.0
    assert O.mx_scale_exp(0.0) == -127


def test_mx_quantize_rows_blocks():
    rng = np.random.default_rng(2)
    a = f32_to_bf16_bits(rng.standard_normal((7, 96)).astype(np.float32) * 3)
    codes, scales, deq = O.mx_quantize_rows(a)
    af = bf16_bits_to_f32(a).astype(np.float64)
    for r, b in itertools.product(range(7), range(3)):
        blk = af[r, 32 * b:32 * b + 32]
        X = int(scales[r, b]) - 127
        assert X == O.mx_scale_exp(np.abs(blk).max())
        for i in range(32):
            assert codes[r, 32 * b + i] == O.e4m3_encode(blk[i] / 2.0 ** X)
            assert deq[r, 32 * b + i] == O.e4m3_decode(codes[r, 32 * b + i]) * 2.0 ** X
    rel = np.abs(deq - af) / np.abs(af).max()
    assert rel.max() <= 2.0 ** -4  # half an E4M3 step at the block scale


def test_fp8_bwd_mode_changes_backward_by_quantisation_error_only():
    shape = MoEShape(T=128, H=64, I=64, E=4, k=2)
    inp = synth.make_inputs_shape(shape, 21)
    idx, w = O.route(inp["logits"], shape.k)
    args = (shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    ex = O.backward_tokens(*args)
    qt = O.backward_tokens(*args, quant=True)
    dwa = (shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    exw, qtw = O.dw_full(*dwa), O.dw_full(*dwa, quant=True)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    for a, b in [(qt[0], ex[0])] + list(zip(qtw, exw)):
        assert 5e-3 < rel(a, b) < 1.2e-1
    # quantised weights: exactly on the E4M3 x 2^X grid, and idempotent under re-quantisation
    qW = O.quant_weights(inp["W_gate"], inp["W_up"], inp["W_down"])
    again = O.mx_quantize_rows(f32_to_bf16_bits(qW[2]))[2]
    np.testing.assert_array_equal(again, qW[2])


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        (rng.standard_normal(4000) * np.exp2(rng.integers(-140, 127, 4000))).astype(np.float32),
        np.float32([3.0e38, -3.39e38, 1e-45, -3e-41, 0.0, 1.0, 2.0 ** -126, 2.0 ** -127])])
    # exact ties between two bf16 neighbours: both tie-to-even directions
    base = f32_to_bf16_bits(rng.standard_normal(500).astype(np.float32)).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([O.round_bf16(float(a)) for a in v])
    np.testing.assert_array_equal(got, ref)


def _deq_cols(bits, seg, n, table):
    codes, scales = O.mx_quantize_cols(bits, seg, n)
    return (table[codes] * np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=0))[:n]


def test_fp8_bwd_composition():
    """backward_tokens/dw_full in quant mode against the same chain written with
    numpy matrix products over the oracle's pinned quantiser and bf16 rounding."""
    shape = MoEShape(T=96, H=64, I=96, E=4, k=2)
    inp = synth.make_inputs_shape(shape, 23, w_scale=0.3)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    idx, w = O.route(inp["logits"], k)
    f = lambda b: bf16_bits_to_f32(b).astype(np.float64)
    x, Wg, Wu, Wd, dy = (f(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dy"))
    qWg, qWu, qWd = (q.astype(np.float64) for q in O.quant_weights(inp["W_gate"], inp["W_up"], inp["W_down"]))
    rb = np.vectorize(O.round_bf16)
    table = np.array([O.e4m3_decode(c) for c in range(256)])
    q_rows = lambda v: O.mx_quantize_rows(f32_to_bf16_bits(np.atleast_2d(v).astype(np.float32)))[2].astype(np.float64)
    sig = lambda z: 1 / (1 + np.exp(-z))
    dx = np.zeros((T, H))
    rows = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(k):
            e, wt = idx[t, j], w[t, j]
            g, u = x[t] @ Wg[e], x[t] @ Wu[e]
            da = wt * (q_rows(dy[t])[0] @ qWd[e].T)
            gb, ub = rb(g), rb(u)
            dg = rb(da * ub * sig(gb) * (1 + gb * (1 - sig(gb))))
            du = rb(da * gb * sig(gb))
            dx[t] += q_rows(dg)[0] @ qWg[e].T + q_rows(du)[0] @ qWu[e].T
            rows[e].append((t, rb(wt * g * sig(g) * u), dg, du))
    ref_dx = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                               inp["W_down"], inp["dy"], quant=True)[0]
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(dx, ref_dx) < 1e-12
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"],
                              quant=True)
    for e in range(E):
        toks = [r[0] for r in rows[e]]
        n = len(toks)
        bits = lambda m: f32_to_bf16_bits(np.asarray(m, np.float32).reshape(n, -1))
        Xq = _deq_cols(inp["x"][toks], 0, n, table)
        DYq = _deq_cols(inp["dy"][toks], 0, n, table)
        Aq = _deq_cols(bits([r[1] for r in rows[e]]), 0, n, table)
        DGq = _deq_cols(bits([r[2] for r in rows[e]]), 0, n, table)
        DUq = _deq_cols(bits([r[3] for r in rows[e]]), 0, n, table)
        assert rel(Xq.T @ DGq, dWg[e]) < 1e-12
        assert rel(Xq.T @ DUq, dWu[e]) < 1e-12
        assert rel(Aq.T @ DYq, dWd[e]) < 1e-12
    # the element-wise path agrees with the full one
    rng = np.random.default_rng(3)
    which = rng.integers(0, 3, 60).astype(np.int32)
    ee = rng.integers(0, E, 60).astype(np.int32)
    rr = np.where(which == 2, rng.integers(0, I, 60), rng.integers(0, H, 60)).astype(np.int32)
    cc = np.where(which == 2, rng.integers(0, H, 60), rng.integers(0, I, 60)).astype(np.int32)
    got = O.dw_elements(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"],
                        which, ee, rr, cc, quant=True)
    full = np.stack([dWg, dWu])
    exp = np.array([dWd[e, r, c] if wh == 2 else full[wh, e, r, c] for wh, e, r, c in zip(which, ee, rr, cc)])
    np.testing.assert_allclose(got, exp, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------- router projection

def test_router_forward_exact_on_integers():
    """Small-integer bf16 inputs: every product and partial sum is exact, so the
    oracle's logits equal an integer matrix product exactly."""
    rng = np.random.default_rng(12)
    xi = rng.integers(-8, 9, (37, 96))
    wi = rng.integers(-8, 9, (96, 24))
    x = f32_to_bf16_bits(xi.astype(np.float32))
    W = f32_to_bf16_bits(wi.astype(np.float32))
    np.testing.assert_array_equal(O.router_forward(x, W), (xi @ wi).astype(np.float64))


def test_router_backward_through_the_layer_matches_torch_autograd():
    """The router projection in front of the layer: torch autograd through
    logits = x . W_r and the whole MoE layer (fp64) gives d(W_r) and the total dx;
    the oracle composes router_forward, backward_tokens and router_backward."""
    shape = MoEShape(T=40, H=32, I=16, E=6, k=2)
    inp = small_inputs(shape, c=13)
    rng = np.random.default_rng(14)
    # x on a 1/64 grid and W_r on a 1/256 grid: every logit is exact in fp32, so
    # routing on fp32 logits and differentiating in fp64 see the same numbers
    inp["x"] = f32_to_bf16_bits((rng.integers(-64, 65, (shape.T, shape.H)) / 64.0).astype(np.float32))
    W_r = f32_to_bf16_bits((rng.integers(-128, 129, (shape.H, shape.E)) / 256.0).astype(np.float32))
    logits64 = O.router_forward(inp["x"], W_r)
    inp["logits"] = logits64.astype(np.float32)
    assert np.array_equal(inp["logits"].astype(np.float64), logits64)
    idx, w = O.route(inp["logits"], shape.k)
    srt = np.sort(logits64, axis=1)[:, ::-1]
    assert np.all(srt[:, shape.k - 1] - srt[:, shape.k] > 1e-4)  # no near tie at the cut
    dx, dl, _ = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                  inp["W_down"], inp["dy"])
    dWr, dx_router = O.router_backward(inp["x"], W_r, dl)
    # torch: the same layer with the logits computed from x and W_r inside the graph
    f = lambda b: torch.from_numpy(bf16_bits_to_f32(b).astype(np.float64)).requires_grad_(True)
    x, Wg, Wu, Wd, Wr = (f(a) for a in (inp["x"], inp["W_gate"], inp["W_up"], inp["W_down"], W_r))
    dy = torch.from_numpy(bf16_bits_to_f32(inp["dy"]).astype(np.float64))
    sel = torch.from_numpy(idx.astype(np.int64))
    p = torch.softmax(x @ Wr, dim=1)
    ps = torch.gather(p, 1, sel)
    wt = ps / ps.sum(1, keepdim=True)
    g = torch.einsum("th,tkhi->tki", x, Wg[sel])
    u = torch.einsum("th,tkhi->tki", x, Wu[sel])
    y = torch.einsum("tki,tkih->tkh", torch.nn.functional.silu(g) * u, Wd[sel])
    ((wt.unsqueeze(-1) * y).sum(1) * dy).sum().backward()
    np.testing.assert_allclose(dWr, Wr.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dx + dx_router, x.grad.numpy(), rtol=1e-10, atol=1e-13)


# ----------------------------------------------------------------------------- mxfp8 forward


def _fwd_weights_by_cols(W, table):
    """Dequantised W [E, R, C] quantised along R (blocks of 32 rows of each
    column) through the column quantiser."""
    E, R, C = W.shape
    return np.stack([_deq_cols(W[e], 0, R, table) for e in range(E)])


def _mxfp8_chain(inp, shape, idx, w):
    """The mxfp8 forward written out with numpy products: Q(x) . Q(W_gate) (both
    along H), a = silu(g) u, y = Q(bf16(a)) . Q(W_down) (both along I)."""
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    table = np.array([O.e4m3_decode(c) for c in range(256)])
    f = lambda b: bf16_bits_to_f32(b).astype(np.float64)
    q_rows = lambda v: O.mx_quantize_rows(f32_to_bf16_bits(np.atleast_2d(v).astype(np.float32)))[2].astype(np.float64)
    rb = np.vectorize(O.round_bf16)
    xq = O.mx_quantize_rows(inp["x"])[2].astype(np.float64)
    Wg, Wu, Wd = (_fwd_weights_by_cols(inp[n], table) for n in ("W_gate", "W_up", "W_down"))
    sig = lambda z: 1 / (1 + np.exp(-z))
    out = np.zeros((T, H))
    per = {}
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            g, u = xq[t] @ Wg[e], xq[t] @ Wu[e]
            a = g * sig(g) * u
            y = q_rows(rb(a))[0] @ Wd[e]
            out[t] += w[t, j] * y
            per[(t, j)] = (g, u, a, y)
    return out, per


def test_mxfp8_forward_composition():
    shape = MoEShape(T=96, H=64, I=96, E=4, k=2)
    inp = synth.make_inputs_shape(shape, 31, w_scale=0.3)
    idx, w = O.route(inp["logits"], shape.k)
    ref, per = _mxfp8_chain(inp, shape, idx, w)
    got, y = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], want_y=True,
                       fwd_quant=True)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(got, ref) < 1e-12
    toks = np.repeat(np.arange(shape.T), shape.k)
    g, u, a, yy = O.expert_rows(shape, inp["x"], inp["W_gate"], inp["W_up"], inp["W_down"], toks, idx.ravel(),
                                fwd_quant=True)
    for q, (t, j) in enumerate(zip(toks, np.tile(np.arange(shape.k), shape.T))):
        for got_v, ref_v in zip((g[q], u[q], a[q], yy[q], y[t, j]), per[(t, j)] + (per[(t, j)][3],)):
            np.testing.assert_allclose(got_v, ref_v, rtol=1e-12, atol=1e-12)
    # the quantised forward differs from the exact one by quantisation error only
    exact = O.forward(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    assert 5e-3 < rel(got, exact) < 1.2e-1
    # the forward-quantised weights sit on the E4M3 x 2^X grid along the reduction axis
    fWg, fWu, fWd = O.quant_weights_fwd(inp["W_gate"], inp["W_up"], inp["W_down"])
    table = np.array([O.e4m3_decode(c) for c in range(256)])
    np.testing.assert_array_equal(fWg, _fwd_weights_by_cols(inp["W_gate"], table).astype(np.float32))
    np.testing.assert_array_equal(fWd, _fwd_weights_by_cols(inp["W_down"], table).astype(np.float32))


def test_mxfp8_backward_composition():
    """The mxfp8 mode's backward is the fp8_bwd backward on the quantised forward's
    values: gdot = <dy, y_q>, dSwiGLU on bf16(g_q), bf16(u_q), dW_down's operand
    bf16(w a_q)."""
    shape = MoEShape(T=96, H=64, I=96, E=4, k=2)
    inp = synth.make_inputs_shape(shape, 33, w_scale=0.3)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    idx, w = O.route(inp["logits"], k)
    _, per = _mxfp8_chain(inp, shape, idx, w)
    f = lambda b: bf16_bits_to_f32(b).astype(np.float64)
    dy = f(inp["dy"])
    qWg, qWu, qWd = (q.astype(np.float64) for q in O.quant_weights(inp["W_gate"], inp["W_up"], inp["W_down"]))
    rb = np.vectorize(O.round_bf16)
    q_rows = lambda v: O.mx_quantize_rows(f32_to_bf16_bits(np.atleast_2d(v).astype(np.float32)))[2].astype(np.float64)
    sig = lambda z: 1 / (1 + np.exp(-z))
    dx = np.zeros((T, H))
    gd = np.zeros((T, k))
    rows = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(k):
            e, wt = idx[t, j], w[t, j]
            g, u, a, y = per[(t, j)]
            gd[t, j] = dy[t] @ y
            da = wt * (q_rows(dy[t])[0] @ qWd[e].T)
            gb, ub = rb(g), rb(u)
            dg = rb(da * ub * sig(gb) * (1 + gb * (1 - sig(gb))))
            du = rb(da * gb * sig(gb))
            dx[t] += q_rows(dg)[0] @ qWg[e].T + q_rows(du)[0] @ qWu[e].T
            rows[e].append((t, rb(wt * a), dg, du))
    got_dx, got_dl, got_gd = O.backward_tokens(shape, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                               inp["W_down"], inp["dy"], quant=True, fwd_quant=True)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(got_dx, dx) < 1e-12
    assert rel(got_gd, gd) < 1e-12
    dWg, dWu, dWd = O.dw_full(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"],
                              quant=True, fwd_quant=True)
    table = np.array([O.e4m3_decode(c) for c in range(256)])
    for e in range(E):
        toks = [r[0] for r in rows[e]]
        n = len(toks)
        bits = lambda m: f32_to_bf16_bits(np.asarray(m, np.float32).reshape(n, -1))
        Xq = _deq_cols(inp["x"][toks], 0, n, table)
        DYq = _deq_cols(inp["dy"][toks], 0, n, table)
        Aq = _deq_cols(bits([r[1] for r in rows[e]]), 0, n, table)
        DGq = _deq_cols(bits([r[2] for r in rows[e]]), 0, n, table)
        DUq = _deq_cols(bits([r[3] for r in rows[e]]), 0, n, table)
        assert rel(Xq.T @ DGq, dWg[e]) < 1e-12
        assert rel(Xq.T @ DUq, dWu[e]) < 1e-12
        assert rel(Aq.T @ DYq, dWd[e]) < 1e-12
    rng = np.random.default_rng(4)
    which = rng.integers(0, 3, 60).astype(np.int32)
    ee = rng.integers(0, E, 60).astype(np.int32)
    rr = np.where(which == 2, rng.integers(0, I, 60), rng.integers(0, H, 60)).astype(np.int32)
    cc = np.where(which == 2, rng.integers(0, H, 60), rng.integers(0, I, 60)).astype(np.int32)
    got = O.dw_elements(shape, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"],
                        which, ee, rr, cc, quant=True, fwd_quant=True)
    full = np.stack([dWg, dWu])
    exp = np.array([dWd[e, r, c] if wh == 2 else full[wh, e, r, c] for wh, e, r, c in zip(which, ee, rr, cc)])
    np.testing.assert_allclose(got, exp, rtol=1e-12, atol=1e-14)
