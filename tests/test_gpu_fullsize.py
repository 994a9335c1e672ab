"""Full-size workloads (T=16384, the 30B- and 235B-shaped layers) through the C ABI,
in the launch configuration the benchmark times.

Routing and the permutation are compared in full (bit-exact).  Floating-point
outputs are compared on samples the oracle computes one by one: whole output
rows of sampled tokens (out, dx, d_logits, d_topk_w) and sampled weight-gradient
elements, including the largest and smallest experts; experts that received no
token must have exactly zero weight gradients."""
import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from oracle import oracle as O
from tests import gpu_util as G

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WORKLOADS = ["qwen3_30b_a3b_layer_t16384", "qwen3_30b_a3b_layer_t16384_zipf",
             "qwen3_235b_a22b_layer_t16384", "qwen3_30b_a3b_layer_t16384_fp8_bwd",
             "qwen3_30b_a3b_layer_t16384_mxfp8"]


def sample_tokens(T, counts, idx, rng, n=64):
    toks = {0, T - 1}
    toks |= set(int(t) for t in rng.integers(0, T, n))
    nz = np.flatnonzero(counts)
    for e in (nz[np.argmax(counts[nz])], nz[np.argmin(counts[nz])]):
        on = np.flatnonzero((idx == e).any(1))
        toks |= set(int(t) for t in on[:: max(1, len(on) // 3)][:3])
    return np.array(sorted(toks), dtype=np.int64)


def sample_dw(shape, counts, rng, n_uniform=384):
    """Per weight gradient: n_uniform elements drawn uniformly over all of it (every
    expert equally likely, empty ones included), whose relative L2 error estimates the
    whole tensor's; plus corner and random elements of the largest, smallest, first and
    last non-empty experts, held to the max-error bound."""
    nz = np.flatnonzero(counts)
    special = [int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]), int(nz[0]), int(nz[-1])]
    which, ee, rr, cc, uni = [], [], [], [], []
    for wh in range(3):
        R, C = (shape.I, shape.H) if wh == 2 else (shape.H, shape.I)
        for q in range(n_uniform):
            which.append(wh), ee.append(int(rng.integers(shape.E))), rr.append(int(rng.integers(R)))
            cc.append(int(rng.integers(C))), uni.append(True)
        for e in special:
            for r, c in ((0, 0), (R - 1, C - 1), (0, C - 1), (R - 1, 0),
                         (int(rng.integers(R)), int(rng.integers(C)))):
                which.append(wh), ee.append(e), rr.append(r), cc.append(c), uni.append(False)
    return [np.array(a, np.int32) for a in (which, ee, rr, cc)] + [np.array(uni)]


def run_workload(name):
    w = synth.WORKLOADS[name]
    shape = w.shape
    inp = synth.make_inputs(w)
    layer, out, grads = G.run_layer(shape, inp, precision=w.precision)
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    return w, shape, inp, layer, out, grads


@pytest.mark.parametrize("name", WORKLOADS)
def test_fullsize_sampled_parity(name):
    w, shape, inp, layer, out, grads = run_workload(name)
    quant = w.precision in ("fp8_bwd", "mxfp8")
    fq = w.precision == "mxfp8"  # the forward quantised too
    tol = dict(rel_l2=G.FP8_REL_L2, max_rel=G.FP8_MAX_REL) if quant else {}
    ftol = tol if fq else {}
    qW = O.quant_weights(inp["W_gate"], inp["W_up"], inp["W_down"]) if quant else None
    fW = O.quant_weights_fwd(inp["W_gate"], inp["W_up"], inp["W_down"]) if fq else None
    idx, wts, counts, offsets, ros, sor = G.check_routing(shape, inp, layer)
    assert counts.sum() == shape.T * shape.k
    if w.routing == "zipf":
        assert (counts == 0).sum() >= 1 and counts.max() > 8 * counts[counts > 0].min()
    rng = np.random.default_rng(7)
    toks = sample_tokens(shape.T, counts, idx, rng)
    ref_out = O.forward(shape, inp["x"], idx, wts, inp["W_gate"], inp["W_up"], inp["W_down"], tokens=toks,
                        fwd_quant=fq, fW=fW)
    G.close("out[sampled tokens]", G.bf(out[torch.from_numpy(toks).cuda()]), ref_out, **ftol)
    dx, dl, gd = O.backward_tokens(shape, inp["x"], inp["logits"], idx, wts, inp["W_gate"], inp["W_up"],
                                   inp["W_down"], inp["dy"], tokens=toks, quant=quant, qW=qW, fwd_quant=fq,
                                   fW=fW)
    tk = torch.from_numpy(toks).cuda()
    G.close("dx[sampled tokens]", G.bf(grads["dx"][tk]), dx, **tol)
    G.close("d_logits[sampled tokens]", grads["d_logits"][tk].cpu().numpy(), dl, **ftol)
    G.close("d_topk_w[sampled tokens]", grads["d_topk_w"][tk].cpu().numpy(), gd, **ftol)
    which, ee, rr, cc, uni = sample_dw(shape, counts, rng)
    ref = O.dw_elements(shape, inp["x"], idx, wts, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"],
                        which, ee, rr, cc, quant=quant, qW=qW, fwd_quant=fq, fW=fW)
    names = ["dW_gate", "dW_up", "dW_down"]
    for wh in range(3):
        m = which == wh
        t = grads[names[wh]]
        got = G.bf(t[torch.from_numpy(ee[m]).long().cuda(), torch.from_numpy(rr[m]).long().cuda(),
                     torch.from_numpy(cc[m]).long().cuda()])
        u = uni[m]
        G.close(f"{names[wh]}[uniform sample]", got[u], ref[m][u], **tol)
        bound = (G.FP8_MAX_REL if quant else G.MAX_REL) * np.abs(ref[m]).max()
        worst = np.abs(got[~u] - ref[m][~u]).max()
        assert worst <= bound, f"{names[wh]}[edge elements]: max|diff| {worst:.3e} > {bound:.3e}"
    for e in np.flatnonzero(counts == 0):
        for n in names:
            assert int(grads[n][int(e)].abs().sum()) == 0, (n, e)
    # every output is finite at full size
    for n in ("dx",) + tuple(names):
        assert torch.isfinite(grads[n].view(torch.bfloat16).float()).all(), n
    assert torch.isfinite(out.view(torch.bfloat16).float()).all()
