"""GPU path against the fp64 oracle, every output element, on small seeded shapes
that span several tiles and ragged tails, plus the method's degenerate cases."""
import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe, synth
from dropless_mixture_experts_top_gb300.synth import MoEShape
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SHAPES = [
    ("tiny", MoEShape(T=512, H=128, I=64, E=8, k=2)),
    ("ragged_tiles", MoEShape(T=700, H=256, I=192, E=6, k=2)),   # several M/N/K tiles, ragged tails
    ("wide", MoEShape(T=300, H=576, I=320, E=16, k=4)),          # N/K not multiples of the tile
    ("k1", MoEShape(T=200, H=128, I=128, E=4, k=1)),
    ("k_eq_E", MoEShape(T=130, H=128, I=64, E=3, k=3)),
    ("single_expert", MoEShape(T=333, H=192, I=128, E=1, k=1)),
    ("E256_k16_max", MoEShape(T=300, H=128, I=128, E=256, k=16)),  # the largest E and k: most experts empty
]


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


@pytest.mark.parametrize("name,shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_layer_matches_oracle(name, shape):
    inp = synth.make_inputs_shape(shape, 31)
    layer, out, grads = G.run_layer(shape, inp)
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    G.check_full(shape, inp, layer, out, grads)


def test_workload_tiny_config():
    w = synth.WORKLOADS["tiny_t512_h128_i64_e8_k2"]
    inp = synth.make_inputs(w)
    layer, out, grads = G.run_layer(w.shape, inp)
    G.check_full(w.shape, inp, layer, out, grads)


def test_empty_experts_and_hot_expert():
    shape = MoEShape(T=640, H=128, I=128, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 41)
    inp["logits"][:, 2] -= 30.0   # never chosen
    inp["logits"][:, 5] -= 30.0   # never chosen
    inp["logits"][:, 6] += 12.0   # chosen by every token, weight close to 1
    layer, out, grads = G.run_layer(shape, inp)
    idx, _ = G.check_full(shape, inp, layer, out, grads)
    counts = layer.routing["counts"].cpu().numpy()
    assert counts[2] == 0 and counts[5] == 0 and counts[6] == shape.T


def test_all_tokens_one_expert_tail():
    # T not a multiple of 128, every token on expert 0 (k=1): one long ragged segment
    shape = MoEShape(T=1000, H=128, I=64, E=4, k=1)
    inp = synth.make_inputs_shape(shape, 43)
    inp["logits"][:, 0] += 100.0
    layer, out, grads = G.run_layer(shape, inp)
    G.check_full(shape, inp, layer, out, grads)


def test_hot_experts_weight_gradients_bitwise():
    """Skewed routing (the weight gradients' longest-first order and snake assignment of
    tiles to CTA pairs): every element against the oracle, and a second step gives the
    same bits."""
    shape = MoEShape(T=2048, H=256, I=256, E=16, k=2)  # mean 256 rows per expert
    inp = synth.make_inputs_shape(shape, 61)
    inp["logits"][:, 3] += 6.0   # in nearly every token's top 2: ~8x the mean
    inp["logits"][:, 11] += 2.0  # a second hot expert
    layer, out, grads = G.run_layer(shape, inp)
    G.check_full(shape, inp, layer, out, grads)
    counts = layer.routing["counts"].cpu().numpy()
    assert counts[3] > 6 * counts.mean() and counts[11] > 2 * counts.mean()
    first = {n: grads[n].clone() for n in ("dW_gate", "dW_up", "dW_down")}
    _, _, grads2 = G.run_layer(shape, inp, layer=layer)
    for n, v in first.items():
        assert torch.equal(grads2[n], v), n


def test_many_hot_experts():
    """Twenty hot experts among sixty-four: every element against the oracle."""
    shape = MoEShape(T=2048, H=128, I=128, E=64, k=4)  # mean 128 rows per expert
    inp = synth.make_inputs_shape(shape, 67)
    inp["logits"][:, :20] += 4.0  # each of the twenty takes about 3x the mean
    layer, out, grads = G.run_layer(shape, inp)
    G.check_full(shape, inp, layer, out, grads)
    counts = layer.routing["counts"].cpu().numpy()
    assert (counts > 2 * counts.mean()).sum() > 16


PRECISIONS = ["bf16", "fp8_bwd", "mxfp8"]


# expert segments ending at and around every 32-row boundary of a 256-row tile:
# a CTA of a ragged tile loads 1-4 of its 32-row A boxes, or none
BOX_COUNTS = [1, 31, 32, 33, 63, 64, 65, 96, 97, 127, 128, 129, 160, 255, 256, 257]


@pytest.mark.parametrize("precision", PRECISIONS)
def test_segments_ending_at_every_box_boundary(precision):
    shape = MoEShape(T=sum(BOX_COUNTS), H=128, I=128, E=len(BOX_COUNTS), k=1)
    inp = synth.make_inputs_shape(shape, 71)
    owner = np.repeat(np.arange(shape.E), BOX_COUNTS)
    np.random.default_rng(71).shuffle(owner)  # tokens of an expert spread over the batch
    inp["logits"][np.arange(shape.T), owner] += 100.0
    layer, out, grads = G.run_layer(shape, inp, precision=precision)
    G.check_full(shape, inp, layer, out, grads, precision=precision)
    assert list(layer.routing["counts"].cpu().numpy()) == BOX_COUNTS


@pytest.mark.parametrize("precision", PRECISIONS)
def test_zero_tokens(precision):
    shape = MoEShape(T=0, H=128, I=128, E=4, k=2)
    layer = moe.MoELayer(shape, precision=precision)
    dev = "cuda"
    logits = torch.empty((0, 4), dtype=torch.float32, device=dev)
    x = torch.empty((0, 128), dtype=torch.int16, device=dev)
    W = [torch.ones((4, 128, 128), dtype=torch.int16, device=dev)] * 3
    layer.route(logits)
    out = layer.forward(x, *W, save=False)  # the checkpointing calls accept an empty batch too
    layer.recompute(x, *W)
    out = layer.forward(x, *W)
    grads = {"dx": x.clone(), "dW_gate": torch.full((4, 128, 128), 7, dtype=torch.int16, device=dev),
             "dW_up": torch.full((4, 128, 128), 7, dtype=torch.int16, device=dev),
             "dW_down": torch.full((4, 128, 128), 7, dtype=torch.int16, device=dev),
             "d_logits": logits.clone(), "d_topk_w": torch.empty((0, 2), dtype=torch.float32, device=dev)}
    layer.backward(x, x, *W, grads=grads)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert layer.routing["offsets"].cpu().tolist() == [0] * 5
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert int(grads[n].abs().sum()) == 0


def test_nonfinite_logits_flagged_not_trapped():
    shape = MoEShape(T=256, H=128, I=64, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 47)
    inp["logits"][3, 1] = np.nan
    inp["logits"][7, 4] = np.inf
    t = G.to_dev(inp)
    layer = moe.MoELayer(shape)
    layer.route(t["logits"])
    code = moe.get_device_status(layer.route_scratch)
    assert code & moe.DEV_NONFINITE_LOGIT
    idx = layer.routing["topk_idx"].cpu().numpy()
    assert idx.min() >= 0 and idx.max() < shape.E
    assert np.all(np.sort(idx, 1)[:, 0] != np.sort(idx, 1)[:, 1])  # distinct experts per token
    # the permutation is still a bijection
    sor = layer.routing["slot_of_row"].cpu().numpy()
    assert np.array_equal(np.sort(sor), np.arange(shape.T * shape.k))
    # a clean call afterwards reports no anomaly (the status word is reset per call)
    inp["logits"] = np.nan_to_num(inp["logits"], nan=0.0, posinf=0.0)
    layer.route(G.to_dev(inp)["logits"])
    assert moe.get_device_status(layer.route_scratch) == 0


@pytest.mark.parametrize("precision", PRECISIONS)
def test_deterministic_bitwise(precision):
    shape = MoEShape(T=700, H=256, I=256, E=6, k=2)
    inp = synth.make_inputs_shape(shape, 53)
    _, out1, g1 = G.run_layer(shape, inp, precision=precision)
    _, out2, g2 = G.run_layer(shape, inp, precision=precision)
    assert torch.equal(out1, out2)
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("precision", PRECISIONS)
def test_two_layers_on_two_streams_concurrently(precision):
    """The library keeps no per-call state: two layers with different shapes and
    inputs, their calls interleaved on two streams, give the bits each gives alone."""
    shapes = [MoEShape(T=700, H=256, I=256, E=6, k=2), MoEShape(T=512, H=384, I=128, E=16, k=4)]
    inps = [synth.make_inputs_shape(sh, 73 + i) for i, sh in enumerate(shapes)]
    alone = [G.run_layer(sh, inp, precision=precision) for sh, inp in zip(shapes, inps)]
    layers = [moe.MoELayer(sh, precision=precision) for sh in shapes]
    ts = [G.to_dev(inp) for inp in inps]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs, grads = [None, None], [None, None]
    for i in (0, 1):
        layers[i].route(ts[i]["logits"], streams[i])
    for i in (0, 1):
        outs[i] = layers[i].forward(ts[i]["x"], ts[i]["W_gate"], ts[i]["W_up"], ts[i]["W_down"], stream=streams[i])
    for i in (1, 0):
        grads[i] = layers[i].backward(ts[i]["dy"], ts[i]["x"], ts[i]["W_gate"], ts[i]["W_up"], ts[i]["W_down"],
                                      stream=streams[i])
    torch.cuda.synchronize()
    for i in (0, 1):
        assert layers[i].status(streams[i]) == {"route": 0, "forward": 0, "backward": 0}
        _, out_a, g_a = alone[i]
        assert torch.equal(outs[i], out_a), i
        for n in g_a:
            assert torch.equal(grads[i][n], g_a[n]), (i, n)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_cuda_graph_capture_and_replay_with_new_routing(precision):
    shape = MoEShape(T=512, H=128, I=128, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 59)
    t = G.to_dev(inp)
    layer = moe.MoELayer(shape, precision=precision)
    s = torch.cuda.Stream()
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    grads = None
    with torch.cuda.stream(s):  # warm-up outside capture (first-call attribute setup)
        layer.route(t["logits"], s)
        layer.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"], out=out, stream=s)
        grads = layer.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"], stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.route(t["logits"], s)
        layer.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"], out=out, stream=s)
        layer.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"], grads=grads, stream=s)
    # new routing (different loads, including an empty expert) replayed through the same graph
    inp2 = dict(inp)
    lg = np.random.default_rng(5).standard_normal(inp["logits"].shape).astype(np.float32)
    lg[:, 3] -= 50.0
    inp2["logits"] = lg
    t["logits"].copy_(torch.from_numpy(lg).cuda())
    g.replay()
    torch.cuda.synchronize()
    G.check_full(shape, inp2, layer, out, grads, precision=precision)


@pytest.mark.parametrize("precision", ["bf16", "fp8_bwd", "mxfp8"])
def test_cuda_graph_checkpointed_step(precision):
    """The activation-checkpointed sequence (route, forward without saving,
    recompute, backward) captured once and replayed with new routing."""
    shape = MoEShape(T=512, H=128, I=128, E=8, k=2)
    inp = synth.make_inputs_shape(shape, 61)
    t = G.to_dev(inp)
    layer = moe.MoELayer(shape, precision=precision)
    s = torch.cuda.Stream()
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")

    def step(grads=None):
        layer.route(t["logits"], s)
        layer.forward(t["x"], t["W_gate"], t["W_up"], t["W_down"], out=out, stream=s, save=False)
        layer.recompute(t["x"], t["W_gate"], t["W_up"], t["W_down"], stream=s)
        return layer.backward(t["dy"], t["x"], t["W_gate"], t["W_up"], t["W_down"], grads=grads, stream=s)

    with torch.cuda.stream(s):  # warm-up outside capture (first-call attribute setup)
        grads = step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(grads)
    inp2 = dict(inp)
    lg = np.random.default_rng(6).standard_normal(inp["logits"].shape).astype(np.float32)
    lg[:, 5] -= 50.0  # an empty expert
    inp2["logits"] = lg
    t["logits"].copy_(torch.from_numpy(lg).cuda())
    g.replay()
    torch.cuda.synchronize()
    assert layer.status() == {"route": 0, "forward": 0, "backward": 0}
    G.check_full(shape, inp2, layer, out, grads, precision=precision, check_saved=False)
