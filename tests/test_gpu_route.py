"""Routing alone (softmax, top-k, renormalise, count, scan, permutation) through
the C ABI against the oracle, bit for bit, on the shapes that take the route
kernel's other paths: the 16-entry lists (k > 8), the largest expert count,
expert counts that are not a multiple of 32 or of 4 (unaligned logit rows),
ragged last blocks, more blocks than the histogram scan keeps in registers,
and exact ties between logits (the lower expert wins)."""
import zlib

import numpy as np
import pytest
import torch

from dropless_mixture_experts_top_gb300 import moe
from dropless_mixture_experts_top_gb300.synth import MoEShape
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from dropless_mixture_experts_top_gb300 import _build as B
    B.build()


CASES = [
    ("E256_k16", 1000, 256, 16),
    ("E200_k9", 777, 200, 9),
    ("E13_k5_unaligned_rows", 300, 13, 5),
    ("E64_k8_one_past_a_block", 129, 64, 8),
    ("E256_k8_long_scan", 9000, 256, 8),   # 71 blocks, 2 partial sums per expert: 36 blocks each
    ("E8_k2_many_blocks", 20000, 8, 2),    # 157 blocks, 64 partial sums per expert
    ("E128_k8_t16384", 16384, 128, 8),     # the 30B-shaped layer's routing, in full
    ("E256_k16_t131072", 131072, 256, 16),  # 2 M slots, 1024 blocks: 16 register batches per scan
]


def _route(T, E, k, logits):
    shape = MoEShape(T=T, H=64, I=64, E=E, k=k)
    layer = moe.MoELayer(shape)
    layer.route(torch.from_numpy(logits).cuda())
    torch.cuda.synchronize()
    return shape, layer


@pytest.mark.parametrize("name,T,E,k", CASES, ids=[c[0] for c in CASES])
def test_route_bit_exact(name, T, E, k):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    shape, layer = _route(T, E, k, logits)
    assert layer.status()["route"] == 0
    G.check_routing(shape, {"logits": logits}, layer)


@pytest.mark.parametrize("E,k", [(128, 8), (256, 16), (13, 5)])
def test_route_exact_ties(E, k):
    """Logits on a grid of five values: most tokens have ties inside and across
    the cut, which the lower expert index decides."""
    rng = np.random.default_rng(E * 100 + k)
    T = 640
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    shape, layer = _route(T, E, k, logits)
    assert layer.status()["route"] == 0
    G.check_routing(shape, {"logits": logits}, layer)


def test_route_twice_bitwise():
    """A second call on the same logits gives the same bits (every scratch
    value a call reads, it wrote first)."""
    rng = np.random.default_rng(5)
    T, E, k = 5000, 128, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    shape, layer = _route(T, E, k, logits)
    first = {n: v.clone() for n, v in layer.routing.items()}
    layer.route(torch.from_numpy(logits).cuda())
    torch.cuda.synchronize()
    for n, v in layer.routing.items():
        assert torch.equal(v, first[n]), n
