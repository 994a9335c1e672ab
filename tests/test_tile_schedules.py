"""Host-side checks of the work split inside the forward GEMMs that quantise the
weights for an MXFP8 backward (no GPU needed).

The grouped GEMM hands out 256-row x 256-column tiles round-robin over the CTA
pairs (`tile = it * pairs + pair`, row tiles of each expert from its first row);
of tile (expert e, row tile m, column tile n) the weight K blocks of stage ks
(128 of K, two 64-row blocks) with ks mod (e's row tiles) = m are quantised,
in 32-row units shared round-robin by the epilogue warps ((unit + tile index)
mod warps).  Every weight element of every expert that received rows must be
quantised exactly once, each unit by exactly one warp, and nothing outside the
weights may be touched.  The rules are restated here from the kernel's comments
and walked over the routing of the 30B-shaped workload, a skewed one and small
ragged cases."""
import numpy as np
import pytest

from dropless_mixture_experts_top_gb300 import synth
from oracle import oracle as O

PAIRS = 76  # CTA pairs of a 152-SM part


def walk(counts, H, I, mode, epi_warps=8):
    """Coverage count per (weight row block of 32, 128-column block, CTA) and the
    number of units each (pair, warp) takes."""
    E = len(counts)
    tiles_e = (counts + 255) // 256
    tp = np.concatenate([[0], np.cumsum(tiles_e)])
    if mode == "gateup":  # B = W_gate (CTA 0) and W_up (CTA 1): [E*H, I]; 128 columns per tile
        rows_e, ld, n_tiles, ncta = H, I, I // 128, 2
    else:  # down: B = W_down [E*I, H]; 256 columns per tile, 128 per CTA
        rows_e, ld, n_tiles, ncta = I, H, (H + 255) // 256, 2
    nkb = rows_e // 64
    cover = np.zeros((ncta, E * rows_e // 32, (ld + 127) // 128), np.int32)
    total = int(tp[E]) * n_tiles
    for pair in range(PAIRS):
        it = 0
        while it * PAIRS + pair < total:
            tile = it * PAIRS + pair
            mt_lin, nt = divmod(tile, n_tiles)
            e = int(np.searchsorted(tp, mt_lin, side="right") - 1)
            nmt, mtl = int(tiles_e[e]), mt_lin - int(tp[e])
            for rank in range(ncta):
                col0 = nt * 128 if mode == "gateup" else nt * 256 + 128 * rank
                if col0 >= ld:
                    continue
                u = 0
                ks = mtl
                while ks * 2 < nkb:
                    for kb in range(2 * ks, min(2 * ks + 2, nkb)):
                        for q in range(2):
                            owner = (u + it) % epi_warps
                            assert 0 <= owner < epi_warps
                            r0 = e * rows_e + kb * 64 + 32 * q
                            assert r0 + 32 <= E * rows_e and col0 + 128 <= ld
                            cover[rank if mode == "gateup" else 0, r0 // 32, col0 // 128] += 1
                            u += 1
                    ks += nmt
            it += 1
    return cover, rows_e


def check(counts, H, I):
    for mode in ("gateup", "down"):
        cover, rows_e = walk(counts, H, I, mode)
        ncta = 2 if mode == "gateup" else 1
        for e, c in enumerate(counts):
            blk = cover[:ncta, e * rows_e // 32:(e + 1) * rows_e // 32]
            if c > 0:
                assert (blk == 1).all(), (mode, e, int(blk.min()), int(blk.max()))
            else:
                assert (blk == 0).all(), (mode, e)  # no tile, no rows: never read, never written


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_layer_t16384", "qwen3_30b_a3b_layer_t16384_zipf"])
def test_weight_quantisation_covers_each_element_once(name):
    w = synth.WORKLOADS[name]
    s = w.shape
    inp = synth.make_inputs(w, parts=("logits",))
    idx, _ = O.route(inp["logits"], s.k)
    counts, _, _, _ = O.dispatch(idx, s.E)
    check(counts, s.H, s.I)


@pytest.mark.parametrize("counts,H,I", [
    ([1024, 0, 1, 255, 256, 257, 2048, 3000], 768, 768),  # empty, 1-row, exact and ragged tiles, deep experts
    ([1, 1, 1], 256, 128),
    ([5000], 2048, 384),   # one expert with 20 row tiles: more row tiles than stages in the down GEMM
    ([700, 700], 384, 384),
])
def test_weight_quantisation_covers_ragged_cases(counts, H, I):
    check(np.array(counts), H, I)
