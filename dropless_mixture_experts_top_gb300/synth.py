"""Seeded synthetic inputs for the dropless MoE expert layer.

This module only draws random numbers and shapes them into the layer's inputs
(token activations x, router logits, expert weights, upstream gradient dy).  It
holds none of the layer's arithmetic: no routing, no expert MLP, no gradients.
Both the CUDA path (through the tests and the benchmark) and the fp64 oracle
read the arrays it returns, so the two sides always see identical inputs.

Workloads follow the layer shapes quoted for the Qwen3 MoE models in the
"Prime Mega MoE" write-ups (128 experts, top-8, 16,384-token sequences,
"random routing" in the single-layer table), with hidden/intermediate sizes of
the two Qwen3 models.  No public dataset or trained weight is involved; the
synthetic draws below stand in for them.

Recipe (all arrays row-major):
  * x, dy      [T, H]    bf16, N(0, 1)
  * logits     [T, E]    fp32, N(0, 1)   (+ a per-expert bias for the skewed case)
  * W_gate     [E, H, I] bf16, N(0, 0.02)
  * W_up       [E, H, I] bf16, N(0, 0.02)
  * W_down     [E, I, H] bf16, N(0, 0.02)
Draws are float32 standard normals from numpy's PCG64 generator, scaled in
float32 and rounded to bf16 with round-to-nearest-even.  Weights are drawn per
expert from the stream SeedSequence([seed, e]) so that large tensors can be
generated in parallel and still be reproducible.

Bf16 arrays are returned as uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import functools
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEShape:
    T: int  # tokens
    H: int  # hidden size
    I: int  # expert intermediate size
    E: int  # experts
    k: int  # experts per token

    @property
    def M(self) -> int:
        """Permuted rows: every token appears once per selected expert."""
        return self.T * self.k

    def gemm_flops(self) -> tuple[float, float]:
        """Algorithmic grouped-GEMM flops (forward, backward).

        Forward: gate and up projections (2*M*H*I each) plus down (2*M*I*H).
        Backward: twice that (data gradients and weight gradients).
        """
        fwd = 6.0 * self.M * self.H * self.I
        return fwd, 2.0 * fwd


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: MoEShape
    seed_index: int          # selects the seed family (x 1000+c, logits 2000+c, ...)
    routing: str             # "uniform" or "zipf"
    precision: str           # "bf16", "fp8_bwd" or "mxfp8"
    description: str


_TINY = MoEShape(T=512, H=128, I=64, E=8, k=2)
_Q30 = MoEShape(T=16384, H=2048, I=768, E=128, k=8)
_Q235 = MoEShape(T=16384, H=4096, I=1536, E=128, k=8)

WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_t512_h128_i64_e8_k2", _TINY, 1, "uniform", "bf16",
                 "tiny layer, T=512 H=128 I=64 E=8 top-2"),
        Workload("qwen3_30b_a3b_layer_t16384", _Q30, 2, "uniform", "bf16",
                 "Qwen3-30B-A3B-shaped layer, T=16384 H=2048 I=768 E=128 top-8, uniform routing"),
        Workload("qwen3_30b_a3b_layer_t16384_zipf", _Q30, 3, "zipf", "bf16",
                 "same shape, Zipf(s=1.2) expert loads with 8 empty experts"),
        Workload("qwen3_235b_a22b_layer_t16384", _Q235, 4, "uniform", "bf16",
                 "Qwen3-235B-A22B-shaped layer, T=16384 H=4096 I=1536 E=128 top-8, uniform routing"),
        Workload("qwen3_30b_a3b_layer_t16384_fp8_bwd", _Q30, 2, "uniform", "fp8_bwd",
                 "30B shape, BF16 forward, MXFP8 backward grouped GEMMs (same inputs as the uniform 30B case)"),
        Workload("qwen3_30b_a3b_layer_t16384_mxfp8", _Q30, 2, "uniform", "mxfp8",
                 "30B shape, forward and backward grouped GEMMs in MXFP8 (same inputs as the uniform 30B case)"),
    ]
}

WORKLOAD_ORDER = list(WORKLOADS)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round-to-nearest-even), returned as uint16 bits.

    Inputs here are finite normals, so no NaN handling is needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_bf16(seed, shape, scale: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence(seed))
    a = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return f32_to_bf16_bits(a).reshape(shape)


def _weights(seed: int, E: int, rows: int, cols: int, scale: float = 0.02) -> np.ndarray:
    out = np.empty((E, rows, cols), dtype=np.uint16)

    def one(e):
        out[e] = _normal_bf16([seed, e], (rows, cols), scale)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(E)))
    return out


def _rows_normal_bf16(seed: int, T: int, H: int) -> np.ndarray:
    # chunked by 1024 rows, each chunk its own stream, for parallel generation
    out = np.empty((T, H), dtype=np.uint16)
    chunks = [(c, min(T, c + 1024)) for c in range(0, T, 1024)]

    def one(ci):
        a, b = chunks[ci]
        out[a:b] = _normal_bf16([seed, ci], (b - a, H))

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(len(chunks))))
    return out


# --------------------------------------------------------------------------------------
# Skewed routing: per-expert logit bias so that expected loads follow a capped Zipf law.
# --------------------------------------------------------------------------------------

def zipf_targets(E: int, k: int, s: float = 1.2, n_empty: int = 8) -> np.ndarray:
    """Target selection probability per load rank (rank 1 = hottest).

    An expert can be chosen at most once per token, so a load share above 1/k of
    the selections is impossible.  The target is a Zipf law capped at
    probability 1 per token: q_r = min(1, c * r**-s) for the E - n_empty
    non-empty ranks, with c set by bisection so that the q sum to k.
    """
    r = np.arange(1, E - n_empty + 1, dtype=np.float64)
    lo, hi = 1e-6, 1e3
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(1.0, c * r ** -s).sum() > k:
            hi = c
        else:
            lo = c
    return np.minimum(1.0, 0.5 * (lo + hi) * r ** -s)


def _topk_counts(z: np.ndarray, k: int) -> np.ndarray:
    # load counting for bias calibration only (input shaping, not part of the layer)
    sel = np.argpartition(-z, k - 1, axis=1)[:, :k]
    return np.bincount(sel.ravel(), minlength=z.shape[1])


@functools.lru_cache(maxsize=None)
def zipf_bias(T: int, E: int, k: int, s: float = 1.2, n_empty: int = 8, iters: int = 200) -> np.ndarray:
    """Per-expert fp32 logit bias producing Zipf(s) loads with n_empty empty experts.

    The rank-to-expert map is a seeded permutation (seed 1234) so hot and empty
    experts are interleaved in expert-index order.  Calibration runs on a
    separate batch of T x E normals (seed 99): start from log q (centred), then
    repeatedly move each bias by half the log-ratio of target to measured load.
    """
    q = zipf_targets(E, k, s, n_empty)
    perm = np.random.default_rng(1234).permutation(E)
    hot, empty = perm[: E - n_empty], perm[E - n_empty:]
    target = np.zeros(E)
    target[hot] = q
    z0 = np.random.default_rng(99).standard_normal((T, E), dtype=np.float32).astype(np.float64)
    b = np.zeros(E)
    b[hot] = np.log(q) - np.log(q).mean()
    for _ in range(iters):
        counts = _topk_counts(z0 + np.where(np.isin(np.arange(E), empty), -1e4, b), k)
        frac = np.clip(counts[hot] / T, 1e-4, 0.999)
        b[hot] += 0.5 * (np.log(np.minimum(q, 0.999)) - np.log(frac))
    b[empty] = -1e4
    return b.astype(np.float32)


# --------------------------------------------------------------------------------------

def make_inputs(workload: str | Workload, parts=("x", "logits", "weights", "dy")) -> dict:
    """Inputs for one of the named workloads.

    Seeds for seed index c: x 1000+c, logits 2000+c, W_gate 3000+c, W_up 3100+c,
    W_down 3200+c, dy 4000+c.
    """
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    return make_inputs_shape(w.shape, w.seed_index, routing=w.routing, parts=parts)


def make_inputs_shape(shape: MoEShape, c: int, routing: str = "uniform",
                      parts=("x", "logits", "weights", "dy"), w_scale: float = 0.02,
                      logit_scale: float = 1.0) -> dict:
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    out: dict = {"shape": shape}
    if "x" in parts:
        out["x"] = _rows_normal_bf16(1000 + c, T, H)
    if "logits" in parts:
        rng = np.random.default_rng(2000 + c)
        lg = rng.standard_normal((T, E), dtype=np.float32)
        if logit_scale != 1.0:
            lg *= np.float32(logit_scale)
        if routing == "zipf":
            lg = lg + zipf_bias(T, E, k)[None, :]
        elif routing != "uniform":
            raise ValueError(routing)
        out["logits"] = np.ascontiguousarray(lg, dtype=np.float32)
    if "weights" in parts:
        out["W_gate"] = _weights(3000 + c, E, H, I, w_scale)
        out["W_up"] = _weights(3100 + c, E, H, I, w_scale)
        out["W_down"] = _weights(3200 + c, E, I, H, w_scale)
    if "dy" in parts:
        out["dy"] = _rows_normal_bf16(4000 + c, T, H)
    return out


def topk_gap_ok(logits: np.ndarray, k: int, gap: float = 1e-3) -> bool:
    """True when every token's k-th and (k+1)-th largest logits differ by more than gap.

    Finite-difference checks perturb logits by tiny amounts; this guarantees the
    selected set cannot change under such perturbations.
    """
    E = logits.shape[1]
    if k >= E:
        return True
    s = -np.sort(-logits.astype(np.float64), axis=1)
    return bool(np.all(s[:, k - 1] - s[:, k] > gap))
