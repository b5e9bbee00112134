"""Seeded synthetic inputs and the workload shapes, shared by the tests and the benchmark.

This module holds no quantization or matmul arithmetic: it only draws float32
arrays from numpy's PCG64 generator and names the shapes.  Both the CUDA path
and the CPU oracle consume the same float32 arrays (the oracle never sees a
GPU-produced input, and the GPU never sees an oracle-produced one).

Recipe (the pages' workloads are model matrices, not datasets):
  weights      f32 N(0, 0.02) per element; the decoder-layer set multiplies
               each row's standard deviation by U(0.5, 2).
  activations  f32 N(0, 1); each entry independently, with probability 0.01,
               is multiplied by 20 (an outlier).
Shapes (N rows x K input dim, M tokens):
  q4_0 matvec       4864 x 896, M=1            (a 0.5B-class MLP matrix)
  q8_0 matvec       12288 x 4096, M=1          (an 8B-class FFN gate, one token)
  q4_K_M layer set  hidden 4096: Wq, Wo 4096x4096, Wk, Wv 1024x4096,
                    W_gate, W_up 12288x4096 in Q4_K; W_down 4096x12288 in Q6_K
  q2_K matvec       12288 x 4096, M=1
  q4_0 prefill      M in {128, 512, 2048} x 12288 x 4096
  q4_1 / q5_0 / q5_1 / q5_K matvecs   12288 x 4096, M=1 (the other formats the
                    pages list, on the FFN shape)
  Q8 KV cache       32 query heads, 8 KV heads, head_dim 128, 4096 cached
                    positions (an 8B-class layer at the page's 4096-position
                    context): q, K, V ~ the activation recipe; the attention
                    weights a softmax of N(0, 2^2) logits per query head
"""
from __future__ import annotations

import numpy as np

WEIGHT_STD = 0.02
OUTLIER_P = 0.01
OUTLIER_SCALE = 20.0

# name -> (weight type, N, K); the layer set lists its seven matrices.
LAYER_SET = [
    ("Wq", "q4_K", 4096, 4096),
    ("Wk", "q4_K", 1024, 4096),
    ("Wv", "q4_K", 1024, 4096),
    ("Wo", "q4_K", 4096, 4096),
    ("W_gate", "q4_K", 12288, 4096),
    ("W_up", "q4_K", 12288, 4096),
    ("W_down", "q6_K", 4096, 12288),
]

WORKLOADS = {
    "q4_0_matvec_4864x896": dict(kind="matvec", wtype="q4_0", M=1, N=4864, K=896, seed=0xC0FFEE + 0),
    "q8_0_matvec_12288x4096": dict(kind="matvec", wtype="q8_0", M=1, N=12288, K=4096, seed=0xC0FFEE + 1),
    "q4_K_M_layer_4096": dict(kind="layer", matrices=LAYER_SET, M=1, seed=0xC0FFEE + 2),
    "q2_K_matvec_12288x4096": dict(kind="matvec", wtype="q2_K", M=1, N=12288, K=4096, seed=0xC0FFEE + 3),
    "q4_0_prefill_512x12288x4096": dict(kind="matmul", wtype="q4_0", M=512, N=12288, K=4096,
                                        seed=0xC0FFEE + 4, M_sweep=(128, 512, 2048)),
    "q4_1_matvec_12288x4096": dict(kind="matvec", wtype="q4_1", M=1, N=12288, K=4096, seed=0xC0FFEE + 5),
    "q5_0_matvec_12288x4096": dict(kind="matvec", wtype="q5_0", M=1, N=12288, K=4096, seed=0xC0FFEE + 6),
    "q5_1_matvec_12288x4096": dict(kind="matvec", wtype="q5_1", M=1, N=12288, K=4096, seed=0xC0FFEE + 7),
    "q5_K_matvec_12288x4096": dict(kind="matvec", wtype="q5_K", M=1, N=12288, K=4096, seed=0xC0FFEE + 8),
    "q8_kv_cache_32x8x4096x128": dict(kind="kv", Hq=32, Hkv=8, P=4096, hd=128, seed=0xC0FFEE + 9),
}


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """An independent PCG64 stream per (seed, stream)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def weights_f32(N: int, K: int, seed: int, stream: int = 0, row_jitter: bool = False) -> np.ndarray:
    """f32 [N, K] ~ N(0, 0.02); with row_jitter each row's std is scaled by U(0.5, 2)."""
    g = rng(seed, 2 * stream)
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(WEIGHT_STD)
    if row_jitter:
        w *= g.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    return w


def activations_f32(M: int, K: int, seed: int, stream: int = 0) -> np.ndarray:
    """f32 [M, K] ~ N(0, 1) with 1% of entries multiplied by 20."""
    g = rng(seed, 2 * stream + 1)
    x = g.standard_normal((M, K), dtype=np.float32)
    mask = g.random((M, K)) < OUTLIER_P
    x[mask] *= np.float32(OUTLIER_SCALE)
    return x


def uniform_f32(shape, lo: float, hi: float, seed: int) -> np.ndarray:
    return rng(seed, 99).uniform(lo, hi, size=shape).astype(np.float32)


def kv_inputs(Hq: int, Hkv: int, P: int, hd: int, seed: int):
    """Decode-attention inputs: q f32 [Hq, hd], K and V f32 [P * Hkv, hd] (row p * Hkv + kvh),
    attention weights f32 [Hq, P] (each row a softmax of N(0, 4) logits, summing to 1)."""
    q = activations_f32(Hq, hd, seed, stream=0)
    k = activations_f32(P * Hkv, hd, seed, stream=1)
    v = activations_f32(P * Hkv, hd, seed, stream=2)
    z = rng(seed, 6).standard_normal((Hq, P)) * 2.0
    e = np.exp(z - z.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return q, k, v, w
