"""Seeded synthetic inputs: quantized weight bytes, activations and routing.

This module holds no decoding or product arithmetic.  Weight blocks are random
bytes placed at each field's byte offset:

* code fields (Q4_K/Q5_K ``qs``/``qh``, Q6_K ``ql``/``qh``) are uniform random
  bytes, so every 4/5/6-bit code is uniform over its full range;
* the 12-byte Q4_K/Q5_K scale field is uniform random bytes -- its 16 six-bit
  scales and mins are a bijective re-arrangement of those 96 bits, so each is
  uniform over 0..63 and independent;
* Q6_K scales are int8 drawn uniformly from a given range;
* ``d`` / ``dmin`` are ``|N(0, sigma)|`` rounded to fp16 (round to nearest even).

IA4 (group-affine INT4) blocks put bf16 scales ``|N(0, sigma)|`` and biases
``-8 * scale * (1 + N(0, 1)/4)`` in the header and uniform random code bytes
after it; ``gen_ia4_mlx`` draws the same kind of matrix in MLX's layout (code
words, scales, biases).

Activations are fp32 N(0, 1), optionally rounded to bfloat16 (nearest even) and
returned as raw bit patterns.  Routing inputs are drawn directly: distinct
expert ids uniform per token and flat-Dirichlet gate weights, or router logits
(N(0, 1), integer-valued, or with a component shared by all tokens).

Used by the tests (feeding the oracle and the CUDA path the same bytes) and by
the benchmark.
"""
from __future__ import annotations

import numpy as np
import torch

Q4_K, Q5_K, Q6_K, IA4 = 1, 2, 3, 4
TYPE_NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", IA4: "IA4"}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, IA4: 144}
QK = 256

# byte offsets of the fields of one block (format reading; see the design notes)
_D_OFF = {Q4_K: 0, Q5_K: 0, Q6_K: 208}
_DMIN_OFF = {Q4_K: 2, Q5_K: 2}
_SCALES = {Q4_K: (4, 12), Q5_K: (4, 12), Q6_K: (192, 16)}


def rng(seed: int, *stream: int) -> np.random.Generator:
    """An independent generator per (seed, stream...) tuple."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, stream)])))


def n_blocks_per_row(K: int) -> int:
    return (K + QK - 1) // QK


def matrix_bytes(qtype: int, N: int, K: int) -> int:
    return N * n_blocks_per_row(K) * BLOCK_BYTES[qtype]


def _half_bits(g: np.random.Generator, n: int, sigma: float) -> np.ndarray:
    return np.abs(g.normal(0.0, sigma, n)).astype(np.float16).view(np.uint16)


def gen_blocks(qtype: int, n_blocks: int, g: np.random.Generator, *, d_sigma: float = 0.002,
               q6_scale_range: tuple[int, int] = (-128, 127)) -> np.ndarray:
    """``n_blocks`` random blocks as a (n_blocks, block_bytes) uint8 array."""
    nbytes = BLOCK_BYTES[qtype]
    out = g.integers(0, 256, size=(n_blocks, nbytes), dtype=np.uint8)
    if qtype == IA4:
        s, b = _ia4_scale_bias(g, n_blocks * 4, d_sigma)
        out[:, 0:8] = s.reshape(n_blocks, 4).astype("<u2").view(np.uint8).reshape(n_blocks, 8)
        out[:, 8:16] = b.reshape(n_blocks, 4).astype("<u2").view(np.uint8).reshape(n_blocks, 8)
        return out
    d = _half_bits(g, n_blocks, d_sigma)
    o = _D_OFF[qtype]
    out[:, o] = (d & 0xFF).astype(np.uint8)
    out[:, o + 1] = (d >> 8).astype(np.uint8)
    if qtype in _DMIN_OFF:
        dm = _half_bits(g, n_blocks, d_sigma)
        o = _DMIN_OFF[qtype]
        out[:, o] = (dm & 0xFF).astype(np.uint8)
        out[:, o + 1] = (dm >> 8).astype(np.uint8)
    if qtype == Q6_K:
        lo, hi = q6_scale_range
        off, cnt = _SCALES[Q6_K]
        sc = g.integers(lo, hi + 1, size=(n_blocks, cnt), dtype=np.int64).astype(np.int8)
        out[:, off:off + cnt] = sc.view(np.uint8)
    return out


def _bf16_bits_of(v: np.ndarray) -> np.ndarray:
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _ia4_scale_bias(g: np.random.Generator, n: int, sigma: float):
    """bf16 bit patterns of n scales |N(0, sigma)| and biases -8 * scale * (1 + N(0,1)/4)."""
    s = np.abs(g.normal(0.0, sigma, n)).astype(np.float32)
    b = (-8.0 * s * (1.0 + 0.25 * g.standard_normal(n))).astype(np.float32)
    return _bf16_bits_of(s), _bf16_bits_of(b)


def gen_ia4_mlx(N: int, K: int, g: np.random.Generator, sigma: float = 0.002):
    """A group-affine INT4 matrix in MLX's layout: (code words uint32 [N, K/8],
    scales bf16 bits [N, K/64], biases bf16 bits [N, K/64]); K a multiple of 64."""
    q = g.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s, b = _ia4_scale_bias(g, N * (K // 64), sigma)
    return q, s.reshape(N, K // 64), b.reshape(N, K // 64)


def gen_matrix(qtype: int, N: int, K: int, g: np.random.Generator, **kw) -> np.ndarray:
    """A row-major N x ceil(K/256) matrix of blocks, flattened to bytes."""
    return gen_blocks(qtype, N * n_blocks_per_row(K), g, **kw).reshape(-1)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 (round to nearest even) bit patterns as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def gen_x(M: int, K: int, g: np.random.Generator, dtype: str = "f32") -> np.ndarray:
    """M x K activations: float32, or bfloat16 bit patterns (uint16) if dtype == 'bf16'."""
    x = g.standard_normal((M, K), dtype=np.float32)
    if dtype == "bf16":
        return to_bf16_bits(x)
    return x


def gen_routing(M: int, n_experts: int, top_k: int, g: np.random.Generator):
    """(ids int32 [M, top_k], gate float32 [M, top_k]): top_k distinct experts
    per token drawn uniformly, positive gates summing to about 1 (a flat
    Dirichlet draw).  Drawn directly, not by routing logits."""
    ids = np.stack([g.permutation(n_experts)[:top_k] for _ in range(M)]).astype(np.int32).reshape(M, top_k)
    gate = g.dirichlet(np.ones(top_k), size=M).astype(np.float32).reshape(M, top_k)
    return ids, gate


def gen_logits(M: int, n_experts: int, g: np.random.Generator, ties: bool = False, rho: float = 0.0) -> np.ndarray:
    """Router logits [M, n_experts] fp32: N(0, 1), or small integers (-4..4)
    so that equal logits are common.  rho > 0 correlates the tokens (as
    neighbouring tokens of a verify block are): sqrt(rho) z + sqrt(1 - rho) z_m
    with one N(0, 1) draw z shared by all tokens; rho = 0.62 makes 8 tokens'
    top-8 of 128 cover about 29 distinct experts."""
    if ties:
        return g.integers(-4, 5, size=(M, n_experts)).astype(np.float32)
    if rho > 0.0:
        z = g.standard_normal(n_experts)
        return (np.sqrt(rho) * z + np.sqrt(1.0 - rho) * g.standard_normal((M, n_experts))).astype(np.float32)
    return g.standard_normal((M, n_experts), dtype=np.float32)


# --------------------------------------------------------------------------
# Workload shapes (synthetic stand-ins for the checkpoints the pages load).
# --------------------------------------------------------------------------

def dense_layer_sweep(n_layers: int = 36, hidden: int = 2560, q_out: int = 4096, kv_out: int = 1024,
                      ffn: int = 9728, vocab: int = 151936):
    """4B-class dense decoder in a Q4_K_M mix: a list of stages, each a list of
    (name, qtype, N, K) matrices that share one input vector.  Q6_K holds v_proj
    and down_proj on even layers and the LM head; everything else is Q4_K."""
    stages = []
    for layer in range(n_layers):
        hi = (layer % 2 == 0)
        v_t = Q6_K if hi else Q4_K
        d_t = Q6_K if hi else Q4_K
        stages.append([(f"L{layer}.q_proj", Q4_K, q_out, hidden),
                       (f"L{layer}.k_proj", Q4_K, kv_out, hidden),
                       (f"L{layer}.v_proj", v_t, kv_out, hidden)])
        stages.append([(f"L{layer}.o_proj", Q4_K, hidden, q_out)])
        stages.append([(f"L{layer}.gate_proj", Q4_K, ffn, hidden),
                       (f"L{layer}.up_proj", Q4_K, ffn, hidden)])
        stages.append([(f"L{layer}.down_proj", d_t, hidden, ffn)])
    stages.append([("lm_head", Q6_K, vocab, hidden)])
    return stages
