"""Oracle for k-quant decoding and products: ctypes wrapper around kq_oracle.c.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library never
does, and the two share no code.  ``build()`` compiles the C source with gcc
(fp64 loops, OpenMP over output rows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kq_oracle.c")
LIB = os.path.join(HERE, "libkq_oracle.so")

Q4_K, Q5_K, Q6_K, IA4 = 1, 2, 3, 4
X_F32, X_BF16 = 0, 1
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, IA4: 144}


def build(force: bool = False) -> str:
    """Compile the oracle into libkq_oracle.so next to its source."""
    hdr = os.path.join(HERE, "kq_oracle.h")
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(hdr))):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                           "-o", tmp, SRC, "-lm"])
    os.replace(tmp, LIB)
    return LIB


class _Fields(ctypes.Structure):
    _fields_ = [("d_bits", ctypes.c_uint16), ("dmin_bits", ctypes.c_uint16),
                ("sc", ctypes.c_int * 16), ("m", ctypes.c_int * 8), ("q", ctypes.c_int * 256)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = bind(LIB)
    return _lib


def use_library(path: str | None):
    """Point this wrapper at another build of the oracle source (the pin tests
    use this to check that deliberately broken copies fail); None restores."""
    global _lib
    _lib = bind(path) if path else None


def bind(path: str):
    """Load one build of the oracle and declare its C signatures."""
    L = ctypes.CDLL(path)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.oracle_block_bytes.argtypes = [I]
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_half_to_double.restype = ctypes.c_double
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_unpack.argtypes = [I, P, ctypes.POINTER(_Fields)]
    L.oracle_pack.argtypes = [I, ctypes.POINTER(_Fields), P]
    L.oracle_dequant_block_f64.argtypes = [I, P, P]
    L.oracle_dequant.argtypes = [I, P, I64, P]
    L.oracle_dequant_f64.argtypes = [I, P, I64, P]
    L.oracle_matvec.argtypes = [I, P, I64, I64, P, I, I64, P, P, I]
    L.oracle_moe_matvec.argtypes = [I, P, I, P, P, P, I, I, I64, I64, I64, I, P, P, I]
    return L


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def unpack(qtype: int, blk: np.ndarray) -> dict:
    """Integer fields of one block: d_bits, dmin_bits, sc, m, q (unbiased codes)."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == BLOCK_BYTES[qtype]
    f = _Fields()
    rc = lib().oracle_unpack(qtype, _ptr(blk), ctypes.byref(f))
    assert rc == 0
    nsc = 16 if qtype == Q6_K else 8
    return {"d_bits": f.d_bits, "dmin_bits": f.dmin_bits,
            "sc": np.array(f.sc[:nsc], dtype=np.int32), "m": np.array(f.m[:8], dtype=np.int32),
            "q": np.array(f.q[:], dtype=np.int32)}


def pack(qtype: int, d_bits: int, sc, q, dmin_bits: int = 0, m=None) -> np.ndarray:
    """Build one block's bytes from integer fields."""
    f = _Fields()
    f.d_bits, f.dmin_bits = int(d_bits), int(dmin_bits)
    for i, v in enumerate(sc):
        f.sc[i] = int(v)
    if m is not None:
        for i, v in enumerate(m):
            f.m[i] = int(v)
    for i, v in enumerate(q):
        f.q[i] = int(v)
    out = np.zeros(BLOCK_BYTES[qtype], dtype=np.uint8)
    assert lib().oracle_pack(qtype, ctypes.byref(f), _ptr(out)) == 0
    return out


def dequant_block_f64(qtype: int, blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    w = np.zeros(256, dtype=np.float64)
    assert lib().oracle_dequant_block_f64(qtype, _ptr(blk), _ptr(w)) == 0
    return w


def dequant(qtype: int, blocks: np.ndarray) -> np.ndarray:
    """All blocks (any shape ending in a multiple of the block size) -> fp32 weights."""
    raw = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    nb = raw.size // BLOCK_BYTES[qtype]
    assert nb * BLOCK_BYTES[qtype] == raw.size
    out = np.zeros(nb * 256, dtype=np.float32)
    assert lib().oracle_dequant(qtype, _ptr(raw), nb, _ptr(out)) == 0
    return out


def dequant_f64(qtype: int, blocks: np.ndarray) -> np.ndarray:
    """All blocks -> their exact weights in fp64 (before any fp32 rounding)."""
    raw = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    nb = raw.size // BLOCK_BYTES[qtype]
    assert nb * BLOCK_BYTES[qtype] == raw.size
    out = np.zeros(nb * 256, dtype=np.float64)
    assert lib().oracle_dequant_f64(qtype, _ptr(raw), nb, _ptr(out)) == 0
    return out


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, rounded to nearest, ties to even (the
    plain definition: keep the top 16 bits after adding half an ulp of the
    kept part, plus one if that part is odd); a NaN stays a NaN (quiet, sign
    kept)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x7FFFFF) != 0)
    r[nan] = ((u[nan] >> 16) | 0x0040).astype(np.uint16)
    return r


def dequant_bf16(qtype: int, blocks: np.ndarray) -> np.ndarray:
    """All blocks -> the fp32 weights of dequant, rounded to bfloat16 (bit patterns).
    "GGUF in transformers", "Load GGUF with transformers": GgufConfig(dequantize=True,
    dtype=torch.bfloat16) expands the weights to bf16."""
    return f32_to_bf16_bits(dequant(qtype, blocks))


def _x_arg(x: np.ndarray):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, X_F32
    if x.dtype == np.uint16:  # bfloat16 bit patterns
        return x, X_BF16
    raise TypeError("x must be float32 or uint16 (bfloat16 bits)")


def matvec(qtype: int, W: np.ndarray, N: int, K: int, x: np.ndarray, threads: int = 1):
    """Returns (y, s), both float64 of shape (M, N); x has shape (M, K)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x, xd = _x_arg(x)
    M = x.size // K if K else (x.shape[0] if x.ndim == 2 else 0)
    y = np.zeros((M, N), dtype=np.float64)
    s = np.zeros((M, N), dtype=np.float64)
    rc = lib().oracle_matvec(qtype, _ptr(W), N, K, _ptr(x), xd, M, _ptr(y), _ptr(s), threads)
    assert rc == 0, rc
    return y, s


def moe_matvec(qtype: int, W_experts: np.ndarray, n_experts: int, ids: np.ndarray,
               gate, x: np.ndarray, x_per_slot: bool, N: int, K: int, M: int, top_k: int,
               threads: int = 1):
    """Routed-expert product; returns (y, s) float64 ([M,top_k,N] without gate, [M,N] with)."""
    W_experts = np.ascontiguousarray(W_experts, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    x, xd = _x_arg(x)
    shape = (M, N) if gate is not None else (M, top_k, N)
    y = np.zeros(shape, dtype=np.float64)
    s = np.zeros(shape, dtype=np.float64)
    g = None
    if gate is not None:
        g = np.ascontiguousarray(gate, dtype=np.float32)
    rc = lib().oracle_moe_matvec(qtype, _ptr(W_experts), n_experts, _ptr(ids),
                                 _ptr(g) if g is not None else None, _ptr(x), xd,
                                 int(bool(x_per_slot)), N, K, M, top_k, _ptr(y), _ptr(s), threads)
    if rc != 0:
        raise ValueError(f"oracle_moe_matvec failed: {rc}")
    return y, s


def moe_route(logits: np.ndarray, top_k: int):
    """The MoE router by definition (plain numpy, fp64 arithmetic).

    "GGUF in transformers", "Reusing ggml's Metal kernels": a kernel combining
    softmax and top-k routing; "ANE Fieldfare" README, "How it works": each
    token picks 8 of 128 experts.  Reading: the top_k largest logits of a row in
    descending order, equal logits in ascending index order, a NaN below every
    number; gate_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the selected.
    Returns (ids int32 [M, top_k], gate float64 [M, top_k])."""
    logits = np.asarray(logits, dtype=np.float32)
    M, E = logits.shape
    ids = np.zeros((M, top_k), dtype=np.int32)
    gate = np.zeros((M, top_k), dtype=np.float64)
    for m in range(M):
        row = logits[m].astype(np.float64)
        nan = np.isnan(row)
        neg = np.where(nan, 0.0, -row)  # ascending -value = descending value
        order = np.lexsort((np.arange(E), neg, nan))  # NaN last, then value desc, then index asc
        sel = order[:top_k]
        ids[m] = sel
        l = row[sel]
        with np.errstate(invalid="ignore"):  # an infinite or NaN leading logit gives NaN gates
            ex = np.exp(l - l[0])
            gate[m] = ex / np.sum(ex)
    return ids, gate


def moe_group(ids: np.ndarray, n_experts: int):
    """Grouping of routed (token, slot) pairs by expert, by its definition:
    the distinct valid ids in ascending order, and for each the pair indices
    m*top_k + j holding it, in (m, j) order.  Ids outside [0, n_experts) are
    left out.  Returns (experts, offsets, pairs) as Python lists."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    experts = sorted({v for v in flat if 0 <= v < n_experts})
    pairs, offsets = [], []
    for e in experts:
        offsets.append(len(pairs))
        pairs.extend(i for i, v in enumerate(flat) if v == e)
    offsets.append(len(pairs))
    return experts, offsets, pairs


def ffn_act(act: int, g: np.ndarray) -> np.ndarray:
    """The FFN activations by definition, fp64: 0 = SiLU g / (1 + e^-g);
    1 = GELU in its tanh form, 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))."""
    g = np.asarray(g, dtype=np.float64)
    if act == 1:
        return 0.5 * g * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (g + 0.044715 * g ** 3)))
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def _x_f64(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:  # bfloat16 bits: the high half of an fp32
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def _matrix_f64(qtype: int, W: np.ndarray, row0: int, N: int, K: int) -> np.ndarray:
    """Rows row0 .. row0+N of a block matrix with K columns, as fp64 [N, K]."""
    nb = (K + 255) // 256
    rb = nb * BLOCK_BYTES[qtype]
    raw = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)[row0 * rb:(row0 + N) * rb]
    return dequant_f64(qtype, raw).reshape(N, nb * 256)[:, :K]


def moe_ffn(type_gu: int, W_gate, W_up, type_dn: int, W_down, n_experts: int, ids, gate, x, act: int,
            H: int, F: int, M: int, top_k: int, shared=None):
    """The expert FFN of one MoE layer by its definition (fp64, numpy matmul on
    the exact weights, as every product here uses them).

    "ANE Fieldfare" README, "How it works": a shared FFN every token goes
    through plus the routed experts each token picked.  Reading: gated FFN
    blocks, h = act(W_gate x) * (W_up x), y = sum_j g_j W_down[e_j] h_j + shared.
    shared = (Ws_gate, Ws_up, Ws_down, SH) or None.  Ids outside
    [0, n_experts) are dropped.  Returns a dict: y, s (sum of |g_j| |W_down| |h_j|
    plus the shared |Ws_down| |hs|), h, g, u [M*top_k, F] (NaN for dropped
    pairs: h and the gate and up products), sg, su (their |W| |x| sums), and
    hs, gs, us, sgs, sus for the shared expert."""
    ids = np.asarray(ids, dtype=np.int64).reshape(M, top_k)
    gate = np.asarray(gate, dtype=np.float32).astype(np.float64).reshape(M, top_k)
    X = _x_f64(x).reshape(M, H)
    AX = np.abs(X)
    MK = M * top_k
    out = {"y": np.zeros((M, H)), "s": np.zeros((M, H)), "h": np.full((MK, F), np.nan),
           "g": np.full((MK, F), np.nan), "u": np.full((MK, F), np.nan),
           "sg": np.zeros((MK, F)), "su": np.zeros((MK, F))}
    for e in sorted({int(v) for v in ids.reshape(-1) if 0 <= v < n_experts}):
        pairs = [i for i in range(MK) if ids.reshape(-1)[i] == e]
        ms = [p // top_k for p in pairs]
        Wg = _matrix_f64(type_gu, W_gate, e * F, F, H)
        Wu = _matrix_f64(type_gu, W_up, e * F, F, H)
        g, u = X[ms] @ Wg.T, X[ms] @ Wu.T
        h = ffn_act(act, g) * u
        out["h"][pairs], out["g"][pairs], out["u"][pairs] = h, g, u
        out["sg"][pairs], out["su"][pairs] = AX[ms] @ np.abs(Wg).T, AX[ms] @ np.abs(Wu).T
        del Wg, Wu
        Wd = _matrix_f64(type_dn, W_down, e * H, H, F)
        d, sd = h @ Wd.T, np.abs(h) @ np.abs(Wd).T
        for k, p in enumerate(pairs):
            m, j = divmod(p, top_k)
            out["y"][m] += gate[m, j] * d[k]
            out["s"][m] += abs(gate[m, j]) * sd[k]
    if shared is not None:
        Wsg, Wsu, Wsd, SH = shared
        A = _matrix_f64(type_gu, Wsg, 0, SH, H)
        B = _matrix_f64(type_gu, Wsu, 0, SH, H)
        g, u = X @ A.T, X @ B.T
        hs = ffn_act(act, g) * u
        out.update(hs=hs, gs=g, us=u, sgs=AX @ np.abs(A).T, sus=AX @ np.abs(B).T)
        Cd = _matrix_f64(type_dn, Wsd, 0, H, SH)
        out["y"] += hs @ Cd.T
        out["s"] += np.abs(hs) @ np.abs(Cd).T
    return out


def _bf16_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def ia4_dequant_mlx(q: np.ndarray, scales: np.ndarray, biases: np.ndarray, N: int, K: int) -> np.ndarray:
    """Group-affine INT4 by its definition, straight from MLX's arrays (fp64
    [N, K]): code k of row n = bits 4(k%8).. of word q[n, k//8], w = scale *
    code + bias with the bf16 scale and bias of group k//64.  "ANE Fieldfare"
    README, "Requirements": the experts are an mlx-community 4-bit
    checkpoint; reading: MLX's affine form, groups of 64."""
    q = np.asarray(q, dtype=np.uint32).reshape(N, K // 8)
    k = np.arange(K)
    codes = (q[:, k // 8] >> (4 * (k % 8)).astype(np.uint32)) & 15
    s = _bf16_f64(np.asarray(scales).reshape(N, K // 64))[:, k // 64]
    b = _bf16_f64(np.asarray(biases).reshape(N, K // 64))[:, k // 64]
    return s * codes.astype(np.float64) + b


def ia4_pack(q: np.ndarray, scales: np.ndarray, biases: np.ndarray, N: int, K: int) -> np.ndarray:
    """MLX's arrays -> IA4 blocks (uint8, N * ceil(K/256) * 144 bytes), by the
    block layout: per block, 4 bf16 scales, 4 bf16 biases, then for group g
    and l < 32 the byte (code of weight 64g+l) | (code of weight 64g+32+l) << 4;
    groups past K are zero."""
    q = np.asarray(q, dtype=np.uint32).reshape(N, K // 8)
    scales = np.asarray(scales, dtype=np.uint16).reshape(N, K // 64)
    biases = np.asarray(biases, dtype=np.uint16).reshape(N, K // 64)
    nb = (K + 255) // 256
    out = np.zeros((N, nb, 144), dtype=np.uint8)
    for n in range(N):
        for G in range(K // 64):
            b, g = divmod(G, 4)
            out[n, b, 2 * g:2 * g + 2] = np.array([scales[n, G]], dtype="<u2").view(np.uint8)
            out[n, b, 8 + 2 * g:10 + 2 * g] = np.array([biases[n, G]], dtype="<u2").view(np.uint8)
            for l in range(32):
                lo_k, hi_k = 64 * G + l, 64 * G + 32 + l
                lo = (int(q[n, lo_k // 8]) >> (4 * (lo_k % 8))) & 15
                hi = (int(q[n, hi_k // 8]) >> (4 * (hi_k % 8))) & 15
                out[n, b, 16 + 32 * g + l] = lo | (hi << 4)
    return out.reshape(-1)
