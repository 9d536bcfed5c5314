"""Activation outliers inside a 128-value run, on every path that stages x.

x = N(0,1) with one large value in each 128-run (bf16 x: 2^12, fp32 x: 2^14),
and a third of the rows have weight exactly 0 at every outlier's column
(Q6_K code 32; Q4_K/Q5_K dmin = d, m_j = sc_j and code 1; IA4 bias = -8 scale
and code 8), so the outlier adds nothing to sum|w x| and every other term
must be carried to the tolerance.  Elementwise against the oracle at
max |y_gpu - y_ref| / sum_k |w x| <= 1e-4 (fp32 x) / 4e-3 (bf16 x):

* one-token products, two to four tokens (rows bit-identical to one token),
  the tensor cores (M = 5..16), the batched fp32 product (M >= 2), chains;
* routed-expert products in both forms and the expert FFN;
* blocks with 0..21 values off the image's grid (the entry list fills at 20;
  one more keeps the block as raw bf16) and runs whose outlier leaves every
  other value off the grid.
"""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, rel_err, require_gpu, x_dev

pytestmark = pytest.mark.gpu
Q4_K, Q5_K, Q6_K, IA4 = 1, 2, 3, 4
TYPES = [Q4_K, Q5_K, Q6_K, IA4]
MAG = {"bf16": 2.0 ** 12, "f32": 2.0 ** 14}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    kq.kq_device_error(clear=True)
    yield
    assert kq.kq_device_error() == 0, "device error word set"


def outlier_x(M, K, g, xd, mag=None):
    """M x K: N(0,1) with one value of magnitude mag at a random place in each
    128-run; returns (x in the dtype's encoding, the outlier columns per row)."""
    mag = MAG[xd] if mag is None else mag
    x = g.standard_normal((M, K), dtype=np.float32)
    cols = []
    for m in range(M):
        c = [r + int(g.integers(0, min(128, K - r))) for r in range(0, K, 128)]
        x[m, c] = mag * np.where(g.random(len(c)) < 0.5, -1.0, 1.0)
        cols.append(c)
    return (synth.to_bf16_bits(x) if xd == "bf16" else x), cols


def zero_weights(qtype, W, N, K, rows, cols):
    """W with the weight at (row, col) made exactly zero for every row in rows
    and col in cols (each block's other weights keep their codes)."""
    W = W.copy()
    BB = synth.BLOCK_BYTES[qtype]
    nb = (K + 255) // 256
    blk = W.reshape(N, nb, BB)
    by_block = {}
    for k in sorted(set(int(c) for c in cols)):
        by_block.setdefault(k // 256, []).append(k % 256)
    for r in rows:
        for b, idx in by_block.items():
            if qtype == IA4:
                hdr = blk[r, b, :16].copy().view("<u2")
                for i in idx:
                    grp = i // 64
                    sc = float(np.array([np.uint32(hdr[grp]) << np.uint32(16)], dtype=np.uint32).view(np.float32)[0])
                    hdr[4 + grp] = synth.to_bf16_bits(np.array([-8.0 * sc], dtype=np.float32))[0]
                    ci = 16 + 32 * (i >> 6) + (i & 31)
                    sh = 4 * ((i >> 5) & 1)
                    blk[r, b, ci] = (int(blk[r, b, ci]) & ~(15 << sh) | (8 << sh)) & 0xFF
                blk[r, b, :16] = hdr.view(np.uint8)
                continue
            f = oracle.unpack(qtype, blk[r, b])
            q = f["q"].copy()
            if qtype == Q6_K:
                q[idx] = 32
                blk[r, b] = oracle.pack(qtype, f["d_bits"], f["sc"], q)
            else:
                sc, m = f["sc"].copy(), f["m"].copy()
                for i in idx:
                    j = i // 32
                    sc[j] = max(int(sc[j]), 1)
                    m[j] = sc[j]
                    q[i] = 1
                blk[r, b] = oracle.pack(qtype, f["d_bits"], sc, q, f["d_bits"], m)
    return W


def case(qtype, N, K, M, xd, seed, zero_every=3, mag=None):
    g = synth.rng(seed, qtype, N, K, M)
    x, cols = outlier_x(M, K, g, xd, mag)
    W = synth.gen_matrix(qtype, N, K, g)
    allc = [c for cs in cols for c in cs]
    W = zero_weights(qtype, W, N, K, range(0, N, zero_every), allc)
    return W, x


def check(qtype, W, N, K, x, y, xd):
    yr, sr = oracle.matvec(qtype, W, N, K, x, threads=8)
    err = rel_err(np.asarray(y).reshape(yr.shape), yr, sr)
    assert err <= TOL[xd], err
    return err


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("xd", ["bf16", "f32"])
@pytest.mark.parametrize("K", [256, 768, 2560])
def test_one_token(qtype, xd, K):
    N = 99
    W, x = case(qtype, N, K, 1, xd, 700)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    check(qtype, W, N, K, x, y, xd)


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [2, 3, 4])
def test_few_tokens_bit_identical(qtype, M):
    N, K = 77, 768
    W, x = case(qtype, N, K, M, "bf16", 701)
    Wd, xd_ = dev(W), x_dev(x)
    y = kq.matvec(qtype, Wd, xd_, N, K)
    check(qtype, W, N, K, x, y.cpu().numpy(), "bf16")
    for m in range(M):
        assert torch.equal(y[m], kq.matvec(qtype, Wd, xd_[m:m + 1], N, K)[0]), m


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [5, 8, 16])
def test_tensor_cores(qtype, M):
    N, K = 300, 2560
    W, x = case(qtype, N, K, M, "bf16", 702)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    check(qtype, W, N, K, x, y, "bf16")


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [2, 5])
def test_batched_fp32(qtype, M):
    N, K = 150, 768
    W, x = case(qtype, N, K, M, "f32", 703)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    check(qtype, W, N, K, x, y, "f32")


def test_chain_mixed_dtypes():
    """A chain with bf16 and fp32 ops (the fp32 ones as two images), with and
    without grid barriers and split K."""
    specs = [(Q4_K, 1000, 2560, "bf16", 0), (Q6_K, 512, 2560, "f32", 0), (Q5_K, 700, 4096, "bf16", 1),
             (Q4_K, 2560, 9728, "bf16", 1), (Q6_K, 96, 768, "f32", 0)]
    ops, ref = [], []
    for i, (qt, N, K, xd, wait) in enumerate(specs):
        W, x = case(qt, N, K, 1, xd, 704 + i)
        y = torch.full((N,), np.nan, device="cuda")
        ops.append({"type": qt, "x_dtype": kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, "W": dev(W),
                    "x": x_dev(x), "y": y, "N": N, "K": K, "wait_previous": wait})
        ref.append((qt, W, N, K, x, xd))
    ch = kq.Chain(ops)
    ch.run()
    torch.cuda.synchronize()
    for o, (qt, W, N, K, x, xd) in zip(ops, ref):
        check(qt, W, N, K, x, o["y"].cpu().numpy(), xd)


@pytest.mark.parametrize("qtype", [Q4_K, Q6_K, IA4])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("xd", ["bf16", "f32"])
def test_moe(qtype, gated, xd):
    E, M, top_k = 32, 4, 4
    N, K = (768, 704) if gated else (704, 768)
    g = synth.rng(710, qtype, int(gated))
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x, cols = outlier_x(M * top_k if gated else M, K, g, xd)
    We = synth.gen_matrix(qtype, E * N, K, g)
    allc = [c for cs in cols for c in cs]
    We = zero_weights(qtype, We, E * N, K, range(0, E * N, 3), allc)
    ws = kq.moe_workspace(N, M, top_k, E)
    shape = (M, N) if gated else (M, top_k, N)
    y = torch.full(shape, np.nan, device="cuda")
    kq.kq_moe_matvec(qtype, dev(We), E, dev(ids), dev(gate) if gated else None, x_dev(x),
                     kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, gated, y, N, K, M, top_k, ws, ws.numel())
    kq.kq_moe_check(ws)
    yr, sr = oracle.moe_matvec(qtype, We, E, ids, gate if gated else None, x, gated, N, K, M, top_k, threads=8)
    assert rel_err(y.cpu().numpy(), yr, sr) <= TOL[xd]


def test_expert_ffn():
    """The expert FFN with outliers in x: h against the fp64 definition, the
    down stage (fp32 h as x: two images) against the oracle on the same h."""
    from tests import test_gpu_ffn as F
    c = F._case(720, 16, 512, 320, 288, 4, 4, Q4_K, Q6_K, "bf16")
    c["x"], _ = outlier_x(4, 512, synth.rng(721), "bf16")
    y, h, hs, ws = F._run(c, kq.KQ_ACT_SILU)
    r = F._ref(c, kq.KQ_ACT_SILU)
    F._check_h(c, kq.KQ_ACT_SILU, h, hs, r)
    F._check_down(c, y, h, hs)
    kq.kq_moe_check(ws)


def listed_x(K, n_off, g):
    """bf16 x of one row whose first 128-run has a maximum of 2^12 (grid step
    2^-9) and exactly n_off values off that grid (magnitudes near 0.1); every
    other value is on the grid of its run (|v| >= 0.25, bf16)."""
    x = g.standard_normal(K).astype(np.float32)
    x = np.where(np.abs(x) < 0.25, np.sign(x + 1e-9) * 0.25, x)
    x[0] = 2.0 ** 12
    pos = 1 + g.permutation(127)[:n_off]
    # odd multiples of 2^-11 near 0.1: exact in bf16, never multiples of 2^-9
    x[pos] = (4 * g.integers(48, 56, n_off) + 1) * 2.0 ** -11 * np.where(g.random(n_off) < 0.5, -1.0, 1.0)
    xb = synth.to_bf16_bits(x[None, :])
    v = (xb.astype(np.uint32) << 16).view(np.float32)[0]
    off = np.count_nonzero(v[:128] * 512.0 != np.rint(v[:128] * 512.0))
    assert off == n_off
    return xb


@pytest.mark.parametrize("n_off", [0, 1, 4, 5, 19, 20, 21, 64, 127])
@pytest.mark.parametrize("qtype", TYPES)
def test_entry_list_and_raw_blocks(qtype, n_off):
    N, K = 64, 768
    g = synth.rng(730, qtype, n_off)
    x = listed_x(K, n_off, g)
    W = zero_weights(qtype, synth.gen_matrix(qtype, N, K, g), N, K, range(0, N, 2), [0])
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    check(qtype, W, N, K, x, y, "bf16")
    if n_off in (20, 21):  # the same rows through the routed-expert kernel
        ws = kq.moe_workspace(N, 1, 1, 1)
        ym = torch.full((1, 1, N), np.nan, device="cuda")
        kq.kq_moe_matvec(qtype, dev(W), 1, dev(np.zeros((1, 1), np.int32)), None, x_dev(x), kq.KQ_BF16, 0, ym,
                         N, K, 1, 1, ws, ws.numel())
        check(qtype, W, N, K, x, ym.cpu().numpy()[0], "bf16")


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("xd,mag", [("bf16", 2.0 ** 16), ("bf16", 2.0 ** 40), ("f32", 2.0 ** 20),
                                    ("f32", 2.0 ** 60)])
def test_huge_outliers(qtype, xd, mag):
    """Outliers so large that nearly every other value of their run is off the
    grid (raw blocks)."""
    N, K = 64, 1024
    W, x = case(qtype, N, K, 1, xd, 740, zero_every=2, mag=mag)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    check(qtype, W, N, K, x, y, xd)
