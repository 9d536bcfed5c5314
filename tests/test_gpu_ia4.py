"""Parity of the group-affine INT4 format (KQ_IA4) through the C ABI with the
oracle: regrouping from MLX's arrays (bit-exact), dequantization (bit-exact),
products for M = 1..16 with fp32 and bf16 x (the few-token rows bit-identical
to one-token products), routed-expert products and the expert FFN with IA4
experts."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, rel_err, require_gpu, x_dev

pytestmark = pytest.mark.gpu
IA4 = 4


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    yield
    assert kq.kq_device_error() == 0, "device error word set"


def _mlx_dev(q, s, b):
    return (torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(s.view(np.int16)).cuda(),
            torch.from_numpy(b.view(np.int16)).cuda())


@pytest.mark.parametrize("NK", [(1, 64), (3, 320), (17, 704), (64, 2816), (5, 4096 + 192)])
def test_ia4_pack_bit_exact(NK):
    N, K = NK
    q, s, b = synth.gen_ia4_mlx(N, K, synth.rng(401, N, K))
    blk = kq.ia4_pack(*_mlx_dev(q, s, b)).cpu().numpy()
    assert np.array_equal(blk, oracle.ia4_pack(q, s, b, N, K))


@pytest.mark.parametrize("nblocks", [1, 7, 1000])
def test_ia4_dequant_bit_exact(nblocks):
    blocks = synth.gen_blocks(IA4, nblocks, synth.rng(402, nblocks)).reshape(-1)
    w = kq.dequant(IA4, dev(blocks), 256 * nblocks).cpu().numpy()
    assert np.array_equal(w.view(np.uint32), oracle.dequant(IA4, blocks).view(np.uint32))
    wb = kq.dequant_bf16(IA4, dev(blocks), 256 * nblocks).cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wb, oracle.dequant_bf16(IA4, blocks))


def _case(N, K, M, xd, seed):
    g = synth.rng(seed, N, K, M)
    W = synth.gen_matrix(IA4, N, K, g)
    x = synth.gen_x(M, K, g, xd)
    y = kq.matvec(IA4, dev(W), x_dev(x), N, K).cpu().numpy()
    yr, sr = oracle.matvec(IA4, W, N, K, x, threads=8)
    return y, yr, sr


@pytest.mark.parametrize("xd", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("NK", [(1, 256), (33, 704), (130, 2560), (300, 2816), (64, 4096 + 96)])
def test_ia4_matvec(NK, M, xd):
    """Every path: one-token kernel (M = 1; M = 2..4 with bf16 x), tensor
    cores (bf16 x, M > 4), batched CUDA-core product (fp32 x, M > 1)."""
    N, K = NK
    y, yr, sr = _case(N, K, M, xd, 403)
    assert rel_err(y, yr, sr) <= TOL[xd]


@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("NK", [(300, 2816), (4096, 4096)])
def test_ia4_few_tokens_bit_identical_to_one(NK, M):
    N, K = NK
    g = synth.rng(404, N, K, M)
    W = dev(synth.gen_matrix(IA4, N, K, g))
    x = x_dev(synth.gen_x(M, K, g, "bf16"))
    yM = kq.matvec(IA4, W, x, N, K)
    for m in range(M):
        assert torch.equal(yM[m], kq.matvec(IA4, W, x[m:m + 1], N, K)[0]), m


def test_ia4_packed_mlx_matrix_product():
    """From MLX's arrays to a product: pack on the GPU, multiply, compare with
    the MLX definition's weights times x (fp64)."""
    N, K = 704, 2816
    q, s, b = synth.gen_ia4_mlx(N, K, synth.rng(405))
    x = synth.gen_x(1, K, synth.rng(406), "bf16")
    blk = kq.ia4_pack(*_mlx_dev(q, s, b))
    y = kq.matvec(IA4, blk, x_dev(x), N, K).cpu().numpy().astype(np.float64)
    w = oracle.ia4_dequant_mlx(q, s, b, N, K)
    xf = oracle._x_f64(x)
    yr, sr = xf @ w.T, np.abs(xf) @ np.abs(w).T
    assert np.max(np.abs(y - yr) / sr) <= TOL["bf16"]


@pytest.mark.parametrize("xd", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 16])
def test_ia4_moe_products(M, xd):
    """Routed IA4 experts: per-slot gate/up form and gated down form."""
    E, top_k, H, F = 32, 4, 1024, 320
    g = synth.rng(407, M)
    Wg = synth.gen_matrix(IA4, E * F, H, g)
    Wd = synth.gen_matrix(IA4, E * H, F, g)
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = synth.gen_x(M, H, g, xd)
    xs = synth.gen_x(M * top_k, F, g, xd)
    xdt = kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32
    ws = kq.moe_workspace(max(F, H), M, top_k, E)
    yg = torch.full((M, top_k, F), np.nan, device="cuda")
    kq.kq_moe_matvec(IA4, dev(Wg), E, dev(ids), None, x_dev(x), xdt, 0, yg, F, H, M, top_k, ws, ws.numel())
    yd = torch.full((M, H), np.nan, device="cuda")
    kq.kq_moe_matvec(IA4, dev(Wd), E, dev(ids), dev(gate), x_dev(xs), xdt, 1, yd, H, F, M, top_k, ws, ws.numel())
    torch.cuda.synchronize()
    kq.kq_moe_check(ws)
    rg, sg = oracle.moe_matvec(IA4, Wg, E, ids, None, x, False, F, H, M, top_k)
    rd, sd = oracle.moe_matvec(IA4, Wd, E, ids, gate, xs, True, H, F, M, top_k)
    assert np.max(np.abs(yg.cpu().numpy() - rg) / sg) <= TOL[xd]
    assert np.max(np.abs(yd.cpu().numpy() - rd) / sd) <= TOL[xd]


def test_ia4_expert_ffn():
    """The expert FFN with IA4 routed and shared experts against the fp64
    definition (whole layer, the intermediate h in fp32)."""
    E, H, F, SH, M, top_k = 16, 512, 320, 256, 4, 4
    g = synth.rng(408)
    Wg, Wu = synth.gen_matrix(IA4, E * F, H, g), synth.gen_matrix(IA4, E * F, H, g)
    Wd = synth.gen_matrix(IA4, E * H, F, g)
    Sg, Su, Sd = synth.gen_matrix(IA4, SH, H, g), synth.gen_matrix(IA4, SH, H, g), synth.gen_matrix(IA4, H, SH, g)
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = synth.gen_x(M, H, g, "f32")
    t = [dev(a) for a in (Wg, Wu, Wd, Sg, Su, Sd)]
    w = kq.ffn_weights(IA4, IA4, E, kq.KQ_ACT_GELU_TANH, F, t[0], t[1], t[2], SH, t[3], t[4], t[5])
    ws = kq.moe_ffn_workspace(H, F, SH, M, top_k, E)
    y = torch.full((M, H), np.nan, device="cuda")
    kq.kq_moe_ffn(w, dev(ids), dev(gate), x_dev(x), kq.KQ_F32, y, H, M, top_k, ws, ws.numel())
    torch.cuda.synchronize()
    kq.kq_moe_check(ws)
    h_off, hs_off = kq.kq_moe_ffn_offsets(H, F, SH, M, top_k, E)
    wsn = ws.cpu().numpy()
    h = wsn[h_off:h_off + 4 * M * top_k * F].view(np.float32).reshape(M * top_k, F)
    hs = wsn[hs_off:hs_off + 4 * M * SH].view(np.float32).reshape(M, SH)
    # the down stage against the oracle's products on the same h
    yr, sr = oracle.moe_matvec(IA4, Wd, E, ids, gate, np.ascontiguousarray(h), True, H, F, M, top_k)
    ys, ss = oracle.matvec(IA4, Sd, H, SH, np.ascontiguousarray(hs))
    assert np.all(np.abs(y.cpu().numpy() - (yr + ys)) <= TOL["f32"] * (sr + ss) + 1e-30)
    # h against the fp64 definition (fp32 x: the products' bound carried through the activation)
    r = oracle.moe_ffn(IA4, Wg, Wu, IA4, Wd, E, ids, gate, x, kq.KQ_ACT_GELU_TANH, H, F, M, top_k,
                       shared=(Sg, Su, Sd, SH))
    eps = TOL["f32"]
    act = oracle.ffn_act(1, r["g"])
    bound = eps * (1.13 * np.abs(r["u"]) * r["sg"] + np.abs(act) * r["su"]) + 2e-6 * np.abs(r["h"]) + 1e-30
    assert np.all(np.abs(h - r["h"]) <= bound)
