"""Parity of the CUDA path (through the C ABI) with the oracle.

* unpack: codes, scales, mins, d, dmin bit-exact;
* dequant: fp32 weights bit-exact;
* matvec: max |y_gpu - y_oracle| / sum_k |w x| <= 1e-4 (fp32 x) / 4e-3 (bf16 x),
  on sizes that span several tiles and a ragged tail, the degenerate shapes,
  and the full-size matrices of the benchmark workloads (sampled rows);
* rows of a batched product match the one-token product within tolerance;
* no writes outside y.
"""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, rel_err, require_gpu, x_dev

pytestmark = pytest.mark.gpu
Q4_K, Q5_K, Q6_K = 1, 2, 3
TYPES = [Q4_K, Q5_K, Q6_K]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    assert kq.kq_device_error(clear=True) in (0, 1, 2, 3)
    yield
    assert kq.kq_device_error() == 0, "device error word set"


@pytest.mark.parametrize("qtype", TYPES)
def test_unpack_bit_exact(qtype):
    g = synth.rng(200, qtype)
    nb = 1000
    blocks = g.integers(0, 256, size=(nb, synth.BLOCK_BYTES[qtype]), dtype=np.uint8)
    bd = dev(blocks.reshape(-1))
    codes = torch.zeros(nb * 256, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(nb * 16, dtype=torch.int8, device="cuda")
    mins = torch.zeros(nb * 8, dtype=torch.uint8, device="cuda")
    d = torch.zeros(nb, dtype=torch.int16, device="cuda")
    dm = torch.zeros(nb, dtype=torch.int16, device="cuda")
    kq.kq_unpack(qtype, bd, nb, codes, scales, mins, d, dm)
    codes, scales, mins = codes.cpu().numpy(), scales.cpu().numpy(), mins.cpu().numpy()
    d, dm = d.cpu().numpy().view(np.uint16), dm.cpu().numpy().view(np.uint16)
    nsc = 16 if qtype == Q6_K else 8
    for b in range(nb):
        f = oracle.unpack(qtype, blocks[b])
        assert np.array_equal(codes[b * 256:(b + 1) * 256], f["q"])
        assert np.array_equal(scales[b * 16:b * 16 + nsc], f["sc"])
        assert d[b] == f["d_bits"]
        if qtype != Q6_K:
            assert np.array_equal(mins[b * 8:(b + 1) * 8], f["m"])
            assert dm[b] == f["dmin_bits"]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("dist", ["workload", "random_bytes"])
def test_dequant_bf16_bit_exact(qtype, dist):
    """bf16 weights: the fp32 weights rounded to nearest even, bit for bit
    (NaN blocks from random bytes stay NaN)."""
    g = synth.rng(205, qtype)
    nb = 4099
    if dist == "workload":
        blocks = synth.gen_blocks(qtype, nb, g)
    else:
        blocks = g.integers(0, 256, size=(nb, synth.BLOCK_BYTES[qtype]), dtype=np.uint8)
    ref = oracle.dequant_bf16(qtype, blocks)
    got = kq.dequant_bf16(qtype, dev(blocks.reshape(-1)), nb * 256).cpu().view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())
    gnan = np.isnan(torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy())
    assert np.array_equal(gnan, nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("dist", ["workload", "random_bytes"])
def test_dequant_bit_exact(qtype, dist):
    g = synth.rng(201, qtype)
    nb = 4099
    if dist == "workload":
        blocks = synth.gen_blocks(qtype, nb, g)
    else:  # any fp16 d/dmin, including subnormals, infinities and NaNs
        blocks = g.integers(0, 256, size=(nb, synth.BLOCK_BYTES[qtype]), dtype=np.uint8)
    ref = oracle.dequant(qtype, blocks)
    got = kq.dequant(qtype, dev(blocks.reshape(-1)), nb * 256).cpu().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def _matvec_case(qtype, N, K, M, xd, seed, rows=None):
    g = synth.rng(seed, qtype, N, K, M)
    W = synth.gen_matrix(qtype, N, K, g)
    x = synth.gen_x(M, K, g, xd)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    if rows is None:
        yr, sr = oracle.matvec(qtype, W, N, K, x, threads=8)
        return y, yr, sr
    rb = synth.matrix_bytes(qtype, 1, K)
    Wsub = np.concatenate([W[r * rb:(r + 1) * rb] for r in rows])
    yr, sr = oracle.matvec(qtype, Wsub, len(rows), K, x, threads=8)
    return y[:, rows], yr, sr


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("xd", ["f32", "bf16"])
@pytest.mark.parametrize("NK", [(1, 256), (7, 512), (33, 704), (130, 2560), (64, 32), (5, 4096 + 96)])
def test_matvec_small_shapes(qtype, xd, NK):
    N, K = NK
    y, yr, sr = _matvec_case(qtype, N, K, 1, xd, 202)
    assert rel_err(y, yr, sr) <= TOL[xd]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 16])
def test_matvec_batched(qtype, M):
    for xd in ("f32", "bf16"):
        y, yr, sr = _matvec_case(qtype, 97, 1536, M, xd, 203)
        assert rel_err(y, yr, sr) <= TOL[xd]


@pytest.mark.parametrize("qtype", TYPES)
def test_matvec_batch_rows_match_single_token(qtype):
    """Row m of a batched product equals the one-token product of x[m] within
    the tolerance (different kernels serve M = 1 and M > 1)."""
    N, K = 300, 2816
    g = synth.rng(204, qtype)
    Wn = synth.gen_matrix(qtype, N, K, g)
    W = dev(Wn)
    x = synth.gen_x(16, K, g, "bf16")
    xt = x_dev(x)
    _, sr = oracle.matvec(qtype, Wn, N, K, x, threads=8)
    ref = [kq.matvec(qtype, W, xt[m:m + 1], N, K).cpu().numpy()[0] for m in range(16)]
    for M in (2, 3, 4, 7, 8, 16):
        y = kq.matvec(qtype, W, xt[:M], N, K).cpu().numpy()
        for m in range(M):
            assert rel_err(y[m], ref[m].astype(np.float64), sr[m]) <= 2 * TOL["bf16"], (M, m)


def test_matvec_large_row_count():
    """Many rows (no K split): matches the oracle."""
    qtype, N, K = Q4_K, 40000, 512
    y, yr, sr = _matvec_case(qtype, N, K, 1, "bf16", 205)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


def test_matvec_does_not_write_outside_y():
    qtype, N, K, M = Q6_K, 77, 768, 3
    g = synth.rng(206)
    W = dev(synth.gen_matrix(qtype, N, K, g))
    x = x_dev(synth.gen_x(M, K, g, "bf16"))
    buf = torch.full((M * N + 64,), 1234.5, dtype=torch.float32, device="cuda")
    y = buf[32:32 + M * N]
    kq.kq_matvec(qtype, W, x, kq.KQ_BF16, y, N, K, M)
    b = buf.cpu()
    assert torch.all(b[:32] == 1234.5) and torch.all(b[32 + M * N:] == 1234.5)


def test_matvec_zero_x_and_zero_K():
    qtype, N, K = Q4_K, 50, 512
    g = synth.rng(207)
    W = dev(synth.gen_matrix(qtype, N, K, g))
    y = kq.matvec(qtype, W, torch.zeros((2, K), device="cuda"), N, K)
    assert torch.all(y == 0)
    y = torch.full((2, N), 7.0, device="cuda")
    kq.kq_matvec(qtype, W, torch.zeros((2, 32), device="cuda"), kq.KQ_F32, y, N, 0, 2)
    assert torch.all(y == 0)


def test_matvec_errors_on_gpu():
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, device="cuda")
    y = torch.zeros(4, device="cuda")
    with pytest.raises(kq.KQError):
        kq.kq_matvec(9, W, x, 0, y, 4, 256, 1)
    with pytest.raises(kq.KQError):
        kq.kq_matvec(1, W[1:], x, 0, y, 4, 256, 1)
    with pytest.raises(kq.KQError):
        kq.kq_matvec(1, W, x, 0, y, 4, 256, 17)


# ---------------------------------------------------------------------------
# Full-size matrices of the benchmark workloads, in the launch configuration
# the benchmark uses; the oracle runs on sampled rows.
# ---------------------------------------------------------------------------

def test_full_q4k_4096x4096_fp32_all_rows():
    """Single Q4_K 4096 x 4096 product, fp32 x, seed 0: every output checked."""
    y, yr, sr = _matvec_case(Q4_K, 4096, 4096, 1, "f32", 0)
    assert rel_err(y, yr, sr) <= TOL["f32"]


DENSE_SHAPES = sorted({(t, N, K) for st in synth.dense_layer_sweep(n_layers=2) for (_, t, N, K) in st})


@pytest.mark.parametrize("qtype,N,K", DENSE_SHAPES)
def test_full_dense_layer_matrices(qtype, N, K):
    rows = sorted(set(np.random.default_rng(N + K).integers(0, N, 512).tolist()) | {0, N - 1})
    y, yr, sr = _matvec_case(qtype, N, K, 1, "bf16", 208, rows=rows)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_full_format_sweep_4096x14336(qtype, M):
    N, K = 4096, 14336
    rows = sorted(set(np.random.default_rng(M).integers(0, N, 256).tolist()) | {0, N - 1})
    y, yr, sr = _matvec_case(qtype, N, K, M, "bf16", 1, rows=rows)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_full_verify_block_m16(N, K):
    """Speculative-verify block: M = 16 tokens against the gate/up and down
    shapes (Q4_K, bf16 x) -- the tensor-core path; sampled rows."""
    rows = sorted(set(np.random.default_rng(N).integers(0, N, 256).tolist()) | {0, N - 1})
    y, yr, sr = _matvec_case(Q4_K, N, K, 16, "bf16", 3, rows=rows)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("NK", [(1, 256), (129, 704), (300, 2816), (128, 4096 + 96)])
def test_matvec_m16_ragged(qtype, NK):
    """Ragged row tiles (N not a multiple of 128) and K tails on the M = 16 path."""
    N, K = NK
    y, yr, sr = _matvec_case(qtype, N, K, 16, "bf16", 209)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("NK", [(300, 2816), (4096, 4096), (2560, 9728), (14336, 4096), (1024, 2560)])
@pytest.mark.parametrize("M", [2, 3, 4])
def test_matvec_few_tokens_bit_identical_to_one(qtype, NK, M):
    """Two to four tokens (bf16 x) run the one-token arithmetic on M x images:
    each row equals that token's one-token product bit for bit (the property
    the ANE page tests for its kernel of up to 4 tokens).  Four tokens at
    K = 9728 do not fit beside the weight ring and go to the tensor cores."""
    N, K = NK
    if M == 4 and K > 4096:
        pytest.skip("four x images of K = 9728 do not fit: tensor-core path")
    g = synth.rng(212, qtype, N, K)
    W = dev(synth.gen_matrix(qtype, N, K, g))
    x = x_dev(synth.gen_x(M, K, g, "bf16"))
    yM = kq.matvec(qtype, W, x, N, K)
    for m in range(M):
        assert torch.equal(yM[m], kq.matvec(qtype, W, x[m:m + 1], N, K)[0]), m


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("NK", [(1, 256), (129, 704), (300, 2816), (128, 4096 + 96), (2600, 9728)])
@pytest.mark.parametrize("M", [2, 3, 4])
def test_matvec_few_tokens_ragged(qtype, NK, M):
    """M = 2..4 with bf16 x runs the one-token kernel with M x images: ragged
    tiles, K tails, and tile heights of 32, 16 and 8 rows."""
    N, K = NK
    y, yr, sr = _matvec_case(qtype, N, K, M, "bf16", 211)
    assert rel_err(y, yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("xd", ["f32", "bf16"])
def test_matvec_x_extreme_runs(qtype, xd):
    """Runs of x whose maximum is subnormal, tiny, huge or zero take the
    block-float staging's slow path; every product must still match."""
    N, K = 70, 1536
    g = synth.rng(210, qtype)
    W = synth.gen_matrix(qtype, N, K, g)
    x = g.standard_normal((1, K)).astype(np.float32)
    x[0, 0:128] *= 1e-39      # subnormal run
    x[0, 128:256] *= 1e-30    # tiny normal run
    x[0, 256:384] *= 1e30     # huge run
    x[0, 384:512] = 0.0       # zero run
    x[0, 512:640] *= 1e-20
    if xd == "bf16":
        x = synth.to_bf16_bits(x)
    y = kq.matvec(qtype, dev(W), x_dev(x), N, K).cpu().numpy()
    yr, sr = oracle.matvec(qtype, W, N, K, x, threads=8)
    assert rel_err(y, yr, sr) <= TOL[xd]
    if xd == "bf16":  # the two-token path stages each token's runs on its own
        x2 = np.concatenate([synth.gen_x(1, K, g, "bf16"), x], axis=0)
        y2 = kq.matvec(qtype, dev(W), x_dev(x2), N, K).cpu().numpy()
        yr2, sr2 = oracle.matvec(qtype, W, N, K, x2, threads=8)
        assert rel_err(y2, yr2, sr2) <= TOL[xd]
