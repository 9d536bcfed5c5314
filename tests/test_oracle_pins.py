"""Pins for the oracle: each checks it against something other than itself.

* IEEE-754 decoders against numpy's float16 and torch's bfloat16 (all patterns);
* the integer field decoder against an independent bit-position reader;
* pack <-> unpack round trips in both directions (the layouts are bijections);
* hand-built blocks with closed-form weights (tests/golden/handbuilt_blocks.txt);
* closed forms: constant fields, one-hot scales and mins, the Q6_K zero point;
* the product against plain integer / float matrix products (numpy matmul) on
  tiny matrices, linearity in x, zero x, weights past K ignored;
* the routed-expert product against per-slot products and brute force;
* the bf16 rounding of dequantized weights against torch's bfloat16 conversion
  and hand-worked ties;
* the router against a hand-worked table and brute-force order checks.

All run on the CPU.
"""
import os

import numpy as np
import pytest
import torch

import tests.bitref as bitref
from gguf_quant_weight_super_gb300 import synth

Q4_K, Q5_K, Q6_K = 1, 2, 3
TYPES = [Q4_K, Q5_K, Q6_K]
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "handbuilt_blocks.txt")


def test_block_sizes(orc):
    lib = orc.lib()
    assert [lib.oracle_block_bytes(t) for t in TYPES] == [144, 176, 210]
    assert lib.oracle_block_bytes(0) == 0 and lib.oracle_block_bytes(5) == 0
    assert lib.oracle_block_bytes(4) == 144  # IA4: 4 + 4 bf16 scales and biases, 128 code bytes
    # bits per weight: 4.5, 5.5, 6.5625
    assert [lib.oracle_block_bytes(t) * 8 / 256 for t in TYPES] == [4.5, 5.5, 6.5625]


def test_half_decoder_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("qtype", TYPES)
def test_unpack_matches_bit_reader(orc, qtype):
    g = synth.rng(100, qtype)
    blocks = g.integers(0, 256, size=(3000, synth.BLOCK_BYTES[qtype]), dtype=np.uint8)
    if qtype == Q6_K:
        d, sc, q = bitref.q6k(blocks)
    else:
        d, dmin, sc, m, q = bitref.q4k_like(blocks, five_bit=(qtype == Q5_K))
    for i in range(len(blocks)):
        f = orc.unpack(qtype, blocks[i])
        assert f["d_bits"] == d[i]
        assert np.array_equal(f["sc"], sc[i])
        assert np.array_equal(f["q"], q[i])
        if qtype != Q6_K:
            assert f["dmin_bits"] == dmin[i]
            assert np.array_equal(f["m"], m[i])


@pytest.mark.parametrize("qtype", TYPES)
def test_bytes_unpack_pack_roundtrip(orc, qtype):
    g = synth.rng(101, qtype)
    blocks = g.integers(0, 256, size=(500, synth.BLOCK_BYTES[qtype]), dtype=np.uint8)
    for blk in blocks:
        f = orc.unpack(qtype, blk)
        again = orc.pack(qtype, f["d_bits"], f["sc"], f["q"], f["dmin_bits"], f["m"])
        assert np.array_equal(again, blk)


@pytest.mark.parametrize("qtype", TYPES)
def test_fields_pack_unpack_roundtrip(orc, qtype):
    g = synth.rng(102, qtype)
    qmax = {Q4_K: 15, Q5_K: 31, Q6_K: 63}[qtype]
    for _ in range(300):
        q = g.integers(0, qmax + 1, 256)
        if qtype == Q6_K:
            sc = g.integers(-128, 128, 16)
            m = None
        else:
            sc = g.integers(0, 64, 8)
            m = g.integers(0, 64, 8)
        d, dm = (int(v) for v in g.integers(0, 65536, 2))
        blk = orc.pack(qtype, d, sc, q, dm, m)
        f = orc.unpack(qtype, blk)
        assert f["d_bits"] == d and np.array_equal(f["q"], q) and np.array_equal(f["sc"], sc)
        if m is not None:
            assert f["dmin_bits"] == dm and np.array_equal(f["m"], m)


def _golden_cases():
    cases = []
    with open(GOLDEN) as fh:
        lines = [ln.rstrip("\n") for ln in fh if not ln.startswith("#")]
    for i in range(0, len(lines), 3):
        name = lines[i].split()[1]
        blk = np.frombuffer(bytes.fromhex(lines[i + 1].split()[1]), dtype=np.uint8)
        w = np.array([float(v) for v in lines[i + 2].split()[1:]])
        cases.append(({"Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K}[name], blk, w, lines[i]))
    return cases


def test_golden_handbuilt_blocks(orc):
    cases = _golden_cases()
    assert len(cases) >= 5
    for qtype, blk, w, desc in cases:
        got = orc.dequant_block_f64(qtype, blk)
        assert np.array_equal(got, w), desc
        assert np.array_equal(orc.dequant(qtype, blk), w.astype(np.float32)), desc
        assert np.array_equal(bitref.dequant_f64(qtype, blk[None])[0], w), desc


@pytest.mark.parametrize("qtype", [Q4_K, Q5_K])
def test_closed_form_constant_fields(orc, qtype):
    g = synth.rng(103, qtype)
    qmax = 15 if qtype == Q4_K else 31
    for _ in range(50):
        q0, s, t = int(g.integers(0, qmax + 1)), int(g.integers(0, 64)), int(g.integers(0, 64))
        dh, mh = np.abs(g.normal(0, 0.01, 2)).astype(np.float16)
        blk = orc.pack(qtype, int(dh.view(np.uint16)), [s] * 8, [q0] * 256, int(mh.view(np.uint16)), [t] * 8)
        expect = float(dh) * s * q0 - float(mh) * t
        assert np.all(orc.dequant_block_f64(qtype, blk) == expect)


@pytest.mark.parametrize("qtype", [Q4_K, Q5_K])
def test_one_hot_scale_and_min(orc, qtype):
    g = synth.rng(104, qtype)
    qmax = 15 if qtype == Q4_K else 31
    q = g.integers(0, qmax + 1, 256)
    for j in range(8):
        sc = [0] * 8
        sc[j] = 1
        blk = orc.pack(qtype, 0x3C00, sc, q, 0x3C00, [0] * 8)
        w = orc.dequant_block_f64(qtype, blk)
        inside = np.zeros(256, bool)
        inside[32 * j:32 * j + 32] = True
        assert np.array_equal(w[inside], q[inside].astype(np.float64))
        assert np.all(w[~inside] == 0)
        m = [0] * 8
        m[j] = 1
        blk = orc.pack(qtype, 0x3C00, [0] * 8, q, 0x3C00, m)
        w = orc.dequant_block_f64(qtype, blk)
        assert np.all(w[inside] == -1.0) and np.all(w[~inside] == 0)


def test_q6k_zero_point_and_one_hot(orc):
    g = synth.rng(105)
    sc = g.integers(-128, 128, 16)
    blk = orc.pack(Q6_K, 0x3C00, sc, [32] * 256)
    assert np.all(orc.dequant_block_f64(Q6_K, blk) == 0)
    q = g.integers(0, 64, 256)
    for j in range(16):
        s = [0] * 16
        s[j] = 1
        w = orc.dequant_block_f64(Q6_K, orc.pack(Q6_K, 0x3C00, s, q))
        inside = np.zeros(256, bool)
        inside[16 * j:16 * j + 16] = True
        assert np.array_equal(w[inside], (q[inside] - 32).astype(np.float64))
        assert np.all(w[~inside] == 0)


@pytest.mark.parametrize("qtype", TYPES)
def test_dequant_matches_bit_reader_and_rounds_once(orc, qtype):
    g = synth.rng(106, qtype)
    blocks = synth.gen_blocks(qtype, 400, g)
    ref = bitref.dequant_f64(qtype, blocks)
    w64 = np.stack([orc.dequant_block_f64(qtype, b) for b in blocks])
    assert np.array_equal(w64, ref)
    assert np.array_equal(orc.dequant(qtype, blocks).reshape(-1, 256), ref.astype(np.float32))


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
def test_matvec_integer_special_case(orc, qtype, x_dtype):
    """d = 1, sc = 1, m = 0: weights are the integer codes (minus 32 for Q6_K), so
    the product is a plain integer-matrix times vector (numpy matmul)."""
    g = synth.rng(107, qtype)
    N, K = 5, 512
    qmax = {Q4_K: 15, Q5_K: 31, Q6_K: 63}[qtype]
    codes = g.integers(0, qmax + 1, (N, K))
    blocks = []
    for n in range(N):
        for b in range(K // 256):
            q = codes[n, 256 * b:256 * b + 256]
            if qtype == Q6_K:
                blocks.append(orc.pack(qtype, 0x3C00, [1] * 16, q))
            else:
                blocks.append(orc.pack(qtype, 0x3C00, [1] * 8, q, 0x3C00, [0] * 8))
    W = np.concatenate(blocks)
    x = synth.gen_x(3, K, g, x_dtype)
    xf = x.astype(np.float64) if x_dtype == "f32" else \
        torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    wint = (codes - 32) if qtype == Q6_K else codes
    y, s = orc.matvec(qtype, W, N, K, x)
    ref = xf @ wint.T.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-12)
    assert np.allclose(s, np.abs(xf) @ np.abs(wint).T, rtol=1e-13)


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("NK", [(1, 256), (3, 512), (4, 768)])
def test_matvec_brute_force(orc, qtype, NK):
    N, K = NK
    g = synth.rng(108, qtype, N, K)
    W = synth.gen_matrix(qtype, N, K, g)
    x = synth.gen_x(2, K, g, "f32")
    wd = bitref.dequant_f64(qtype, W.reshape(-1, synth.BLOCK_BYTES[qtype])).reshape(N, -1)[:, :K]
    y, s = orc.matvec(qtype, W, N, K, x)
    ref = x.astype(np.float64) @ wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(s, np.abs(x.astype(np.float64)) @ np.abs(wd).T, rtol=1e-12)


@pytest.mark.parametrize("qtype", TYPES)
def test_matvec_linearity_and_zero(orc, qtype):
    N, K = 6, 768
    g = synth.rng(109, qtype)
    W = synth.gen_matrix(qtype, N, K, g)
    x1 = synth.gen_x(1, K, g)
    x2 = synth.gen_x(1, K, g)
    y1, _ = orc.matvec(qtype, W, N, K, x1)
    y2, _ = orc.matvec(qtype, W, N, K, x2)
    # power-of-two coefficients keep a*x1 + b*x2 nearly exact in fp32
    x3 = (np.float32(2.0) * x1 - np.float32(0.5) * x2).astype(np.float32)
    y3, _ = orc.matvec(qtype, W, N, K, x3)
    assert np.allclose(y3, 2.0 * y1 - 0.5 * y2, rtol=1e-6, atol=1e-9)
    y0, s0 = orc.matvec(qtype, W, N, K, np.zeros((1, K), np.float32))
    assert np.all(y0 == 0) and np.all(s0 == 0)


@pytest.mark.parametrize("qtype", TYPES)
def test_matvec_weights_past_K_ignored(orc, qtype):
    N, K = 3, 704          # 3 blocks per row, the last one covers 192 weights
    g = synth.rng(110, qtype)
    W = synth.gen_matrix(qtype, N, K, g)
    x = synth.gen_x(2, K, g)
    y, _ = orc.matvec(qtype, W, N, K, x)
    wd = bitref.dequant_f64(qtype, W.reshape(-1, synth.BLOCK_BYTES[qtype])).reshape(N, -1)[:, :K]
    assert np.allclose(y, x.astype(np.float64) @ wd.T, rtol=1e-12, atol=1e-15)
    # rewriting the codes of the part of each row past K changes nothing
    nbytes = synth.BLOCK_BYTES[qtype]
    W2 = W.copy().reshape(N, 3, nbytes)
    if qtype == Q4_K:
        W2[:, 2, 16 + 96:16 + 128] ^= 0xFF      # chunk 3 = weights 192..255
    elif qtype == Q6_K:
        W2[:, 2, 64 + 0:64 + 64] ^= 0xF0        # high nibbles of half 1 = weights 192..255
    y2, _ = orc.matvec(qtype, W2.reshape(-1), N, K, x)
    assert np.array_equal(y, y2)


@pytest.mark.parametrize("with_gate", [False, True])
@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_matches_per_slot_products(orc, with_gate, x_per_slot):
    qtype, E, N, K, M, top_k = Q4_K, 6, 5, 512, 3, 2
    g = synth.rng(111, int(with_gate), int(x_per_slot))
    We = synth.gen_matrix(qtype, E * N, K, g)
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = synth.gen_x(M * top_k if x_per_slot else M, K, g, "bf16")
    y, s = orc.moe_matvec(qtype, We, E, ids, gate if with_gate else None, x, x_per_slot, N, K, M, top_k)
    eb = N * 2 * 144
    per = np.zeros((M, top_k, N))
    per_abs = np.zeros((M, top_k, N))
    for m in range(M):
        for t in range(top_k):
            e = ids[m, t]
            xr = x[m * top_k + t] if x_per_slot else x[m]
            yy, ss = orc.matvec(qtype, We[e * eb:(e + 1) * eb], N, K, xr[None])
            per[m, t], per_abs[m, t] = yy[0], ss[0]
    if with_gate:
        ref = (gate.astype(np.float64)[:, :, None] * per).sum(axis=1)
        ref_abs = (np.abs(gate.astype(np.float64))[:, :, None] * per_abs).sum(axis=1)
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-15) and np.allclose(s, ref_abs, rtol=1e-13)
    else:
        assert np.array_equal(y, per) and np.array_equal(s, per_abs)


def test_moe_rejects_bad_expert_id(orc):
    g = synth.rng(112)
    We = synth.gen_matrix(Q4_K, 2 * 4, 256, g)
    x = synth.gen_x(1, 256, g)
    with pytest.raises(ValueError):
        orc.moe_matvec(Q4_K, We, 2, np.array([[0, 2]], np.int32), None, x, False, 4, 256, 1, 2)


def test_routing_generator_shape():
    g = synth.rng(113)
    ids, gate = synth.gen_routing(16, 128, 8, g)
    assert ids.shape == (16, 8) and gate.shape == (16, 8)
    assert all(len(set(r)) == 8 for r in ids) and ids.min() >= 0 and ids.max() < 128
    assert np.allclose(gate.sum(axis=1), 1.0, atol=1e-6) and np.all(gate > 0)


def test_moe_group_by_definition():
    import oracle
    """Grouping pin: a hand-worked routing table (3 tokens, top-2, 5 experts,
    one id out of range)."""
    ids = np.array([[4, 1], [1, 0], [9, 4]], dtype=np.int32)
    experts, offsets, pairs = oracle.moe_group(ids, 5)
    assert experts == [0, 1, 4]
    assert offsets == [0, 1, 3, 5]
    assert pairs == [3, 1, 2, 0, 5]


def test_bf16_rounding_against_torch_and_ties():
    """f32 -> bf16 rounding (used by the bf16 dequant oracle): every one of a
    few hundred thousand patterns -- random bits, exact ties, subnormals,
    infinities, the largest floats -- agrees with torch's conversion, and the
    hand-worked ties go to the even neighbour."""
    import oracle
    g = np.random.default_rng(114)
    u = g.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (g.integers(0, 2**16, size=50000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    special = np.array([0, 0x80000000, 0x00000001, 0x007FFFFF, 0x00008000, 0x00018000, 0x7F7FFFFF,
                        0x7F7F8000, 0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x3F808000, 0x3F818000,
                        0x3F808001, 0x3F807FFF], dtype=np.uint32)
    allu = np.concatenate([u, ties, special])
    f = allu.view(np.float32)
    got = oracle.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(torch.from_numpy(got[nan].view(np.int16)).view(torch.bfloat16).float().numpy()))
    # ties to even: 1 + 2^-8 -> 1.0 (0x3F80), 1 + 3*2^-8 -> 1 + 2^-6 (0x3F82); just past a tie rounds up
    t = np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF], dtype=np.uint32).view(np.float32)
    assert oracle.f32_to_bf16_bits(t).tolist() == [0x3F80, 0x3F82, 0x3F81, 0x3F80]


@pytest.mark.parametrize("qtype", TYPES)
def test_dequant_bf16_is_the_fp32_weights_rounded(orc, qtype):
    """The bf16 dequant oracle equals the fp32 oracle's weights converted by
    torch (round to nearest even)."""
    g = synth.rng(115, qtype)
    blocks = synth.gen_blocks(qtype, 64, g)
    w = orc.dequant(qtype, blocks)
    ref = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.dequant_bf16(qtype, blocks), ref)


def test_route_hand_worked():
    """Router pin: a hand-worked row -- equal logits in index order, -inf after
    every finite logit, a NaN after everything -- with closed-form gates."""
    import oracle
    l = np.array([[1.0, 3.0, 3.0, 0.0, np.nan, -np.inf],
                  [2.0, 2.0, 2.0, 2.0, 2.0, 2.0]], dtype=np.float32)
    ids, gate = oracle.moe_route(l, 4)
    assert ids.tolist() == [[1, 2, 0, 3], [0, 1, 2, 3]]
    e = np.exp(np.array([0.0, 0.0, -2.0, -3.0]))
    assert np.allclose(gate[0], e / e.sum(), rtol=1e-15, atol=0)
    assert np.allclose(gate[1], 0.25, rtol=1e-15, atol=0)
    ids5, _ = oracle.moe_route(l, 6)
    assert ids5[0].tolist() == [1, 2, 0, 3, 5, 4]


def test_route_brute_force_order():
    """Every selected logit ranks at or above every unselected one, equal
    logits are taken in index order, the gates are a softmax of the selected
    logits (sum 1, ratios exp(l_i - l_j)); integer logits force many ties."""
    import oracle
    g = np.random.default_rng(116)
    for E, k in ((128, 8), (16, 16), (300, 5)):
        l = g.integers(-4, 5, size=(40, E)).astype(np.float32)
        ids, gate = oracle.moe_route(l, k)
        for m in range(40):
            sel = list(ids[m])
            rest = [e for e in range(E) if e not in sel]
            vals = l[m, sel]
            assert all(vals[i] >= vals[i + 1] for i in range(k - 1))
            for i in range(k - 1):  # ties in index order
                if vals[i] == vals[i + 1]:
                    assert sel[i] < sel[i + 1]
            if rest:
                worst = vals[-1]
                assert all(l[m, e] < worst or (l[m, e] == worst and e > sel[-1]) for e in rest)
            assert abs(gate[m].sum() - 1.0) < 1e-12
            assert np.allclose(gate[m] / gate[m][0], np.exp(vals.astype(np.float64) - vals[0]), rtol=1e-12)


def test_ffn_activations():
    """Activation pins: SiLU at closed-form points; the tanh form of GELU
    within 5e-4 of the erf form (its known approximation error, 4.7e-4 at
    most) over [-8, 8]; both satisfy act(x) - act(-x) = x, act(0) = 0, and
    tend to x for large x and to 0 for very negative x."""
    import math
    import oracle
    assert abs(oracle.ffn_act(0, np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(oracle.ffn_act(0, np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15  # sigma(ln 3) = 3/4
    x = np.linspace(-8, 8, 20001)
    erf_gelu = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in x])
    assert np.max(np.abs(oracle.ffn_act(1, x) - erf_gelu)) < 5e-4
    for act in (0, 1):
        a = oracle.ffn_act(act, x)
        assert np.allclose(a - oracle.ffn_act(act, -x), x, rtol=0, atol=1e-12)
        assert oracle.ffn_act(act, np.array([0.0]))[0] == 0.0
        assert abs(oracle.ffn_act(act, np.array([40.0]))[0] - 40.0) < 1e-12
        assert abs(oracle.ffn_act(act, np.array([-40.0]))[0]) < 1e-12


def _ffn_case(seed, E=4, H=512, F=96, SH=64, M=3, top_k=2, qg=Q4_K, qd=Q6_K):
    g = synth.rng(seed)
    Wg = synth.gen_matrix(qg, E * F, H, g)
    Wu = synth.gen_matrix(qg, E * F, H, g)
    Wd = synth.gen_matrix(qd, E * H, F, g)
    sh = (synth.gen_matrix(qg, SH, H, g), synth.gen_matrix(qg, SH, H, g), synth.gen_matrix(qd, H, SH, g), SH)
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = synth.gen_x(M, H, g)
    return dict(Wg=Wg, Wu=Wu, Wd=Wd, sh=sh, ids=ids, gate=gate, x=x, E=E, H=H, F=F, M=M, top_k=top_k, qg=qg, qd=qd)


def test_moe_ffn_matches_composed_dense_products():
    """FFN pin: the oracle's layer (numpy matmul on dequantized weights)
    against the same layer composed from the C dense product oracle.matvec
    (its own decode and loops): gate and up per pair, the activation, down
    with h rounded to fp32, the gated sum and the shared term."""
    import oracle
    c = _ffn_case(131)
    E, H, F, M, k = c["E"], c["H"], c["F"], c["M"], c["top_k"]
    for act in (0, 1):
        r = oracle.moe_ffn(c["qg"], c["Wg"], c["Wu"], c["qd"], c["Wd"], E, c["ids"], c["gate"], c["x"], act,
                           H, F, M, k, shared=c["sh"])
        rb_g = synth.matrix_bytes(c["qg"], F, H)
        rb_d = synth.matrix_bytes(c["qd"], H, F)
        y = np.zeros((M, H))
        for m in range(M):
            for j in range(k):
                e = int(c["ids"][m, j])
                gg, _ = oracle.matvec(c["qg"], c["Wg"][e * rb_g:(e + 1) * rb_g], F, H, c["x"][m:m + 1])
                uu, _ = oracle.matvec(c["qg"], c["Wu"][e * rb_g:(e + 1) * rb_g], F, H, c["x"][m:m + 1])
                h = oracle.ffn_act(act, gg) * uu
                p = m * k + j  # the two sum orders differ by fp64 rounding, relative to sum |w x|
                bound = 1e-12 * (1.2 * np.abs(uu[0]) * r["sg"][p] + np.abs(oracle.ffn_act(act, gg[0])) * r["su"][p])
                assert np.all(np.abs(h[0] - r["h"][p]) <= bound)
                dd, _ = oracle.matvec(c["qd"], c["Wd"][e * rb_d:(e + 1) * rb_d], H, F, h.astype(np.float32))
                y[m] += np.float64(c["gate"][m, j]) * dd[0]
            Wsg, Wsu, Wsd, SH = c["sh"]
            gs, _ = oracle.matvec(c["qg"], Wsg, SH, H, c["x"][m:m + 1])
            us, _ = oracle.matvec(c["qg"], Wsu, SH, H, c["x"][m:m + 1])
            hs = oracle.ffn_act(act, gs) * us
            ds, _ = oracle.matvec(c["qd"], Wsd, H, SH, hs.astype(np.float32))
            y[m] += ds[0]
        assert np.all(np.abs(y - r["y"]) <= 1e-6 * r["s"])


def test_moe_ffn_brute_force_tiny():
    """FFN pin on a tiny layer with pure-Python loops over the per-block
    exact weights (one routed slot with its gate, no shared expert)."""
    import oracle
    c = _ffn_case(132, E=2, H=256, F=32, M=1, top_k=1)
    r = oracle.moe_ffn(c["qg"], c["Wg"], c["Wu"], c["qd"], c["Wd"], 2, c["ids"], c["gate"], c["x"], 1,
                       256, 32, 1, 1)
    e = int(c["ids"][0, 0])
    wg = np.array([oracle.dequant_block_f64(c["qg"], b) for b in c["Wg"].reshape(-1, 144)]).reshape(2, 32, 256)[e]
    wu = np.array([oracle.dequant_block_f64(c["qg"], b) for b in c["Wu"].reshape(-1, 144)]).reshape(2, 32, 256)[e]
    wd = np.array([oracle.dequant_block_f64(c["qd"], b) for b in c["Wd"].reshape(-1, 210)]).reshape(2, 256, 256)[e]
    wd = wd[:, :32]
    xs = [float(v) for v in c["x"][0]]
    import math
    h = []
    for f in range(32):
        gv = sum(float(wg[f, k]) * xs[k] for k in range(256))
        uv = sum(float(wu[f, k]) * xs[k] for k in range(256))
        h.append(0.5 * gv * (1 + math.tanh(math.sqrt(2 / math.pi) * (gv + 0.044715 * gv ** 3))) * uv)
    for n in (0, 17, 255):
        yv = float(c["gate"][0, 0]) * sum(float(wd[n, f]) * h[f] for f in range(32))
        assert abs(yv - r["y"][0, n]) <= 1e-12 * r["s"][0, n]


def test_moe_ffn_invariants():
    """Gate linearity (the routed part doubles with the gates), slot order
    (a consistent permutation of each token's slots changes nothing), dropped
    ids (an id out of range equals a zero gate), and no valid id (only the
    shared term remains)."""
    import oracle
    c = _ffn_case(133, M=4, top_k=3)
    args = (c["qg"], c["Wg"], c["Wu"], c["qd"], c["Wd"], c["E"])
    dims = (c["H"], c["F"], c["M"], c["top_k"])
    base = oracle.moe_ffn(*args, c["ids"], c["gate"], c["x"], 0, *dims, shared=c["sh"])
    none = oracle.moe_ffn(*args, np.full_like(c["ids"], -1), c["gate"], c["x"], 0, *dims, shared=c["sh"])
    dbl = oracle.moe_ffn(*args, c["ids"], 2 * c["gate"], c["x"], 0, *dims, shared=c["sh"])
    assert np.allclose(dbl["y"] - none["y"], 2 * (base["y"] - none["y"]), rtol=0, atol=1e-12 * base["s"].max())
    perm = np.array([2, 0, 1])
    pr = oracle.moe_ffn(*args, c["ids"][:, perm], c["gate"][:, perm], c["x"], 0, *dims, shared=c["sh"])
    assert np.allclose(pr["y"], base["y"], rtol=0, atol=1e-12 * base["s"].max())
    ids2, g2 = c["ids"].copy(), c["gate"].copy()
    ids2[1, 2] = c["E"] + 5
    g2[1, 2] = 0.0
    dropped = oracle.moe_ffn(*args, ids2, c["gate"], c["x"], 0, *dims, shared=c["sh"])
    zero_gate = oracle.moe_ffn(*args, c["ids"], g2, c["x"], 0, *dims, shared=c["sh"])
    assert np.allclose(dropped["y"], zero_gate["y"], rtol=0, atol=1e-12 * base["s"].max())
    Wsg, Wsu, Wsd, SH = c["sh"]
    gs, _ = oracle.matvec(c["qg"], Wsg, SH, c["H"], c["x"])
    us, _ = oracle.matvec(c["qg"], Wsu, SH, c["H"], c["x"])
    assert np.allclose(none["hs"], oracle.ffn_act(0, gs) * us, rtol=1e-12, atol=0)


def test_dequant_f64_is_exact_weights():
    """dequant_f64 equals the per-block exact weights, and rounded to fp32 it
    equals dequant (the fp32 weights are the exact ones rounded once)."""
    import oracle
    g = synth.rng(134)
    for qt in (Q4_K, Q5_K, Q6_K):
        blocks = synth.gen_blocks(qt, 40, g)
        w = oracle.dequant_f64(qt, blocks)
        ref = np.concatenate([oracle.dequant_block_f64(qt, b) for b in blocks.reshape(40, -1)])
        assert np.array_equal(w, ref)
        assert np.array_equal(w.astype(np.float32), oracle.dequant(qt, blocks))


# ---------------------------------------------------------------- IA4
def test_ia4_pack_then_block_decode_equals_mlx_definition(orc):
    """IA4 pin: regrouping MLX's arrays into blocks and decoding the blocks
    (the C decoder) gives exactly the weights of the MLX definition computed
    from the arrays themselves (numpy), for ragged K too."""
    for N, K in ((3, 320), (2, 704), (1, 2816), (4, 64)):
        q, s, b = synth.gen_ia4_mlx(N, K, synth.rng(140, N, K))
        blk = orc.ia4_pack(q, s, b, N, K)
        assert blk.size == N * ((K + 255) // 256) * 144
        w = orc.dequant_f64(4, blk).reshape(N, -1)
        assert np.array_equal(w[:, :K], orc.ia4_dequant_mlx(q, s, b, N, K))
        assert np.array_equal(w.astype(np.float32).reshape(-1), orc.dequant(4, blk))
        tail = blk.reshape(N, -1, 144)[:, -1]  # groups past K in the last block are all zero
        for g in range((K % 256) // 64 if K % 256 else 4, 4):
            assert not tail[:, 2 * g:2 * g + 2].any() and not tail[:, 8 + 2 * g:10 + 2 * g].any()
            assert not tail[:, 16 + 32 * g:48 + 32 * g].any()


def test_ia4_hand_worked_block(orc):
    """One group by hand: codes k % 16 for k = 0..63, scale 1.0 (bf16 0x3F80),
    bias -1.0 (0xBF80).  Block byte 16 + l = (l % 16) | ((32 + l) % 16) << 4
    = 0x11 * (l % 16); weights are (k % 16) - 1."""
    words = np.array([[sum(((8 * i + j) % 16) << (4 * j) for j in range(8)) for i in range(8)]], dtype=np.uint32)
    blk = orc.ia4_pack(words, np.array([[0x3F80]], np.uint16), np.array([[0xBF80]], np.uint16), 1, 64)
    assert list(blk[0:4]) == [0x80, 0x3F, 0, 0] and list(blk[8:12]) == [0x80, 0xBF, 0, 0]
    assert list(blk[16:48]) == [0x11 * (l % 16) for l in range(32)]
    assert not blk[48:].any()
    w = orc.dequant_f64(4, blk)[:64]
    assert np.array_equal(w, np.array([(k % 16) - 1.0 for k in range(64)]))
    # closed forms: scale 0 leaves the bias; all codes 15 give 15 s + b
    blk2 = blk.copy()
    blk2[0:2] = [0, 0]
    assert np.all(orc.dequant_f64(4, blk2)[:64] == -1.0)
    blk3 = blk.copy()
    blk3[16:48] = 0xFF
    assert np.all(orc.dequant_f64(4, blk3)[:64] == 14.0)


def test_ia4_matvec_reduces_to_dense_integer_product(orc):
    """With scale 1 and bias 0 everywhere the IA4 product is the integer code
    matrix times x (numpy, fp64)."""
    N, K = 5, 512
    q, _, _ = synth.gen_ia4_mlx(N, K, synth.rng(141))
    ones = np.full((N, K // 64), 0x3F80, np.uint16)
    zeros = np.zeros((N, K // 64), np.uint16)
    blk = orc.ia4_pack(q, ones, zeros, N, K)
    x = synth.gen_x(2, K, synth.rng(142))
    codes = orc.ia4_dequant_mlx(q, ones, zeros, N, K)
    assert np.all((codes == np.round(codes)) & (codes >= 0) & (codes <= 15))
    y, _ = orc.matvec(4, blk, N, K, x)
    assert np.allclose(y, x.astype(np.float64) @ codes.T, rtol=1e-13, atol=1e-12)
