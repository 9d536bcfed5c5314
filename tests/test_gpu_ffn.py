"""Parity of the expert FFN of an MoE layer (kq_moe_ffn through the C ABI)
with the oracle: the intermediate h = act(W_gate x) * (W_up x) against the
fp64 definition, the down stage with the gated combine and the shared term
against the oracle's products on the same h, the whole layer against the fp64
definition, dropped ids, repeated calls, and that only routed experts' bytes
are used."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, require_gpu, x_dev

pytestmark = pytest.mark.gpu
Q4_K, Q5_K, Q6_K = 1, 2, 3
LIP = 1.13  # |act'| <= 1.13 for both activations (SiLU: 1.0998, tanh-form GELU: 1.1289)


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    yield
    assert kq.kq_device_error() == 0, "device error word set"


def _case(seed, E, H, F, SH, M, top_k, qg, qd, xd):
    g = synth.rng(seed, E, H, F, SH, M, top_k, qg, qd)
    c = dict(E=E, H=H, F=F, SH=SH, M=M, top_k=top_k, qg=qg, qd=qd, xd=xd)
    c["Wg"] = synth.gen_matrix(qg, E * F, H, g)
    c["Wu"] = synth.gen_matrix(qg, E * F, H, g)
    c["Wd"] = synth.gen_matrix(qd, E * H, F, g)
    c["sh"] = (synth.gen_matrix(qg, SH, H, g), synth.gen_matrix(qg, SH, H, g), synth.gen_matrix(qd, H, SH, g),
               SH) if SH else None
    c["ids"], c["gate"] = synth.gen_routing(M, E, top_k, g)
    c["x"] = synth.gen_x(M, H, g, xd)
    return c


def _run(c, act, ids=None, Wg=None, Wu=None, Wd=None, ws=None, y=None):
    E, H, F, SH, M, k = c["E"], c["H"], c["F"], c["SH"], c["M"], c["top_k"]
    dW = [dev(a) for a in (Wg if Wg is not None else c["Wg"], Wu if Wu is not None else c["Wu"],
                           Wd if Wd is not None else c["Wd"])]
    dS = [dev(a) for a in c["sh"][:3]] if SH else [None] * 3
    w = kq.ffn_weights(c["qg"], c["qd"], E, act, F, *dW, SH, *dS)
    if ws is None:
        ws = kq.moe_ffn_workspace(H, F, SH, M, k, E)
    if y is None:
        y = torch.full((M, H), np.nan, device="cuda")
    keep = (dW, dS)
    kq.kq_moe_ffn(w, dev(c["ids"] if ids is None else ids), dev(c["gate"]), x_dev(c["x"]),
                  kq.KQ_BF16 if c["xd"] == "bf16" else kq.KQ_F32, y, H, M, k, ws, ws.numel())
    torch.cuda.synchronize()
    del keep
    h_off, hs_off = kq.kq_moe_ffn_offsets(H, F, SH, M, k, E)
    wsn = ws.cpu().numpy()
    h = wsn[h_off:h_off + 4 * M * k * F].view(np.float32).reshape(M * k, F)
    hs = wsn[hs_off:hs_off + 4 * M * SH].view(np.float32).reshape(M, SH) if SH else None
    return y.cpu().numpy().astype(np.float64), h, hs, ws


def _ref(c, act, ids=None, gate=None):
    return oracle.moe_ffn(c["qg"], c["Wg"], c["Wu"], c["qd"], c["Wd"], c["E"],
                          c["ids"] if ids is None else ids, c["gate"] if gate is None else gate, c["x"], act,
                          c["H"], c["F"], c["M"], c["top_k"], shared=c["sh"])


def _h_bound(g, u, sg, su, act, eps):
    """|h_gpu - h| for h = act(g) u when g and u carry errors up to eps * sg and
    eps * su, plus a few fp32 ulps of the activation and the product."""
    return (eps * (LIP * np.abs(u) * sg + np.abs(oracle.ffn_act(act, g)) * su) + LIP * eps * eps * sg * su
            + 2e-6 * np.abs(oracle.ffn_act(act, g) * u) + 1e-30)


def _check_h(c, act, h, hs, r):
    eps = TOL[c["xd"]]
    valid = (c["ids"].reshape(-1) >= 0) & (c["ids"].reshape(-1) < c["E"])
    b = _h_bound(r["g"], r["u"], r["sg"], r["su"], act, eps)
    assert np.all(np.abs(h[valid] - r["h"][valid]) <= b[valid])
    if c["SH"]:
        bs = _h_bound(r["gs"], r["us"], r["sgs"], r["sus"], act, eps)
        assert np.all(np.abs(hs - r["hs"]) <= bs)


def _check_down(c, y, h, hs, ids=None, gate=None):
    """The down stage against the oracle's products applied to the GPU's own h."""
    ids = c["ids"] if ids is None else ids
    gate = c["gate"] if gate is None else gate
    E, H, F, M, k = c["E"], c["H"], c["F"], c["M"], c["top_k"]
    yr, sr = oracle.moe_matvec(c["qd"], c["Wd"], E, ids, gate, np.ascontiguousarray(h), True, H, F, M, k)
    if c["SH"]:
        ys, ss = oracle.matvec(c["qd"], c["sh"][2], H, c["SH"], np.ascontiguousarray(hs))
        yr, sr = yr + ys, sr + ss
    assert np.all(np.abs(y - yr) <= TOL["f32"] * sr + 1e-30)


def _check_layer(c, act, y, r):
    """The whole layer against fp64: the down products' own error plus what
    the error bound of h carries through |W_down|."""
    eps = TOL[c["xd"]]
    E, H, F, M, k = c["E"], c["H"], c["F"], c["M"], c["top_k"]
    bound = TOL["f32"] * r["s"] * 1.01 + 1e-30
    hb = _h_bound(r["g"], r["u"], r["sg"], r["su"], act, eps)
    for e in sorted(set(int(v) for v in c["ids"].reshape(-1))):
        Wd = np.abs(oracle._matrix_f64(c["qd"], c["Wd"], e * H, H, F))
        for p in np.nonzero(c["ids"].reshape(-1) == e)[0]:
            m, j = divmod(int(p), k)
            bound[m] += abs(float(c["gate"][m, j])) * (Wd @ hb[p])
    if c["SH"]:
        Ws = np.abs(oracle._matrix_f64(c["qd"], c["sh"][2], 0, H, c["SH"]))
        bound += (_h_bound(r["gs"], r["us"], r["sgs"], r["sus"], act, eps)) @ Ws.T
    assert np.all(np.abs(y - r["y"]) <= bound)


SMALL = [  # (E, H, F, SH, M, top_k, gate|up type, down type, x)
    (16, 512, 320, 288, 1, 4, Q4_K, Q6_K, "f32"),
    (16, 512, 320, 288, 5, 4, Q4_K, Q4_K, "bf16"),
    (16, 512, 320, 0, 16, 4, Q5_K, Q4_K, "bf16"),
    (8, 768, 224, 96, 3, 8, Q6_K, Q5_K, "f32"),
    (32, 256, 512, 256, 16, 2, Q4_K, Q6_K, "bf16"),
]


@pytest.mark.parametrize("act", [kq.KQ_ACT_SILU, kq.KQ_ACT_GELU_TANH])
@pytest.mark.parametrize("shape", SMALL)
def test_ffn_matches_definition(shape, act):
    c = _case(301, *shape)
    y, h, hs, ws = _run(c, act)
    r = _ref(c, act)
    _check_h(c, act, h, hs, r)
    _check_down(c, y, h, hs)
    _check_layer(c, act, y, r)
    kq.kq_moe_check(ws)


@pytest.mark.parametrize("M", [1, 16])
def test_ffn_full_size_layer(M):
    """The MoE benchmark's layer: 128 experts top-8, hidden 2816, expert width
    704, shared width 2112, Q4_K, bf16 x, the tanh-form GELU."""
    c = _case(302, 128, 2816, 704, 2112, M, 8, Q4_K, Q4_K, "bf16")
    y, h, hs, ws = _run(c, kq.KQ_ACT_GELU_TANH)
    r = _ref(c, kq.KQ_ACT_GELU_TANH)
    _check_h(c, kq.KQ_ACT_GELU_TANH, h, hs, r)
    _check_down(c, y, h, hs)
    _check_layer(c, kq.KQ_ACT_GELU_TANH, y, r)


def test_ffn_dropped_id_equals_zero_gate():
    c = _case(303, 16, 512, 320, 288, 4, 4, Q4_K, Q6_K, "f32")
    ids = c["ids"].copy()
    ids[2, 1] = 99
    y, h, hs, ws = _run(c, kq.KQ_ACT_SILU, ids=ids)
    with pytest.raises(RuntimeError):
        kq.kq_moe_check(ws)
    gate = c["gate"].copy()
    gate[2, 1] = 0.0
    r = _ref(c, kq.KQ_ACT_SILU, gate=gate)
    _check_h(dict(c, ids=ids), kq.KQ_ACT_SILU, h, hs, r)
    _check_down(c, y, h, hs, gate=gate)


@pytest.mark.parametrize("SH", [0, 288])
def test_ffn_no_valid_id(SH):
    """No valid routed id: only the shared term remains (zero without one)."""
    c = _case(304, 16, 512, 320, SH, 3, 4, Q4_K, Q4_K, "f32")
    ids = np.full_like(c["ids"], -1)
    y, h, hs, ws = _run(c, kq.KQ_ACT_SILU, ids=ids)
    with pytest.raises(RuntimeError):
        kq.kq_moe_check(ws)
    if SH == 0:
        assert np.all(y == 0.0)
    else:
        ys, ss = oracle.matvec(Q4_K, c["sh"][2], 512, SH, np.ascontiguousarray(hs))
        assert np.all(np.abs(y - ys) <= TOL["f32"] * ss + 1e-30)


def test_ffn_repeats_identically_and_reads_only_routed_experts():
    """Two calls on one workspace give identical bits (the arrival counters
    return to zero); replacing every unrouted expert's bytes with 0xFF (NaN
    scales) changes nothing."""
    c = _case(305, 16, 512, 320, 288, 2, 4, Q4_K, Q6_K, "bf16")
    y1, _, _, ws = _run(c, kq.KQ_ACT_GELU_TANH)
    y2, _, _, _ = _run(c, kq.KQ_ACT_GELU_TANH, ws=ws)
    assert np.array_equal(y1, y2)
    used = set(int(v) for v in c["ids"].reshape(-1))
    Wg, Wu, Wd = c["Wg"].copy(), c["Wu"].copy(), c["Wd"].copy()
    bg, bd = synth.matrix_bytes(Q4_K, 320, 512), synth.matrix_bytes(Q6_K, 512, 320)
    for e in range(16):
        if e not in used:
            Wg[e * bg:(e + 1) * bg] = 0xFF
            Wu[e * bg:(e + 1) * bg] = 0xFF
            Wd[e * bd:(e + 1) * bd] = 0xFF
    y3, _, _, _ = _run(c, kq.KQ_ACT_GELU_TANH, Wg=Wg, Wu=Wu, Wd=Wd)
    assert np.array_equal(y1, y3)
