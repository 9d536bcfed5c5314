"""Parity of the routed-expert products (kq_moe_matvec through the C ABI)
with the oracle: gate/up form (per-slot outputs) and down form (per-slot x,
gate-weighted combine), the expert grouping it plans, bad ids, repeated calls,
and that only routed experts' bytes are used."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, require_gpu, x_dev

pytestmark = pytest.mark.gpu
Q4_K, Q5_K, Q6_K = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    yield
    assert kq.kq_device_error() == 0, "device error word set"


def _moe(qtype, E, N, K, M, top_k, xd, gated, seed, ids=None):
    g = synth.rng(seed, qtype, N, K, M)
    We = synth.gen_matrix(qtype, E * N, K, g)          # E experts of N rows, back to back
    if ids is None:
        ids, gate = synth.gen_routing(M, E, top_k, g)
    else:
        gate = synth.gen_routing(M, E, top_k, g)[1]
    x = synth.gen_x(M * top_k if gated else M, K, g, xd)
    ws = kq.moe_workspace(N, M, top_k, E)
    shape = (M, N) if gated else (M, top_k, N)
    y = torch.full(shape, np.nan, device="cuda")
    args = (qtype, dev(We), E, dev(ids), dev(gate) if gated else None, x_dev(x),
            kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, gated, y, N, K, M, top_k, ws, ws.numel())
    return We, ids, gate, x, ws, y, args


def _rel(y, yr, sr, mask=None):
    y = np.asarray(y, np.float64)
    if mask is not None:
        y, yr, sr = y[mask], yr[mask], sr[mask]
    nz = sr > 0
    assert np.all(y[~nz] == 0)
    return float(np.max(np.abs(y[nz] - yr[nz]) / sr[nz])) if nz.any() else 0.0


@pytest.mark.parametrize("M", [1, 3, 16])
def test_moe_gate_up_form(M):
    """Config-4 expert gate/up shape: 704 x 2816 Q4_K, 128 experts, top-8."""
    E, N, K, top_k = 128, 704, 2816, 8
    We, ids, gate, x, ws, y, args = _moe(Q4_K, E, N, K, M, top_k, "bf16", False, 400)
    kq.kq_moe_matvec(*args)
    kq.kq_moe_check(ws)
    yr, sr = oracle.moe_matvec(Q4_K, We, E, ids, None, x, False, N, K, M, top_k, threads=8)
    assert _rel(y.cpu().numpy(), yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("M", [1, 16])
def test_moe_down_form_gated(M):
    """Config-4 expert down shape: 2816 x 704 Q4_K (K not a multiple of 256),
    per-slot inputs, gate-weighted sum over the 8 slots."""
    E, N, K, top_k = 128, 2816, 704, 8
    We, ids, gate, x, ws, y, args = _moe(Q4_K, E, N, K, M, top_k, "bf16", True, 401)
    kq.kq_moe_matvec(*args)
    kq.kq_moe_check(ws)
    yr, sr = oracle.moe_matvec(Q4_K, We, E, ids, gate, x, True, N, K, M, top_k, threads=8)
    assert _rel(y.cpu().numpy(), yr, sr) <= TOL["bf16"]


@pytest.mark.parametrize("qtype", [Q5_K, Q6_K])
@pytest.mark.parametrize("xd", ["f32", "bf16"])
def test_moe_formats_and_dtypes(qtype, xd):
    E, N, K, M, top_k = 20, 70, 1024 + 32, 5, 4
    for gated in (False, True):
        We, ids, gate, x, ws, y, args = _moe(qtype, E, N, K, M, top_k, xd, gated, 402)
        kq.kq_moe_matvec(*args)
        kq.kq_moe_check(ws)
        yr, sr = oracle.moe_matvec(qtype, We, E, ids, gate if gated else None, x, gated, N, K, M, top_k,
                                   threads=8)
        assert _rel(y.cpu().numpy(), yr, sr) <= TOL[xd]


def test_moe_grouping_plan_matches_definition():
    """The plan left in the workspace equals the grouping by definition (ids
    shared across tokens, a repeated id within a token)."""
    E, N, K, M, top_k = 40, 64, 512, 6, 3
    ids = np.array([[3, 7, 39], [7, 3, 0], [12, 12, 5], [39, 0, 1], [5, 6, 7], [7, 8, 3]], dtype=np.int32)
    We, ids, gate, x, ws, y, args = _moe(Q4_K, E, N, K, M, top_k, "bf16", False, 403, ids=ids)
    kq.kq_moe_matvec(*args)
    kq.kq_moe_check(ws)
    experts, offsets, pairs = oracle.moe_group(ids, E)
    Dmax = min(E, M * top_k)
    plan = ws[256:256 + 4 * (2 + 2 * Dmax + M * top_k)].cpu().numpy().view(np.int32)
    D = int(plan[0])
    assert D == len(experts)
    assert plan[1:1 + D].tolist() == experts
    assert plan[1 + Dmax:1 + Dmax + D + 1].tolist() == offsets
    assert plan[2 + 2 * Dmax:2 + 2 * Dmax + len(pairs)].tolist() == pairs
    yr, sr = oracle.moe_matvec(Q4_K, We, E, ids, None, x, False, N, K, M, top_k, threads=8)
    assert _rel(y.cpu().numpy(), yr, sr) <= TOL["bf16"]


def test_moe_bad_ids_are_dropped_and_reported():
    E, N, K, M, top_k = 16, 96, 768, 4, 4
    ids = np.array([[1, 2, 3, 4], [5, 16, 6, 7], [-1, 8, 9, 10], [11, 12, 13, 2]], dtype=np.int32)
    bad = (ids < 0) | (ids >= E)
    for gated in (False, True):
        We, ids_, gate, x, ws, y, args = _moe(Q6_K, E, N, K, M, top_k, "bf16", gated, 404, ids=ids)
        kq.kq_moe_matvec(*args)
        with pytest.raises(kq.KQError) as ex:
            kq.kq_moe_check(ws)
        assert ex.value.status == -8
        kq.kq_moe_check(ws)                            # cleared by the first check
        ok_ids = np.where(bad, 0, ids)
        g2 = np.where(bad, 0.0, gate).astype(np.float32)
        yr, sr = oracle.moe_matvec(Q6_K, We, E, ok_ids, g2 if gated else None, x, gated, N, K, M, top_k, threads=8)
        yg = y.cpu().numpy()
        if gated:
            assert _rel(yg, yr, sr) <= TOL["bf16"]
        else:
            assert np.all(np.isnan(yg[bad]))          # dropped pairs are not written
            assert _rel(yg, yr, sr, mask=~bad) <= TOL["bf16"]


def test_moe_all_ids_bad_gives_zero_gated_output():
    """Every routed id out of range: no pair survives, every gated output is the
    empty sum (0), and the bad ids are reported."""
    E, N, K, M, top_k = 8, 80, 512, 3, 2
    ids = np.array([[8, -1], [9, 100], [-5, 8]], dtype=np.int32)
    We, ids_, gate, x, ws, y, args = _moe(Q4_K, E, N, K, M, top_k, "f32", True, 406, ids=ids)
    y.fill_(np.nan)
    kq.kq_moe_matvec(*args)
    with pytest.raises(kq.KQError) as ex:
        kq.kq_moe_check(ws)
    assert ex.value.status == -8
    assert torch.count_nonzero(y).item() == 0


def test_moe_reads_only_routed_experts_and_repeats_identically():
    """Unrouted experts hold blocks whose d is NaN: any use of them would
    poison the outputs.  Repeated calls give identical outputs (the arrival
    counters return to zero)."""
    E, N, K, M, top_k = 32, 256, 1024, 2, 4
    We, ids, gate, x, ws, y, args = _moe(Q4_K, E, N, K, M, top_k, "bf16", True, 405)
    rb = synth.matrix_bytes(Q4_K, N, K)
    routed = set(ids.reshape(-1).tolist())
    poisoned = We.copy()
    for e in range(E):
        if e not in routed:
            blk = poisoned[e * rb:(e + 1) * rb].reshape(-1, 144)
            blk[:, 0:2] = np.frombuffer(np.array([0x7E00], np.uint16).tobytes(), np.uint8)  # d = NaN
    args = (args[0], dev(poisoned)) + args[2:]
    kq.kq_moe_matvec(*args)
    first = y.clone()
    kq.kq_moe_check(ws)
    yr, sr = oracle.moe_matvec(Q4_K, We, E, ids, gate, x, True, N, K, M, top_k, threads=8)
    assert np.all(np.isfinite(first.cpu().numpy()))
    assert _rel(first.cpu().numpy(), yr, sr) <= TOL["bf16"]
    for _ in range(3):
        y.fill_(np.nan)
        kq.kq_moe_matvec(*args)
        assert torch.equal(y, first)
