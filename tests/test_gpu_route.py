"""Parity of the MoE router (kq_moe_route through the C ABI) with the oracle:
expert ids exact, gates within fp32 rounding of the fp64 definition, equal
logits, NaN and infinite logits, the limits of the path, and the grouping plan
it leaves in a workspace against the grouping by definition."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import dev, require_gpu

pytestmark = pytest.mark.gpu

# gate_j = exp(l_j - l_0) / sum: the fp32 difference rounds by at most
# |l_j - l_0| * 2^-24, expf and the division add a few ulps, the fp32 sum of
# <= 32 terms at most 32 * 2^-24 relative; logits here stay within |d| < 64.
GATE_RTOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()


def _route(logits, top_k, plan=False):
    M, E = logits.shape
    ws = kq.moe_workspace(1, max(M, 1), top_k, E) if plan else None
    if ws is not None:
        ws.fill_(0x7F)  # the plan must overwrite what it reports
    ids, gate = kq.moe_route(dev(logits), top_k, workspace=ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), gate.cpu().numpy(), ws


def _check(logits, top_k):
    ids, gate, _ = _route(logits, top_k)
    rid, rgate = oracle.moe_route(logits, top_k)
    assert np.array_equal(ids, rid)
    np.testing.assert_allclose(gate, rgate, rtol=GATE_RTOL, atol=0, equal_nan=True)


@pytest.mark.parametrize("E,top_k,M", [(8, 1, 1), (8, 8, 3), (128, 8, 1), (128, 8, 16), (128, 8, 64),
                                       (128, 1, 512), (128, 32, 16), (4096, 8, 5), (4096, 32, 16),
                                       (300, 7, 33), (33, 32, 2), (64, 6, 16), (256, 8, 16), (200, 32, 4),
                                       (257, 8, 3)])
def test_route_matches_definition(E, top_k, M):
    g = synth.rng(201, E, top_k, M)
    _check(synth.gen_logits(M, E, g), top_k)


@pytest.mark.parametrize("E,top_k", [(128, 8), (16, 16), (4096, 32), (256, 32), (48, 4)])
def test_route_equal_logits_take_lower_index(E, top_k):
    g = synth.rng(202, E, top_k)
    _check(synth.gen_logits(min(40, 512 // top_k), E, g, ties=True), top_k)


def test_route_nan_and_infinite_logits():
    """NaN ranks below every number (-inf included), +inf above; a row whose
    leading logit is infinite or NaN has NaN gates on both sides."""
    g = synth.rng(203)
    E, top_k = 64, 8
    l = synth.gen_logits(8, E, g)
    l[0, ::3] = np.nan                    # NaN never beats a number
    l[1, :] = -np.inf; l[1, 5] = 0.0      # one finite logit, the rest -inf: gates 1, 0, ...
    l[2, :] = np.nan                      # all NaN: ids 0..7, NaN gates
    l[3, 7] = np.inf                      # +inf leads: NaN gates
    l[4, :] = 1.5                         # all equal: ids 0..7, gates 1/8
    l[5, :20] = -np.inf; l[5, 20:] = np.nan  # -inf above NaN
    l[6, 40:] = 0.0; l[6, :40] = -1.0     # ties at the top spill over in index order
    _check(l, top_k)
    ids, gate, _ = _route(l, top_k)
    assert ids[1].tolist()[0] == 5 and gate[1, 0] == 1.0 and np.all(gate[1, 1:] == 0.0)
    assert ids[2].tolist() == list(range(8)) and np.all(np.isnan(gate[2]))
    assert ids[4].tolist() == list(range(8)) and np.all(gate[4] == np.float32(0.125))
    assert ids[5].tolist() == list(range(8))


@pytest.mark.parametrize("E,top_k,M", [(128, 8, 16), (128, 8, 1), (8, 8, 64), (4096, 8, 64), (4096, 1, 1)])
def test_route_grouping_plan_matches_definition(E, top_k, M):
    g = synth.rng(204, E, top_k, M)
    logits = synth.gen_logits(M, E, g, ties=(E == 8))
    ids, gate, ws = _route(logits, top_k, plan=True)
    rid, _ = oracle.moe_route(logits, top_k)
    assert np.array_equal(ids, rid)
    experts, offsets, pairs = oracle.moe_group(rid, E)
    Dmax = min(M * top_k, E)
    plan = ws[256:256 + 4 * (2 + 2 * Dmax + M * top_k)].cpu().numpy().view(np.int32)
    D = int(plan[0])
    assert D == len(experts)
    assert plan[1:1 + D].tolist() == experts
    assert plan[1 + Dmax:1 + Dmax + D + 1].tolist() == offsets
    assert plan[2 + 2 * Dmax:2 + 2 * Dmax + len(pairs)].tolist() == pairs


def test_route_feeds_the_expert_products():
    """Router ids and gates drive kq_moe_matvec to the oracle's combined output."""
    from tests.gpu_util import TOL, x_dev
    Q4_K, E, N, K, M, top_k = 1, 32, 256, 512, 4, 4
    g = synth.rng(205)
    logits = synth.gen_logits(M, E, g)
    We = synth.gen_matrix(Q4_K, E * N, K, g)
    x = synth.gen_x(M * top_k, K, g, "f32")
    ids_d, gate_d = kq.moe_route(dev(logits), top_k)
    ws = kq.moe_workspace(N, M, top_k, E)
    y = torch.full((M, N), np.nan, device="cuda")
    kq.kq_moe_matvec(Q4_K, dev(We), E, ids_d, gate_d, x_dev(x), kq.KQ_F32, 1, y, N, K, M, top_k, ws, ws.numel())
    torch.cuda.synchronize()
    rid, rgate = oracle.moe_route(logits, top_k)
    gate = gate_d.cpu().numpy()
    assert np.array_equal(ids_d.cpu().numpy(), rid)
    np.testing.assert_allclose(gate, rgate, rtol=GATE_RTOL, atol=0)
    yr, sr = oracle.moe_matvec(Q4_K, We, E, rid, gate, x, True, N, K, M, top_k)
    assert np.all(sr > 0)
    assert np.max(np.abs(y.cpu().numpy().astype(np.float64) - yr) / sr) <= TOL["f32"]


def test_route_empty_and_limits():
    ids, gate = kq.moe_route(torch.zeros((0, 128), device="cuda"), 8)
    assert ids.shape == (0, 8)
    with pytest.raises(RuntimeError):
        kq.moe_route(torch.zeros((65, 128), device="cuda"), 8)      # 520 pairs > 512
    with pytest.raises(RuntimeError):
        kq.moe_route(torch.zeros((1, 8192), device="cuda"), 8)      # > 4096 experts
