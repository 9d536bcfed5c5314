"""Parity of chains of one-token products (kq_chain_* through the C ABI)
with the oracle: mixed block types and x dtypes, ragged shapes, grid-barrier
ordering (an op whose x is an earlier op's y), split-K outputs, repeated runs
(bit-identical: counters reset, fixed summation order), CUDA graph replay."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, rel_err, require_gpu, x_dev

pytestmark = pytest.mark.gpu
Q4_K, Q5_K, Q6_K = 1, 2, 3


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


def _op(qtype, N, K, xd, g, x=None, wait=0):
    Wn = synth.gen_matrix(qtype, N, K, g)
    xn = synth.gen_x(1, K, g, xd) if x is None else None
    return {"type": qtype, "x_dtype": kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, "W": dev(Wn),
            "x": x_dev(xn) if x is None else x, "y": torch.full((N,), np.nan, device="cuda"),
            "N": N, "K": K, "wait_previous": wait, "_Wn": Wn, "_xn": xn, "_xd": xd}


def _strip(ops):
    return [{k: v for k, v in o.items() if not k.startswith("_")} for o in ops]


def _check_independent(o):
    yr, sr = oracle.matvec(o["type"], o["_Wn"], o["N"], o["K"], o["_xn"], threads=8)
    assert rel_err(o["y"].cpu().numpy(), yr[0], sr[0]) <= TOL[o["_xd"]]
    return yr[0], sr[0]


def test_chain_mixed_ops_match_oracle():
    g = synth.rng(300)
    ops = [_op(Q4_K, 4096, 2560, "bf16", g), _op(Q4_K, 1024, 2560, "bf16", g), _op(Q6_K, 1024, 2560, "bf16", g),
           _op(Q4_K, 2560, 4096, "bf16", g, wait=1), _op(Q5_K, 333, 704, "f32", g, wait=1),
           _op(Q6_K, 2560, 9728, "bf16", g, wait=1), _op(Q4_K, 97, 4096 + 96, "f32", g),
           _op(Q5_K, 3000, 2816, "bf16", g, wait=1)]
    ch = kq.Chain(_strip(ops))
    ch.run()
    torch.cuda.synchronize()
    for o in ops:
        _check_independent(o)


def test_chain_dependent_op_reads_earlier_output():
    """x of op 2 is y of op 0 (wait_previous): compared with the oracle run on
    the oracle's own y of op 0; the tolerance adds the propagated error of that
    input (|dy_2| <= sum|w2| * max|dy_0|)."""
    g = synth.rng(301)
    a = _op(Q4_K, 2560, 2560, "bf16", g)                   # y_a: 2560 values, feeds op c
    b = _op(Q6_K, 777, 2560, "bf16", g)
    c = _op(Q5_K, 1500, 2560, "f32", g, x=a["y"], wait=1)
    ch = kq.Chain(_strip([a, b, c]))
    ch.run()
    torch.cuda.synchronize()
    ya, sa = _check_independent(a)
    _check_independent(b)
    xa = ya.astype(np.float32).reshape(1, -1)              # the oracle's own input for op c
    yc, sc = oracle.matvec(c["type"], c["_Wn"], c["N"], c["K"], xa, threads=8)
    # sum_k |w_c| per row: the oracle's product with |x| = 1
    _, wabs = oracle.matvec(c["type"], c["_Wn"], c["N"], c["K"], np.ones((1, c["K"]), np.float32), threads=8)
    dx = TOL["bf16"] * float(np.max(sa)) + float(np.max(np.abs(ya - ya.astype(np.float32))))
    err = np.abs(c["y"].cpu().numpy().astype(np.float64) - yc[0])
    assert np.all(err <= TOL["f32"] * sc[0] + wabs[0] * dx)


def test_chain_repeated_runs_identical_and_graph_replay():
    g = synth.rng(302)
    ops = [_op(Q4_K, 2560, 9728, "bf16", g), _op(Q6_K, 4096, 2560, "bf16", g, wait=1),
           _op(Q4_K, 1024, 4096, "bf16", g, wait=1)]
    ch = kq.Chain(_strip(ops))
    ch.run()
    torch.cuda.synchronize()
    first = [o["y"].clone() for o in ops]
    for o in ops:
        _check_independent(o)
    for _ in range(3):
        for o in ops:
            o["y"].fill_(np.nan)
        ch.run()
        torch.cuda.synchronize()
        for o, f in zip(ops, first):
            assert torch.equal(o["y"], f)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            ch.run(stream=s)
    for _ in range(2):
        for o in ops:
            o["y"].fill_(np.nan)
        graph.replay()
        torch.cuda.synchronize()
        for o, f in zip(ops, first):
            assert torch.equal(o["y"], f)


def test_chain_dense_layer_sweep_two_layers():
    """Two layers of the dense sweep with stage barriers, as the benchmark
    runs them; sampled rows of every matrix against the oracle."""
    g = synth.rng(303)
    ops = []
    for stage in synth.dense_layer_sweep(n_layers=2, vocab=4096):
        xs = None
        for j, (_, t, N, K) in enumerate(stage):
            o = _op(t, N, K, "bf16", g, x=xs, wait=1 if (j == 0 and ops) else 0)
            if xs is None:
                xs = o["x"]
            else:
                o["_xn"] = ops[-1]["_xn"]
            ops.append(o)
    ch = kq.Chain(_strip(ops))
    ch.run()
    torch.cuda.synchronize()
    for o in ops:
        N, K = o["N"], o["K"]
        rows = sorted(set(np.random.default_rng(N + K).integers(0, N, 128).tolist()) | {0, N - 1})
        rb = synth.matrix_bytes(o["type"], 1, K)
        Wsub = np.concatenate([o["_Wn"][r * rb:(r + 1) * rb] for r in rows])
        yr, sr = oracle.matvec(o["type"], Wsub, len(rows), K, o["_xn"], threads=8)
        assert rel_err(o["y"].cpu().numpy()[rows], yr[0], sr[0]) <= TOL["bf16"]


def test_chain_rejects_races_and_small_workspace():
    g = synth.rng(304)
    a = _op(Q4_K, 512, 512, "f32", g)
    c = _op(Q4_K, 64, 512, "f32", g, x=a["y"], wait=0)     # reads a's y without waiting
    with pytest.raises(kq.KQError):
        kq.Chain(_strip([a, c]))
    n = kq.kq_chain_workspace_size(_strip([a]))
    assert n > 0
    ws = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
    p = ws.data_ptr() + (-ws.data_ptr()) % 256
    with pytest.raises(kq.KQError):
        kq.kq_chain_prepare(_strip([a]), p, n - 1, kq.KqChainPlan())
