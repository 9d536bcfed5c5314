"""The allocation-free routed-expert call (kq_moe_matvec_noalloc) against the
workspace call (kq_moe_matvec) on the same inputs.

Both calls run the same kernel with the same grouping and summation order, so
the outputs must be bit-identical; they are also checked elementwise against
the oracle.  The library-owned array is laid out per call shape, so calls of
different shapes (M, top_k, gated or not) are interleaved: a gated call after
one of another shape must start from cleared arrival counters.  Collected last
on purpose; it also passes on its own."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, rel_err, require_gpu, x_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    yield


def _case(M, top_k, gated, seed, E=128, qtype=synth.Q4_K):
    """The MoE workload's expert shapes: gate/up 704 x 2816, down 2816 x 704."""
    N, K = (2816, 704) if gated else (704, 2816)
    g = synth.rng(500, seed, M, top_k, int(gated))
    We = synth.gen_matrix(qtype, E * N, K, g)
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = synth.gen_x(M * top_k if gated else M, K, g, "bf16")
    c = dict(qtype=qtype, E=E, N=N, K=K, M=M, top_k=top_k, gated=gated, We=We, ids=ids, gate=gate, x=x)
    c["dev"] = (dev(We), dev(ids), dev(gate) if gated else None, x_dev(x))
    c["shape"] = (M, N) if gated else (M, top_k, N)
    return c


def _workspace_call(c):
    We, ids, gate, x = c["dev"]
    y = torch.full(c["shape"], np.nan, device="cuda")
    ws = kq.moe_workspace(c["N"], c["M"], c["top_k"], c["E"])
    kq.kq_moe_matvec(c["qtype"], We, c["E"], ids, gate, x, kq.KQ_BF16, c["gated"], y, c["N"], c["K"], c["M"],
                     c["top_k"], ws, ws.numel())
    kq.kq_moe_check(ws)
    return y


def _noalloc_call(c):
    We, ids, gate, x = c["dev"]
    y = torch.full(c["shape"], np.nan, device="cuda")
    kq.kq_moe_matvec_noalloc(c["qtype"], We, c["E"], ids, gate, x, kq.KQ_BF16, c["gated"], y, c["N"], c["K"],
                             c["M"], c["top_k"])
    torch.cuda.synchronize()
    return y


def _oracle(c):
    return oracle.moe_matvec(c["qtype"], c["We"], c["E"], c["ids"], c["gate"] if c["gated"] else None, c["x"],
                             c["gated"], c["N"], c["K"], c["M"], c["top_k"], threads=8)


@pytest.mark.parametrize("gated", [False, True])
def test_noalloc_matches_workspace_call(gated):
    """Two calls in a row, each bit-identical to the workspace call and within
    the bf16 tolerance of the oracle elementwise."""
    c = _case(16, 8, gated, 0)
    y_ws = _workspace_call(c)
    yr, sr = _oracle(c)
    for _ in range(2):
        y = _noalloc_call(c)
        assert torch.equal(y, y_ws)
        assert rel_err(y.cpu().numpy(), yr, sr) <= TOL["bf16"]
    assert kq.kq_device_error() == 0


def test_noalloc_calls_of_different_shapes_interleaved():
    """Gated M = 16, gated M = 1, ungated M = 16, gated M = 1, gated M = 3
    (top_k 4), gated M = 16 again: each equal to its workspace call.  The
    shapes lay the array out differently (plan, counters and partial sums move
    with M and top_k), so a gated call finds counters another shape left."""
    seq = [(16, 8, True), (1, 8, True), (16, 8, False), (1, 8, True), (3, 4, True), (16, 8, True)]
    cases = [_case(M, k, gt, i) for i, (M, k, gt) in enumerate(seq)]
    refs = [_workspace_call(c) for c in cases]
    for c, r in zip(cases, refs):
        assert torch.equal(_noalloc_call(c), r), (c["M"], c["top_k"], c["gated"])
    yr, sr = _oracle(cases[-1])
    assert rel_err(refs[-1].cpu().numpy(), yr, sr) <= TOL["bf16"]
    assert kq.kq_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    W = torch.zeros(144, dtype=torch.uint8, device="cuda")
    ids = torch.zeros((512, 1), dtype=torch.int32, device="cuda")
    x = torch.zeros((512, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((512, 4096), device="cuda")
    with pytest.raises(kq.KQError) as ex:   # 512 pairs x 4096 outputs: 8 MiB of partial sums
        kq.kq_moe_matvec_noalloc(synth.Q4_K, W, 1, ids, None, x, kq.KQ_BF16, 0, y, 4096, 256, 512, 1)
    assert ex.value.status == -7
