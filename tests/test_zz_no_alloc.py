"""The allocation-free routed-expert call (kq_moe_matvec_noalloc) against the
workspace call (kq_moe_matvec) on the same inputs: both forms, two
consecutive calls each, within the bf16 tolerance.  Collected last on
purpose; it also passes on its own."""
import numpy as np
import pytest
import torch

from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, require_gpu, x_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    kq.lib()
    yield


@pytest.mark.parametrize("gated", [False, True])
def test_noalloc_matches_workspace_call(gated):
    qtype, E, top_k = synth.Q4_K, 128, 8
    M = 16
    N, K = (2816, 704) if gated else (704, 2816)
    g = synth.rng(500, int(gated))
    We = dev(synth.gen_matrix(qtype, E * N, K, g))
    ids, gate = synth.gen_routing(M, E, top_k, g)
    x = x_dev(synth.gen_x(M * top_k if gated else M, K, g, "bf16"))
    ids_d, gate_d = dev(ids), dev(gate)
    shape = (M, N) if gated else (M, top_k, N)
    y_ws = torch.empty(shape, device="cuda")
    ws = kq.moe_workspace(N, M, top_k, E)
    kq.kq_moe_matvec(qtype, We, E, ids_d, gate_d if gated else None, x, kq.KQ_BF16, gated, y_ws, N, K, M, top_k,
                     ws, ws.numel())
    kq.kq_moe_check(ws)
    ref = y_ws.double()
    # scale of the outputs for the tolerance: |W| |x| products, bounded by the reference itself
    scale = ref.abs().max().item() + 1e-30
    for _ in range(2):
        y = torch.full(shape, np.nan, device="cuda")
        kq.kq_moe_matvec_noalloc(qtype, We, E, ids_d, gate_d if gated else None, x, kq.KQ_BF16, gated, y, N, K, M,
                                 top_k)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all()
        assert (y.double() - ref).abs().max().item() <= TOL["bf16"] * scale
    assert kq.kq_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    W = torch.zeros(144, dtype=torch.uint8, device="cuda")
    ids = torch.zeros((512, 1), dtype=torch.int32, device="cuda")
    x = torch.zeros((512, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((512, 4096), device="cuda")
    with pytest.raises(kq.KQError) as ex:   # 512 pairs x 4096 outputs: 8 MiB of partial sums
        kq.kq_moe_matvec_noalloc(synth.Q4_K, W, 1, ids, None, x, kq.KQ_BF16, 0, y, 4096, 256, 512, 1)
    assert ex.value.status == -7
