"""Guard bands and failure paths on the GPU: outputs written through the C ABI
stay inside their buffers (canary words around y untouched on every path), and
the kernels' bounded waits, made to run out on a flag nothing sets, record a
timeout and return with the context usable."""
import numpy as np
import pytest
import torch

import oracle
from gguf_quant_weight_super_gb300 import kq, synth
from tests.gpu_util import TOL, dev, require_gpu, x_dev

pytestmark = pytest.mark.gpu
CANARY = 0x7FC0DEAD  # a NaN pattern no product writes
PAD = 64             # canary words on each side


@pytest.fixture(scope="module", autouse=True)
def _setup():
    require_gpu()
    from gguf_quant_weight_super_gb300 import build
    build.build()
    oracle.build()
    kq.lib()
    yield
    assert kq.kq_device_error() == 0, "device error word set"


def _guarded(n):
    """An fp32 view of n elements with PAD canary words on each side."""
    buf = torch.full((n + 2 * PAD,), CANARY, dtype=torch.int32, device="cuda")
    return buf, buf[PAD:PAD + n].view(torch.float32)


def _intact(buf, n):
    b = buf.cpu().numpy()
    return bool(np.all(b[:PAD] == CANARY) and np.all(b[PAD + n:] == CANARY))


@pytest.mark.parametrize("qtype,M,xd", [(1, 1, "bf16"), (3, 1, "f32"), (2, 3, "bf16"), (1, 8, "bf16"),
                                        (3, 16, "bf16"), (1, 4, "f32"), (4, 1, "bf16"), (4, 16, "bf16")])
def test_products_write_only_their_output(qtype, M, xd):
    N, K = 300, 2816  # ragged row tiles and a K tail
    g = synth.rng(501, qtype, M)
    W = synth.gen_matrix(qtype, N, K, g)
    x = synth.gen_x(M, K, g, xd)
    buf, y = _guarded(M * N)
    kq.kq_matvec(qtype, dev(W), x_dev(x), kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, y, N, K, M)
    torch.cuda.synchronize()
    assert _intact(buf, M * N)
    yr, sr = oracle.matvec(qtype, W, N, K, x)
    assert np.max(np.abs(y.cpu().numpy().reshape(M, N) - yr) / sr) <= TOL[xd]


def test_moe_ffn_route_and_dequant_write_only_their_outputs():
    E, H, F, SH, M, k = 16, 512, 320, 288, 3, 4
    g = synth.rng(502)
    mats = [synth.gen_matrix(1, n, kk, g) for n, kk in ((E * F, H), (E * F, H), (E * H, F), (SH, H), (SH, H),
                                                         (H, SH))]
    dm = [dev(m) for m in mats]
    logits = synth.gen_logits(M, E, g)
    x = synth.gen_x(M, H, g, "bf16")
    ibuf = torch.full((M * k + 2 * PAD,), CANARY, dtype=torch.int32, device="cuda")
    ids = ibuf[PAD:PAD + M * k]
    gbuf, gate = _guarded(M * k)
    kq.kq_moe_route(dev(logits), M, E, k, ids, gate)
    ybuf, y = _guarded(M * H)
    w = kq.ffn_weights(1, 1, E, kq.KQ_ACT_SILU, F, dm[0], dm[1], dm[2], SH, dm[3], dm[4], dm[5])
    ws = kq.moe_ffn_workspace(H, F, SH, M, k, E)
    kq.kq_moe_ffn(w, ids, gate, x_dev(x), kq.KQ_BF16, y, H, M, k, ws, ws.numel())
    pbuf, yp = _guarded(M * k * F)
    wsm = kq.moe_workspace(F, M, k, E)
    kq.kq_moe_matvec(1, dm[0], E, ids, None, x_dev(x), kq.KQ_BF16, 0, yp, F, H, M, k, wsm, wsm.numel())
    dbuf, wd = _guarded(4 * 256)
    kq.kq_dequant(1, dm[0], wd, 4 * 256)
    torch.cuda.synchronize()
    kq.kq_moe_check(ws)
    kq.kq_moe_check(wsm)
    assert _intact(ibuf, M * k) and _intact(gbuf, M * k) and _intact(ybuf, M * H)
    assert _intact(pbuf, M * k * F) and _intact(dbuf, 4 * 256)
    assert np.array_equal(ids.cpu().numpy().reshape(M, k), oracle.moe_route(logits, k)[0])


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_wait_runs_out_and_context_survives(kind):
    """kind 0: an mbarrier no copy completes; kind 1: a grid barrier no CTA
    reaches.  The wait records a timeout (code 1) and the kernel returns; the
    next product runs normally and the library's error word is untouched."""
    assert kq.kq_selftest_wait(kind) == 1
    N, K = 64, 512
    g = synth.rng(503, kind)
    W = synth.gen_matrix(1, N, K, g)
    x = synth.gen_x(1, K, g, "f32")
    y = kq.matvec(1, dev(W), x_dev(x), N, K).cpu().numpy()
    yr, sr = oracle.matvec(1, W, N, K, x)
    assert np.max(np.abs(y - yr) / sr) <= TOL["f32"]
    assert kq.kq_device_error() == 0
