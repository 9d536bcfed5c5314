"""CPU checks of the C ABI: libkq builds for sm_103a, loads, exports every
function include/kq.h declares, and rejects bad arguments before touching the
GPU (these paths make no CUDA call)."""
import ctypes
import os
import re

import pytest

from gguf_quant_weight_super_gb300 import build as kqbuild
from gguf_quant_weight_super_gb300 import kq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(kq_[a-z0-9_]+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def L():
    kqbuild.build()
    return kq.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"kq_matvec", "kq_dequant", "kq_unpack", "kq_block_bytes"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(kq.SIGNATURES) >= names


def test_block_bytes(L):
    assert [L.kq_block_bytes(t) for t in (1, 2, 3, 4)] == [144, 176, 210, 144]
    assert L.kq_block_bytes(0) == 0 and L.kq_block_bytes(9) == 0


def test_status_strings(L):
    for s in range(0, -9, -1):
        assert L.kq_status_string(s)


def test_argument_errors_without_gpu(L):
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert L.kq_matvec(7, fake, fake, 0, fake, 4, 256, 1, None) == -2         # type
    assert L.kq_matvec(1, fake, fake, 5, fake, 4, 256, 1, None) == -1         # x dtype
    assert L.kq_matvec(1, fake, fake, 0, fake, 4, 250, 1, None) == -3         # K % 32
    assert L.kq_matvec(1, fake, fake, 0, fake, 4, 256, 17, None) == -4        # M > 16
    assert L.kq_matvec(1, fake, fake, 0, fake, -1, 256, 1, None) == -1        # N < 0
    assert L.kq_matvec(1, fake, fake, 0, fake, 0, 256, 1, None) == 0          # empty: no-op
    assert L.kq_matvec(1, None, fake, 0, fake, 4, 256, 1, None) == -1         # null W
    assert L.kq_matvec(1, P(0x1001), fake, 0, fake, 4, 256, 1, None) == -5    # W alignment
    assert L.kq_dequant(1, fake, fake, 100, None) == -3                        # n % 256
    assert L.kq_dequant(3, fake, P(0x1004), 256, None) == -5                   # out alignment
    assert L.kq_dequant(3, fake, fake, 0, None) == 0
    assert L.kq_dequant_bf16(7, fake, fake, 256, None) == -2                   # type
    assert L.kq_dequant_bf16(1, fake, fake, 300, None) == -3                   # n % 256
    assert L.kq_dequant_bf16(2, fake, P(0x1008), 256, None) == -5              # out alignment
    assert L.kq_dequant_bf16(2, None, fake, 256, None) == -1                   # null blocks
    assert L.kq_dequant_bf16(3, fake, fake, 0, None) == 0
    assert L.kq_unpack(4, fake, 1, None, None, None, None, None, None) == -2   # IA4: no k-quant fields
    assert L.kq_unpack(5, fake, 1, None, None, None, None, None, None) == -2
    assert L.kq_matvec(5, fake, fake, 0, fake, 4, 256, 1, None) == -2         # unknown type
    assert L.kq_ia4_pack(fake, fake, fake, 2, 96, fake, None) == -3           # K % 64
    assert L.kq_ia4_pack(fake, fake, fake, -1, 64, fake, None) == -1          # N < 0
    assert L.kq_ia4_pack(fake, fake, fake, 0, 64, fake, None) == 0            # empty: no-op
    assert L.kq_ia4_pack(None, fake, fake, 2, 64, fake, None) == -1           # null codes
    assert L.kq_ia4_pack(P(0x1002), fake, fake, 2, 64, fake, None) == -5      # codes alignment
    assert L.kq_ia4_pack(fake, P(0x1001), fake, 2, 64, fake, None) == -5      # scales alignment
    assert L.kq_ia4_pack(fake, fake, fake, 2, 64, P(0x1008), None) == -5      # blocks alignment
    assert L.kq_unpack(1, fake, -1, None, None, None, None, None, None) == -1


def test_chain_argument_errors_without_gpu(L):
    """Chain checks that run before any CUDA call (fake device addresses)."""
    def ops(**kw):
        o = dict(type=1, x_dtype=1, wait_previous=0, W=0x100000, x=0x200000, y=0x300000, N=64, K=512)
        o.update(kw)
        return o
    assert kq.kq_chain_workspace_size([ops(type=9)]) == 0
    assert kq.kq_chain_workspace_size([ops(type=4)]) == 0               # IA4 is not taken by chains
    assert kq.kq_chain_workspace_size([ops(K=500)]) == 0
    assert kq.kq_chain_workspace_size([ops(K=16384 + 32)]) == 0
    assert kq.kq_chain_workspace_size([ops(x=0x200008)]) == 0          # x alignment
    assert kq.kq_chain_workspace_size([ops(y=0x200000)]) == 0          # y overlaps x
    # op 2 reads op 1's output without a barrier
    assert kq.kq_chain_workspace_size([ops(), ops(x=0x300000, x_dtype=0, W=0x400000, y=0x500000)]) == 0
    plan = kq.KqChainPlan()
    with pytest.raises(kq.KQError):
        kq.kq_chain_prepare([ops(type=9)], 0x800000, 1 << 20, plan, stream=0)
    with pytest.raises(kq.KQError):                                      # workspace alignment
        kq.kq_chain_prepare([ops()], 0x800010, 1 << 20, plan, stream=0)


def test_selftest_argument_errors_without_gpu(L):
    code = ctypes.c_int(0)
    assert L.kq_selftest_wait(2, ctypes.byref(code), None) == -1     # unknown kind
    assert L.kq_selftest_wait(0, None, None) == -1                   # no output


def test_route_argument_errors_without_gpu(L):
    P = ctypes.c_void_p
    fake = P(0x1000)
    r = L.kq_moe_route
    assert r(fake, -1, 128, 8, fake, fake, None, 0, None) == -1        # M < 0
    assert r(fake, 0, 128, 8, fake, fake, None, 0, None) == 0          # empty: no-op
    assert r(fake, 4, 0, 8, fake, fake, None, 0, None) == -1           # no experts
    assert r(fake, 4, 128, 0, fake, fake, None, 0, None) == -1         # top_k < 1
    assert r(fake, 4, 6, 8, fake, fake, None, 0, None) == -4           # top_k > n_experts
    assert r(fake, 4, 128, 33, fake, fake, None, 0, None) == -4        # top_k > 32
    assert r(fake, 65, 128, 8, fake, fake, None, 0, None) == -4        # M*top_k > 512
    assert r(fake, 4, 8192, 8, fake, fake, None, 0, None) == -4        # n_experts > 4096
    assert r(None, 4, 128, 8, fake, fake, None, 0, None) == -1         # null logits
    assert r(P(0x1002), 4, 128, 8, fake, fake, None, 0, None) == -5    # logits alignment
    assert r(fake, 4, 128, 8, fake, fake, P(0x1080), 1 << 20, None) == -7  # workspace alignment
    assert r(fake, 4, 128, 8, fake, fake, fake, 64, None) == -7        # workspace too small


def test_ffn_argument_errors_without_gpu(L):
    f = 0x1000
    def call(w, ids=f, gate=f, x=f, xd=0, y=f, H=512, M=2, k=4, ws=f, wsb=1 << 30):
        return kq.lib().kq_moe_ffn(None if w is None else ctypes.cast(ctypes.pointer(w), ctypes.c_void_p),
                                   ids, gate, x, xd, y, H, M, k, ws, wsb, None)
    def w(**kw):
        a = dict(type_gate_up=1, type_down=3, n_experts=16, act=1, F=320, W_gate=f, W_up=f, W_down=f, SH=0)
        a.update(kw)
        return kq.ffn_weights(a["type_gate_up"], a["type_down"], a["n_experts"], a["act"], a["F"], a["W_gate"],
                              a["W_up"], a["W_down"], a["SH"], a.get("Ws_gate"), a.get("Ws_up"), a.get("Ws_down"))
    assert call(None) == -1                                  # no weights struct
    assert call(w(type_down=9)) == -2                        # unknown block type
    assert call(w(act=7)) == -1                              # unknown activation
    assert call(w(), xd=5) == -1                             # bad x dtype
    assert call(w(F=100)) == -3                              # F not a multiple of 32
    assert call(w(), H=500) == -3                            # H not a multiple of 32
    assert call(w(), M=0) == 0                               # empty: no-op
    assert call(w(), M=200, k=4) == -4                       # 800 pairs > 512
    assert call(w(SH=64)) == -1                              # shared width without shared weights
    assert call(w(W_up=None)) == -1                          # null weight
    assert call(w(W_gate=0x1008)) == -5                      # weight alignment
    assert call(w(), ws=0x1080) == -7                        # workspace alignment
    assert call(w(), wsb=64) == -7                           # workspace too small
    assert kq.kq_moe_ffn_workspace_size(512, 320, 0, 2, 4, 16) > 0
    assert kq.kq_moe_ffn_workspace_size(512, 320, 0, 200, 4, 16) == 0
    h_off, hs_off = kq.kq_moe_ffn_offsets(512, 320, 288, 2, 4, 16)
    assert h_off % 256 == 0 and hs_off >= h_off + 4 * 8 * 320


def test_moe_argument_errors_without_gpu(L):
    f = 0x100000
    def call(**kw):
        a = dict(type=1, W=f, E=128, ids=f, gate=None, x=f, xd=1, per_slot=0, y=0x200000, N=704, K=2816, M=1,
                 top_k=8, ws=0x300000, wsb=1 << 24)
        a.update(kw)
        return L.kq_moe_matvec(a["type"], a["W"], a["E"], a["ids"], a["gate"], a["x"], a["xd"], a["per_slot"],
                               a["y"], a["N"], a["K"], a["M"], a["top_k"], a["ws"], a["wsb"], None)
    assert call(type=0) == -2
    assert call(xd=3) == -1
    assert call(K=700) == -3
    assert call(M=0) == 0                                   # empty: no-op
    assert call(top_k=0) == -1
    assert call(M=100, top_k=8) == -4                       # more than 512 pairs
    assert call(K=16384, type=3) == -4                      # 32 rows over the tile limit
    assert call(W=0x100008) == -5
    assert call(ws=None) == -7
    assert call(ws=0x300010) == -7                          # workspace alignment
    assert call(wsb=100) == -7
    assert L.kq_moe_workspace_size(704, 1, 8, 128) > 0
    assert L.kq_moe_workspace_size(704, 100, 8, 128) == 0


def test_header_is_plain_c_and_links(L, tmp_path):
    """include/kq.h compiles as C99 and a C program links against libkq.so and
    calls it (argument-error paths only: no CUDA call is made)."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    src = tmp_path / "use_kq.c"
    src.write_text(
        '#include "kq.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "  kq_moe_ffn_weights w = {0};\n"
        "  int code = 0;\n"
        "  if (kq_block_bytes(KQ_Q4_K) != 144 || kq_block_bytes(KQ_IA4) != 144) return 1;\n"
        "  if (kq_matvec(KQ_Q6_K, 0, 0, KQ_BF16, 0, 4, 250, 1, 0) != KQ_ERR_SHAPE) return 2;\n"
        "  if (kq_moe_ffn(&w, 0, 0, 0, KQ_F32, 0, 512, 2, 4, 0, 0, 0) != KQ_ERR_TYPE) return 3;\n"
        "  if (kq_selftest_wait(7, &code, 0) != KQ_ERR_ARG) return 4;\n"
        "  printf(\"%s\\n\", kq_status_string(KQ_ERR_WORKSPACE));\n"
        "  return 0;\n"
        "}\n")
    exe = tmp_path / "use_kq"
    libdir = os.path.dirname(kq.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), "-L", libdir, "-lkq", "-Wl,-rpath," + libdir])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip()
