"""Thin Python binding of libkq's C ABI (include/kq.h): argument marshalling only.

Every function named ``kq_*`` here calls the C function of the same name with
the device pointers of the given torch tensors and the current CUDA stream;
all computation happens in libkq's CUDA kernels.  There is no fallback: if
libkq.so is missing or fails to load, importing the library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkq.so")

KQ_Q4_K, KQ_Q5_K, KQ_Q6_K, KQ_IA4 = 1, 2, 3, 4
KQ_F32, KQ_BF16 = 0, 1
KQ_ACT_SILU, KQ_ACT_GELU_TANH = 0, 1
KQ_OK = 0
STATUS = {0: "KQ_OK", -1: "KQ_ERR_ARG", -2: "KQ_ERR_TYPE", -3: "KQ_ERR_SHAPE", -4: "KQ_ERR_UNSUPPORTED",
          -5: "KQ_ERR_ALIGN", -6: "KQ_ERR_CUDA", -7: "KQ_ERR_WORKSPACE", -8: "KQ_ERR_DEVICE"}

# exported symbols and their C signatures (kept in step with include/kq.h)
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "kq_block_bytes": (_SZ, [_I]),
    "kq_ia4_pack": (_I, [_P, _P, _P, _I64, _I64, _P, _P]),
    "kq_unpack": (_I, [_I, _P, _I64, _P, _P, _P, _P, _P, _P]),
    "kq_dequant": (_I, [_I, _P, _P, _I64, _P]),
    "kq_dequant_bf16": (_I, [_I, _P, _P, _I64, _P]),
    "kq_moe_route": (_I, [_P, _I64, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _SZ, _P]),
    "kq_matvec": (_I, [_I, _P, _P, _I, _P, _I64, _I64, _I64, _P]),
    "kq_chain_workspace_size": (_SZ, [_P, _I]),
    "kq_chain_prepare": (_I, [_P, _I, _P, _SZ, _P, _P]),
    "kq_chain_run": (_I, [_P, _P, _P]),
    "kq_moe_workspace_size": (_SZ, [_I64, _I64, ctypes.c_int32, ctypes.c_int32]),
    "kq_moe_matvec": (_I, [_I, _P, ctypes.c_int32, _P, _P, _P, _I, _I, _P, _I64, _I64, _I64, ctypes.c_int32,
                           _P, _SZ, _P]),
    "kq_moe_check": (_I, [_P, _P]),
    "kq_selftest_wait": (_I, [_I, ctypes.POINTER(ctypes.c_int), _P]),
    "kq_moe_ffn_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, ctypes.c_int32, ctypes.c_int32]),
    "kq_moe_ffn_offsets": (_I, [_I64, _I64, _I64, _I64, ctypes.c_int32, ctypes.c_int32,
                                ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "kq_moe_ffn": (_I, [_P, _P, _P, _P, _I, _P, _I64, _I64, ctypes.c_int32, _P, _SZ, _P]),
    "kq_moe_matvec_noalloc": (_I, [_I, _P, ctypes.c_int32, _P, _P, _P, _I, _I, _P, _I64, _I64, _I64,
                                   ctypes.c_int32, _P]),
    "kq_device_error": (_I, [ctypes.POINTER(ctypes.c_int), _I]),
    "kq_last_cuda_error": (_I, []),
    "kq_status_string": (ctypes.c_char_p, [_I]),
}


# The sources each kernel family is compiled from (the one-token / program
# kernel: kq_gemv_kernel.cuh, the translation units that instantiate it and
# the headers it includes).
KERNEL_SOURCES = {
    "prog_kernel": ("kq_gemv_kernel.cuh", "kq_gemv.cu", "kq_gemv_q4k.cu", "kq_gemv_q5k.cu", "kq_gemv_q6k.cu",
                    "kq_gemv_ia4.cu", "kq_lane.cuh", "kq_ptx.cuh", "kq_internal.h", "kq_decode.cuh"),
}


def build_id(kernel=None) -> str:
    """Hash of the kernel sources (identifies which code a profile was taken
    on): all of csrc, or only the files of one kernel family."""
    import glob
    import hashlib
    h = hashlib.sha256()
    if kernel is None:
        files = sorted(glob.glob(os.path.join(PKG, "csrc", "*")))
    else:
        files = [os.path.join(PKG, "csrc", n) for n in KERNEL_SOURCES[kernel]]
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


class KQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _lib.kq_status_string(status).decode() if _lib is not None else ""
        extra = ""
        if status == -6 and _lib is not None:
            extra = f" (cudaError {_lib.kq_last_cuda_error()})"
        super().__init__(f"{fn}: {STATUS.get(status, status)} -- {msg}{extra}")


_lib = None


def use_timeline_library() -> ctypes.CDLL:
    """Build and load libkq_timeline.so (the library with the one-token
    kernel's per-CTA timer stamps) in place of libkq.so; call before any other
    use of the library in the process."""
    global LIB_PATH
    if _lib is not None:
        raise RuntimeError("the library is already loaded")
    from . import build
    LIB_PATH = build.build(timeline=True)
    L = lib()
    L.kq_timeline_read.restype = ctypes.c_int
    L.kq_timeline_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    return L


def lib() -> ctypes.CDLL:
    """Load libkq.so (built in-tree by ``gguf_quant_weight_super_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkq.so not built ({LIB_PATH}); run gguf_quant_weight_super_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libkq takes device tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, status: int):
    if status != KQ_OK:
        raise KQError(fn, status)


def kq_block_bytes(qtype: int) -> int:
    return lib().kq_block_bytes(qtype)


def kq_unpack(qtype, blocks, n_blocks, codes=None, scales=None, mins=None, d_bits=None, dmin_bits=None,
              stream=None):
    _check("kq_unpack", lib().kq_unpack(qtype, _ptr(blocks), n_blocks, _ptr(codes), _ptr(scales), _ptr(mins),
                                        _ptr(d_bits), _ptr(dmin_bits), _stream(stream)))


def kq_dequant(qtype, blocks, out, n, stream=None):
    _check("kq_dequant", lib().kq_dequant(qtype, _ptr(blocks), _ptr(out), n, _stream(stream)))


def kq_moe_route(logits, M, n_experts, top_k, expert_ids, gate_w, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kq_moe_route", lib().kq_moe_route(_ptr(logits), M, n_experts, top_k, _ptr(expert_ids), _ptr(gate_w),
                                              _ptr(workspace), ws_bytes, _stream(stream)))


def moe_route(logits: torch.Tensor, top_k: int, workspace=None, stream=None):
    """(ids int32 [M, top_k], gate fp32 [M, top_k]) for logits [M, n_experts] (kq_moe_route)."""
    M, E = logits.shape
    ids = torch.empty((M, top_k), dtype=torch.int32, device=logits.device)
    gate = torch.empty((M, top_k), dtype=torch.float32, device=logits.device)
    kq_moe_route(logits, M, E, top_k, ids, gate, workspace, stream)
    return ids, gate


def kq_ia4_pack(q, scales, biases, N, K, blocks, stream=None):
    _check("kq_ia4_pack", lib().kq_ia4_pack(_ptr(q), _ptr(scales), _ptr(biases), N, K, _ptr(blocks),
                                            _stream(stream)))


def ia4_pack(q: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor) -> torch.Tensor:
    """MLX group-affine INT4 arrays (int32 codes [N, K/8], bf16-bit scales and
    biases [N, K/64] as int16 or bfloat16) -> KQ_IA4 blocks (uint8)."""
    N, K = q.shape[0], q.shape[1] * 8
    out = torch.empty(N * ((K + 255) // 256) * 144, dtype=torch.uint8, device=q.device)
    kq_ia4_pack(q, scales, biases, N, K, out)
    return out


def kq_dequant_bf16(qtype, blocks, out, n, stream=None):
    _check("kq_dequant_bf16", lib().kq_dequant_bf16(qtype, _ptr(blocks), _ptr(out), n, _stream(stream)))


def kq_matvec(qtype, W, x, x_dtype, y, N, K, M, stream=None):
    _check("kq_matvec", lib().kq_matvec(qtype, _ptr(W), _ptr(x), x_dtype, _ptr(y), N, K, M, _stream(stream)))


class KqOp(ctypes.Structure):
    """struct kq_op of include/kq.h."""
    _fields_ = [("type", ctypes.c_int32), ("x_dtype", ctypes.c_int32), ("wait_previous", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("W", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class KqChainPlan(ctypes.Structure):
    """struct kq_chain_plan of include/kq.h (opaque)."""
    _fields_ = [("opaque", ctypes.c_int64 * 8)]


def _op_array(ops):
    arr = (KqOp * len(ops))()
    for i, o in enumerate(ops):
        arr[i] = KqOp(o["type"], o["x_dtype"], int(o.get("wait_previous", 0)), 0, _ptr(o["W"]), _ptr(o["x"]),
                      _ptr(o["y"]), o["N"], o["K"])
    return arr


def kq_chain_workspace_size(ops) -> int:
    arr = _op_array(ops)
    return lib().kq_chain_workspace_size(ctypes.cast(arr, ctypes.c_void_p), len(ops))


def kq_chain_prepare(ops, workspace, workspace_bytes, plan: KqChainPlan, stream=None):
    arr = _op_array(ops)
    _check("kq_chain_prepare", lib().kq_chain_prepare(ctypes.cast(arr, ctypes.c_void_p), len(ops), _ptr(workspace),
                                                      workspace_bytes, ctypes.cast(ctypes.pointer(plan), ctypes.c_void_p),
                                                      _stream(stream)))


def kq_chain_run(plan: KqChainPlan, workspace, stream=None):
    _check("kq_chain_run", lib().kq_chain_run(ctypes.cast(ctypes.pointer(plan), ctypes.c_void_p), _ptr(workspace),
                                              _stream(stream)))


def kq_moe_workspace_size(N, M, top_k, n_experts) -> int:
    return lib().kq_moe_workspace_size(N, M, top_k, n_experts)


def kq_moe_matvec(qtype, W_experts, n_experts, expert_ids, gate_w, x, x_dtype, x_per_slot, y, N, K, M, top_k,
                  workspace, workspace_bytes, stream=None):
    _check("kq_moe_matvec", lib().kq_moe_matvec(qtype, _ptr(W_experts), n_experts, _ptr(expert_ids), _ptr(gate_w),
                                                _ptr(x), x_dtype, int(x_per_slot), _ptr(y), N, K, M, top_k,
                                                _ptr(workspace), workspace_bytes, _stream(stream)))


def kq_moe_matvec_noalloc(qtype, W_experts, n_experts, expert_ids, gate_w, x, x_dtype, x_per_slot, y, N, K, M,
                          top_k, stream=None):
    _check("kq_moe_matvec_noalloc",
           lib().kq_moe_matvec_noalloc(qtype, _ptr(W_experts), n_experts, _ptr(expert_ids), _ptr(gate_w), _ptr(x),
                                       x_dtype, int(x_per_slot), _ptr(y), N, K, M, top_k, _stream(stream)))


def kq_moe_check(workspace, stream=None):
    _check("kq_moe_check", lib().kq_moe_check(_ptr(workspace), _stream(stream)))


def moe_workspace(N, M, top_k, n_experts, device="cuda") -> torch.Tensor:
    """A zero-filled workspace tensor for kq_moe_matvec (the caching allocator aligns it to 512 bytes)."""
    n = kq_moe_workspace_size(N, M, top_k, n_experts)
    if n == 0:
        raise KQError("kq_moe_workspace_size", -4)
    return torch.zeros(n, dtype=torch.uint8, device=device)


class KqMoeFfnWeights(ctypes.Structure):
    """struct kq_moe_ffn_weights of include/kq.h."""
    _fields_ = [("type_gate_up", ctypes.c_int32), ("type_down", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("act", ctypes.c_int32), ("F", ctypes.c_int64), ("SH", ctypes.c_int64),
                ("W_gate", ctypes.c_void_p), ("W_up", ctypes.c_void_p), ("W_down", ctypes.c_void_p),
                ("Ws_gate", ctypes.c_void_p), ("Ws_up", ctypes.c_void_p), ("Ws_down", ctypes.c_void_p)]


def ffn_weights(type_gate_up, type_down, n_experts, act, F, W_gate, W_up, W_down, SH=0, Ws_gate=None, Ws_up=None,
                Ws_down=None) -> KqMoeFfnWeights:
    return KqMoeFfnWeights(type_gate_up, type_down, n_experts, act, F, SH, _ptr(W_gate), _ptr(W_up), _ptr(W_down),
                           _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down))


def kq_moe_ffn_workspace_size(H, F, SH, M, top_k, n_experts) -> int:
    return lib().kq_moe_ffn_workspace_size(H, F, SH, M, top_k, n_experts)


def kq_moe_ffn_offsets(H, F, SH, M, top_k, n_experts):
    """(byte offset of h [M*top_k][F], byte offset of hs [M][SH]) in the workspace."""
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("kq_moe_ffn_offsets", lib().kq_moe_ffn_offsets(H, F, SH, M, top_k, n_experts, ctypes.byref(a),
                                                          ctypes.byref(b)))
    return a.value, b.value


def moe_ffn_workspace(H, F, SH, M, top_k, n_experts, device="cuda") -> torch.Tensor:
    """A zero-filled workspace tensor for kq_moe_ffn."""
    n = kq_moe_ffn_workspace_size(H, F, SH, M, top_k, n_experts)
    if n == 0:
        raise KQError("kq_moe_ffn_workspace_size", -4)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def kq_moe_ffn(weights: KqMoeFfnWeights, expert_ids, gate_w, x, x_dtype, y, H, M, top_k, workspace,
               workspace_bytes, stream=None):
    _check("kq_moe_ffn", lib().kq_moe_ffn(ctypes.cast(ctypes.pointer(weights), ctypes.c_void_p), _ptr(expert_ids),
                                          _ptr(gate_w), _ptr(x), x_dtype, _ptr(y), H, M, top_k, _ptr(workspace),
                                          workspace_bytes, _stream(stream)))


def kq_selftest_wait(kind: int, stream=None) -> int:
    """Run the bounded-wait self-test (0: mbarrier, 1: grid barrier); returns the observed error code."""
    code = ctypes.c_int(-1)
    _check("kq_selftest_wait", lib().kq_selftest_wait(kind, ctypes.byref(code), _stream(stream)))
    return code.value


def kq_device_error(clear: bool = False) -> int:
    code = ctypes.c_int(0)
    st = lib().kq_device_error(ctypes.byref(code), int(clear))
    if st not in (KQ_OK, -8):
        raise KQError("kq_device_error", st)
    return code.value


# ---------------------------------------------------------------------------
# Convenience wrappers that allocate outputs with torch (still one C call each).
# ---------------------------------------------------------------------------

def x_dtype_of(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return KQ_F32
    if x.dtype == torch.bfloat16:
        return KQ_BF16
    raise TypeError("x must be float32 or bfloat16")


def matvec(qtype: int, W: torch.Tensor, x: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None):
    """y = W x for x of shape (M, K) (or (K,)); returns fp32 (M, N)."""
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    kq_matvec(qtype, W, x2, x_dtype_of(x2), y, N, K, M)
    return y


class Chain:
    """A prepared chain of one-token products (kq_chain_* of include/kq.h).

    ops: dicts with keys type, x_dtype, W, x, y, N, K and optionally
    wait_previous; the tensors must stay alive while the chain is used.
    The workspace is a torch uint8 tensor owned by this object.
    """

    def __init__(self, ops, device=None, stream=None):
        self.ops = list(ops)
        n = kq_chain_workspace_size(self.ops)
        if n == 0:
            raise KQError("kq_chain_workspace_size", -4)
        dev = device if device is not None else self.ops[0]["y"].device
        self.workspace = torch.empty(n + 256, dtype=torch.uint8, device=dev)
        off = (-self.workspace.data_ptr()) % 256
        self._ws_ptr = self.workspace.data_ptr() + off
        self._ws_bytes = n
        self.plan = KqChainPlan()
        kq_chain_prepare(self.ops, self._ws_ptr, self._ws_bytes, self.plan, stream)

    def run(self, stream=None):
        kq_chain_run(self.plan, self._ws_ptr, stream)


def dequant(qtype: int, blocks: torch.Tensor, n: int) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.float32, device=blocks.device)
    kq_dequant(qtype, blocks, out, n)
    return out


def dequant_bf16(qtype: int, blocks: torch.Tensor, n: int) -> torch.Tensor:
    """The weights as a torch.bfloat16 tensor (kq_dequant_bf16)."""
    out = torch.empty(n, dtype=torch.bfloat16, device=blocks.device)
    kq_dequant_bf16(qtype, blocks, out, n)
    return out
