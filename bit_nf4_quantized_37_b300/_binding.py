"""ctypes binding of libqlora_nf4.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# QLORA_NF4_LIB may name another build of the same library (the bounds-checked variant,
# libqlora_nf4_checked.so, built by `python -m bit_nf4_quantized_37_b300.build --checked`)
LIB_PATH = os.environ.get("QLORA_NF4_LIB") or os.path.join(_HERE, "libqlora_nf4.so")

NF4_BLOCKSIZE = 64
NF4_DQ_BLOCK = 256
NF4_NO_DQ = 0

_STATUS = {0: "QLORA_OK", -1: "QLORA_ERR_INVALID_ARG", -2: "QLORA_ERR_UNSUPPORTED",
           -3: "QLORA_ERR_MISALIGNED", -4: "QLORA_ERR_WORKSPACE", -5: "QLORA_ERR_CUDA",
           -6: "QLORA_ERR_DEVICE_TIMEOUT", -7: "QLORA_ERR_NO_DEVICE", -8: "QLORA_ERR_TOO_LARGE"}
NF4_NOALLOC_MAX_NUMEL = 1 << 26

# Every symbol include/qlora_nf4.h declares.
EXPORTS = ["nf4_storage_bytes", "nf4_quantize_workspace_bytes", "nf4_quantize",
           "nf4_dequantize", "qlora_workspace_bytes", "qlora_linear_fwd", "qlora_linear_bwd",
           "nf4_level_table", "qlora_device_status", "qlora_status_str", "qlora_version",
           "qlora_profile_start", "qlora_profile_stop", "nf4_quantize_noalloc",
           "nf4_merge_lora", "nf4_int4_error_workspace_bytes", "nf4_int4_error_stats",
           "qlora_linear_fwd_multi", "nf4_dequantize_f16", "qlora_linear_fwd_f16",
           "qlora_linear_bwd_f16", "qlora_wait_timeout_selftest"]


class QLoRAError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {_STATUS.get(status, status)} "
                         f"({status_str(status) if _lib is not None else ''})")


class _NF4Struct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale_codes", ctypes.c_void_p),
                ("scale_steps", ctypes.c_void_p), ("scale_mean", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("blocksize", ctypes.c_int32), ("dq_block", ctypes.c_int32),
                ("dq_type", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bit_nf4_quantized_37_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u64p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        sp = ctypes.POINTER(_NF4Struct)
        sig = {
            "nf4_storage_bytes": [i64, i64, i32, i32, u64p, u64p],
            "nf4_quantize_workspace_bytes": [i64, u64p],
            "nf4_quantize": [vp, sp, vp, ctypes.c_uint64, vp],
            "nf4_dequantize": [sp, vp, vp],
            "nf4_dequantize_f16": [sp, vp, vp],
            "qlora_workspace_bytes": [i64, i64, i64, i32, u64p],
            "qlora_linear_fwd": [vp, i64, sp, vp, vp, i32, ctypes.c_float, vp, vp, vp,
                                 ctypes.c_uint64, vp],
            "qlora_linear_bwd": [vp, vp, i64, sp, vp, vp, i32, ctypes.c_float, vp, vp, vp, vp,
                                 vp, ctypes.c_uint64, vp],
            "qlora_linear_fwd_f16": [vp, i64, sp, vp, vp, i32, ctypes.c_float, vp, vp, vp,
                                     ctypes.c_uint64, vp],
            "qlora_linear_bwd_f16": [vp, vp, i64, sp, vp, vp, i32, ctypes.c_float, vp, vp, vp,
                                     vp, vp, ctypes.c_uint64, vp],
            "nf4_level_table": [vp, vp],
            "qlora_device_status": [vp, vp],
            "qlora_wait_timeout_selftest": [vp],
            "qlora_status_str": [ctypes.c_int],
            "qlora_version": [],
            "qlora_profile_start": [],
            "qlora_profile_stop": [vp, i32, vp],
            "nf4_quantize_noalloc": [vp, sp, vp],
            "nf4_merge_lora": [sp, vp, vp, i32, ctypes.c_float, vp, vp, vp],
            "qlora_linear_fwd_multi": [vp, i64, sp, vp, vp, i32, i32, vp, vp, vp, vp,
                                       ctypes.c_uint64, vp],
            "nf4_int4_error_workspace_bytes": [u64p],
            "nf4_int4_error_stats": [vp, i64, vp, vp, ctypes.c_uint64, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "qlora_status_str" else ctypes.c_int
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().qlora_status_str(int(status)).decode()


def _check(call: str, status: int):
    if status != 0:
        raise QLoRAError(call, status)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream() -> int:
    return int(torch.cuda.current_stream().cuda_stream)


def _u64() -> ctypes.c_uint64:
    return ctypes.c_uint64(0)


# ------------------------------------------------------------------------- NF4 tensor
@dataclass
class NF4Tensor:
    """Blockwise NF4 weights with double-quantized scales (device tensors)."""
    codes: torch.Tensor        # uint8 [ceil(numel/2)]
    scale_codes: torch.Tensor  # int8  [ceil(numel/64)]
    scale_steps: torch.Tensor  # fp32  [ceil(numel/16384)]
    scale_mean: torch.Tensor   # fp32  [1]
    rows: int
    cols: int
    dq_block: int = NF4_DQ_BLOCK  # NF4_NO_DQ: scale_steps holds the fp32 block absmax
    dq_type: int = 0              # 1: second-level codes are E4M3 8-bit floats (else int8)

    @property
    def numel(self) -> int:
        return self.rows * self.cols

    def c_struct(self) -> _NF4Struct:
        def p(t):
            return _ptr(t) if t is not None and t.numel() > 0 else 0
        return _NF4Struct(p(self.codes), p(self.scale_codes), p(self.scale_steps),
                          p(self.scale_mean), self.rows, self.cols, NF4_BLOCKSIZE, self.dq_block,
                          self.dq_type)

    def storage_bytes(self) -> int:
        return nf4_storage_bytes(self.rows, self.cols, self.dq_block)[1]

    @staticmethod
    def empty(rows: int, cols: int, device, double_quant: bool = True,
              fp8_second_level: bool = False) -> "NF4Tensor":
        dq = NF4_DQ_BLOCK if double_quant else NF4_NO_DQ
        sizes, _ = nf4_storage_bytes(rows, cols, dq)
        return NF4Tensor(torch.empty(sizes[0], dtype=torch.uint8, device=device),
                         torch.empty(sizes[1], dtype=torch.int8, device=device),
                         torch.empty(sizes[2] // 4, dtype=torch.float32, device=device),
                         torch.empty(sizes[3] // 4, dtype=torch.float32, device=device), rows, cols,
                         dq, 1 if (fp8_second_level and double_quant) else 0)


def nf4_storage_bytes(rows: int, cols: int, dq_block: int = 256) -> tuple[list[int], int]:
    sizes = (ctypes.c_uint64 * 4)()
    total = _u64()
    _check("nf4_storage_bytes", lib().nf4_storage_bytes(rows, cols, NF4_BLOCKSIZE, dq_block,
                                                         sizes, ctypes.byref(total)))
    return [int(s) for s in sizes], int(total.value)


def nf4_quantize_workspace_bytes(numel: int) -> int:
    out = _u64()
    _check("nf4_quantize_workspace_bytes", lib().nf4_quantize_workspace_bytes(numel, ctypes.byref(out)))
    return int(out.value)


def qlora_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    out = _u64()
    _check("qlora_workspace_bytes", lib().qlora_workspace_bytes(M, N, K, r, ctypes.byref(out)))
    return int(out.value)


def level_table():
    L = (ctypes.c_float * 16)()
    T = (ctypes.c_float * 15)()
    _check("nf4_level_table", lib().nf4_level_table(L, T))
    return list(L), list(T)


# Workspaces are caller-owned device memory; the binding keeps one growing buffer per device.
_ws_cache: dict = {}


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (torch.device(device).index, torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _shape(t, want: tuple, name: str):
    """Raise ValueError unless t has exactly the shape `want` (checked before any launch: a
    mismatched buffer would make a kernel read or write past its allocation)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(want):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(want)}")


def _numel(t, want: int, name: str):
    if t is not None and t.numel() != want:
        raise ValueError(f"{name} has {t.numel()} elements, expected {want}")


def _check_nf4(q: "NF4Tensor"):
    """The NF4 buffers hold at least the sizes rows x cols needs in its format."""
    if q.rows < 1 or q.cols < 1:
        raise ValueError(f"NF4Tensor has shape ({q.rows}, {q.cols})")
    sizes, _ = nf4_storage_bytes(q.rows, q.cols, q.dq_block)
    need = [("codes", q.codes, sizes[0], 1), ("scale_codes", q.scale_codes, sizes[1], 1),
            ("scale_steps", q.scale_steps, sizes[2], 4), ("scale_mean", q.scale_mean, sizes[3], 4)]
    for name, t, nbytes, esz in need:
        have = 0 if t is None else t.numel() * t.element_size()
        if have < nbytes:
            raise ValueError(f"NF4Tensor.{name} holds {have} bytes, its {q.rows} x {q.cols} "
                             f"tensor needs {nbytes}")


def _rank2(t, name: str):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    return t.shape


def _req(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def nf4_quantize(W: torch.Tensor, out: NF4Tensor | None = None,
                 workspace: torch.Tensor | None = None, double_quant: bool = True,
                 fp8_second_level: bool = False) -> NF4Tensor:
    """Quantize fp32 weights [rows, cols] (CUDA) to NF4 with double-quantized scales (int8, or
    E4M3 with fp8_second_level), or with fp32 block absmax scales when double_quant is False
    (an `out` tensor brings its own variant)."""
    rows, cols = (W.shape[0], W.shape[1]) if W.dim() == 2 else (1, W.numel())
    if out is not None:
        _numel(W, out.rows * out.cols, "W")
        _check_nf4(out)
    _req(W, torch.float32, "W")
    q = out if out is not None else NF4Tensor.empty(rows, cols, W.device, double_quant,
                                                    fp8_second_level)
    nb = nf4_quantize_workspace_bytes(rows * cols)
    ws = workspace if workspace is not None else _workspace(nb, W.device)
    s = q.c_struct()
    _check("nf4_quantize", lib().nf4_quantize(_ptr(W), ctypes.byref(s), _ptr(ws),
                                              ws.numel() * ws.element_size(), _stream()))
    return q


def nf4_quantize_noalloc(W: torch.Tensor, out: NF4Tensor) -> NF4Tensor:
    """nf4_quantize for callers that must not allocate device memory: the output buffers
    are the caller's and the scratch is the library's fixed device array (up to
    NF4_NOALLOC_MAX_NUMEL weights).  Calls overlapping on the GPU race on that array."""
    _numel(W, out.rows * out.cols, "W")
    _check_nf4(out)
    _req(W, torch.float32, "W")
    s = out.c_struct()
    _check("nf4_quantize_noalloc", lib().nf4_quantize_noalloc(_ptr(W), ctypes.byref(s), _stream()))
    return out


def _dequantize(call: str, dtype, q: NF4Tensor, out: torch.Tensor | None) -> torch.Tensor:
    _check_nf4(q)
    _numel(out, q.rows * q.cols, "out")
    o = out if out is not None else torch.empty(q.rows, q.cols, dtype=dtype,
                                                device=q.codes.device)
    _req(o, dtype, "out")
    s = q.c_struct()
    _check(call, getattr(lib(), call)(ctypes.byref(s), _ptr(o), _stream()))
    return o


def nf4_dequantize(q: NF4Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [rows, cols] dequantization of an NF4Tensor."""
    return _dequantize("nf4_dequantize", torch.bfloat16, q, out)


def nf4_dequantize_f16(q: NF4Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp16 [rows, cols] dequantization of an NF4Tensor (the fp16 compute type)."""
    return _dequantize("nf4_dequantize_f16", torch.float16, q, out)


def _linear_shapes(X, q, A, B):
    """(M, N, K, r) of a LoRA-wrapped linear call; ValueError on any mismatch with the NF4
    base [N, K]: X [M, K], A [r, K], B [N, r]."""
    _check_nf4(q)
    M, K = _rank2(X, "X")
    N = q.rows
    if K != q.cols:
        raise ValueError(f"X has {K} columns, the NF4 base has {q.cols}")
    r = _rank2(A, "A")[0]
    _shape(A, (r, K), "A")
    _shape(B, (N, r), "B")
    return M, N, K, r


def _linear_fwd(call: str, dtype, X, q, A, B, scale, save_u, out):
    M, N, K, r = _linear_shapes(X, q, A, B)
    _shape(out, (M, N), "out")
    for t, n in ((X, "X"), (A, "A"), (B, "B")):
        _req(t, dtype, n)
    Y = out if out is not None else torch.empty(M, N, dtype=dtype, device=X.device)
    _req(Y, dtype, "out")
    U = torch.empty(M, r, dtype=torch.float32, device=X.device) if save_u else None
    nb = qlora_workspace_bytes(M, N, K, r)
    ws = _workspace(nb, X.device)
    s = q.c_struct()
    _check(call, getattr(lib(), call)(
        _ptr(X), M, ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale), _ptr(Y), _ptr(U),
        _ptr(ws), ws.numel(), _stream()))
    return Y, U


def qlora_linear_fwd(X: torch.Tensor, q: NF4Tensor, A: torch.Tensor, B: torch.Tensor,
                     scale: float, save_u: bool = True, out: torch.Tensor | None = None):
    """Y = X W'^T + scale (X A^T) B^T.  Returns (Y bf16 [M, N], U fp32 [M, r] or None)."""
    return _linear_fwd("qlora_linear_fwd", torch.bfloat16, X, q, A, B, scale, save_u, out)


def qlora_linear_fwd_f16(X: torch.Tensor, q: NF4Tensor, A: torch.Tensor, B: torch.Tensor,
                         scale: float, save_u: bool = True, out: torch.Tensor | None = None):
    """qlora_linear_fwd in the fp16 compute type: X, A, B and Y are fp16."""
    return _linear_fwd("qlora_linear_fwd_f16", torch.float16, X, q, A, B, scale, save_u, out)


def qlora_linear_fwd_multi(X: torch.Tensor, q: NF4Tensor, A_all: torch.Tensor,
                           B_all: torch.Tensor, adapter_idx: torch.Tensor, scales: torch.Tensor,
                           out: torch.Tensor | None = None) -> torch.Tensor:
    """Y_t = X_t W'^T + s_a (X_t A_a^T) B_a^T with a = adapter_idx[t], for M <= 16 tokens.
    A_all [n, r, K], B_all [n, N, r] bf16; adapter_idx int32 [M]; scales fp32 [n]."""
    _check_nf4(q)
    M, K = _rank2(X, "X")
    N = q.rows
    if K != q.cols:
        raise ValueError(f"X has {K} columns, the NF4 base has {q.cols}")
    if A_all.dim() != 3:
        raise ValueError(f"A_all must be 3-D [n, r, K], got shape {tuple(A_all.shape)}")
    n_ad, r, _ = A_all.shape
    _shape(A_all, (n_ad, r, K), "A_all")
    _shape(B_all, (n_ad, N, r), "B_all")
    _shape(adapter_idx, (M,), "adapter_idx")
    _shape(scales, (n_ad,), "scales")
    _shape(out, (M, N), "out")
    for t, n in ((X, "X"), (A_all, "A_all"), (B_all, "B_all")):
        _req(t, torch.bfloat16, n)
    _req(adapter_idx, torch.int32, "adapter_idx")
    _req(scales, torch.float32, "scales")
    Y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=X.device)
    nb = qlora_workspace_bytes(M, N, K, r)
    ws = _workspace(nb, X.device)
    s = q.c_struct()
    _check("qlora_linear_fwd_multi", lib().qlora_linear_fwd_multi(
        _ptr(X), M, ctypes.byref(s), _ptr(A_all), _ptr(B_all), r, n_ad, _ptr(adapter_idx),
        _ptr(scales), _ptr(Y), _ptr(ws), ws.numel(), _stream()))
    return Y


def _linear_bwd(call: str, dtype, dY, X, q, A, B, scale, U, need_dx):
    M, N, K, r = _linear_shapes(X, q, A, B)
    _shape(dY, (M, N), "dY")
    _shape(U, (M, r), "U")
    for t, n in ((dY, "dY"), (X, "X"), (A, "A"), (B, "B")):
        _req(t, dtype, n)
    if U is not None:
        _req(U, torch.float32, "U")
    dX = torch.empty(M, K, dtype=dtype, device=X.device) if need_dx else None
    dA = torch.empty(r, K, dtype=torch.float32, device=X.device)
    dB = torch.empty(N, r, dtype=torch.float32, device=X.device)
    nb = qlora_workspace_bytes(M, N, K, r)
    ws = _workspace(nb, X.device)
    s = q.c_struct()
    _check(call, getattr(lib(), call)(
        _ptr(dY), _ptr(X), M, ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale), _ptr(U),
        _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws), ws.numel(), _stream()))
    return dX, dA, dB


def qlora_linear_bwd(dY: torch.Tensor, X: torch.Tensor, q: NF4Tensor, A: torch.Tensor,
                     B: torch.Tensor, scale: float, U: torch.Tensor | None = None,
                     need_dx: bool = True):
    """Returns (dX bf16 [M, K] or None, dA fp32 [r, K], dB fp32 [N, r]); the base is frozen."""
    return _linear_bwd("qlora_linear_bwd", torch.bfloat16, dY, X, q, A, B, scale, U, need_dx)


def qlora_linear_bwd_f16(dY: torch.Tensor, X: torch.Tensor, q: NF4Tensor, A: torch.Tensor,
                         B: torch.Tensor, scale: float, U: torch.Tensor | None = None,
                         need_dx: bool = True):
    """qlora_linear_bwd in the fp16 compute type: dY, X, A, B and dX are fp16."""
    return _linear_bwd("qlora_linear_bwd_f16", torch.float16, dY, X, q, A, B, scale, U, need_dx)


def nf4_merge_lora(q: NF4Tensor, A: torch.Tensor, B: torch.Tensor, scale: float,
                   bf16: bool = True, f32: bool = False,
                   out: torch.Tensor | None = None, out_f32: torch.Tensor | None = None):
    """W_merged = bf16(W' + scale B A) for the NF4 base q, A [r, K], B [N, r] bf16.
    Returns (bf16 [N, K] or None, the same values as fp32 [N, K] or None)."""
    _check_nf4(q)
    r = _rank2(A, "A")[0]
    _shape(A, (r, q.cols), "A")
    _shape(B, (q.rows, r), "B")
    _shape(out, (q.rows, q.cols), "out")
    _shape(out_f32, (q.rows, q.cols), "out_f32")
    for t, n in ((A, "A"), (B, "B")):
        _req(t, torch.bfloat16, n)
    dev = q.codes.device
    o16 = out if out is not None else (
        torch.empty(q.rows, q.cols, dtype=torch.bfloat16, device=dev) if bf16 else None)
    o32 = out_f32 if out_f32 is not None else (
        torch.empty(q.rows, q.cols, dtype=torch.float32, device=dev) if f32 else None)
    if o16 is not None:
        _req(o16, torch.bfloat16, "out")
    if o32 is not None:
        _req(o32, torch.float32, "out_f32")
    s = q.c_struct()
    _check("nf4_merge_lora", lib().nf4_merge_lora(ctypes.byref(s), _ptr(A), _ptr(B), r,
                                                  float(scale), _ptr(o16), _ptr(o32), _stream()))
    return o16, o32


def nf4_int4_error_stats(W: torch.Tensor) -> torch.Tensor:
    """fp64 [3] on the device: sum w^2, NF4 and INT4 (absmax, 64-blocks) squared errors."""
    _req(W, torch.float32, "W")
    n = _u64()
    _check("nf4_int4_error_workspace_bytes", lib().nf4_int4_error_workspace_bytes(ctypes.byref(n)))
    ws = _workspace(n.value, W.device)
    out = torch.empty(3, dtype=torch.float64, device=W.device)
    _check("nf4_int4_error_stats", lib().nf4_int4_error_stats(
        _ptr(W), W.numel(), _ptr(out), _ptr(ws), ws.numel(), _stream()))
    return out


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32),
                ("total_ms", ctypes.c_double)]


def profile_start() -> None:
    """Bracket every library kernel launch with CUDA events until profile_stop()."""
    _check("qlora_profile_start", lib().qlora_profile_start())


def profile_stop() -> dict:
    """{kernel name: (launches, summed device ms)} since profile_start (synchronizes)."""
    cap = 64
    buf = (_KernelTime * cap)()
    n = ctypes.c_int32(0)
    _check("qlora_profile_stop", lib().qlora_profile_stop(buf, cap, ctypes.byref(n)))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n.value, cap))}


def wait_timeout_selftest() -> None:
    """Enqueue the bounded-wait self-test on the current stream: one wait that nothing
    completes, which gives up after its limit (about 2 s) and sets wait code 8; read it with
    device_status()."""
    _check("qlora_wait_timeout_selftest", lib().qlora_wait_timeout_selftest(_stream()))


def device_status() -> int:
    """Synchronizes the current stream; returns the kernels' bounded-wait error word."""
    out = ctypes.c_int32(0)
    st = lib().qlora_device_status(ctypes.byref(out), _stream())
    if st not in (0, -6):
        raise QLoRAError("qlora_device_status", st)
    return int(out.value)
