"""Python binding of the GB300 FP8 block-scaled GEMM C ABI (include/dgfp8.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libdgfp8.so``. PyTorch supplies device memory and the current stream. There
is no CPU fallback: if the shared library is missing or fails to load, import
of the compute functions raises.

The three compute calls carry the C names:

* ``dg_quantize_fp8_block(x, scale_mode)`` -> ``(q, scales)``: 128x128 block
  quantization (lpnh.cn DeepGEMM walkthrough §4.2).
* ``dg_fp8_gemm_nt(c, a, b, sa, sb, scale_mode)``: C = A . B^T with per-block
  scales, the argument order of fp8_gemm_nt(c, a_fp8, b_fp8, a_sf, b_sf) on
  pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §4.1.
* ``dg_fp8_grouped_gemm_contiguous(c, a, b, sa, sb, m_indices, scale_mode)``:
  the M-grouped contiguous MoE variant (same page §2.3, §3.2).
* ``dg_fp8_gemm(c, a, b, sa, sb, layout, scale_mode)``: the dense GEMM in any of
  the layouts NT, TN, NN, TT; ``dg_fp8_k_grouped_gemm_tn(c, a, b, sa, sb,
  k_sizes, scale_mode)``: the K-grouped GEMM (same page §3.1, §3.2).
* ``dg_fp8_gemm_nt_requant`` / ``dg_fp8_grouped_gemm_contiguous_requant``: the
  same GEMMs with the FP32 accumulators requantized to E4M3 codes plus block
  scales in the epilogue (walkthrough §2.2, §6); they return ``(cq, cs)``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

__all__ = [
    "DG_OK", "DG_SCALE_FP32", "DG_SCALE_UE8M0", "DG_INPUT_FP32", "DG_INPUT_BF16", "DgError", "lib",
    "library_path",
    "dg_get_abi_version", "dg_status_string", "dg_get_mk_alignment_for_contiguous_layout",
    "dg_set_num_sms", "dg_get_num_sms", "dg_quantize_fp8_block", "dg_fp8_gemm_nt",
    "dg_fp8_grouped_gemm_contiguous", "dg_get_device_status", "dg_selftest_wait_timeout",
    "dg_quantize_fp8_1x128", "dg_fp8_gemm_nt_1x128", "dg_fp8_grouped_gemm_contiguous_1x128",
    "dg_fp8_gemm_nt_requant", "dg_fp8_grouped_gemm_contiguous_requant", "dg_fp8_gemm",
    "dg_fp8_k_grouped_gemm_tn", "dg_fp8_gemm_requant", "DG_LAYOUT_NT", "DG_LAYOUT_TN", "DG_LAYOUT_NN", "DG_LAYOUT_TT",
    "declared_functions",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libdgfp8.so")
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "dgfp8.h")

DG_OK = 0
DG_ERR_INVALID_ARG = 1
DG_ERR_UNSUPPORTED_SHAPE = 2
DG_ERR_MISALIGNED = 3
DG_ERR_CUDA = 4
DG_ERR_NO_DEVICE = 5
DG_ERR_TIMEOUT = 6
DG_ERR_BAD_GROUP = 7
DG_SCALE_FP32 = 0
DG_SCALE_UE8M0 = 1
DG_INPUT_FP32 = 0
DG_INPUT_BF16 = 1
DG_LAYOUT_NT = 0
DG_LAYOUT_TN = 1
DG_LAYOUT_NN = 2
DG_LAYOUT_TT = 3
_LAYOUTS = {"NT": DG_LAYOUT_NT, "TN": DG_LAYOUT_TN, "NN": DG_LAYOUT_NN, "TT": DG_LAYOUT_TT}
BLOCK = 128

_lock = threading.Lock()
_lib = None


class DgError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {dg_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.dg_get_abi_version.restype = ctypes.c_uint32
        L.dg_status_string.restype = ctypes.c_char_p
        L.dg_status_string.argtypes = [i32]
        L.dg_get_mk_alignment_for_contiguous_layout.restype = i32
        L.dg_set_num_sms.argtypes = [i32]
        L.dg_set_num_sms.restype = i32
        L.dg_get_num_sms.restype = i32
        L.dg_quantize_fp8_block.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp]
        L.dg_quantize_fp8_block.restype = i32
        L.dg_fp8_gemm_nt.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp, i64, i64, i64, i32, vp]
        L.dg_fp8_gemm_nt.restype = i32
        L.dg_fp8_grouped_gemm_contiguous.argtypes = [vp, i64, vp, i64, vp, vp, vp, i32, vp,
                                                     i64, i64, i64, i32, vp]
        L.dg_fp8_grouped_gemm_contiguous.restype = i32
        L.dg_quantize_fp8_1x128.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, i32, vp]
        L.dg_quantize_fp8_1x128.restype = i32
        L.dg_fp8_gemm_nt_1x128.argtypes = L.dg_fp8_gemm_nt.argtypes
        L.dg_fp8_gemm_nt_1x128.restype = i32
        L.dg_fp8_grouped_gemm_contiguous_1x128.argtypes = L.dg_fp8_grouped_gemm_contiguous.argtypes
        L.dg_fp8_grouped_gemm_contiguous_1x128.restype = i32
        L.dg_fp8_gemm_nt_requant.argtypes = [vp, i64, vp, i32, i32, vp, i64, vp, i32, vp, i64, vp,
                                             i64, i64, i64, i32, vp]
        L.dg_fp8_gemm_nt_requant.restype = i32
        L.dg_fp8_grouped_gemm_contiguous_requant.argtypes = [vp, i64, vp, i32, i32, vp, i64, vp, i32, vp, vp,
                                                             i32, vp, i64, i64, i64, i32, vp]
        L.dg_fp8_grouped_gemm_contiguous_requant.restype = i32
        L.dg_fp8_gemm.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp, i64, i64, i64, i32, i32, vp]
        L.dg_fp8_gemm.restype = i32
        L.dg_fp8_gemm_requant.argtypes = [vp, i64, vp, i32, i32, vp, i64, vp, i32, vp, i64, vp,
                                          i64, i64, i64, i32, i32, vp]
        L.dg_fp8_gemm_requant.restype = i32
        L.dg_fp8_k_grouped_gemm_tn.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp, i32, vp, i64, i64, i32, vp]
        L.dg_fp8_k_grouped_gemm_tn.restype = i32
        L.dg_get_device_status.argtypes = [vp]
        L.dg_get_device_status.restype = i32
        L.dg_selftest_wait_timeout.argtypes = [i64, vp]
        L.dg_selftest_wait_timeout.restype = i32
        _lib = L
        return L


def declared_functions() -> list[str]:
    """Names of the entry points that include/dgfp8.h declares."""
    with open(_HEADER) as f:
        text = f.read()
    return re.findall(r"DG_API\s+[\w\s\*]+?\b(dg_\w+)\s*\(", text)


def dg_get_abi_version() -> int:
    return int(lib().dg_get_abi_version())


def dg_status_string(status: int) -> str:
    return lib().dg_status_string(int(status)).decode()


def dg_get_mk_alignment_for_contiguous_layout() -> int:
    return int(lib().dg_get_mk_alignment_for_contiguous_layout())


def dg_set_num_sms(n: int) -> None:
    _check(lib().dg_set_num_sms(int(n)), "dg_set_num_sms")


def dg_get_num_sms() -> int:
    return int(lib().dg_get_num_sms())


def _check(status: int, what: str) -> None:
    if status != DG_OK:
        raise DgError(status, what)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ld(t: torch.Tensor, name: str, empty_ld: int = 16) -> int:
    """Row stride in elements; an empty matrix gets a placeholder stride."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.numel() == 0:
        return max(empty_ld, (t.shape[1] + empty_ld - 1) // empty_ld * empty_ld)
    if t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor with unit column stride")
    return int(t.stride(0))


def _cuda(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _u8(t: torch.Tensor) -> torch.Tensor:
    """Codes may come as uint8 or torch.float8_e4m3fn; both are passed as bytes."""
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def dg_quantize_fp8_block(x: torch.Tensor, scale_mode: int = DG_SCALE_FP32,
                          q: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """Quantize a float32 CUDA matrix; returns (q uint8 [rows, cols], scales float32)."""
    _cuda(x, torch.float32, "x")
    rows, cols = x.shape
    ld_x = _ld(x, "x", 4)
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(((rows + BLOCK - 1) // BLOCK, (cols + BLOCK - 1) // BLOCK),
                             dtype=torch.float32, device=x.device)
    qb = _u8(q)
    _cuda(qb, torch.uint8, "q")
    _cuda(scales, torch.float32, "scales")
    ld_q = _ld(qb, "q", 4)
    st = lib().dg_quantize_fp8_block(ctypes.c_void_p(x.data_ptr()), rows, cols, ld_x,
                                     ctypes.c_void_p(qb.data_ptr()), ld_q,
                                     ctypes.c_void_p(scales.data_ptr()), int(scale_mode), _stream(x))
    _check(st, "dg_quantize_fp8_block")
    return q, scales


def dg_quantize_fp8_1x128(x: torch.Tensor, scale_mode: int = DG_SCALE_FP32,
                          q: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """Row-wise quantization (one scale per row and 128 columns) of a float32
    or bfloat16 CUDA matrix; returns (q uint8 [rows, cols], scales float32
    [rows, ceil(cols/128)])."""
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
    _cuda(x, x.dtype, "x")
    rows, cols = x.shape
    ld_x = _ld(x, "x", 8)
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, (cols + BLOCK - 1) // BLOCK), dtype=torch.float32, device=x.device)
    qb = _u8(q)
    _cuda(qb, torch.uint8, "q")
    _cuda(scales, torch.float32, "scales")
    if tuple(scales.shape) != (rows, (cols + BLOCK - 1) // BLOCK) or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous [rows, ceil(cols/128)] tensor")
    dtype = DG_INPUT_BF16 if x.dtype == torch.bfloat16 else DG_INPUT_FP32
    st = lib().dg_quantize_fp8_1x128(ctypes.c_void_p(x.data_ptr()), dtype, rows, cols, ld_x,
                                     ctypes.c_void_p(qb.data_ptr()), _ld(qb, "q", 4),
                                     ctypes.c_void_p(scales.data_ptr()), int(scale_mode), _stream(x))
    _check(st, "dg_quantize_fp8_1x128")
    return q, scales


def dg_fp8_gemm_nt(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor,
                   sb: torch.Tensor, scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """c[M, N] (bf16) = block-scaled A[M, K] . B[N, K]^T; returns c."""
    return _gemm_nt(c, a, b, sa, sb, scale_mode, False)


def dg_fp8_gemm_nt_1x128(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor,
                         sb: torch.Tensor, scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """As dg_fp8_gemm_nt with one A scale per row and K block (sa [M, K/128])."""
    return _gemm_nt(c, a, b, sa, sb, scale_mode, True)


def _gemm_nt(c, a, b, sa, sb, scale_mode, a_1x128):
    a, b = _u8(a), _u8(b)
    _cuda(c, torch.bfloat16, "c")
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k or tuple(c.shape) != (m, n):
        raise ValueError("shape mismatch between c, a and b")
    kb = k // BLOCK
    sa_rows = m if a_1x128 else (m + BLOCK - 1) // BLOCK
    if tuple(sa.shape) != (sa_rows, kb) or tuple(sb.shape) != ((n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (sa.is_contiguous() and sb.is_contiguous()):
        raise ValueError("scales must be contiguous")
    fn = lib().dg_fp8_gemm_nt_1x128 if a_1x128 else lib().dg_fp8_gemm_nt
    st = fn(ctypes.c_void_p(c.data_ptr()), _ld(c, "c", 8),
            ctypes.c_void_p(a.data_ptr()), _ld(a, "a"),
            ctypes.c_void_p(sa.data_ptr()),
            ctypes.c_void_p(b.data_ptr()), _ld(b, "b"),
            ctypes.c_void_p(sb.data_ptr()), m, n, k, int(scale_mode), _stream(c))
    _check(st, "dg_fp8_gemm_nt_1x128" if a_1x128 else "dg_fp8_gemm_nt")
    return c


def dg_fp8_grouped_gemm_contiguous(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor,
                                   sa: torch.Tensor, sb: torch.Tensor, m_indices: torch.Tensor,
                                   scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """c[M_tot, N] = A[M_tot, K] . B[g(i)]^T per row i, zero for padding rows."""
    return _grouped(c, a, b, sa, sb, m_indices, scale_mode, False)


def dg_fp8_grouped_gemm_contiguous_1x128(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor,
                                         sa: torch.Tensor, sb: torch.Tensor, m_indices: torch.Tensor,
                                         scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """As dg_fp8_grouped_gemm_contiguous with sa [M_tot, K/128] (one A scale per row and K block)."""
    return _grouped(c, a, b, sa, sb, m_indices, scale_mode, True)


def _grouped(c, a, b, sa, sb, m_indices, scale_mode, a_1x128):
    a, b = _u8(a), _u8(b)
    _cuda(c, torch.bfloat16, "c")
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    _cuda(m_indices, torch.int32, "m_indices")
    m_tot, k = a.shape
    g, n, k2 = b.shape
    if k2 != k or tuple(c.shape) != (m_tot, n) or tuple(m_indices.shape) != (m_tot,):
        raise ValueError("shape mismatch")
    kb = k // BLOCK
    sa_rows = m_tot if a_1x128 else (m_tot + BLOCK - 1) // BLOCK
    if tuple(sa.shape) != (sa_rows, kb) or tuple(sb.shape) != (g, (n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (b.is_contiguous() and sa.is_contiguous() and sb.is_contiguous() and m_indices.is_contiguous()):
        raise ValueError("b, sa, sb and m_indices must be contiguous")
    fn = lib().dg_fp8_grouped_gemm_contiguous_1x128 if a_1x128 else lib().dg_fp8_grouped_gemm_contiguous
    st = fn(
        ctypes.c_void_p(c.data_ptr()), _ld(c, "c", 8), ctypes.c_void_p(a.data_ptr()), _ld(a, "a"),
        ctypes.c_void_p(sa.data_ptr()), ctypes.c_void_p(b.data_ptr()),
        ctypes.c_void_p(sb.data_ptr()), g, ctypes.c_void_p(m_indices.data_ptr()),
        m_tot, n, k, int(scale_mode), _stream(c))
    _check(st, "dg_fp8_grouped_gemm_contiguous_1x128" if a_1x128 else "dg_fp8_grouped_gemm_contiguous")
    return c


def dg_fp8_gemm(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor, sb: torch.Tensor,
                layout="NT", scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """c[M, N] (bf16) = op(A) . op(B) with per-block scales in layout NT, TN,
    NN or TT (a dg_layout value or its name): a is [M, K] for N-A and [K, M]
    for T-A; b is [N, K] for T-B and [K, N] for N-B. sa [ceil(M/128), K/128],
    sb [ceil(N/128), K/128] whatever the layout. Returns c."""
    lay = _LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    if lay not in _LAYOUTS.values():
        raise ValueError(f"unknown layout {layout}")
    a_t = lay in (DG_LAYOUT_TN, DG_LAYOUT_TT)
    b_n = lay in (DG_LAYOUT_TN, DG_LAYOUT_NN)
    a, b = _u8(a), _u8(b)
    _cuda(c, torch.bfloat16, "c")
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    m, n = c.shape
    k = a.shape[0] if a_t else a.shape[1]
    if (a.shape[1] if a_t else a.shape[0]) != m:
        raise ValueError("a does not match c's M")
    if tuple(b.shape) != ((k, n) if b_n else (n, k)):
        raise ValueError("b does not match the layout, K or c's N")
    kb = k // BLOCK
    if tuple(sa.shape) != ((m + BLOCK - 1) // BLOCK, kb) or tuple(sb.shape) != ((n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (sa.is_contiguous() and sb.is_contiguous()):
        raise ValueError("scales must be contiguous")
    st = lib().dg_fp8_gemm(ctypes.c_void_p(c.data_ptr()), _ld(c, "c", 8), ctypes.c_void_p(a.data_ptr()),
                           _ld(a, "a"), ctypes.c_void_p(sa.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                           _ld(b, "b"), ctypes.c_void_p(sb.data_ptr()), m, n, k, lay, int(scale_mode),
                           _stream(c))
    _check(st, "dg_fp8_gemm")
    return c


def dg_fp8_gemm_requant(a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor, sb: torch.Tensor, m: int, n: int,
                        layout="NT", scale_mode: int = DG_SCALE_FP32, out_block_rows: int = 1,
                        out_scale_mode: int = DG_SCALE_FP32, a_scale_rows: int = BLOCK,
                        cq: torch.Tensor | None = None, cs: torch.Tensor | None = None):
    """op(A) . op(B) in layout NT, TN, NN or TT (as dg_fp8_gemm) with the FP32
    result requantized to E4M3 in the epilogue; returns (cq uint8 [m, n], cs).
    sa is [ceil(m/128), K/128], or [m, K/128] with a_scale_rows = 1."""
    lay = _LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    if lay not in _LAYOUTS.values():
        raise ValueError(f"unknown layout {layout}")
    a_t = lay in (DG_LAYOUT_TN, DG_LAYOUT_TT)
    b_n = lay in (DG_LAYOUT_TN, DG_LAYOUT_NN)
    a, b = _u8(a), _u8(b)
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    k = a.shape[0] if a_t else a.shape[1]
    if tuple(a.shape) != ((k, m) if a_t else (m, k)) or tuple(b.shape) != ((k, n) if b_n else (n, k)):
        raise ValueError("a or b does not match the layout, m, n and K")
    kb = k // BLOCK
    if a_scale_rows not in (1, BLOCK):
        raise ValueError("a_scale_rows must be 1 or 128")
    sa_rows = m if a_scale_rows == 1 else (m + BLOCK - 1) // BLOCK
    if tuple(sa.shape) != (sa_rows, kb) or tuple(sb.shape) != ((n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (sa.is_contiguous() and sb.is_contiguous()):
        raise ValueError("scales must be contiguous")
    cq, qb, cs = _requant_out(cq, cs, m, n, out_block_rows, a.device)
    st = lib().dg_fp8_gemm_requant(
        ctypes.c_void_p(qb.data_ptr()), _ld(qb, "cq"), ctypes.c_void_p(cs.data_ptr()), int(out_block_rows),
        int(out_scale_mode), ctypes.c_void_p(a.data_ptr()), _ld(a, "a"), ctypes.c_void_p(sa.data_ptr()),
        int(a_scale_rows), ctypes.c_void_p(b.data_ptr()), _ld(b, "b"), ctypes.c_void_p(sb.data_ptr()),
        m, n, k, lay, int(scale_mode), _stream(a))
    _check(st, "dg_fp8_gemm_requant")
    return cq, cs


def dg_fp8_k_grouped_gemm_tn(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor,
                             sb: torch.Tensor, k_sizes, scale_mode: int = DG_SCALE_FP32) -> torch.Tensor:
    """K-grouped TN GEMM: c[g] (bf16 [M, N]) = A[k range g]^T . B[k range g]
    for a [K_tot, M], b [K_tot, N], sa [ceil(M/128), K_tot/128],
    sb [ceil(N/128), K_tot/128] and host group sizes k_sizes (multiples of
    128). c is [G, M, N] with contiguous groups. Returns c."""
    sizes = [int(v) for v in k_sizes]
    arr = (ctypes.c_int64 * max(1, len(sizes)))(*sizes)
    a, b = _u8(a), _u8(b)
    _cuda(c, torch.bfloat16, "c")
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    g, m, n = c.shape
    k_tot = a.shape[0]
    if g != len(sizes) or sum(sizes) != k_tot or tuple(a.shape) != (k_tot, m) or tuple(b.shape) != (k_tot, n):
        raise ValueError("shape mismatch")
    if c.stride(2) != 1 or c.stride(0) != m * c.stride(1):
        raise ValueError("c must be [G, M, N] with unit column stride and groups M rows apart")
    kb = k_tot // BLOCK
    if tuple(sa.shape) != ((m + BLOCK - 1) // BLOCK, kb) or tuple(sb.shape) != ((n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (sa.is_contiguous() and sb.is_contiguous()):
        raise ValueError("scales must be contiguous")
    st = lib().dg_fp8_k_grouped_gemm_tn(ctypes.c_void_p(c.data_ptr()), int(c.stride(1)),
                                        ctypes.c_void_p(a.data_ptr()), _ld(a, "a"), ctypes.c_void_p(sa.data_ptr()),
                                        ctypes.c_void_p(b.data_ptr()), _ld(b, "b"), ctypes.c_void_p(sb.data_ptr()),
                                        len(sizes), arr, m, n, int(scale_mode), _stream(c))
    _check(st, "dg_fp8_k_grouped_gemm_tn")
    return c


def _requant_out(cq, cs, m, n, out_block_rows, device):
    """Output tensors of a requantizing GEMM: codes [m, n] (row stride a
    multiple of 16) and scales [m or ceil(m/128), ceil(n/128)]."""
    if out_block_rows not in (1, BLOCK):
        raise ValueError("out_block_rows must be 1 or 128")
    nbc = (n + BLOCK - 1) // BLOCK
    s_rows = m if out_block_rows == 1 else (m + BLOCK - 1) // BLOCK
    if cq is None:
        ld = max(16, (n + 15) // 16 * 16)
        cq = torch.empty((m, ld), dtype=torch.uint8, device=device)[:, :n]
    if cs is None:
        cs = torch.empty((s_rows, nbc), dtype=torch.float32, device=device)
    qb = _u8(cq)
    _cuda(qb, torch.uint8, "cq")
    _cuda(cs, torch.float32, "cs")
    if tuple(qb.shape) != (m, n):
        raise ValueError("cq shape mismatch")
    if tuple(cs.shape) != (s_rows, nbc) or not cs.is_contiguous():
        raise ValueError(f"cs must be a contiguous [{s_rows}, {nbc}] tensor")
    return cq, qb, cs


def dg_fp8_gemm_nt_requant(a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor, sb: torch.Tensor,
                           scale_mode: int = DG_SCALE_FP32, out_block_rows: int = 1,
                           out_scale_mode: int = DG_SCALE_FP32, cq: torch.Tensor | None = None,
                           cs: torch.Tensor | None = None):
    """Block-scaled A[M, K] . B[N, K]^T with the FP32 result requantized to
    E4M3 in the epilogue: returns (cq uint8 [M, N], cs float32) with one scale
    per out_block_rows x 128 block. sa is [ceil(M/128), K/128] or, for
    row-wise activation scales, [M, K/128]."""
    a, b = _u8(a), _u8(b)
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k:
        raise ValueError("shape mismatch between a and b")
    kb = k // BLOCK
    if tuple(sa.shape) == (m, kb) and m != (m + BLOCK - 1) // BLOCK:
        a_scale_rows = 1
    elif tuple(sa.shape) == ((m + BLOCK - 1) // BLOCK, kb):
        a_scale_rows = BLOCK
    else:
        raise ValueError("sa must be [ceil(M/128), K/128] or [M, K/128]")
    if tuple(sb.shape) != ((n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (sa.is_contiguous() and sb.is_contiguous()):
        raise ValueError("scales must be contiguous")
    cq, qb, cs = _requant_out(cq, cs, m, n, out_block_rows, a.device)
    st = lib().dg_fp8_gemm_nt_requant(
        ctypes.c_void_p(qb.data_ptr()), _ld(qb, "cq"), ctypes.c_void_p(cs.data_ptr()), int(out_block_rows),
        int(out_scale_mode), ctypes.c_void_p(a.data_ptr()), _ld(a, "a"), ctypes.c_void_p(sa.data_ptr()),
        a_scale_rows, ctypes.c_void_p(b.data_ptr()), _ld(b, "b"), ctypes.c_void_p(sb.data_ptr()),
        m, n, k, int(scale_mode), _stream(a))
    _check(st, "dg_fp8_gemm_nt_requant")
    return cq, cs


def dg_fp8_grouped_gemm_contiguous_requant(a: torch.Tensor, b: torch.Tensor, sa: torch.Tensor,
                                           sb: torch.Tensor, m_indices: torch.Tensor,
                                           scale_mode: int = DG_SCALE_FP32, out_block_rows: int = 1,
                                           out_scale_mode: int = DG_SCALE_FP32,
                                           cq: torch.Tensor | None = None, cs: torch.Tensor | None = None):
    """The M-grouped contiguous GEMM with its output requantized to E4M3
    (padding rows: codes 0); returns (cq, cs) as dg_fp8_gemm_nt_requant."""
    a, b = _u8(a), _u8(b)
    _cuda(a, torch.uint8, "a")
    _cuda(b, torch.uint8, "b")
    _cuda(sa, torch.float32, "sa")
    _cuda(sb, torch.float32, "sb")
    _cuda(m_indices, torch.int32, "m_indices")
    m_tot, k = a.shape
    g, n, k2 = b.shape
    if k2 != k or tuple(m_indices.shape) != (m_tot,):
        raise ValueError("shape mismatch")
    kb = k // BLOCK
    if tuple(sa.shape) == (m_tot, kb) and m_tot != (m_tot + BLOCK - 1) // BLOCK:
        a_scale_rows = 1
    elif tuple(sa.shape) == ((m_tot + BLOCK - 1) // BLOCK, kb):
        a_scale_rows = BLOCK
    else:
        raise ValueError("sa must be [M_tot/128, K/128] or [M_tot, K/128]")
    if tuple(sb.shape) != (g, (n + BLOCK - 1) // BLOCK, kb):
        raise ValueError("scale shape mismatch")
    if not (b.is_contiguous() and sa.is_contiguous() and sb.is_contiguous() and m_indices.is_contiguous()):
        raise ValueError("b, sa, sb and m_indices must be contiguous")
    cq, qb, cs = _requant_out(cq, cs, m_tot, n, out_block_rows, a.device)
    st = lib().dg_fp8_grouped_gemm_contiguous_requant(
        ctypes.c_void_p(qb.data_ptr()), _ld(qb, "cq"), ctypes.c_void_p(cs.data_ptr()), int(out_block_rows),
        int(out_scale_mode), ctypes.c_void_p(a.data_ptr()), _ld(a, "a"), ctypes.c_void_p(sa.data_ptr()),
        a_scale_rows, ctypes.c_void_p(b.data_ptr()), ctypes.c_void_p(sb.data_ptr()), g,
        ctypes.c_void_p(m_indices.data_ptr()), m_tot, n, k, int(scale_mode), _stream(a))
    _check(st, "dg_fp8_grouped_gemm_contiguous_requant")
    return cq, cs


def dg_get_device_status(device=None) -> int:
    """Synchronize the current stream and return (and clear) the device status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    return int(lib().dg_get_device_status(s))


def dg_selftest_wait_timeout(limit_ns: int, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _check(lib().dg_selftest_wait_timeout(int(limit_ns), s), "dg_selftest_wait_timeout")
