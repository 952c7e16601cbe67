"""CPU oracle for FP8 E4M3 128x128 block quantization and the block-scaled NT GEMM.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import this package. The product
path (``block_quantize_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``dgfp8_oracle.c`` (plain C, FP64 accumulation, IEEE
FP32 division, no fast-math); this module compiles it with gcc and wraps it for
numpy arrays. Every function cites the page section it follows:

* lpnh.cn DeepGEMM walkthrough (untitled), §3.1 and §4.2: scale = block
  max|x| / 448 in FP32, divide, round to nearest-even E4M3; §5.4 all-zero block.
* pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析", §3.1: NT layout, FP32 or
  power-of-two (UE8M0) scales; §2.3/§3.2: M-grouped GEMM for MoE experts.
* pzsr.cn page §3.1 (all four layouts NT, TN, NN, TT from SM100 on) and §3.2
  (grouping along K): ``gemm_layout`` and ``k_grouped_gemm_tn``.
* lpnh.cn walkthrough §2.2 (accumulate in FP32, quantize on demand at
  write-back) and §6 (fuse the scale computation into the kernel): the
  requantized GEMM output, ``requantize_output`` / ``gemm_nt_requant``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgfp8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128
SCALE_FP32 = 0
SCALE_UE8M0 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, IEEE arithmetic) if stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, f32p, u8p, f64p, i64p = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p)
        lib.oracle_e4m3_table.argtypes = [f64p]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_array.argtypes = [f32p, i64, u8p]
        lib.oracle_pow2_ceil.argtypes = [ctypes.c_float]
        lib.oracle_pow2_ceil.restype = ctypes.c_float
        lib.oracle_quantize.argtypes = [f32p, i64, i64, i64, ctypes.c_int, u8p, i64, f32p]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_quantize_1x128.argtypes = [f32p, i64, i64, i64, ctypes.c_int, u8p, i64, f32p]
        lib.oracle_quantize_1x128.restype = ctypes.c_int
        lib.oracle_gemm_nt_rows_a1x128.argtypes = [u8p, i64, f32p, u8p, i64, f32p,
                                                   i64, i64, i64, i64p, i64, f64p, f64p]
        lib.oracle_grouped_gemm_rows_a1x128.argtypes = [u8p, i64, f32p, u8p, f32p, i64,
                                                        ctypes.c_void_p, i64, i64, i64,
                                                        i64p, i64, f64p, f64p]
        lib.oracle_grouped_gemm_rows_a1x128.restype = ctypes.c_int
        lib.oracle_gemm_nt_rows.argtypes = [u8p, i64, f32p, u8p, i64, f32p,
                                            i64, i64, i64, i64p, i64, f64p, f64p]
        lib.oracle_grouped_gemm_rows.argtypes = [u8p, i64, f32p, u8p, f32p, i64,
                                                 ctypes.c_void_p, i64, i64, i64,
                                                 i64p, i64, f64p, f64p]
        lib.oracle_grouped_gemm_rows.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def e4m3_table() -> np.ndarray:
    """The 256 E4M3 code values as float64 (NaN for 0x7F and 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    """Nearest E4M3 code (ties to even, saturating to +-448) of float32 values."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def pow2_ceil(s: float) -> float:
    """Smallest power of two >= s, clamped to >= 2^-127 (UE8M0 scale)."""
    return float(_load().oracle_pow2_ceil(ctypes.c_float(s)))


def quantize(x: np.ndarray, mode: int = SCALE_FP32):
    """128x128 block quantization of a float32 matrix.

    Returns (q uint8 [rows, cols], scales float32 [ceil(rows/128), ceil(cols/128)]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(((rows + BLOCK - 1) // BLOCK, (cols + BLOCK - 1) // BLOCK), dtype=np.float32)
    rc = _load().oracle_quantize(_ptr(x), rows, cols, cols, int(mode), _ptr(q), cols, _ptr(s))
    if rc != 0:
        raise ValueError("oracle.quantize: input holds a non-finite value")
    return q, s


def quantize_1x128(x: np.ndarray, mode: int = SCALE_FP32):
    """Row-wise 1x128 quantization of a float32 matrix (one scale per row and
    128-column block).

    Returns (q uint8 [rows, cols], scales float32 [rows, ceil(cols/128)]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty((rows, (cols + BLOCK - 1) // BLOCK), dtype=np.float32)
    rc = _load().oracle_quantize_1x128(_ptr(x), rows, cols, cols, int(mode), _ptr(q), cols, _ptr(s))
    if rc != 0:
        raise ValueError("oracle.quantize_1x128: input holds a non-finite value")
    return q, s


def _rows_arg(rows, m):
    if rows is None:
        rows = np.arange(m, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= m):
        raise IndexError("row index out of range")
    return rows


def gemm_nt(qa, sa, qb, sb, rows=None, want_e: bool = True, a_1x128: bool = False):
    """Block-scaled NT GEMM in float64: C[r, j] for i = rows[r] and all j.

    qa uint8 [M, K], sa float32 [ceil(M/128), K/128] (or [M, K/128] with
    a_1x128: one A scale per row and K block), qb uint8 [N, K],
    sb float32 [ceil(N/128), K/128]. Returns (C, E) (E None if not wanted).
    """
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    m, k = qa.shape
    n, k2 = qb.shape
    if k != k2 or k % BLOCK:
        raise ValueError("K mismatch or not a multiple of 128")
    sa_rows = m if a_1x128 else (m + BLOCK - 1) // BLOCK
    if sa.shape != (sa_rows, k // BLOCK) or sb.shape != ((n + BLOCK - 1) // BLOCK, k // BLOCK):
        raise ValueError("scale shape mismatch")
    rows = _rows_arg(rows, m)
    c = np.empty((rows.size, n), dtype=np.float64)
    e = np.empty((rows.size, n), dtype=np.float64) if want_e else None
    fn = _load().oracle_gemm_nt_rows_a1x128 if a_1x128 else _load().oracle_gemm_nt_rows
    fn(_ptr(qa), k, _ptr(sa), _ptr(qb), k, _ptr(sb), m, n, k, _ptr(rows), rows.size, _ptr(c),
       _ptr(e) if want_e else None)
    return c, e


def grouped_gemm_contiguous(qa, sa, qb, sb, m_indices, rows=None, want_e: bool = True,
                            a_1x128: bool = False):
    """M-grouped contiguous GEMM in float64 (rows with index -1 are zero).

    qa uint8 [M_tot, K], sa float32 [M_tot/128, K/128] (or [M_tot, K/128] with
    a_1x128), qb uint8 [G, N, K], sb float32 [G, ceil(N/128), K/128],
    m_indices int32 [M_tot].
    """
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    mi = np.ascontiguousarray(m_indices, dtype=np.int32)
    m_tot, k = qa.shape
    g, n, k2 = qb.shape
    if k != k2 or k % BLOCK or mi.shape != (m_tot,):
        raise ValueError("shape mismatch")
    if sb.shape != (g, (n + BLOCK - 1) // BLOCK, k // BLOCK):
        raise ValueError("sb shape mismatch")
    if sa.shape != ((m_tot if a_1x128 else m_tot // BLOCK), k // BLOCK):
        raise ValueError("sa shape mismatch")
    rows = _rows_arg(rows, m_tot)
    c = np.empty((rows.size, n), dtype=np.float64)
    e = np.empty((rows.size, n), dtype=np.float64) if want_e else None
    fn = _load().oracle_grouped_gemm_rows_a1x128 if a_1x128 else _load().oracle_grouped_gemm_rows
    rc = fn(_ptr(qa), k, _ptr(sa), _ptr(qb), _ptr(sb), g, _ptr(mi), m_tot, n, k, _ptr(rows), rows.size,
            _ptr(c), _ptr(e) if want_e else None)
    if rc != 0:
        raise ValueError("m_indices holds an expert id >= G")
    return c, e


def dequantize(q, s) -> np.ndarray:
    """float64 values dec(q) * s for each 128x128 block (a test helper)."""
    t = e4m3_table()
    q = np.asarray(q, dtype=np.uint8)
    vals = t[q]
    rows, cols = q.shape
    expand = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), BLOCK, axis=0), BLOCK, axis=1)
    return vals * expand[:rows, :cols]


def dequantize_1x128(q, s) -> np.ndarray:
    """float64 values dec(q) * s with one scale per row and 128 columns (a test helper)."""
    t = e4m3_table()
    q = np.asarray(q, dtype=np.uint8)
    expand = np.repeat(np.asarray(s, dtype=np.float64), BLOCK, axis=1)
    return t[q] * expand[:, :q.shape[1]]


def requantize_output(c, out_block_rows: int = 1, mode: int = SCALE_FP32):
    """The GEMM result requantized at write-back (walkthrough §2.2: the product
    is accumulated in FP32 and quantized on demand when written back; §6: the
    scale computation fused into the kernel). The value quantized is the FP32
    accumulator: the float64 result c rounded once to FP32. The steps are those
    of §4.2 with blocks of out_block_rows x 128 (1: per-row activation scales,
    pzsr.cn page §3.1; 128: the 128 x 128 blocks of §4.2).

    Returns (q uint8, scales float32 [rows or ceil(rows/128), ceil(cols/128)]).
    """
    v = np.asarray(c, dtype=np.float64).astype(np.float32)
    if out_block_rows == 1:
        return quantize_1x128(v, mode)
    if out_block_rows == BLOCK:
        return quantize(v, mode)
    raise ValueError("out_block_rows must be 1 or 128")


def gemm_nt_requant(qa, sa, qb, sb, out_block_rows: int = 1, mode: int = SCALE_FP32, rows=None,
                    a_1x128: bool = False):
    """gemm_nt followed by requantize_output on the selected rows (for
    out_block_rows = 128 the rows must be whole 128-row blocks in order, a
    short last block only at the end). Returns (q, scales, C, E)."""
    c, e = gemm_nt(qa, sa, qb, sb, rows=rows, a_1x128=a_1x128)
    q, s = requantize_output(c, out_block_rows, mode)
    return q, s, c, e


def grouped_gemm_requant(qa, sa, qb, sb, m_indices, out_block_rows: int = 1, mode: int = SCALE_FP32,
                         rows=None, a_1x128: bool = False):
    """grouped_gemm_contiguous followed by requantize_output (padding rows are
    zeros, so their codes are 0). Returns (q, scales, C, E)."""
    c, e = grouped_gemm_contiguous(qa, sa, qb, sb, m_indices, rows=rows, a_1x128=a_1x128)
    q, s = requantize_output(c, out_block_rows, mode)
    return q, s, c, e


LAYOUTS = ("NT", "TN", "NN", "TT")


def gemm_layout(qa, sa, qb, sb, layout: str, rows=None):
    """The block-scaled GEMM C = op(A) . op(B) in one of the layouts of
    pzsr.cn page §3.1, named op(A) op(B): A is stored [M, K] for "N" and
    [K, M] for "T" as first letter; B is stored [N, K] for "T" and [K, N] for
    "N" as second letter (NT is gemm_nt). Scales are per 128 x 128 block of
    the logical operands: sa [ceil(M/128), K/128], sb [ceil(N/128), K/128].
    By definition this is gemm_nt on the operands brought to [M, K] and
    [N, K]. Returns (C, E)."""
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout}")
    a_nk = np.asarray(qa).T if layout[0] == "T" else np.asarray(qa)
    b_nk = np.asarray(qb).T if layout[1] == "N" else np.asarray(qb)
    return gemm_nt(np.ascontiguousarray(a_nk), sa, np.ascontiguousarray(b_nk), sb, rows=rows)


def k_grouped_gemm_tn(qa, sa, qb, sb, k_sizes, rows=None):
    """K-grouped GEMM (pzsr.cn page §3.2, grouping along K): with A stored
    [K_tot, M] and B [K_tot, N], group g owns the K range of its size and gets
    C_g = A[range]^T . B[range] with those K blocks' scales (sa [ceil(M/128),
    K_tot/128], sb [ceil(N/128), K_tot/128]); sizes are multiples of 128 and a
    group of size 0 gives zeros. Returns (C [G, rows, N], E)."""
    qa = np.asarray(qa)
    qb = np.asarray(qb)
    k_tot, m = qa.shape
    n = qb.shape[1]
    sizes = [int(v) for v in k_sizes]
    if sum(sizes) != k_tot or any(v < 0 or v % BLOCK for v in sizes):
        raise ValueError("group sizes must be multiples of 128 summing to K_tot")
    nr = m if rows is None else len(rows)
    cs = np.zeros((len(sizes), nr, n))
    es = np.zeros((len(sizes), nr, n))
    off = 0
    for g, kg in enumerate(sizes):
        if kg:
            kb0, kb1 = off // BLOCK, (off + kg) // BLOCK
            c, e = gemm_nt(np.ascontiguousarray(qa[off:off + kg].T), np.ascontiguousarray(sa[:, kb0:kb1]),
                           np.ascontiguousarray(qb[off:off + kg].T), np.ascontiguousarray(sb[:, kb0:kb1]),
                           rows=rows)
            cs[g], es[g] = c, e
        off += kg
    return cs, es
