"""CPU checks of the C-ABI library: it loads, exports every entry point that
include/dgfp8.h declares, and rejects bad arguments before touching CUDA (so
these run without a GPU). Calls with valid arguments on a machine without a GPU
return DG_ERR_NO_DEVICE and launch nothing."""
import ctypes

import pytest
import torch

import block_quantize_gb300 as bq
from block_quantize_gb300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return bq.lib()


def test_every_declared_symbol_is_exported(L):
    names = bq.declared_functions()
    assert {"dg_quantize_fp8_block", "dg_fp8_gemm_nt", "dg_fp8_grouped_gemm_contiguous"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_version_strings_alignment(L):
    assert bq.dg_get_abi_version() == 6
    assert bq.dg_get_mk_alignment_for_contiguous_layout() == 128
    for s in range(8):
        assert bq.dg_status_string(s)
    assert bq.dg_status_string(99) == "unknown status"
    assert "expert id" in bq.dg_status_string(bq.DG_ERR_BAD_GROUP)


def test_num_sms_knob(L):
    assert bq.dg_get_num_sms() == 0
    bq.dg_set_num_sms(64)
    assert bq.dg_get_num_sms() == 64
    with pytest.raises(bq.DgError):
        bq.dg_set_num_sms(-1)
    bq.dg_set_num_sms(0)


P = 1 << 20        # fake, 1 MiB-aligned device addresses: never dereferenced
NULL = None


def gemm(L, c=P, ldc=256, a=P, lda=512, sa=P, b=P, ldb=512, sb=P, m=128, n=256, k=512, mode=0):
    return L.dg_fp8_gemm_nt(c, ldc, a, lda, sa, b, ldb, sb, m, n, k, mode, None)


def grouped(L, c=P, ldc=256, a=P, lda=512, sa=P, b=P, sb=P, g=2, mi=P, m=256, n=256, k=512, mode=0):
    return L.dg_fp8_grouped_gemm_contiguous(c, ldc, a, lda, sa, b, sb, g, mi, m, n, k, mode, None)


def quant(L, x=P, rows=128, cols=128, ldx=128, q=P, ldq=128, s=P, mode=0):
    return L.dg_quantize_fp8_block(x, rows, cols, ldx, q, ldq, s, mode, None)


def quant_rows(L, x=P, dtype=0, rows=128, cols=128, ldx=128, q=P, ldq=128, s=P, mode=0):
    return L.dg_quantize_fp8_1x128(x, dtype, rows, cols, ldx, q, ldq, s, mode, None)


def gemm_rows(L, **kw):
    a = dict(c=P, ldc=256, a=P, lda=512, sa=P, b=P, ldb=512, sb=P, m=128, n=256, k=512, mode=0)
    a.update(kw)
    return L.dg_fp8_gemm_nt_1x128(a["c"], a["ldc"], a["a"], a["lda"], a["sa"], a["b"], a["ldb"], a["sb"],
                                  a["m"], a["n"], a["k"], a["mode"], None)


def grouped_rows(L, **kw):
    a = dict(c=P, ldc=256, a=P, lda=512, sa=P, b=P, sb=P, g=2, mi=P, m=256, n=256, k=512, mode=0)
    a.update(kw)
    return L.dg_fp8_grouped_gemm_contiguous_1x128(a["c"], a["ldc"], a["a"], a["lda"], a["sa"], a["b"],
                                                  a["sb"], a["g"], a["mi"], a["m"], a["n"], a["k"],
                                                  a["mode"], None)


def gemm_rq(L, **kw):
    a = dict(q=P, ldq=256, s=P, br=1, omode=0, a=P, lda=512, sa=P, arows=128, b=P, ldb=512, sb=P,
             m=128, n=256, k=512, mode=0)
    a.update(kw)
    return L.dg_fp8_gemm_nt_requant(a["q"], a["ldq"], a["s"], a["br"], a["omode"], a["a"], a["lda"], a["sa"],
                                    a["arows"], a["b"], a["ldb"], a["sb"], a["m"], a["n"], a["k"], a["mode"],
                                    None)


def grouped_rq(L, **kw):
    a = dict(q=P, ldq=256, s=P, br=1, omode=0, a=P, lda=512, sa=P, arows=128, b=P, sb=P, g=2, mi=P,
             m=256, n=256, k=512, mode=0)
    a.update(kw)
    return L.dg_fp8_grouped_gemm_contiguous_requant(a["q"], a["ldq"], a["s"], a["br"], a["omode"], a["a"],
                                                    a["lda"], a["sa"], a["arows"], a["b"], a["sb"], a["g"],
                                                    a["mi"], a["m"], a["n"], a["k"], a["mode"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(c=NULL), bq.DG_ERR_INVALID_ARG), (dict(a=NULL), bq.DG_ERR_INVALID_ARG),
    (dict(sb=NULL), bq.DG_ERR_INVALID_ARG), (dict(m=-1), bq.DG_ERR_INVALID_ARG),
    (dict(mode=7), bq.DG_ERR_INVALID_ARG), (dict(lda=256), bq.DG_ERR_INVALID_ARG),
    (dict(ldc=100), bq.DG_ERR_INVALID_ARG),
    (dict(k=500, lda=512, ldb=512), bq.DG_ERR_UNSUPPORTED_SHAPE),
    (dict(m=1 << 31), bq.DG_ERR_UNSUPPORTED_SHAPE),
    (dict(a=P + 8), bq.DG_ERR_MISALIGNED), (dict(c=P + 2), bq.DG_ERR_MISALIGNED),
    (dict(lda=520), bq.DG_ERR_MISALIGNED), (dict(ldc=260), bq.DG_ERR_MISALIGNED),
    (dict(m=0), bq.DG_OK), (dict(n=0), bq.DG_OK),
])
def test_gemm_argument_errors(L, kw, status):
    assert gemm(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(mi=NULL), bq.DG_ERR_INVALID_ARG), (dict(g=0), bq.DG_ERR_INVALID_ARG),
    (dict(m=200), bq.DG_ERR_UNSUPPORTED_SHAPE), (dict(mi=P + 4), bq.DG_ERR_MISALIGNED),
    (dict(k=384 + 64), bq.DG_ERR_UNSUPPORTED_SHAPE), (dict(m=0), bq.DG_OK),
])
def test_grouped_argument_errors(L, kw, status):
    assert grouped(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(x=NULL), bq.DG_ERR_INVALID_ARG), (dict(s=NULL), bq.DG_ERR_INVALID_ARG),
    (dict(rows=-1), bq.DG_ERR_INVALID_ARG), (dict(ldx=100), bq.DG_ERR_INVALID_ARG),
    (dict(ldq=100), bq.DG_ERR_INVALID_ARG), (dict(mode=2), bq.DG_ERR_INVALID_ARG),
    (dict(x=P + 2), bq.DG_ERR_MISALIGNED), (dict(rows=0), bq.DG_OK), (dict(cols=0), bq.DG_OK),
])
def test_quantize_argument_errors(L, kw, status):
    assert quant(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(x=NULL), bq.DG_ERR_INVALID_ARG), (dict(q=NULL), bq.DG_ERR_INVALID_ARG),
    (dict(dtype=2), bq.DG_ERR_INVALID_ARG), (dict(mode=3), bq.DG_ERR_INVALID_ARG),
    (dict(cols=-5), bq.DG_ERR_INVALID_ARG), (dict(ldx=64), bq.DG_ERR_INVALID_ARG),
    (dict(x=P + 2), bq.DG_ERR_MISALIGNED), (dict(x=P + 1, dtype=1), bq.DG_ERR_MISALIGNED),
    (dict(s=P + 2), bq.DG_ERR_MISALIGNED), (dict(rows=0), bq.DG_OK), (dict(cols=0, x=NULL), bq.DG_OK),
])
def test_rowwise_quantize_argument_errors(L, kw, status):
    assert quant_rows(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(sa=NULL), bq.DG_ERR_INVALID_ARG), (dict(mode=5), bq.DG_ERR_INVALID_ARG),
    (dict(k=500), bq.DG_ERR_UNSUPPORTED_SHAPE), (dict(a=P + 8), bq.DG_ERR_MISALIGNED),
    (dict(m=0), bq.DG_OK),
])
def test_rowwise_gemm_argument_errors(L, kw, status):
    assert gemm_rows(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(sa=NULL), bq.DG_ERR_INVALID_ARG), (dict(mi=NULL), bq.DG_ERR_INVALID_ARG),
    (dict(m=200), bq.DG_ERR_UNSUPPORTED_SHAPE), (dict(mi=P + 4), bq.DG_ERR_MISALIGNED),
    (dict(m=0), bq.DG_OK),
])
def test_rowwise_grouped_argument_errors(L, kw, status):
    assert grouped_rows(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(q=NULL), bq.DG_ERR_INVALID_ARG), (dict(s=NULL), bq.DG_ERR_INVALID_ARG),
    (dict(br=64), bq.DG_ERR_INVALID_ARG), (dict(br=0), bq.DG_ERR_INVALID_ARG),
    (dict(omode=2), bq.DG_ERR_INVALID_ARG), (dict(arows=2), bq.DG_ERR_INVALID_ARG),
    (dict(ldq=192), bq.DG_ERR_INVALID_ARG), (dict(mode=3), bq.DG_ERR_INVALID_ARG),
    (dict(ldq=264), bq.DG_ERR_MISALIGNED), (dict(q=P + 8), bq.DG_ERR_MISALIGNED),
    (dict(s=P + 2), bq.DG_ERR_MISALIGNED), (dict(k=500), bq.DG_ERR_UNSUPPORTED_SHAPE),
    (dict(m=0), bq.DG_OK), (dict(n=0, q=NULL, s=NULL), bq.DG_OK), (dict(m=0, br=3), bq.DG_ERR_INVALID_ARG),
])
def test_requant_gemm_argument_errors(L, kw, status):
    assert gemm_rq(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(mi=NULL), bq.DG_ERR_INVALID_ARG), (dict(br=2), bq.DG_ERR_INVALID_ARG),
    (dict(m=200), bq.DG_ERR_UNSUPPORTED_SHAPE), (dict(ldq=64), bq.DG_ERR_INVALID_ARG),
    (dict(ldq=264), bq.DG_ERR_MISALIGNED), (dict(m=0), bq.DG_OK),
])
def test_requant_grouped_argument_errors(L, kw, status):
    assert grouped_rq(L, **kw) == status


def gemm_lay(L, **kw):
    a = dict(c=P, ldc=256, a=P, lda=512, sa=P, b=P, ldb=512, sb=P, m=128, n=256, k=512, layout=0, mode=0)
    a.update(kw)
    return L.dg_fp8_gemm(a["c"], a["ldc"], a["a"], a["lda"], a["sa"], a["b"], a["ldb"], a["sb"], a["m"], a["n"],
                         a["k"], a["layout"], a["mode"], None)


def rq_lay(L, **kw):
    a = dict(q=P, ldq=256, s=P, br=1, omode=0, a=P, lda=512, sa=P, arows=128, b=P, ldb=512, sb=P,
             m=128, n=256, k=512, layout=0, mode=0)
    a.update(kw)
    return L.dg_fp8_gemm_requant(a["q"], a["ldq"], a["s"], a["br"], a["omode"], a["a"], a["lda"], a["sa"],
                                 a["arows"], a["b"], a["ldb"], a["sb"], a["m"], a["n"], a["k"], a["layout"],
                                 a["mode"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(layout=5), bq.DG_ERR_INVALID_ARG), (dict(br=7), bq.DG_ERR_INVALID_ARG),
    (dict(layout=1, lda=112), bq.DG_ERR_INVALID_ARG), (dict(layout=2, ldb=240), bq.DG_ERR_INVALID_ARG),
    (dict(layout=3, ldq=264), bq.DG_ERR_MISALIGNED), (dict(layout=1, m=0), bq.DG_OK),
])
def test_requant_layout_argument_errors(L, kw, status):
    assert rq_lay(L, **kw) == status


def kgrouped(L, sizes=(256, 128), **kw):
    a = dict(c=P, ldc=256, a=P, lda=128, sa=P, b=P, ldb=256, sb=P, m=128, n=256, mode=0)
    a.update(kw)
    arr = (ctypes.c_int64 * len(sizes))(*sizes) if sizes is not None else None
    return L.dg_fp8_k_grouped_gemm_tn(a["c"], a["ldc"], a["a"], a["lda"], a["sa"], a["b"], a["ldb"], a["sb"],
                                      len(sizes) if sizes is not None else 1, arr, a["m"], a["n"], a["mode"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(layout=4), bq.DG_ERR_INVALID_ARG), (dict(layout=-1), bq.DG_ERR_INVALID_ARG),
    # TN: a is [K][ld_a >= M], b is [K][ld_b >= N]
    (dict(layout=1, lda=64), bq.DG_ERR_INVALID_ARG), (dict(layout=1, lda=128, ldb=128), bq.DG_ERR_INVALID_ARG),
    # NN: b is [K][ld_b >= N]; TT: a is [K][ld_a >= M]
    (dict(layout=2, ldb=240), bq.DG_ERR_INVALID_ARG), (dict(layout=3, lda=112, ldb=512), bq.DG_ERR_INVALID_ARG),
    (dict(layout=1, lda=136, ldb=256), bq.DG_ERR_MISALIGNED), (dict(layout=2, k=500), bq.DG_ERR_UNSUPPORTED_SHAPE),
    (dict(layout=3, m=0), bq.DG_OK),
])
def test_layout_gemm_argument_errors(L, kw, status):
    assert gemm_lay(L, **kw) == status


@pytest.mark.parametrize("sizes,kw,status", [
    ((256, 100), {}, bq.DG_ERR_UNSUPPORTED_SHAPE), ((256, -128), {}, bq.DG_ERR_INVALID_ARG),
    (None, {}, bq.DG_ERR_INVALID_ARG), ((256,), dict(lda=64), bq.DG_ERR_INVALID_ARG),
    ((256,), dict(ldb=128), bq.DG_ERR_INVALID_ARG), ((256,), dict(a=P + 8), bq.DG_ERR_MISALIGNED),
    ((256,), dict(m=0), bq.DG_OK),
])
def test_k_grouped_argument_errors(L, sizes, kw, status):
    assert kgrouped(L, sizes, **kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_arguments_without_gpu_report_no_device(L):
    assert gemm(L) == bq.DG_ERR_NO_DEVICE
    assert grouped(L) == bq.DG_ERR_NO_DEVICE
    assert quant(L) == bq.DG_ERR_NO_DEVICE
    assert quant_rows(L) == bq.DG_ERR_NO_DEVICE
    assert quant_rows(L, dtype=1) == bq.DG_ERR_NO_DEVICE
    assert gemm_rows(L) == bq.DG_ERR_NO_DEVICE
    assert grouped_rows(L) == bq.DG_ERR_NO_DEVICE
    assert gemm_rq(L) == bq.DG_ERR_NO_DEVICE
    assert gemm_rq(L, br=128, omode=1, arows=1) == bq.DG_ERR_NO_DEVICE
    assert grouped_rq(L) == bq.DG_ERR_NO_DEVICE
    for layout in range(4):
        assert gemm_lay(L, layout=layout) == bq.DG_ERR_NO_DEVICE
    assert kgrouped(L) == bq.DG_ERR_NO_DEVICE
    for layout in range(4):
        assert rq_lay(L, layout=layout) == bq.DG_ERR_NO_DEVICE
    assert L.dg_selftest_wait_timeout(1000, None) == bq.DG_ERR_NO_DEVICE


def test_python_binding_rejects_cpu_tensors(L):
    x = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        bq.dg_quantize_fp8_block(x)
