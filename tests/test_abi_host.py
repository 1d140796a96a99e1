"""Host-only checks of the C ABI (no GPU, no compute call): the library
builds and loads, exports every function include/wst.h declares, and rejects
invalid arguments with the documented status before touching the GPU."""
import ctypes
import os
import re

import pytest

import warp_specialized_tensor_gb300 as wst

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return wst.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "wst.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wst_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), "libwst.so does not export %s" % n


def test_status_strings_and_version(lib):
    for code in range(7):
        s = wst.wst_status_string(code)
        assert s.startswith("WST_")
    assert "sm_103a" in wst.wst_version()


def test_workspace_sizes(lib):
    assert wst.wst_workspace_size(0, 0, 0) == 256
    # header + 64 flags padded to 256 B + 64*32*128 fp32 partials
    assert wst.wst_workspace_size(64, 32, 128) == 256 + 256 + 64 * 32 * 128 * 4
    assert wst.wst_workspace_size(65, 32, 128) == 256 + 512 + 65 * 32 * 128 * 4


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def gemm(lib, **kw):
    a = dict(batch=1, M=128, N=128, K=64, A=FAKE, lda=64, sA=0, B=FAKE, ldb=64, sB=0,
             bias=None, sBias=0, C=FAKE, ldc=128, sC=0, ct=1, epi=0, ws=FAKE, st=None)
    a.update(kw)
    return lib.wst_gemm_bf16(a["batch"], a["M"], a["N"], a["K"], a["A"], a["lda"], a["sA"],
                             a["B"], a["ldb"], a["sB"], a["bias"], a["sBias"], a["C"], a["ldc"],
                             a["sC"], a["ct"], a["epi"], a["ws"], a["st"])


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), wst.WST_ERR_INVALID_ARG),
    (dict(K=-1), wst.WST_ERR_INVALID_ARG),
    (dict(batch=0), wst.WST_ERR_INVALID_ARG),
    (dict(A=None), wst.WST_ERR_INVALID_ARG),
    (dict(ws=None), wst.WST_ERR_INVALID_ARG),
    (dict(lda=32), wst.WST_ERR_INVALID_ARG),
    (dict(epi=7), wst.WST_ERR_INVALID_ARG),
    (dict(epi=4), wst.WST_ERR_INVALID_ARG),
    (dict(ct=5), wst.WST_ERR_INVALID_ARG),
    (dict(epi=1), wst.WST_ERR_INVALID_ARG),            # bias missing
    (dict(A=FAKE + 8), wst.WST_ERR_ALIGNMENT),
    (dict(lda=68), wst.WST_ERR_ALIGNMENT),             # 136 B rows
    (dict(N=100, ldc=100), wst.WST_ERR_ALIGNMENT),     # 200 B rows of bf16
    (dict(batch=2, sC=10), wst.WST_ERR_INVALID_ARG),   # overlapping outputs
    (dict(), wst.WST_ERR_INVALID_ARG),                 # not device memory (no GPU here)
])
def test_gemm_rejects(lib, kw, code):
    assert gemm(lib, **kw) == code
    assert lib.wst_last_error().decode() != ""


def test_grouped_and_ikbo_reject(lib):
    g = lib.wst_grouped_gemm_bf16
    assert g(0, 10, 128, 64, FAKE, 64, FAKE, 64, 0, FAKE, None, 0, FAKE, 128, 1, 0, FAKE, None) == wst.WST_ERR_INVALID_ARG
    assert g(2, 10, 128, 64, FAKE, 64, FAKE, 64, 0, FAKE + 2, None, 0, FAKE, 128, 1, 0, FAKE, None) == wst.WST_ERR_ALIGNMENT
    assert g(2, 10, 128, 64, FAKE, 64, FAKE, 64, 0, None, None, 0, FAKE, 128, 1, 0, FAKE, None) == wst.WST_ERR_INVALID_ARG
    k = lib.wst_ikbo_linear_compress
    args = [64, 8192, 256, 64, 128, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None]
    bad = list(args); bad[4] = 96      # D != 128
    assert k(*bad) == wst.WST_ERR_UNSUPPORTED
    bad = list(args); bad[5] = 48      # O not a multiple of 32
    assert k(*bad) == wst.WST_ERR_UNSUPPORTED
    bad = list(args); bad[2] = 250     # Du not a multiple of 8
    assert k(*bad) == wst.WST_ERR_UNSUPPORTED
    bad = list(args); bad[0] = 0
    assert k(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[6] = FAKE + 4
    assert k(*bad) == wst.WST_ERR_ALIGNMENT


def test_ikbo_attention_rejects(lib):
    a = lib.wst_ikbo_attention_bf16
    #       users cand Lq H  Dh   Lkv  Q     K     V     off   scale O     type ws    bytes  stream
    args = [32, 8192, 2, 4, 128, 2048, FAKE, FAKE, FAKE, FAKE, 0.088, FAKE, 1, FAKE, 1 << 24, None]
    bad = list(args); bad[4] = 64            # Dh != 128
    assert a(*bad) == wst.WST_ERR_UNSUPPORTED
    bad = list(args); bad[5] = 0             # empty context
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[2] = 0             # no query rows per candidate
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[10] = float("nan")
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[10] = float("inf")
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[12] = 7            # unknown output type
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[1] = 1 << 30; bad[2] = 4   # 2^32 query rows
    assert a(*bad) == wst.WST_ERR_UNSUPPORTED
    bad = list(args); bad[7] = FAKE + 8      # K not 16-byte aligned
    assert a(*bad) == wst.WST_ERR_ALIGNMENT
    bad = list(args); bad[9] = FAKE + 2      # offsets not 4-byte aligned
    assert a(*bad) == wst.WST_ERR_ALIGNMENT
    bad = list(args); bad[11] = None
    assert a(*bad) == wst.WST_ERR_INVALID_ARG
    bad = list(args); bad[14] = 255          # smaller than the error-word header
    assert a(*bad) == wst.WST_ERR_INVALID_ARG


def test_attention_workspace_size(lib):
    # header + 256 CTAs x 4 flags + 256 slots of O [128][128] fp32, m, l
    assert wst.wst_ikbo_attention_workspace_size() == 256 + 256 * 16 + 256 * (128 * 128 + 256) * 4


def test_layernorm_workspace_size(lib):
    # header + one row of N fp32 sums padded to 4 floats (shared B) ...
    assert wst.wst_gemm_layernorm_workspace_size(1, 100, 0) == 256 + 100 * 4
    assert wst.wst_gemm_layernorm_workspace_size(3, 101, 0) == 256 + 104 * 4
    # ... or one row per batch entry when B has a batch stride
    assert wst.wst_gemm_layernorm_workspace_size(3, 101, 4096) == 256 + 3 * 104 * 4
    assert wst.wst_gemm_layernorm_workspace_size(0, 101, 0) == 0


def test_norm_workspace_size(lib):
    # header, LayerNorm column sums (padded to 4 floats, so the statistics
    # stay 16-byte aligned), then 8 bytes of statistics per row of A
    assert wst.wst_gemm_norm_workspace_size(1, 100, 64) == 256 + 100 * 8
    assert wst.wst_gemm_norm_workspace_size(1, 100, 101, 0, 0, True) == 256 + 104 * 4 + 100 * 8
    assert wst.wst_gemm_norm_workspace_size(1, 100, 100, 0, 0, True) == 256 + 100 * 4 + 100 * 8
    # one row per batch entry when A has a batch stride, else one batch's rows
    assert wst.wst_gemm_norm_workspace_size(3, 100, 64, 6400, 0) == 256 + 3 * 100 * 8
    assert wst.wst_gemm_norm_workspace_size(3, 100, 64, 0, 0) == 256 + 100 * 8
    assert wst.wst_gemm_norm_workspace_size(3, 100, 101, 6400, 4096, True) == 256 + 3 * 104 * 4 + 3 * 100 * 8
    assert wst.wst_gemm_norm_workspace_size(0, 100, 64) == 0
    assert wst.wst_gemm_norm_workspace_size(1, 0, 64) == 0


def norm_gemm(fn, **kw):
    a = dict(batch=1, M=128, N=128, K=64, A=FAKE, lda=64, sA=0, B=FAKE, ldb=64, sB=0, eps=1e-5,
             bias=None, sBias=0, C=FAKE, ldc=128, sC=0, ct=1, epi=0, ws=FAKE, wsb=1 << 20, st=None)
    a.update(kw)
    args = [a["batch"], a["M"], a["N"], a["K"], a["A"], a["lda"], a["sA"], a["B"], a["ldb"],
            a["sB"], a["eps"], a["bias"], a["sBias"], a["C"], a["ldc"], a["sC"], a["ct"],
            a["epi"], a["ws"]]
    return fn(*(args + [a["wsb"], a["st"]]))


@pytest.mark.parametrize("name", ["wst_gemm_rmsnorm_bf16", "wst_gemm_layernorm_bf16"])
@pytest.mark.parametrize("kw,code", [
    (dict(eps=-1.0), wst.WST_ERR_INVALID_ARG),
    (dict(eps=float("nan")), wst.WST_ERR_INVALID_ARG),
    (dict(eps=float("inf")), wst.WST_ERR_INVALID_ARG),
    (dict(N=0), wst.WST_ERR_INVALID_ARG),
    (dict(epi=2), wst.WST_ERR_INVALID_ARG),            # bias missing
    (dict(B=FAKE + 8), wst.WST_ERR_ALIGNMENT),
    (dict(ldb=72, sB=0), wst.WST_ERR_INVALID_ARG),     # not device memory (no GPU here)
])
def test_norm_gemm_rejects(lib, name, kw, code):
    assert norm_gemm(getattr(lib, name), **kw) == code


def test_rmsnorm_rejects_workspace_below_header(lib):
    f = lib.wst_gemm_rmsnorm_bf16
    assert norm_gemm(f, wsb=255) == wst.WST_ERR_INVALID_ARG
    assert "workspace" in lib.wst_last_error().decode()


def test_layernorm_rejects_small_workspace(lib):
    f = lib.wst_gemm_layernorm_bf16
    assert norm_gemm(f, wsb=256 + 127 * 4) == wst.WST_ERR_INVALID_ARG
    assert "workspace" in lib.wst_last_error().decode()
    assert norm_gemm(f, batch=2, sA=8192, sB=8192, sC=16384, wsb=256 + 128 * 4) == wst.WST_ERR_INVALID_ARG
    assert "workspace" in lib.wst_last_error().decode()


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_is_plain_c_and_cpp(lang, std, tmp_path):
    # The boundary is a C ABI: include/wst.h must compile on its own as C99
    # (and as C++) with no warnings.
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "wst.h"\nint main(void) { return (int)wst_workspace_size(0, 0, 0) * 0; }\n')
    r = subprocess.run([cc, "-std=" + std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_options_set_get_and_reject(lib):
    # Process-wide schedule options: values round-trip, bad ones are refused
    # with WST_ERR_INVALID_ARG and leave the option unchanged.  No GPU needed.
    import warp_specialized_tensor_gb300 as w
    assert w.wst_get_option(w.OPT_GROUPED_SCHEDULE) == w.SCHED_STATIC
    assert w.wst_get_option(w.OPT_DENSE_CTA_GROUP) == 0
    with w.option(w.OPT_GROUPED_SCHEDULE, w.SCHED_CLC):
        assert w.wst_get_option(w.OPT_GROUPED_SCHEDULE) == w.SCHED_CLC
    assert w.wst_get_option(w.OPT_GROUPED_SCHEDULE) == w.SCHED_STATIC
    for cg in (1, 2, 0):
        w.wst_set_option(w.OPT_DENSE_CTA_GROUP, cg)
        assert w.wst_get_option(w.OPT_DENSE_CTA_GROUP) == cg
    assert lib.wst_set_option(w.OPT_DENSE_CTA_GROUP, 3) == 1
    assert lib.wst_set_option(w.OPT_GROUPED_SCHEDULE, -1) == 1
    assert lib.wst_set_option(99, 0) == 1
    assert b"unknown option" in lib.wst_last_error()
    assert w.wst_get_option(w.OPT_DENSE_CTA_GROUP) == 0
    assert w.wst_get_option(w.OPT_GROUPED_SCHEDULE) == w.SCHED_STATIC
    assert w.wst_get_option(w.OPT_NORM_STATS) == w.NORM_STATS_AUTO
    for mode in (w.NORM_STATS_FUSED, w.NORM_STATS_PASS):
        with w.option(w.OPT_NORM_STATS, mode):
            assert w.wst_get_option(w.OPT_NORM_STATS) == mode
    assert lib.wst_set_option(w.OPT_NORM_STATS, 3) == 1
    assert w.wst_get_option(w.OPT_NORM_STATS) == w.NORM_STATS_AUTO
