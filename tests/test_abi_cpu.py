"""The C ABI on a machine without a GPU: the library loads, exports every
entry point include/wq.h declares, and rejects bad arguments before touching
CUDA (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

import weight_only_bit_w4a16_gb300 as wq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(wq.SIGNATURES)


def test_library_exports_every_declared_symbol():
    L = wq.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define\s+(WQ_[A-Z0-9_]+)\s+\(?(-?(?:0x)?[0-9A-Fa-f]+)\)?", text))
    for k, v in consts.items():
        assert getattr(wq, k) == int(v, 0), k


def test_status_strings_and_version():
    for st in (wq.WQ_OK, wq.WQ_ERR_INVALID_ARG, wq.WQ_ERR_UNSUPPORTED, wq.WQ_ERR_ALIGN,
               wq.WQ_ERR_CUDA, wq.WQ_ERR_DEVICE_TIMEOUT):
        assert wq.wq_status_string(st).startswith("WQ_")
    assert wq.wq_status_string(12345) == "unknown wq status"
    assert wq.wq_version() >= 100


# Arguments rejected during validation: nothing reaches CUDA.
FAKE = ctypes.c_void_p(0x10000)   # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)


@pytest.mark.parametrize("args,expect", [
    # (A, packed, scales, zeros, C, M, N, K, format, group)
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 7, 16), wq.WQ_ERR_INVALID_ARG),       # bad format
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 0x200, 16), wq.WQ_ERR_INVALID_ARG),   # bad flag
    ((FAKE, FAKE, FAKE, None, FAKE, -1, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),      # M < 0
    ((FAKE, FAKE, FAKE, None, FAKE, 4, -8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),      # N < 0
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 32), wq.WQ_ERR_UNSUPPORTED),       # nvfp4 group
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 1, 16), wq.WQ_ERR_UNSUPPORTED),       # mxfp4 group
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 2, 48), wq.WQ_ERR_UNSUPPORTED),      # int4 group
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 48, 0, 16), wq.WQ_ERR_UNSUPPORTED),       # K % 32
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 192, 2, 128), wq.WQ_ERR_UNSUPPORTED),     # K % group
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 2, 32), wq.WQ_ERR_INVALID_ARG),       # int4 w/o zeros
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),       # fp4 with zeros
    ((FAKE, None, FAKE, None, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),       # NULL packed
    ((FAKE, FAKE, None, None, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),       # NULL scales
    ((None, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),       # NULL A
    ((FAKE, FAKE, FAKE, None, None, 4, 8, 64, 0, 16), wq.WQ_ERR_INVALID_ARG),       # NULL C
    ((ODD, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_ALIGN),              # A alignment
    ((FAKE, ODD, FAKE, None, FAKE, 4, 8, 64, 0, 16), wq.WQ_ERR_ALIGN),              # packed alignment
    ((FAKE, FAKE, FAKE, None, ODD, 4, 8, 64, 0, 16), wq.WQ_ERR_ALIGN),              # C alignment
    ((FAKE, FAKE, ctypes.c_void_p(0x10001), FAKE, FAKE, 4, 8, 64, 2, 32), wq.WQ_ERR_ALIGN),  # int4 scales
    ((FAKE, FAKE, FAKE, None, FAKE, 0, 8, 64, 0, 16), wq.WQ_OK),                    # M == 0: no-op
    ((FAKE, FAKE, FAKE, None, FAKE, 4, 0, 64, 0, 16), wq.WQ_OK),                    # N == 0: no-op
])
def test_gemm_argument_validation(args, expect):
    assert wq.wq_gemm(*args) == expect
    assert wq.wq_gemm_ex(*args, None, wq.WQ_PATH_GEMV) == expect


def test_gemm_bad_path():
    assert wq.wq_gemm_ex(FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 16, None, 9) == wq.WQ_ERR_INVALID_ARG
    assert wq.wq_gemm_ex(FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 16, None, 0x400) == wq.WQ_ERR_INVALID_ARG
    # the overlap flag is a valid path bit (M == 0: validated, nothing launched)
    assert wq.wq_gemm_ex(FAKE, FAKE, FAKE, None, FAKE, 0, 8, 64, 0, 16, None,
                         wq.WQ_PATH_GEMV | wq.WQ_LAUNCH_OVERLAP) == wq.WQ_OK


@pytest.mark.parametrize("args,expect", [
    # (packed, scales, zeros, W, N, K, format, group, stream)
    ((FAKE, FAKE, None, FAKE, 8, 64, 0x100, 16, None), wq.WQ_ERR_INVALID_ARG),   # output flag
    ((FAKE, FAKE, None, None, 8, 64, 0, 16, None), wq.WQ_ERR_INVALID_ARG),       # NULL W
    ((FAKE, FAKE, None, ODD, 8, 64, 0, 16, None), wq.WQ_ERR_ALIGN),              # W alignment
    ((FAKE, FAKE, None, FAKE, 8, 40, 0, 16, None), wq.WQ_ERR_UNSUPPORTED),       # K % 32
    ((FAKE, FAKE, None, FAKE, 0, 64, 0, 16, None), wq.WQ_OK),                    # N == 0
])
def test_dequant_argument_validation(args, expect):
    assert wq.wq_dequant(*args) == expect


def test_tensor_helpers_refuse_cpu_tensors():
    torch = pytest.importorskip("torch")
    A = torch.zeros((1, 64), dtype=torch.bfloat16)
    packed = torch.zeros((8, 32), dtype=torch.uint8)
    scales = torch.zeros((8, 4), dtype=torch.uint8)
    with pytest.raises(ValueError):
        wq.gemm(A, packed, scales, None, "nvfp4")


def test_fused_argument_checks():
    epi = wq.wq_epilogue(None, None, 1)
    args = (FAKE, FAKE, FAKE, None, FAKE, 4, 24, 64, 0, 16)   # N = 24: not a multiple of 16
    assert wq.wq_gemm_fused(*args, ctypes.byref(epi), None, 0, None, 0) == wq.WQ_ERR_UNSUPPORTED
    bad = wq.wq_epilogue(None, None, 2)
    assert wq.wq_gemm_fused(*args, ctypes.byref(bad), None, 0, None, 0) == wq.WQ_ERR_INVALID_ARG
    odd = wq.wq_epilogue(0x10001, None, 0)
    assert wq.wq_gemm_fused(FAKE, FAKE, FAKE, None, FAKE, 4, 32, 64, 0, 16, ctypes.byref(odd), None, 0, None,
                            0) == wq.WQ_ERR_ALIGN
    # M == 0 with an epilogue: validated, nothing launched
    assert wq.wq_gemm_fused(FAKE, FAKE, FAKE, None, FAKE, 0, 32, 64, 0, 16, ctypes.byref(epi), None, 0, None,
                            0) == wq.WQ_OK


def test_prepack_sizes_match_the_oracle_layout():
    from oracle import prepack as opk
    for fmt, code, group in (("int4", 2, 128), ("nvfp4", 0, 16), ("mxfp4", 1, 32)):
        for N, K in ((20, 256), (16, 128), (8192, 3072), (1, 32 if fmt != "int4" else 128)):
            assert wq.wq_prepack_bytes(N, K, code, group) == opk.prepack_bytes(N, K, fmt)
    # descriptions prepack does not take
    assert wq.wq_prepack_bytes(16, 256, 2, 64) == 0         # int4 group other than 128
    assert wq.wq_prepack_bytes(16, 256, 0, 32) == 0         # nvfp4 group
    assert wq.wq_prepack_bytes(0, 256, 0, 16) == 0
    assert wq.wq_prepack_bytes(16, 0, 0, 16) == 0
    assert wq.wq_prepack_bytes(16, 48, 0, 16) == 0          # K not a multiple of 32
    assert wq.wq_prepack_bytes(16, 256, 0x100, 16) == 0     # flags are not a format


def test_prepack_argument_checks():
    nb = wq.wq_prepack_bytes(32, 256, 0, 16)
    # (packed, scales, zeros, prepacked, bytes, N, K, format, group, stream)
    assert wq.wq_prepack(FAKE, FAKE, None, FAKE, nb - 1, 32, 256, 0, 16, None) == wq.WQ_ERR_INVALID_ARG
    assert wq.wq_prepack(FAKE, FAKE, None, None, nb, 32, 256, 0, 16, None) == wq.WQ_ERR_INVALID_ARG
    assert wq.wq_prepack(FAKE, FAKE, None, ODD, nb, 32, 256, 0, 16, None) == wq.WQ_ERR_ALIGN
    assert wq.wq_prepack(FAKE, FAKE, FAKE, FAKE, 1 << 20, 32, 256, 2, 64, None) == wq.WQ_ERR_UNSUPPORTED
    assert wq.wq_prepack(FAKE, FAKE, FAKE, FAKE, nb, 32, 256, 0, 16, None) == wq.WQ_ERR_INVALID_ARG  # zeros for fp4
    assert wq.wq_prepack(FAKE, FAKE, None, FAKE, nb, 32, 256, 0x100, 16, None) == wq.WQ_ERR_INVALID_ARG


def test_gemm_prepacked_argument_checks():
    def f(A, pre, C, M, N, K, fmt, group, epi=None, ws=None, wsb=0, path=0):
        return wq.wq_gemm_prepacked(A, pre, C, M, N, K, fmt, group, epi, ws, wsb, None, path)
    assert f(FAKE, FAKE, FAKE, 0, 32, 256, 0, 16) == wq.WQ_OK                        # M == 0: no-op
    assert f(FAKE, FAKE, FAKE, 4, 0, 256, 0, 16) == wq.WQ_OK                         # N == 0: no-op
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 0, 16, path=7) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 0, 16, path=0x400) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, -1, 32, 256, 0, 16) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 7, 16) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 2, 64) == wq.WQ_ERR_UNSUPPORTED
    assert f(FAKE, ODD, FAKE, 4, 32, 256, 0, 16) == wq.WQ_ERR_ALIGN
    assert f(ODD, FAKE, FAKE, 4, 32, 256, 0, 16) == wq.WQ_ERR_ALIGN
    assert f(None, FAKE, FAKE, 4, 32, 256, 0, 16) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 0, 16, ws=None, wsb=64) == wq.WQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 32, 256, 0, 16, ws=ODD, wsb=64) == wq.WQ_ERR_ALIGN
    epi = wq.wq_epilogue(None, None, 1)
    assert f(FAKE, FAKE, FAKE, 4, 24, 256, 0, 16, ctypes.byref(epi)) == wq.WQ_ERR_UNSUPPORTED


def test_workspace_size_alias():
    """wq_workspace_bytes is wq_gemm_workspace_size under its design name."""
    for args in ((300, 3072, 3072, 2, 128), (4, 512, 1024, 2, 128), (0, 8, 64, 0, 16), (300, 1000, 1024, 1, 32)):
        assert wq.wq_workspace_bytes(*args) == wq.wq_gemm_workspace_size(*args)


def test_cluster_split_plans_need_no_workspace(monkeypatch):
    """Host planning (no GPU needed: the planner assumes an SM count without
    a device).  128 x 3072 x 3072 has 24 tiles of 128 weight rows: too few
    to fill the SMs, so each runs on a thread-block cluster whose CTAs add
    their partial sums on chip -- no workspace.  With the cluster mode off
    the same shape asks for stream-K's workspace, and a forced cluster size
    whose CTAs would not fit on the SMs falls back to stream-K as well."""
    shape = (128, 3072, 3072, wq.WQ_INT4, 128)
    monkeypatch.delenv("WQ_TC_CSK", raising=False)
    assert wq.wq_gemm_workspace_size(*shape) == 0
    monkeypatch.setenv("WQ_TC_CSK", "0")
    assert wq.wq_gemm_workspace_size(*shape) > 0
    monkeypatch.setenv("WQ_TC_CSK", "8")          # 24 tiles x 8 CTAs: more than the SMs
    assert wq.wq_gemm_workspace_size(*shape) > 0
    monkeypatch.setenv("WQ_TC_CSK", "2")          # 48 CTAs fit
    assert wq.wq_gemm_workspace_size(*shape) == 0


def test_full_waves_need_no_workspace_either_way(monkeypatch):
    """Shapes whose whole tiles fill the SMs' waves run whole tiles: no
    workspace with or without the cluster mode."""
    for setting in ("1", "0"):
        monkeypatch.setenv("WQ_TC_CSK", setting)
        assert wq.wq_gemm_workspace_size(8192, 8192, 8192, wq.WQ_NVFP4, 16) == 0
        assert wq.wq_gemm_workspace_size(2048, 128256, 3072, wq.WQ_INT4, 128) == 0
