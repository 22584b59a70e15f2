"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/nvfp4.h declares, and rejects bad arguments synchronously
(these paths return before any CUDA runtime call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_quantization_gb300 import _lib
    from nvfp4_block_quantization_gb300.build import build

    build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+(nvfp4_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("nvfp4_kv_smooth_quant", "nvfp4_kv_dequant", "nvfp4_weight_quant_2d"):
        assert n in names
    from nvfp4_block_quantization_gb300 import _lib

    assert sorted(_lib.EXPORTS) == names


def test_library_exports_every_header_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from nvfp4_block_quantization_gb300 import _lib

    for s in range(6):
        assert _lib.status_string(s).startswith("NVFP4_")
    assert _lib.status_string(99) == "NVFP4_UNKNOWN"
    assert lib.nvfp4_version() >= 100


P = ctypes.c_void_p


def test_kv_quant_argument_errors(lib):
    from nvfp4_block_quantization_gb300 import _lib as L

    good = P(4096)
    q = L.nvfp4_kv_smooth_quant
    # NULL input
    assert q(None, 0, 8, 2, 32, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_EINVAL
    # bad dtype / smooth flag
    assert q(good, 7, 8, 2, 32, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_EINVAL
    assert q(good, 0, 8, 2, 32, 2, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_EINVAL
    # mean pointers without smoothing
    assert q(good, 0, 8, 2, 32, 0, good, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_EINVAL
    # shapes
    assert q(good, 0, 8, 2, 24, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_ESHAPE
    assert q(good, 0, -1, 2, 32, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_ESHAPE
    assert q(good, 0, 8, 0, 32, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_ESHAPE
    # alignment
    assert q(P(4098), 0, 8, 2, 32, 1, None, None, good, good, good, None, good, 1 << 20, None) == L.NVFP4_EALIGN
    assert q(good, 0, 8, 2, 32, 1, None, None, P(4104), good, good, None, good, 1 << 20, None) == L.NVFP4_EALIGN
    assert q(good, 0, 8, 2, 32, 1, None, None, good, good, P(4097), None, good, 1 << 20, None) == L.NVFP4_EALIGN
    assert q(good, 0, 8, 2, 32, 1, None, None, good, good, good, P(4098), good, 1 << 20, None) == L.NVFP4_EALIGN


def test_batched_argument_errors(lib):
    from nvfp4_block_quantization_gb300 import _lib as L

    jobs = (L.nvfp4_kv_job * 2)()
    assert L.nvfp4_kv_smooth_quant_batched(jobs, 0, 0, 8, 2, 32, None, P(4096), 1 << 20, None) == L.NVFP4_EINVAL
    assert L.nvfp4_kv_smooth_quant_batched(None, 2, 0, 8, 2, 32, None, P(4096), 1 << 20, None) == L.NVFP4_EINVAL
    for j in jobs:
        j.x = j.codes = j.scales = j.tensor_scale = 4096
        j.smooth = 1
    jobs[1].smooth = 0
    jobs[1].mean_out = 8192  # mean output on an unsmoothed job
    assert L.nvfp4_kv_smooth_quant_batched(jobs, 2, 0, 8, 2, 32, None, P(4096), 1 << 20, None) == L.NVFP4_EINVAL


def test_dequant_argument_errors(lib):
    from nvfp4_block_quantization_gb300 import _lib as L

    g = P(4096)
    d = L.nvfp4_kv_dequant
    assert d(g, g, g, None, 0, 8, 2, 32, g, None) == L.NVFP4_ESHAPE
    assert d(g, g, None, None, 8, 8, 2, 32, g, None) == L.NVFP4_EINVAL
    assert d(g, g, g, None, 8, 8, 2, 20, g, None) == L.NVFP4_ESHAPE
    assert d(P(4100), g, g, None, 8, 8, 2, 32, g, None) == L.NVFP4_EALIGN


def test_weight_argument_errors(lib):
    from nvfp4_block_quantization_gb300 import _lib as L

    g = P(4096)
    w = L.nvfp4_weight_quant_2d
    assert w(g, 0, 20, 32, g, g, g, None, g, 1 << 20, None) == L.NVFP4_ESHAPE
    assert w(g, 0, 32, 8, g, g, g, None, g, 1 << 20, None) == L.NVFP4_ESHAPE
    assert w(g, 0, 1 << 24, 1 << 24, g, g, g, None, g, 1 << 20, None) == L.NVFP4_ESHAPE  # M * N > 2^46
    assert w(g, 3, 32, 32, g, g, g, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert w(None, 0, 32, 32, g, g, g, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert w(g, 0, 32, 32, P(4097), g, g, None, g, 1 << 20, None) == L.NVFP4_EALIGN
    assert L.nvfp4_weight_dequant_2d(g, g, None, 32, 32, g, None) == L.NVFP4_EINVAL


def test_weight_batched_argument_errors(lib):
    from nvfp4_block_quantization_gb300 import _lib as L

    g = P(4096)

    def jobs(*specs):
        arr = (L.nvfp4_w2d_job * len(specs))()
        for k, (w, M, N, c, s, t) in enumerate(specs):
            arr[k].w, arr[k].M, arr[k].N, arr[k].codes, arr[k].scales, arr[k].tensor_scale = w, M, N, c, s, t
        return arr

    b = L.nvfp4_weight_quant_2d_batched
    ok = (g, 32, 32, g, g, g)
    assert b(None, 1, 0, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert b(jobs(ok), 0, 0, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert b(jobs(ok), 1, 2, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert b(jobs(ok, (g, 20, 32, g, g, g)), 2, 0, None, g, 1 << 20, None) == L.NVFP4_ESHAPE
    assert b(jobs(ok, (g, 32, 8, g, g, g)), 2, 0, None, g, 1 << 20, None) == L.NVFP4_ESHAPE
    assert b(jobs(ok, (None, 32, 32, g, g, g)), 2, 0, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert b(jobs(ok, (g, 32, 32, g, g, None)), 2, 0, None, g, 1 << 20, None) == L.NVFP4_EINVAL
    assert b(jobs((g, 32, 32, P(4097), g, g)), 1, 0, None, g, 1 << 20, None) == L.NVFP4_EALIGN
    assert b(jobs(ok), 1, 0, P(4098), g, 1 << 20, None) == L.NVFP4_EALIGN
    assert L.nvfp4_w2d_batched_workspace_bytes(0) == 0
    assert L.nvfp4_w2d_batched_workspace_bytes(1) == L.nvfp4_w2d_batched_workspace_bytes(64) > 0
    assert b(jobs(ok), 1, 0, None, g, 16, None) == L.NVFP4_EWORKSPACE
    assert b(jobs(ok), 1, 0, None, P(4096 + 128), 1 << 20, None) == L.NVFP4_EWORKSPACE


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "nvfp4_block_quantization_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "nvfp4_oracle" not in txt, f


def test_workloads_are_seeded_and_shaped():
    import numpy as np

    from nvfp4_block_quantization_gb300 import workloads as W

    K1, V1 = W.tiny_kv(0)
    K2, V2 = W.tiny_kv(0)
    assert K1.shape == (64, 1, 64) and K1.dtype == np.float32
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
    assert int((np.abs(K1) > 12).sum()) >= 10  # the outliers are there
    k = W.chunk_k(2000, T=64, H=4, D=32)
    assert k.shape == (64, 4, 32)
    assert W.CHUNK_TOKENS == 7040


def test_missing_library_fails_loudly(tmp_path):
    """Without the compiled library the binding raises; there is no other path to fall back to."""
    from nvfp4_block_quantization_gb300 import _lib

    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            _lib.load(str(tmp_path / "libnvfp4_gb300.so"))
    finally:
        _lib._lib = saved
