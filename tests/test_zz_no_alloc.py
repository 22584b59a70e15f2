"""nvfp4_weight_quant_2d_static (no workspace) against nvfp4_weight_quant_2d, through the C ABI.

The static-scratch call must give the workspace call's bits: codes, scales and
tensor scale identical, status OK, on consecutive calls (different matrices, then
the first matrix again, which also checks that nothing stale survives in the
shared scratch).
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _bf16(a: np.ndarray):
    from nvfp4_block_quantization_gb300 import workloads as W

    return torch.from_numpy(W.to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def _static_call(lib, w):
    M, N = w.shape
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((M // 16, N // 16), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    vp = ctypes.c_void_p
    st = lib.nvfp4_weight_quant_2d_static(vp(w.data_ptr()), 0, M, N, vp(codes.data_ptr()), vp(scales.data_ptr()),
                                          vp(g.data_ptr()), vp(status.data_ptr()),
                                          vp(torch.cuda.current_stream().cuda_stream))
    return st, codes, scales, g, status


def test_static_scratch_matches_workspace_call():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from nvfp4_block_quantization_gb300.build import build

    build()
    import nvfp4_block_quantization_gb300 as nv
    from nvfp4_block_quantization_gb300 import _lib
    from nvfp4_block_quantization_gb300 import workloads as W

    lib = _lib.load()
    mats = [_bf16(W.weight(0, 256, 512)), _bf16(W.weight(1, 3072, 3072))]
    refs = []
    for w in mats:
        r = nv.weight_quant_2d(w)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        refs.append(r)
    for i in (0, 1, 0):  # consecutive calls, the first matrix twice
        st, codes, scales, g, status = _static_call(lib, mats[i])
        assert st == 0, _lib.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = refs[i]
        assert torch.equal(codes, ref.codes)
        assert torch.equal(scales, ref.scales)
        assert torch.equal(g.view(torch.int32), ref.tensor_scale.view(torch.int32))
