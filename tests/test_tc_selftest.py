"""tcgen05 tile product against a CPU product (GPU): checks the shared-memory
descriptor, instruction descriptor and TMEM conventions the tensor-core
kernels rely on, for K-major and MN-major operands and for an A operand held
in tensor memory (a_mn = 2)."""
import ctypes

import numpy as np
import pytest

from state_space_model_sm_gb300 import _native
from state_space_model_sm_gb300.inputs import round_to_bf16

pytestmark = pytest.mark.gpu

CASES = [(0, 0, 64, 64), (0, 0, 256, 128), (0, 0, 128, 16), (1, 0, 64, 64), (0, 1, 128, 64),
         (1, 1, 128, 128), (1, 1, 64, 32), (2, 0, 64, 64), (2, 0, 128, 128), (2, 1, 64, 64),
         (2, 1, 128, 32)]


@pytest.mark.parametrize("a_mn,b_mn,nn,k", CASES)
def test_tile_mma(cuda_lib, a_mn, b_mn, nn, k):
    import torch
    rng = np.random.default_rng(nn * 1000 + k + 10 * a_mn + b_mn)
    A = round_to_bf16(rng.standard_normal((128, k)).astype(np.float32))
    B = round_to_bf16(rng.standard_normal((nn, k)).astype(np.float32))
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    tA = torch.from_numpy(A).to("cuda", torch.bfloat16)
    tB = torch.from_numpy(B).to("cuda", torch.bfloat16)
    results = {}
    for swap in (0, 1) if (a_mn == 1 or b_mn) else (0,):
        D = torch.full((128, nn), float("nan"), device="cuda")
        st = _native.load().ssd_selftest_mma(a_mn, b_mn, swap, nn, k,
                                            ctypes.c_void_p(tA.data_ptr()),
                                            ctypes.c_void_p(tB.data_ptr()),
                                            ctypes.c_void_p(D.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        results[swap] = float(np.nanmax(np.abs(D.cpu().numpy().astype(np.float64) - ref)))
    print(f"a_mn={a_mn} b_mn={b_mn} nn={nn} k={k} max err by offset order: {results}")
    # the unswapped order (LBO = panel stride, SBO = 8-row group) is the one the kernels use
    assert results[0] < 1e-3 * max(1.0, np.abs(ref).max()), results
