"""The no-allocation variant of the fused GEMM + LayerNorm call.

Some callers cannot allocate device memory (an operator or plugin interface
that receives only its input and output buffers, or a runtime that plans all
device memory up front and forbids allocation while serving), so they cannot
provide the workspace the regular call takes.  The variant keeps its scratch
in a fixed array inside the library.  This file is collected last so that a
run stopping at its first failure has run every other test first.
"""
import numpy as np
import pytest

from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    torch = torch_cuda()
    # N = 16384 is wider than any cluster (256 columns x 16 CTAs, or 512 x 16), so the
    # global partial buffer (scratch) is used
    M, N, K = 390, 16384, 128
    d = inputs.gemm_inputs(M, N, K, 31, x_std=K ** -0.5, w_std=K ** -0.5, bias_std=0.1, gamma_std=0.1,
                           beta_std=0.1)
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    b, g, be = dev_f32(d["bias"]), dev_f32(d["gamma"]), dev_f32(d["beta"])
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, 1)
    assert st == cf.CF_OK and plan.groups > 1

    Y_ws = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    assert cf.cf_gemm_fused_rownorm(X, W, b, g, be, Y_ws, M, N, K, 1.0, 1e-5, cf.CF_ACT_GELU_TANH, ws,
                                    ws.numel()) == cf.CF_OK
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    ref = host(Y_ws)

    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = cf.cf_gemm_fused_rownorm_noalloc(X, W, b, g, be, Y, M, N, K, 1.0, 1e-5, cf.CF_ACT_GELU_TANH)
        assert st == cf.CF_OK, (call, cf.status_string(st))
        torch.cuda.synchronize()
        y = host(Y)
        assert np.all(np.isfinite(y)), call
        check_ln(y, ref, f"no-alloc call {call} vs workspace call")


def test_noalloc_rejects_scratch_beyond_its_maximum():
    torch = torch_cuda()
    buf = torch.empty(1024, dtype=torch.float32, device="cuda")
    # N = 16384 plans as 4 cluster groups per 128-row block; 1100 row blocks x 4 x 1 KiB of
    # partials > 4 MiB: refused before anything is launched or read
    M, N, K = 128 * 1100, 16384, 64
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, 0)
    assert st == cf.CF_OK and plan.row_blocks * plan.groups * 1024 > 4 << 20
    st = cf.cf_gemm_fused_rownorm_noalloc(buf, buf, None, buf, buf, buf, M, N, K, 1.0, 1e-5, cf.CF_ACT_NONE)
    assert st == cf.CF_ERR_WORKSPACE_TOO_SMALL
