"""The no-allocation variant of the fused GEMM + LayerNorm call.

Some callers cannot allocate device memory (an operator or plugin interface
that receives only its input and output buffers, or a runtime that plans all
device memory up front and forbids allocation while serving), so they cannot
provide the workspace the regular call takes.  The variant keeps its scratch
in a fixed array inside the library.  Both calls run the same plan on the same
deterministic kernel, so their outputs must agree bit for bit; both are also
held to the oracle's tolerance.  This file is collected last so that a run
stopping at its first failure has run every other test first.
"""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed):
    d = inputs.gemm_inputs(M, N, K, seed, x_std=K ** -0.5, w_std=K ** -0.5, bias_std=0.1, gamma_std=0.1,
                           beta_std=0.1)
    dev = {"X": dev_bf16(d["X"]), "W": dev_bf16(d["W"]), "b": dev_f32(d["bias"]), "g": dev_f32(d["gamma"]),
           "be": dev_f32(d["beta"])}
    ref = oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], eps=1e-5, act="gelu_tanh")
    return dev, ref


def _workspace_call(torch, c, M, N, K):
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    assert cf.cf_gemm_fused_rownorm(c["X"], c["W"], c["b"], c["g"], c["be"], Y, M, N, K, 1.0, 1e-5,
                                    cf.CF_ACT_GELU_TANH, ws, ws.numel()) == cf.CF_OK
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    return host(Y)


def _noalloc_call(torch, c, M, N, K):
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = cf.cf_gemm_fused_rownorm_noalloc(c["X"], c["W"], c["b"], c["g"], c["be"], Y, M, N, K, 1.0, 1e-5,
                                          cf.CF_ACT_GELU_TANH)
    assert st == cf.CF_OK, cf.status_string(st)
    dst, info = cf.cf_gemm_fused_rownorm_noalloc_status()  # waits for the stream
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


# (390, 16384, 128): rows wider than any cluster, so the global partial buffer and
# the barrier counters in the fixed array are used (several cluster groups);
# (128, 512, 256): one row block inside one cluster (no partials, one counter pair)
@pytest.mark.parametrize("M,N,K,groups_gt1", [(390, 16384, 128, True), (128, 512, 256, False)])
def test_noalloc_matches_workspace_entry_point_twice(M, N, K, groups_gt1):
    torch = torch_cuda()
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, 1)
    assert st == cf.CF_OK and (plan.groups > 1) == groups_gt1
    c, ref = _case(M, N, K, 31 + M)
    y_ws = _workspace_call(torch, c, M, N, K)
    check_ln(y_ws, ref, "workspace call")
    for call in range(2):
        y = _noalloc_call(torch, c, M, N, K)
        assert np.array_equal(y, y_ws), f"call {call}: differs from the workspace entry point"
        check_ln(y, ref, f"no-alloc call {call}")


def test_noalloc_large_then_small_back_to_back():
    """A call using many partials and counters, then a smaller one on the same
    array without a sync between them: the second must read nothing stale."""
    torch = torch_cuda()
    shapes = [(1000, 16384, 64), (260, 8192, 128)]
    cases = [_case(M, N, K, 7 + M) for M, N, K in shapes]
    outs = []
    for (M, N, K), (c, _) in zip(shapes, cases):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert cf.cf_gemm_fused_rownorm_noalloc(c["X"], c["W"], c["b"], c["g"], c["be"], Y, M, N, K, 1.0, 1e-5,
                                                cf.CF_ACT_GELU_TANH) == cf.CF_OK
        outs.append(Y)
    assert cf.cf_gemm_fused_rownorm_noalloc_status()[0] == cf.CF_OK
    for (M, N, K), (c, ref), Y in zip(shapes, cases, outs):
        y = host(Y)
        check_ln(y, ref, f"back to back {M}x{N}x{K}")
        assert np.array_equal(y, _workspace_call(torch, c, M, N, K))


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
