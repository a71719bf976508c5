"""GPU parity of the causally masked fused GEMM + row softmax (through the C
ABI) against the fp64 oracle: offsets that keep part, all or none of a row,
ragged row tails, the schedules of the unmasked call (wide tiles, rows over
several clusters, CTA pairs), masked entries exactly zero, and the
attention-score workload on sampled rows."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_softmax, dev_bf16, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    return inputs.gemm_inputs(M, N, K, seed, x_std=1.0, w_std=K ** -0.5, bias_std=0.5, gamma_std=None,
                              beta_std=None)


def _run(d, scale, offset, bias=None, tuning=None, causal=True):
    torch = torch_cuda()
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    if causal:
        st = cf.cf_gemm_fused_rowsoftmax_causal(X, W, dev_f32(bias), Y, M, N, K, scale, offset, ws, ws.numel(),
                                                None, tuning)
    else:
        st = cf.cf_gemm_fused_rowsoftmax(X, W, dev_f32(bias), Y, M, N, K, scale, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


def _check(y, ref, M, N, offset, what):
    keep = np.arange(N)[None, :] <= (np.arange(M)[:, None] + offset)
    assert np.all(y[~keep] == 0.0), f"{what}: masked entries not exactly 0"
    live = keep.any(axis=1)
    if live.any():
        check_softmax(y[live], ref[live], what, bf16_out=True)
    assert np.all(y[~live] == 0.0), f"{what}: fully masked rows not 0"


@pytest.mark.parametrize("M,N,K,offset", [(300, 2048, 128, 0), (300, 2048, 128, -64), (257, 1024, 64, 37),
                                          (130, 512, 128, 600), (200, 512, 128, -250)])
def test_causal_offsets(M, N, K, offset):
    d = _inputs(M, N, K, seed=M + N + offset % 97)
    scale = K ** -0.5
    y = _run(d, scale, offset, bias=d["bias"])
    ref = oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=scale, offset=offset, bias=d["bias"])
    _check(y, ref, M, N, offset, f"causal {M}x{N}x{K} offset {offset}")


@pytest.mark.parametrize("kw", [dict(n_slice=512), dict(n_slice=256, cluster_size=2), dict(cluster_size=2, cluster_m=2),
                                dict(cluster_size=8, peer_max=-1)])
def test_causal_schedules(kw):
    M, N, K = 390, 4096, 128
    d = _inputs(M, N, K, seed=91)
    y = _run(d, K ** -0.5, 1000, tuning=cf.tuning(**kw))
    ref = oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=K ** -0.5, offset=1000)
    _check(y, ref, M, N, 1000, f"causal {kw}")


@pytest.mark.parametrize("offset", [-300, -129, 0, 200, 1500])
def test_causal_row_groups_past_the_mask(offset):
    """Rows over G = 4 cluster groups (1024 columns each, through the global
    barrier): groups lying entirely past a row block's last kept column are all
    zeros, and row blocks whose rows keep nothing are zeros throughout."""
    M, N, K = 650, 4096, 128
    d = _inputs(M, N, K, seed=93 + offset % 89)
    t = cf.tuning(n_slice=256, cluster_size=4)
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, 2, t)
    assert st == cf.CF_OK and plan.groups == 4
    y = _run(d, K ** -0.5, offset, bias=d["bias"], tuning=t)
    ref = oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=K ** -0.5, offset=offset, bias=d["bias"])
    _check(y, ref, M, N, offset, f"causal G=4 offset {offset}")


def test_causal_keeping_everything_is_the_unmasked_kernel():
    """With every column kept the masked kernel does the unmasked one's arithmetic."""
    d = _inputs(300, 2048, 128, seed=92)
    a = _run(d, 0.1, 2047, bias=d["bias"])
    b = _run(d, 0.1, 0, bias=d["bias"], causal=False)
    assert np.array_equal(a, b)


def test_causal_full_workload():
    w = inputs.WORKLOADS["causal_softmax_4096x4096x128"]
    d = inputs.workload_inputs(w.name)
    y = _run(d, w.scale, w.mask_offset)
    rows = sample_rows(w.M, 512, seed=7)
    ref = oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=w.scale, offset=w.mask_offset, rows=rows)
    keep = np.arange(w.N)[None, :] <= (rows[:, None] + w.mask_offset)
    assert np.all(y[rows][~keep] == 0.0)
    check_softmax(y[rows], ref, w.name, bf16_out=True)
