"""The C-ABI library loads, exports every symbol include/cf.h declares, and its
host-only logic (status strings, planner, workspace sizing, argument checks
that return before any CUDA call) behaves.  No compute calls: CPU only."""
import ctypes
import os
import re

import pytest

from memory_fusion_gb300 import cf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from memory_fusion_gb300 import build
    build.build()


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "cf.h")).read()
    return sorted(set(re.findall(r"^CF_API[^(]*?\b(cf_\w+)\(", txt, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    syms = header_symbols()
    for s in ("cf_gemm_fused_rownorm", "cf_gemm_fused_rowsoftmax", "cf_stitch_rowreduce_broadcast",
              "cf_get_device_status", "cf_status_string", "cf_gemm_fused_workspace_size"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(cf.LIB_PATH)
    missing = [s for s in header_symbols() if not hasattr(L, s)]
    assert missing == []


def test_binding_covers_every_declared_symbol():
    assert sorted(cf.declared_symbols()) == header_symbols()


def test_status_strings():
    assert cf.status_string(cf.CF_OK) == "CF_OK"
    assert cf.status_string(cf.CF_ERR_DEVICE_TIMEOUT) == "CF_ERR_DEVICE_TIMEOUT"
    assert cf.status_string(1234) == "CF_ERR_UNKNOWN"
    assert cf.cf_version() >= 100


def test_tuning_default_is_zero():
    t = cf.cf_tuning_default()
    assert all(getattr(t, f) in (0, None) for f, _ in t._fields_)


def _active(d):
    a = [0] * 17
    for k, v in d.items():
        a[k] = v
    return a


# cluster residency measured on a GB300 (152 SMs) for this kernel's shared-memory sizes
GB300 = _active({1: 152, 2: 76, 4: 36, 8: 15, 16: 7})
GB300_LIKE = GB300


def test_plan_forced_single_cluster_rows():
    # N = 2048 -> 8 slices of 256; forcing a cluster of 8 keeps the row in one cluster (peer mode)
    st, p = cf.cf_plan_gemm_fused(4096, 2048, 128, 152, GB300, cf.tuning(cluster_size=8))
    assert st == cf.CF_OK
    assert (p.n_slice, p.ctas_per_row, p.cluster_size, p.groups, p.leader_mode) == (256, 8, 8, 1, 0)
    assert p.row_blocks == 32 and p.clusters == 15
    assert p.smem_bytes <= 232448 and p.stages >= 2


def test_plan_chooses_fastest_predicted():
    """The automatic choice minimises the planner's time model: ceil(T/ncl) tiles per
    CTA in rounds of two (two accumulators, two epilogue groups), each round
    max(2 mainloops, epilogue), plus the global barrier's skew; the epilogue
    grows with the columns of a thread's row slice."""
    cases = {
        (4096, 2048, 128): (4, 1, 1, 32),     # wide tiles: one per CTA, each row in one cluster of 4
        (16384, 4096, 4096): (1, 2, 16, 76),  # CTA pairs (cta_group::2), rows over 16 clusters
        (8192, 16384, 2048): (2, 2, 32, 32),  # CTA pairs, rows over 32 clusters: 32 of the 36 that fit
        (128, 512, 256): (8, 1, 1, 1),        # one row block: 64-column tiles over a cluster of 8, no pair
    }
    for (M, N, K), (C, CM, G, ncl) in cases.items():
        st, p = cf.cf_plan_gemm_fused(M, N, K, 152, GB300)
        assert st == cf.CF_OK
        assert (p.cluster_size, p.cluster_m, p.groups, p.clusters) == (C, CM, G, ncl), (M, N, K, p.as_dict())
        assert p.smem_bytes <= 232448


def test_plan_wide_tile():
    """n_slice 512: one tile fills tensor memory and both epilogue groups share it; the
    row must stay in one cluster (G = 1) of at most 16, with single-CTA MMAs."""
    st, p = cf.cf_plan_gemm_fused(4096, 2048, 128, 152, GB300, cf.tuning(n_slice=512))
    assert st == cf.CF_OK
    assert (p.n_slice, p.ctas_per_row, p.cluster_size, p.groups, p.cluster_m, p.clusters) == (512, 4, 4, 1, 1, 32)
    assert p.stages == 2 and p.smem_bytes <= 232448
    for M, N, kw in [(256, 4096, dict(cluster_size=4)), (256, 16384, {}), (512, 1024, dict(cluster_m=2))]:
        st, _ = cf.cf_plan_gemm_fused(M, N, 128, 152, GB300, cf.tuning(n_slice=512, **kw))
        assert st == cf.CF_ERR_UNSUPPORTED, (M, N, kw)
    # N not a multiple of 512: no wide candidate, and a request for one is refused
    st, _ = cf.cf_plan_gemm_fused(256, 768, 128, 152, GB300, cf.tuning(n_slice=512))
    assert st == cf.CF_ERR_UNSUPPORTED


def test_plan_pair_mode_limits():
    # pairs need two row blocks and tiles of at least 128 columns
    st, p = cf.cf_plan_gemm_fused(128, 4096, 4096, 152, GB300, cf.tuning(cluster_m=2))
    assert st == cf.CF_ERR_NOT_RESIDENT
    st, p = cf.cf_plan_gemm_fused(4096, 4096, 4096, 152, GB300, cf.tuning(cluster_m=2, n_slice=64))
    assert st == cf.CF_ERR_NOT_RESIDENT
    st, p = cf.cf_plan_gemm_fused(4096, 4096, 4096, 152, GB300, cf.tuning(cluster_m=2, n_slice=128))
    assert st == cf.CF_OK and p.cluster_m == 2 and p.stages == 6


def test_plan_leader_mode_above_threshold():
    t = cf.tuning(cluster_size=16)
    st, p = cf.cf_plan_gemm_fused(16384, 4096, 4096, 152, GB300, t)
    assert st == cf.CF_OK
    assert (p.cluster_size, p.groups, p.leader_mode, p.clusters) == (16, 1, 1, 7)
    st, p = cf.cf_plan_gemm_fused(16384, 4096, 4096, 152, GB300, cf.tuning(cluster_size=16, peer_max=16))
    assert p.leader_mode == 0
    st, p = cf.cf_plan_gemm_fused(16384, 4096, 4096, 152, GB300, cf.tuning(cluster_size=2, peer_max=-1))
    assert p.leader_mode == 1


def test_plan_wide_rows_use_global_path():
    # N = 16384 -> 64 slices; a cluster of 16 needs G = 4 resident clusters per row block
    st, p = cf.cf_plan_gemm_fused(8192, 16384, 2048, 152, GB300, cf.tuning(cluster_size=16))
    assert st == cf.CF_OK
    assert (p.cluster_size, p.groups, p.clusters) == (16, 4, 4)
    # cluster 8 forced: G = 8 of the 15 resident clusters
    st, p = cf.cf_plan_gemm_fused(8192, 16384, 2048, 152, GB300, cf.tuning(cluster_size=8))
    assert (p.cluster_size, p.groups, p.clusters) == (8, 8, 8)
    # never more clusters than tickets (one row block: 128-column tiles give
    # every SM work, so G = 64 clusters of 2, one ticket each)
    st, p = cf.cf_plan_gemm_fused(128, 16384, 2048, 152, GB300, cf.tuning(cluster_size=2))
    assert (p.n_slice, p.groups, p.clusters) == (128, 64, 64)
    st, p = cf.cf_plan_gemm_fused(128, 16384, 2048, 152, GB300, cf.tuning(cluster_size=2, n_slice=256))
    assert (p.groups, p.clusters) == (32, 32)


def test_plan_row_groups_keep_one_column_group():
    """A row spanning G > 1 clusters: with fewer than 2G resident clusters the
    grid holds exactly G (each cluster then keeps one column group and the
    static ticket rounds line up with the row groups); with 2G or more, all
    that fit (up to the tickets)."""
    for nres, want in ((32, 32), (36, 32), (63, 32), (64, 64), (76, 76)):
        st, p = cf.cf_plan_gemm_fused(8192, 16384, 2048, 152, _active({4: nres}),
                                      cf.tuning(cluster_size=2, cluster_m=2))
        assert st == cf.CF_OK and p.groups == 32 and p.clusters == want, (nres, p.as_dict())
    # 16 groups of CTA pairs over 4096 columns: 76 pairs fit, more than 2G, all used
    st, p = cf.cf_plan_gemm_fused(16384, 4096, 4096, 152, GB300, cf.tuning(cluster_size=1, cluster_m=2))
    assert (p.groups, p.clusters) == (16, 76)


def test_plan_residency_refused():
    # only 2 clusters of 16 resident but 4 must meet at the barrier
    st, _ = cf.cf_plan_gemm_fused(8192, 16384, 2048, 148, _active({16: 2}), cf.tuning(cluster_size=16))
    assert st == cf.CF_ERR_NOT_RESIDENT
    st, _ = cf.cf_plan_gemm_fused(8192, 16384, 2048, 148, _active({}))
    assert st == cf.CF_ERR_NOT_RESIDENT


def test_plan_shapes():
    assert cf.cf_plan_gemm_fused(128, 100, 256, 148, GB300_LIKE)[0] == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_plan_gemm_fused(128, 512, 100, 148, GB300_LIKE)[0] == cf.CF_ERR_UNSUPPORTED
    st, p = cf.cf_plan_gemm_fused(128, 192, 64, 148, GB300_LIKE)  # 192 = 3 x 64
    assert st == cf.CF_OK
    assert (p.n_slice, p.ctas_per_row) == (64, 3)
    st, p = cf.cf_plan_gemm_fused(1, 384, 64, 152, _active({3: 40}))
    assert (p.n_slice, p.cluster_size, p.row_blocks, p.clusters) == (128, 3, 1, 1)
    # tiny: one row block, too few 256-column tiles to fill the GPU: 64-column
    # tiles over one cluster of 8 (measured 6.8 us against 10.3 us at 256)
    st, p = cf.cf_plan_gemm_fused(128, 512, 256, 152, GB300)
    assert (p.n_slice, p.cluster_size, p.clusters, p.row_blocks) == (64, 8, 1, 1)
    # many row blocks: the widest tile stays (the headline softmax shape)
    st, p = cf.cf_plan_gemm_fused(4096, 2048, 128, 152, GB300)
    assert (p.n_slice, p.cluster_size, p.clusters) == (512, 4, 32)


def test_workspace_sizes():
    # error word + counters + one float2 per row and 64-column group (rounded up to even)
    assert cf.cf_gemm_fused_workspace_size(8192, 16384, 2048) == 256 + 512 + 64 * 257 * 128 * 8
    assert cf.cf_gemm_fused_workspace_size(0, 512, 256) == 256 + 0
    # an odd row-block count is padded to whole CTA pairs
    assert cf.cf_gemm_fused_workspace_size(129, 512, 256) == 256 + 256 + 2 * 9 * 128 * 8
    assert cf.cf_stitch_workspace_size(750000, 32) == 256


def test_argument_errors_need_no_gpu():
    L = cf.lib()
    # null operands
    assert cf.cf_gemm_fused_rownorm(None, None, None, None, None, None, 128, 512, 256, 1.0, 1e-5, 0,
                                    None, 0, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_gemm_fused_rowsoftmax(16, 16, None, 16, -1, 512, 256, 1.0, 16, 4096, 0) == cf.CF_ERR_INVALID_ARG
    # misaligned pointer (checked before any device access)
    assert cf.cf_gemm_fused_rowsoftmax(16 + 2, 16, None, 16, 128, 512, 256, 1.0, 16, 1 << 20, 0) == \
        cf.CF_ERR_MISALIGNED
    # K not a multiple of 64
    assert cf.cf_gemm_fused_rowsoftmax(16, 16, None, 16, 128, 512, 100, 1.0, 16, 1 << 20, 0) == \
        cf.CF_ERR_UNSUPPORTED
    # workspace too small
    assert cf.cf_gemm_fused_rowsoftmax(16, 16, None, 16, 128, 512, 256, 1.0, 16, 8, 0) == \
        cf.CF_ERR_WORKSPACE_TOO_SMALL
    # LayerNorm needs gamma and beta
    assert cf.cf_gemm_fused_rownorm(16, 16, None, None, 16, 16, 128, 512, 256, 1.0, 1e-5, 0,
                                    16, 1 << 20, 0) == cf.CF_ERR_INVALID_ARG
    # bad activation enum
    assert cf.cf_gemm_fused_rownorm(16, 16, None, 16, 16, 16, 128, 512, 256, 1.0, 1e-5, 7,
                                    16, 1 << 20, 0) == cf.CF_ERR_INVALID_ARG
    # M = 0 and empty stitched inputs are no-ops
    assert cf.cf_gemm_fused_rowsoftmax(16, 16, None, 16, 0, 512, 256, 1.0, 16, 1 << 20, 0) == cf.CF_OK
    assert cf.cf_stitch_rowreduce_broadcast(None, None, None, 0, 32, None, 0, 0) == cf.CF_OK
    assert cf.cf_stitch_rowreduce_broadcast(None, None, None, 5, 0, None, 0, 0) == cf.CF_OK
    assert cf.cf_stitch_rowreduce_broadcast(None, None, None, -1, 4, None, 0, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_rowreduce_broadcast(16, 16, 16, 4, 300000, 16, 4096, 0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_stitch_rowreduce_broadcast(18, 16, 16, 4, 32, 16, 4096, 0) == cf.CF_ERR_MISALIGNED
    assert L is not None


def test_newer_entry_points_check_arguments_without_a_gpu():
    big = 1 << 20
    # back-to-back GEMM
    # the error word, then (LayerNorm on the stream kernel) gamma1^T W2 and
    # beta1^T W2, two counters and 32 x 2 x 128 partial sums
    assert cf.cf_b2b_workspace_size() == 256 + 1024 + 256 + 32 * 2 * 128 * 4
    assert cf.cf_b2b_gemm(None, 16, None, 16, 16, 128, 128, 512, 128, 1.0, 0, 16, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 128, 512, 128, 1.0, 7, 16, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm(24, 32, None, 48, 64, 128, 128, 512, 128, 1.0, 0, 16, big, 0) == cf.CF_ERR_MISALIGNED
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 128, 384, 128, 1.0, 0, 16, big, 0) == cf.CF_ERR_UNSUPPORTED
    # the LayerNorm epilogue: N1 in 256-column chunks, N2 in {64, 128}
    assert cf.cf_b2b_gemm_layernorm(16, 32, None, 16, 16, 48, 64, 128, 128, 640, 128, 1.0, 1e-5, 80, big,
                                    0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm_layernorm(16, 32, None, 16, 16, 48, 64, 128, 128, 4096, 96, 1.0, 1e-5, 80, big,
                                    0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 12, 512, 128, 1.0, 0, 16, big, 0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 128, 512, 96, 1.0, 0, 16, big, 0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 128, 512, 128, 1.0, 0, 80, 8, 0) == cf.CF_ERR_WORKSPACE_TOO_SMALL
    # the output may not alias an input
    assert cf.cf_b2b_gemm(16, 32, None, 48, 16, 128, 128, 512, 128, 1.0, 0, 64, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 0, 128, 512, 128, 1.0, 0, 80, big, 0) == cf.CF_OK
    # the LayerNorm epilogue needs gamma1 and beta1, and only has its own entry
    assert cf.cf_b2b_gemm(16, 32, None, 48, 64, 128, 128, 512, 128, 1.0, 2, 80, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm_layernorm(16, 32, None, None, 16, 48, 64, 128, 128, 512, 128, 1.0, 1e-5, 80,
                                    big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm_layernorm(16, 32, None, 16, 16, 48, 64, 0, 128, 512, 128, 1.0, 1e-5, 80,
                                    big, 0) == cf.CF_OK
    # stitched add + LayerNorm
    assert cf.cf_stitch_add_layernorm(16, None, 16, 16, 16, 0, 32, 1e-5, 16, 4096, 0) == cf.CF_OK
    assert cf.cf_stitch_add_layernorm(16, None, None, 16, 16, 4, 32, 1e-5, 16, 4096, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_add_layernorm(18, None, 16, 16, 16, 4, 32, 1e-5, 16, 4096, 0) == cf.CF_ERR_MISALIGNED
    assert cf.cf_stitch_add_layernorm(16, 16, 16, 16, 16, 4, 300000, 1e-5, 16, 4096, 0) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_stitch_add_layernorm(16, 16, 16, 16, 16, 4, 32, 1e-5, 16, 8, 0) == cf.CF_ERR_WORKSPACE_TOO_SMALL
    # stitched BatchNorm: the workspace covers either scheme
    assert cf.cf_stitch_batchnorm_workspace_size(64, 30000) == cf.cf_stitch_batchnorm_workspace_size(750000, 32)
    assert cf.cf_stitch_batchnorm_workspace_size(1, 1) >= 256 + 256 + 1024 * 128 * 8
    assert cf.cf_stitch_batchnorm(16, 16, 16, 16, None, None, 0, 32, 1e-5, 16, 0, 0) == cf.CF_OK
    assert cf.cf_stitch_batchnorm(16, 16, 16, 16, None, None, -2, 32, 1e-5, 16, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_batchnorm(16, None, 16, 16, None, None, 8, 32, 1e-5, 16, big, 0) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_batchnorm(16, 16, 16, 16, 2, None, 8, 32, 1e-5, 16, big, 0) == cf.CF_ERR_MISALIGNED
    assert cf.cf_stitch_batchnorm(16, 16, 16, 16, None, None, 8, 32, 1e-5, 16, 1024, 0) == \
        cf.CF_ERR_WORKSPACE_TOO_SMALL
    # plan queries need the device
    assert cf.cf_query_stitch_batchnorm_plan(8, 32)[0] == cf.CF_ERR_NO_DEVICE
    assert cf.cf_query_b2b_plan(128, 128, 512, 128, 0)[0] == cf.CF_ERR_NO_DEVICE
