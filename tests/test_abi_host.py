"""The C-ABI library on the host (no GPU): it loads, exports every entry
point include/arf.h declares, and its host logic (shape rules, planner, plan
checker, staging layout, argument checks) behaves as documented."""
import ctypes
import os
import re

import pytest

import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "arf.h")

GB300 = arf.DeviceCaps(num_sms=152, max_cluster=16, max_threads_per_sm=2048, max_smem_per_block=232448)
# the bulk kernel's static shared memory: 64 partial pointers, 2 x 16 warp
# sums, 16 mbarriers
BULK_STATIC = 8 * 64 + 2 * 16 * 4 + 8 * 16
K3_M = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048)
SHAPES = [(2, 8, 1024), (2, 128, 4096), *[(8, m, 7168) for m in K3_M], (4, 5851, 7168), (16, 585, 7168),
          (1, 1, 8), (3, 7, 8), (64, 3, 32768), (5, 1000, 1000), (17, 200, 2048),
          (3, 7, 13), (2, 5, 1001), (8, 300, 7170), (1, 2, 1)]


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    arf.load()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(arf_\w+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("arf_workspace_create", "arf_workspace_destroy", "arf_supports", "arf_run", "arf_run_planned",
              "arf_run_host", "arf_status_string", "arf_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(build.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in arf.h but not exported: {missing}"


def test_binding_covers_every_declared_symbol():
    assert sorted(_binding.exported_names()) == declared_functions()
    for n in declared_functions():
        assert callable(getattr(arf, n)), n


def header_constants():
    """Every `#define ARF_...` integer and every enumerator `ARF_... = n` of arf.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, expr in re.findall(r"#define\s+(ARF_\w+)\s+\(?([0-9u <]+)\)?\s*$", text, flags=re.M):
        out[name] = eval(expr.replace("u", ""))  # integer literals and shifts only
    for name, val in re.findall(r"\b(ARF_\w+)\s*=\s*(\d+)", text):
        out[name] = int(val)
    return out


def test_binding_constants_match_the_header():
    consts = header_constants()
    for name in ("ARF_MAX_W", "ARF_MAX_H", "ARF_MAX_H_PER_CTA", "ARF_STATIC_STAGING_BYTES", "ARF_PATH_BULK",
                 "ARF_PATH_ELEM", "ARF_ERR_DEVICE_MISMATCH"):
        assert name in consts, name
    mismatched = {n: (v, getattr(_binding, n)) for n, v in consts.items()
                  if hasattr(_binding, n) and getattr(_binding, n) != v}
    assert not mismatched, f"binding constant differs from arf.h: {mismatched}"
    missing = [n for n in consts if n.startswith(("ARF_PATH_", "ARF_MAX_")) and not hasattr(_binding, n)]
    assert not missing, missing


def test_compiled_rank_counts_match_the_library():
    """arf_plan_check accepts a plan with the rank count compiled in exactly
    for the rank counts COMPILED_W lists."""
    accepted = []
    for W in range(1, arf.ARF_MAX_W + 1):
        p = arf.Plan(path=arf.ARF_PATH_FLAT, threads=128, vpt=1, cluster=1, grid=7, w_spec=W, stages=0)
        if arf.arf_plan_check(GB300, p, arf.ARF_ALLREDUCE, W, 1, 7168, arf.ARF_BF16) == arf.ARF_OK:
            accepted.append(W)
    assert tuple(accepted) == arf.COMPILED_W


def test_static_staging_size_is_the_headers():
    """The library reports the staging size arf.h declares, and the binding's
    copy of the constant agrees with both."""
    assert arf.arf_static_staging_bytes() == header_constants()["ARF_STATIC_STAGING_BYTES"]
    assert arf.arf_static_staging_bytes() == _binding.ARF_STATIC_STAGING_BYTES


def test_read_pass_argument_errors():
    """arf_read_pass checks its arguments before touching a device."""
    assert arf.arf_read_pass(None, 256, 1024, None) == arf.ARF_ERR_INVALID_ARG


def test_wait_timeouts_argument_errors():
    """No workspace or no output: INVALID_ARG, without touching a device."""
    n = ctypes.c_uint(7)
    assert arf.arf_workspace_wait_timeouts(None, n) == arf.ARF_ERR_INVALID_ARG
    assert n.value == 7
    assert arf.load().arf_workspace_wait_timeouts(None, None) == arf.ARF_ERR_INVALID_ARG


def test_status_strings():
    for s in range(5):
        assert arf.arf_status_string(s)
    assert arf.arf_status_string(99) == "unknown status"


@pytest.mark.parametrize("pattern", [arf.ARF_ALLREDUCE, arf.ARF_AR_RESIDUAL_RMSNORM])
def test_supports_rules(pattern):
    S = arf.arf_supports
    bf = arf.ARF_BF16
    assert S(None, pattern, 8, 2048, 7168, bf) == arf.ARF_OK
    assert S(None, pattern, 1, 0, 8, arf.ARF_FP16) == arf.ARF_OK
    assert S(None, pattern, 64, 1, 32768, bf) == arf.ARF_OK
    assert S(None, pattern, 8, 3, 65536, bf) == arf.ARF_OK
    assert S(None, pattern, 0, 1, 8, bf) == arf.ARF_ERR_UNSUPPORTED
    assert S(None, pattern, 65, 1, 8, bf) == arf.ARF_ERR_UNSUPPORTED
    assert S(None, pattern, 2, 1, 12, bf) == arf.ARF_OK                   # H % 8 != 0: elementwise path
    assert S(None, pattern, 2, 1, 1, bf) == arf.ARF_OK
    assert S(None, pattern, 2, 1, 524296, bf) == arf.ARF_ERR_UNSUPPORTED  # H > max
    assert S(None, pattern, 2, 1, 0, bf) == arf.ARF_ERR_INVALID_ARG
    assert S(None, pattern, 2, -1, 8, bf) == arf.ARF_ERR_INVALID_ARG
    assert S(None, pattern, 2, 1, 8, 7) == arf.ARF_ERR_INVALID_ARG
    assert S(None, 9, 2, 1, 8, bf) == arf.ARF_ERR_INVALID_ARG


@pytest.mark.parametrize("pattern", [arf.ARF_ALLREDUCE, arf.ARF_AR_RESIDUAL_RMSNORM])
@pytest.mark.parametrize("W,M,H", SHAPES)
def test_planner_plans_are_legal(pattern, W, M, H):
    for caps in (GB300, arf.DeviceCaps(148, 8, 2048, 232448), arf.DeviceCaps(132, 1, 2048, 101376),
                 arf.DeviceCaps(1, 1, 1024, 49152)):
        p = arf.Plan()
        assert arf.arf_plan_rules(caps, pattern, W, M, H, arf.ARF_BF16, p) == arf.ARF_OK
        assert arf.arf_plan_check(caps, p, pattern, W, M, H, arf.ARF_BF16) == arf.ARF_OK, p
        assert p.grid % p.cluster == 0 and p.threads % 32 == 0
        assert p.w_spec in (0, W)
        per_sm = caps.max_threads_per_sm // p.threads
        if H % 8:
            assert p.path == arf.ARF_PATH_ELEM and p.w_spec == 0 and p.cluster == 1 and p.stages == 0
            continue
        if p.path == arf.ARF_PATH_ASYNC:
            # many rows, compile-time W: one streaming CTA per SM, ring of >= 3 blocks in shared memory
            assert M >= caps.num_sms and W in arf.COMPILED_W and p.grid == caps.num_sms
            ring = p.stages * (W + 1) * 256 * 16 + (H // 8) * 16
            assert 3 <= p.stages <= 8 and ring + 1024 <= caps.max_smem_per_block
            continue
        C = H // 8
        # the row kernel's chunks per thread, and whether it would prefetch
        vpt = 1
        while vpt < 8 and -(-C // vpt) > 512:
            vpt *= 2
        prefetch = W in arf.COMPILED_W and vpt * (W + 1) <= 18
        if p.path == arf.ARF_PATH_BULK:
            # one CTA per row would run without the register prefetch: the bulk ring instead
            assert pattern == arf.ARF_AR_RESIDUAL_RMSNORM and W <= 12 and not prefetch and C <= 4096
            assert not (M < 16 and C >= 512 and caps.max_cluster > 1)  # decode-size wide rows split instead
            assert p.cluster == 1 and p.vpt == 1 and p.threads in (64, 128, 256, 512)
            assert p.threads == min(512, -(-C // 32) * 32) or p.threads < 512
            per_sm = caps.max_smem_per_block + 1024

            def fits(per, stages):
                need = stages * (W + 1) * p.threads * 16 + C * 16 + BULK_STATIC
                room = per_sm // per - 1024 if per > 1 else caps.max_smem_per_block
                return need <= room and per * p.threads <= caps.max_threads_per_sm

            per = max(k for k in (1, 2, 3, 4) if fits(k, 2))  # the most CTAs per SM with 2 slots
            assert p.stages == 2 if per > 1 else (2 <= p.stages <= 4 and fits(1, p.stages))
            assert p.grid == max(1, min(M, caps.num_sms * per))
            continue
        assert p.stages == 0
        if pattern == arf.ARF_ALLREDUCE:
            assert p.path == arf.ARF_PATH_FLAT and p.cluster == 1
            chunks = M * H // 8
            assert p.grid == max(1, -(-chunks // (p.threads * p.vpt)))  # one pass, no grid-stride trips
        else:
            C = H // 8
            assert p.threads * p.vpt * p.cluster >= C
            if p.path == arf.ARF_PATH_CLUSTER:
                # only decode-size batches of few, wide rows split a row
                assert M < 16 and C >= 512 and p.vpt == 1
                assert 2 <= p.cluster <= min(8, caps.max_cluster)
                assert p.grid == p.cluster * min(M, max(1, caps.num_sms * per_sm // p.cluster))
            elif p.vpt == 2 and W in (2, 4) and p.w_spec == W:
                assert p.cluster == 1 and p.grid == M  # one CTA per row: the kernel's one-row form
            else:
                assert p.cluster == 1 and p.grid == max(1, min(M, caps.num_sms * per_sm))


def test_planner_uses_the_sm_count():
    """Few wide rows spread over several SMs; large M fills the device."""
    p = arf.Plan()
    arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 8, 1, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_CLUSTER and p.cluster == 8 and p.threads == 128
    arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 8, 128, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_ROW and (p.threads, p.vpt, p.grid) == (448, 2, 128)
    arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 8, 2048, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_ROW and (p.threads, p.vpt) == (448, 2) and p.grid % 152 == 0
    arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 4, 5851, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_ROW and p.vpt * (4 + 1) <= 18 and p.grid == 5851  # one CTA per row
    arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_ROW and (p.threads, p.vpt) == (448, 2)  # 896 chunks > 512 threads
    no_cluster = arf.DeviceCaps(152, 1, 2048, 232448)
    arf.arf_plan_rules(no_cluster, arf.ARF_AR_RESIDUAL_RMSNORM, 8, 1, 7168, arf.ARF_BF16, p)
    assert p.path == arf.ARF_PATH_ROW and p.grid == 1


@pytest.mark.parametrize("H", [32776, 65536, 131072, 262144, 524288])
@pytest.mark.parametrize("M", [1, 7, 300])
def test_long_rows_split_over_clusters(H, M):
    """Rows longer than one CTA holds: kARResidualRMSNorm splits them over a
    cluster (up to 16 CTAs), or, with rows for half the SMs, streams them
    through the bulk ring where its row buffer fits; kAllReduce is flat and
    takes any H <= ARF_MAX_H."""
    p = arf.Plan()
    bulk = 2 * M >= 152 and (H // 8) * 16 + BULK_STATIC + 2 * 9 * 256 * 16 <= 232448
    assert arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, 8, M, H, arf.ARF_BF16, p) == arf.ARF_OK
    if bulk:
        assert p.path == arf.ARF_PATH_BULK and p.threads <= 512
    else:
        assert p.path == arf.ARF_PATH_CLUSTER and p.threads <= 512
        assert p.threads * p.vpt * p.cluster >= H // 8
    assert arf.arf_plan_check(GB300, p, arf.ARF_AR_RESIDUAL_RMSNORM, 8, M, H, arf.ARF_BF16) == arf.ARF_OK
    assert arf.arf_plan_rules(GB300, arf.ARF_ALLREDUCE, 8, M, H, arf.ARF_BF16, p) == arf.ARF_OK
    # a device with 4-CTA clusters holds rows up to 4 x 32768; longer rows
    # take the elementwise kernel
    small = arf.DeviceCaps(152, 4, 2048, 232448)
    assert arf.arf_plan_rules(small, arf.ARF_AR_RESIDUAL_RMSNORM, 8, M, H, arf.ARF_BF16, p) == arf.ARF_OK
    if H > 4 * 32768:
        assert p.path == arf.ARF_PATH_ELEM
    else:
        assert p.path == (arf.ARF_PATH_BULK if bulk else arf.ARF_PATH_CLUSTER)


def test_elementwise_rmsnorm_plan_shape():
    """Rows with H % 8 != 0: one wide CTA per row while rows are few; from
    3 x SMs rows 256-thread CTAs (at most four per SM), from 7 x SMs
    128-thread CTAs (at most eight per SM)."""
    p = arf.Plan()
    for W, M, H in ((2, 4096, 4098), (4, 2048, 7170), (8, 608, 7175), (3, 128, 4097), (2, 455, 4098),
                    (2, 456, 4098), (8, 1063, 7175), (8, 1064, 7175), (3, 5000, 1001)):
        assert arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16, p) == arf.ARF_OK
        assert p.path == arf.ARF_PATH_ELEM
        if M >= 7 * 152 and H >= 1024:
            assert p.threads == 128 and p.grid == min(M, 8 * 152), (W, M, H, p)
        elif M >= 3 * 152 and H >= 1024:
            assert p.threads == 256 and p.grid == min(M, 4 * 152), (W, M, H, p)
        else:
            assert p.threads == min(512, -(-H // 32) * 32) and p.grid == min(M, 152 * (2048 // p.threads)), (W, M, H, p)
        assert arf.arf_plan_check(GB300, p, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16) == arf.ARF_OK


def test_long_rows_take_the_bulk_ring_when_rows_are_many():
    """Rows of more than 4096 chunks: a cluster per row for fewer rows than
    half the SMs, the bulk ring from there while its row buffer fits."""
    p = arf.Plan()
    for W, M, H in ((2, 16, 32776), (2, 76, 32776), (2, 2048, 32776), (8, 608, 32776), (4, 64, 65536),
                    (4, 152, 65536), (12, 300, 40000), (13, 300, 40000), (2, 500, 131072), (8, 500, 78976),
                    (8, 500, 78984), (8, 500, 106496), (2, 1024, 32776)):
        assert arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16, p) == arf.ARF_OK
        assert arf.arf_plan_check(GB300, p, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16) == arf.ARF_OK
        fits = (H // 8) * 16 + BULK_STATIC + 2 * (W + 1) * 256 * 16 <= 232448  # blocks of >= 256 chunks
        if 2 * M >= 152 and W <= 12 and fits:
            assert p.path == arf.ARF_PATH_BULK, (W, M, H, p)
            if (W, H) == (2, 32776):  # 114 704 B of ring and row buffer: two CTAs per SM, 2 slots
                assert p.threads == 512 and p.stages == 2 and p.grid == min(M, 304), p
        else:
            assert p.path == arf.ARF_PATH_CLUSTER, (W, M, H, p)


def test_long_row_limits():
    S = arf.arf_supports
    assert S(None, arf.ARF_ALLREDUCE, 2, 1, 524288, arf.ARF_BF16) == arf.ARF_OK
    assert S(None, arf.ARF_AR_RESIDUAL_RMSNORM, 2, 1, 524288, arf.ARF_BF16) == arf.ARF_OK
    assert S(None, arf.ARF_ALLREDUCE, 2, 1, 524296, arf.ARF_BF16) == arf.ARF_ERR_UNSUPPORTED
    no_cluster = arf.DeviceCaps(152, 1, 2048, 232448)
    p = arf.Plan()
    assert arf.arf_plan_rules(no_cluster, arf.ARF_AR_RESIDUAL_RMSNORM, 2, 1, 32776, arf.ARF_BF16, p) == arf.ARF_OK
    assert p.path == arf.ARF_PATH_ELEM and p.threads == 512
    assert arf.arf_plan_rules(no_cluster, arf.ARF_ALLREDUCE, 2, 1, 524288, arf.ARF_BF16, p) == arf.ARF_OK


def test_plan_check_rejects_bad_plans():
    good = arf.Plan()
    args = (arf.ARF_AR_RESIDUAL_RMSNORM, 8, 64, 7168, arf.ARF_BF16)
    assert arf.arf_plan_rules(GB300, *args, good) == arf.ARF_OK

    def with_(**kw):
        p = arf.Plan(**good.as_dict())
        for k, v in kw.items():
            setattr(p, k, v)
        return arf.arf_plan_check(GB300, p, *args)

    assert with_() == arf.ARF_OK
    assert with_(threads=48) == arf.ARF_ERR_UNSUPPORTED
    assert with_(threads=1024) == arf.ARF_ERR_UNSUPPORTED
    assert with_(vpt=3) == arf.ARF_ERR_UNSUPPORTED
    assert with_(w_spec=4) == arf.ARF_ERR_UNSUPPORTED
    assert with_(path=arf.ARF_PATH_FLAT) == arf.ARF_ERR_UNSUPPORTED
    assert with_(path=arf.ARF_PATH_CLUSTER, cluster=32, grid=64) == arf.ARF_ERR_UNSUPPORTED
    assert with_(path=arf.ARF_PATH_CLUSTER, cluster=4, grid=6) == arf.ARF_ERR_UNSUPPORTED
    assert with_(path=arf.ARF_PATH_ROW, cluster=1, threads=32, vpt=1) == arf.ARF_ERR_UNSUPPORTED  # 896 chunks
    elem = arf.Plan(path=arf.ARF_PATH_ELEM, threads=256, vpt=1, cluster=1, grid=9, w_spec=0)
    assert arf.arf_plan_check(GB300, elem, *args) == arf.ARF_OK
    assert arf.arf_plan_check(GB300, elem, arf.ARF_AR_RESIDUAL_RMSNORM, 3, 5, 13, arf.ARF_BF16) == arf.ARF_OK
    elem.w_spec = 8
    assert arf.arf_plan_check(GB300, elem, *args) == arf.ARF_ERR_UNSUPPORTED
    row13 = arf.Plan(path=arf.ARF_PATH_ROW, threads=32, vpt=1, cluster=1, grid=5, w_spec=3)
    assert arf.arf_plan_check(GB300, row13, arf.ARF_AR_RESIDUAL_RMSNORM, 3, 5, 13, arf.ARF_BF16) == \
        arf.ARF_ERR_UNSUPPORTED  # 16-byte kernels need H % 8 == 0
    small = arf.DeviceCaps(152, 4, 2048, 232448)
    p = arf.Plan(path=arf.ARF_PATH_CLUSTER, threads=64, vpt=1, cluster=16, grid=16, w_spec=8)
    assert arf.arf_plan_check(small, p, *args) == arf.ARF_ERR_UNSUPPORTED
    flat = arf.Plan(path=arf.ARF_PATH_FLAT, threads=256, vpt=4, cluster=1, grid=10, w_spec=16)
    assert arf.arf_plan_check(GB300, flat, arf.ARF_ALLREDUCE, 16, 4, 64, arf.ARF_BF16) == arf.ARF_ERR_UNSUPPORTED
    flat.vpt = 1
    assert arf.arf_plan_check(GB300, flat, arf.ARF_ALLREDUCE, 16, 4, 64, arf.ARF_BF16) == arf.ARF_OK
    flat.stages = 2
    assert arf.arf_plan_check(GB300, flat, arf.ARF_ALLREDUCE, 16, 4, 64, arf.ARF_BF16) == arf.ARF_ERR_UNSUPPORTED
    a = arf.Plan(path=arf.ARF_PATH_ASYNC, threads=256, vpt=1, cluster=1, grid=152, w_spec=16, stages=3)
    rms16 = (arf.ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7168, arf.ARF_FP16)
    assert arf.arf_plan_check(GB300, a, *rms16) == arf.ARF_OK
    a.stages = 4  # 4 x 17 x 4 KiB does not fit next to the row buffer
    assert arf.arf_plan_check(GB300, a, *rms16) == arf.ARF_ERR_UNSUPPORTED
    a.stages, a.threads = 3, 128
    assert arf.arf_plan_check(GB300, a, *rms16) == arf.ARF_ERR_UNSUPPORTED
    a.threads, a.w_spec = 256, 0
    assert arf.arf_plan_check(GB300, a, *rms16) == arf.ARF_ERR_UNSUPPORTED
    a.w_spec = 16
    assert arf.arf_plan_check(GB300, a, arf.ARF_ALLREDUCE, 16, 585, 7168, arf.ARF_FP16) == arf.ARF_ERR_UNSUPPORTED


def test_bulk_plan_rules():
    """ARF_PATH_BULK: no cluster, vpt 1, 2..16 ring slots, and (W+1) x slots x
    threads x 16 bytes of ring plus the 16-byte row buffer (kAllReduce: W x
    slots x threads x 16 bytes) must fit the opt-in shared memory with the
    kernel's static arrays."""
    rms16 = (arf.ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7168, arf.ARF_FP16)

    def check(caps=GB300, args=rms16, **kw):
        p = arf.Plan(path=arf.ARF_PATH_BULK, threads=128, vpt=1, cluster=1, grid=152, w_spec=16, stages=6)
        for k, v in kw.items():
            setattr(p, k, v)
        return arf.arf_plan_check(caps, p, *args)

    assert check() == arf.ARF_OK
    assert check(w_spec=0) == arf.ARF_OK
    assert check(w_spec=8) == arf.ARF_ERR_UNSUPPORTED
    assert check(stages=1) == arf.ARF_ERR_UNSUPPORTED
    assert check(stages=17) == arf.ARF_ERR_UNSUPPORTED
    assert check(vpt=2) == arf.ARF_ERR_UNSUPPORTED
    assert check(cluster=2, grid=304) == arf.ARF_ERR_UNSUPPORTED
    # kAllReduce form: partials only, no row buffer: 16 x S x 128 x 16 + 768 <= 232448  <=>  S <= 7
    ar16 = (arf.ARF_ALLREDUCE, 16, 585, 7168, arf.ARF_FP16)
    assert check(args=ar16, stages=7) == arf.ARF_OK
    assert check(args=ar16, stages=8) == arf.ARF_ERR_UNSUPPORTED
    assert check(args=(arf.ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7170, arf.ARF_FP16)) == arf.ARF_ERR_UNSUPPORTED
    # shared memory: 17 x S x 128 x 16 + 896 x 16 + 768 <= 232448  <=>  S <= 6
    ring = lambda s, t=128, w=16, c=896: (w + 1) * s * t * 16 + c * 16 + BULK_STATIC  # noqa: E731
    assert ring(6) <= GB300.max_smem_per_block < ring(7)
    assert check(stages=7) == arf.ARF_ERR_UNSUPPORTED
    assert check(threads=64, stages=12) == arf.ARF_OK and ring(12, 64) <= 232448 < ring(13, 64)
    assert check(threads=64, stages=13) == arf.ARF_ERR_UNSUPPORTED
    tight = arf.DeviceCaps(152, 16, 2048, ring(6))
    assert check(caps=tight) == arf.ARF_OK
    tight.max_smem_per_block -= 16
    assert check(caps=tight) == arf.ARF_ERR_UNSUPPORTED
    # the row buffer alone: H = 32768 leaves room for fewer slots
    long_rows = (arf.ARF_AR_RESIDUAL_RMSNORM, 2, 4, 32768, arf.ARF_BF16)
    assert check(args=long_rows, w_spec=2, threads=512, stages=6) == arf.ARF_OK
    assert check(args=long_rows, w_spec=2, threads=512, stages=7) == arf.ARF_ERR_UNSUPPORTED


def test_staging_bytes():
    M, H, W = 128, 4096, 2
    plane = M * H * 2
    ar = arf.arf_host_staging_bytes(arf.ARF_ALLREDUCE, W, M, H, arf.ARF_BF16)
    rms = arf.arf_host_staging_bytes(arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16)
    assert ar == 256 + (W + 1) * plane
    assert rms == 256 + (W + 3) * plane + 8192
    assert arf.arf_host_staging_bytes(arf.ARF_ALLREDUCE, 0, M, H, arf.ARF_BF16) == 0


def test_calls_without_a_workspace_are_rejected():
    assert arf.arf_run(None, 0, 2, None, None, None, 0.0, None, None, 1, 8, 0, None) == arf.ARF_ERR_INVALID_ARG
    assert arf.arf_workspace_destroy(None) == arf.ARF_OK
    assert arf.arf_last_cuda_error(None) == 0
    c = arf.DeviceCaps()
    assert arf.arf_workspace_caps(None, c) == arf.ARF_ERR_INVALID_ARG


def test_workspace_create_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert arf.arf_workspace_create(0, h) == arf.ARF_ERR_CUDA
    assert not h.value


def test_planner_bulk_choices():
    """The bulk ring replaces one-CTA-per-row plans that would run without
    the register prefetch, for up to 12 ranks; prefetching shapes, decode-size
    wide rows (cluster path) and wider rank counts keep their kernels."""
    def plan(W, M, H):
        p = arf.Plan()
        assert arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_BF16, p) == arf.ARF_OK
        return p

    p = plan(3, 2000, 7168)  # rank count not compiled in: 2 x 4 x 8 KiB slots, 2 CTAs per SM
    assert (p.path, p.threads, p.grid, p.w_spec, p.stages) == (arf.ARF_PATH_BULK, 512, 304, 0, 2)
    p = plan(12, 585, 7168)  # 13 x 8 KiB slots: one CTA per SM
    assert (p.path, p.threads, p.grid, p.stages) == (arf.ARF_PATH_BULK, 512, 152, 2)
    p = plan(4, 512, 32768)  # 8 chunks per thread in the row kernel
    assert (p.path, p.threads, p.grid, p.stages, p.w_spec) == (arf.ARF_PATH_BULK, 512, 152, 4, 4)
    for W, M, H, path in ((8, 1024, 7168, arf.ARF_PATH_ROW), (4, 1989, 7168, arf.ARF_PATH_ROW),
                          (16, 585, 7168, arf.ARF_PATH_ROW), (24, 400, 7168, arf.ARF_PATH_ROW),
                          (3, 4, 7168, arf.ARF_PATH_CLUSTER), (2, 128, 4096, arf.ARF_PATH_ROW)):
        assert plan(W, M, H).path == path, (W, M, H)
    # fp16 rows of two chunks per thread: W = 2 and 4 take one CTA per row (the
    # one-row form has no fp16 penalty); W = 1 with many rows takes the bulk ring
    for W, M, H, path, grid in ((2, 3315, 7168, arf.ARF_PATH_ROW, 3315), (4, 5851, 7168, arf.ARF_PATH_ROW, 5851),
                                (1, 4972, 7168, arf.ARF_PATH_BULK, None), (1, 200, 7168, arf.ARF_PATH_ROW, None),
                                (8, 1024, 7168, arf.ARF_PATH_ROW, None), (2, 128, 7168, arf.ARF_PATH_ROW, 128),
                                (2, 8192, 4096, arf.ARF_PATH_ROW, None), (4, 304, 7168, arf.ARF_PATH_ROW, 304)):
        p = arf.Plan()
        assert arf.arf_plan_rules(GB300, arf.ARF_AR_RESIDUAL_RMSNORM, W, M, H, arf.ARF_FP16, p) == arf.ARF_OK
        assert p.path == path, (W, M, H)
        if grid is not None:
            assert p.grid == grid, (W, M, H, p)


def test_workload_tables_agree_with_the_planner():
    """Every extra workload names the kernel path it exists to reach, and the
    planner (on GB300's capabilities) sends each of its patterns there; the
    benchmark can name the kernel of every plan any workload gets."""
    import os
    import sys
    from all_reduce_residual_gb300 import workloads as wl
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert set(wl.EXTRA_PATHS) == set(wl.EXTRA_WORKLOADS)
    want = {"bulk": arf.ARF_PATH_BULK, "elem": arf.ARF_PATH_ELEM, "row, one CTA per row": arf.ARF_PATH_ROW,
            "row": arf.ARF_PATH_ROW, "flat": arf.ARF_PATH_FLAT, "cluster": arf.ARF_PATH_CLUSTER}
    for name, w in {**wl.WORKLOADS, **wl.EXTRA_WORKLOADS}.items():
        dt = arf.ARF_BF16 if w.dtype == "bf16" else arf.ARF_FP16
        for pat in w.patterns:
            p = arf.Plan()
            assert arf.arf_plan_for_caps(GB300, arf.pattern_code(pat), w.W, w.M, w.H, dt, p) == arf.ARF_OK
            table = bench.KERNEL_OF_PATH if pat == "rmsnorm" else bench.AR_KERNEL_OF_PATH
            assert p.path in table, (name, pat, p)
            if name in wl.EXTRA_PATHS:
                assert p.path == want[wl.extra_path(name, pat)], (name, pat, p)
                if wl.extra_path(name, pat) == "row, one CTA per row":
                    assert p.grid == w.M, (name, pat, p)
