"""The C-ABI library builds, loads without a GPU, exports every function that
include/sa.h declares, and rejects bad arguments on the host before any
launch (these calls never reach the GPU)."""
import ctypes
import os

import pytest

from sparse_decode_attention_head_gb300 import build_lib, sa


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sa.LIB_PATH):
        build_lib.build()
    return sa.lib()


def test_exports_every_declared_function(lib):
    names = sa.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def _prob(**kw):
    base = dict(B=2, Hq=8, Hk=2, max_pages_per_seq=64, num_pages=128, sink=4, window=64,
                block_sizes=[16, 16], k_per_head=[3] * 8, kcap=8)
    base.update(kw)
    return sa.Problem(**base)


def test_sizes_of_a_valid_problem(lib):
    p = _prob(block_sizes=[8, 32])
    assert p.block_slots() == 64 * 16 // 8
    assert p.workspace_size() > 0


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=7), sa.SA_ERR_INVALID_ARG),                  # Hq % Hk != 0
    (dict(D=64), sa.SA_ERR_INVALID_ARG),                  # D != 128
    (dict(block_sizes=[16, 12]), sa.SA_ERR_INVALID_ARG),  # Bs not in {8,16,32,64}
    (dict(window=8), sa.SA_ERR_INVALID_ARG),              # W < max Bs
    (dict(k_per_head=[-1] + [3] * 7), sa.SA_ERR_INVALID_ARG),
    (dict(k_per_head=[9] + [3] * 7), sa.SA_ERR_CAPACITY),  # k > kcap
    (dict(page_size=32), sa.SA_ERR_UNSUPPORTED),
    (dict(Hq=32, Hk=2, k_per_head=[1] * 32), sa.SA_ERR_UNSUPPORTED),  # G = 16 > 8
    (dict(kcap=0), sa.SA_ERR_INVALID_ARG),
    (dict(scale=-1.0), sa.SA_ERR_INVALID_ARG),
])
def test_host_validation_before_launch(lib, kw, code):
    p = _prob(**kw)
    assert p.workspace_size() == 0
    vp = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    rc = lib.sa_sparse_decode(p.ref, vp, vp, vp, vp, vp, vp, vp, 0, vp, vp, None, None, vp, None)
    assert rc == code
    rc = lib.sa_select_topk(p.ref, vp, vp, vp, vp, vp, None, vp, None)
    assert rc == code
    rc = lib.sa_block_summarize(p.ref, vp, vp, vp, 0, -1, vp, vp, None)
    assert rc == code


def test_null_pointers_rejected(lib):
    p = _prob()
    vp = ctypes.c_void_p(16)
    assert lib.sa_sparse_decode(p.ref, None, vp, vp, vp, vp, vp, vp, 0, vp, vp, None, None, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_sparse_decode(p.ref, vp, vp, vp, vp, vp, vp, vp, 5, vp, vp, None, None, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_score_blocks(p.ref, vp, vp, vp, None, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_block_summarize(p.ref, vp, vp, vp, -5, -1, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_lse_merge(-1, 128, vp, vp, vp, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_lse_merge(0, 128, None, None, None, None, None, None, None) == sa.SA_OK
    assert lib.sa_workspace_size(None) == 0


def test_status_strings(lib):
    for c in range(7):
        assert sa.status_string(c) not in ("", "unknown status")
    assert sa.status_string(99) == "unknown status"


def test_prepared_step_call_checks_its_tensors_once():
    """DecodeStepCall validates at construction (no GPU needed to reach the checks)."""
    import pytest
    import torch
    from sparse_decode_attention_head_gb300 import sa
    prob = sa.Problem(B=1, Hq=4, Hk=1, max_pages_per_seq=4, num_pages=4, sink=4, window=16, block_sizes=[16],
                      k_per_head=[1] * 4, kcap=1)
    cpu = torch.zeros(1, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        sa.DecodeStepCall(prob, cpu, cpu, cpu, cpu, cpu, cpu, cpu, cpu, cpu, cpu, None)


def test_group_selection_needs_one_budget_per_group():
    import ctypes
    from sparse_decode_attention_head_gb300 import sa
    ok = sa.Problem(B=1, Hq=8, Hk=2, max_pages_per_seq=16, num_pages=16, sink=4, window=64, block_sizes=[16, 16],
                    k_per_head=[3] * 4 + [5] * 4, kcap=8, selection=sa.SELECT_GROUP)
    assert sa.lib().sa_workspace_size(ok.ref) > 0
    bad = sa.Problem(B=1, Hq=8, Hk=2, max_pages_per_seq=16, num_pages=16, sink=4, window=64, block_sizes=[16, 16],
                     k_per_head=[3, 3, 3, 4, 5, 5, 5, 5], kcap=8, selection=sa.SELECT_GROUP)
    assert sa.lib().sa_workspace_size(bad.ref) == 0
    odd = sa.Problem(B=1, Hq=8, Hk=2, max_pages_per_seq=16, num_pages=16, sink=4, window=64, block_sizes=[16, 16],
                     k_per_head=[3] * 8, kcap=8, selection=7)
    assert sa.lib().sa_workspace_size(odd.ref) == 0


def test_bypass_entries_validate_before_launch(lib):
    p = _prob()
    vp = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    # eps outside [0, 1], a missing flag array, missing stats
    assert lib.sa_head_sparsity(p.ref, vp, vp, vp, vp, vp, 1.5, None, vp, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_head_sparsity(p.ref, vp, vp, vp, vp, vp, -0.1, None, vp, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_head_sparsity(p.ref, vp, vp, vp, vp, vp, 0.85, None, None, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_head_sparsity(p.ref, vp, vp, vp, vp, None, 0.85, None, vp, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_kv_stats(p.ref, vp, vp, vp, vp, None, vp, None) == sa.SA_ERR_INVALID_ARG
    step = lib.sa_decode_step_bypass
    assert step(p.ref, vp, None, None, vp, vp, vp, vp, vp, None, 0.85, vp, vp, vp, vp, None, vp, vp, None) \
        == sa.SA_ERR_INVALID_ARG                                            # no stats
    assert step(p.ref, vp, None, None, vp, vp, vp, vp, vp, vp, 0.85, vp, vp, vp, vp, None, None, vp, None) \
        == sa.SA_ERR_INVALID_ARG                                            # no flags
    assert step(p.ref, vp, None, None, vp, vp, vp, vp, vp, vp, 2.0, vp, vp, vp, vp, None, vp, vp, None) \
        == sa.SA_ERR_INVALID_ARG                                            # eps > 1
    assert step(p.ref, vp, vp, None, vp, vp, vp, vp, vp, vp, 0.85, vp, vp, vp, vp, None, vp, vp, None) \
        == sa.SA_ERR_INVALID_ARG                                            # k_new without v_new
    bad = _prob(D=64)
    assert lib.sa_kv_stats(bad.ref, vp, vp, vp, vp, vp, vp, None) == sa.SA_ERR_INVALID_ARG


def test_every_compute_call_refuses_host_tensors():
    # no CPU fallback: each call of the binding wants device tensors and says so
    import torch
    p = _prob()
    t = torch.zeros(4)
    ws = object()   # never reached
    calls = [
        lambda: sa.block_summarize(p, t, t, t, t, ws),
        lambda: sa.select_topk(p, t, t, t, t, t, ws),
        lambda: sa.sparse_decode(p, t, t, t, t, t, t, t, t, t, ws),
        lambda: sa.decode_step(p, t, t, t, t, t, t, t, t, t, t, ws),
        lambda: sa.decode_step_append(p, t, t, t, t, t, t, t, t, t, t, t, t, ws),
        lambda: sa.append_kv(p, t, t, t, t, t, t, ws),
        lambda: sa.select_tokens(p, t, t, t, t, t, t, t, t, ws),
        lambda: sa.update_score_tables(p, t, t, t, t, t, t, t, ws),
        lambda: sa.kv_stats(p, t, t, t, t, t, ws),
        lambda: sa.head_sparsity(p, t, t, t, t, t, t, t, t, ws),
        lambda: sa.decode_step_bypass(p, t, t, t, t, t, t, t, t, t, t, t, t, ws),
        lambda: sa.lse_merge(torch.zeros(2, 128), torch.zeros(2), torch.zeros(2, 128), torch.zeros(2),
                             torch.zeros(2, 128), torch.zeros(2)),
    ]
    for c in calls:
        with pytest.raises(TypeError, match="CUDA tensor"):
            c()


def test_misaligned_out_or_workspace_rejected_before_launch(lib):
    # the kernels store out and the workspace's tiles and partials 16 bytes at
    # a time: a pointer that is only 4-byte aligned is refused on the host
    # (these calls return before any launch; the pointers are never dereferenced)
    p = _prob()
    a, m = ctypes.c_void_p(256), ctypes.c_void_p(260)
    bad = sa.SA_ERR_INVALID_ARG
    assert lib.sa_sparse_decode(p.ref, a, a, a, a, a, a, a, 0, m, a, None, None, a, None) == bad   # out
    assert lib.sa_sparse_decode(p.ref, a, a, a, a, a, a, a, 0, a, a, None, None, m, None) == bad   # ws
    assert lib.sa_decode_step(p.ref, a, a, a, a, a, a, a, a, m, a, a, None) == bad                  # out
    assert lib.sa_decode_step(p.ref, a, a, a, a, a, a, a, a, a, a, m, None) == bad                  # ws
    assert lib.sa_decode_step_append(p.ref, a, a, a, a, a, a, a, a, a, a, m, a, a, None) == bad     # out
    assert lib.sa_decode_step_bypass(p.ref, a, None, None, a, a, a, a, a, a, 0.85, a, a, m, a, None, a, a,
                                     None) == bad                                                   # out
    assert lib.sa_sparse_decode_noalloc(p.ref, a, a, a, a, a, a, a, 0, m, a, None, None, None) == bad
    assert lib.sa_block_summarize(p.ref, a, a, a, 0, -1, a, m, None) == bad                         # ws
    assert lib.sa_score_blocks(p.ref, a, a, a, a, m, None) == bad                                   # ws
    assert lib.sa_select_topk(p.ref, a, a, a, a, a, None, m, None) == bad                           # ws


def test_step_plan_refuses_bad_arguments_before_capture(lib):
    # sa_step_plan_create checks like sa_decode_step and returns before capturing anything
    p = _prob()
    a, m = ctypes.c_void_p(256), ctypes.c_void_p(260)
    h = ctypes.c_void_p()
    bad = sa.SA_ERR_INVALID_ARG
    assert lib.sa_step_plan_create(p.ref, a, a, a, a, a, a, a, a, m, a, a, ctypes.byref(h)) == bad   # out
    assert lib.sa_step_plan_create(p.ref, None, a, a, a, a, a, a, a, a, a, a, ctypes.byref(h)) == bad  # q
    assert lib.sa_step_plan_create(p.ref, a, a, a, a, a, a, a, a, a, a, a, None) == bad               # plan
    assert h.value is None
    assert lib.sa_step_plan_create(_prob(D=64).ref, a, a, a, a, a, a, a, a, a, a, a, ctypes.byref(h)) == bad
    assert lib.sa_step_plan_launch(None, None) == bad
    assert lib.sa_step_plan_destroy(None) == sa.SA_OK


def test_workspace_grows_with_tile_list_windows():
    # tile lists are kept in segments of 4096 pages, with a count and room
    # for a chunk partial per (unit, window): crossing into a new window adds
    # that room, a page inside a window does not
    from sparse_decode_attention_head_gb300 import sa

    def size(mpp):
        p = sa.Problem(B=2, Hq=8, Hk=2, max_pages_per_seq=mpp, num_pages=2 * mpp, sink=4, window=64,
                       block_sizes=[16, 16], k_per_head=[8] * 8, kcap=8)
        n = sa.lib().sa_workspace_size(p.ref)
        assert n > 0
        return n

    inside = size(8192) - size(8191)   # windows 2 -> 2
    across = size(8193) - size(8192)   # windows 2 -> 3
    # 4 units x one partial of G (128 + 2) fp32 = 2080 bytes each, less alignment slack
    assert across - inside > 4 * 2080 - 2048
