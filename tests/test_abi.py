"""The C ABI library builds, loads and exports every declared symbol (CPU only:
no call below reaches the GPU; argument errors are returned before any CUDA
call is made)."""

import ctypes
import os
import re

import pytest

import muon_newton_schulz_expert_gb300 as mk
from muon_newton_schulz_expert_gb300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "muon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    mkbuild.build()
    return mk.lib()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("muon_momentum_update", "muon_ns_batched", "muon_apply_update"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert set(names) == set(mk.SIGNATURES), set(names) ^ set(mk.SIGNATURES)
    raw = ctypes.CDLL(mkbuild.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_library_is_built_for_sm103a_only():
    assert mkbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code, name in mk.STATUS_NAMES.items():
        assert mk.muon_status_string(code) == name
    assert mk.muon_status_string(-99) == "MUON_ERR_UNKNOWN"


def test_default_scale_host_function(lib):
    assert abs(mk.muon_default_scale(6144, 1792) - 1.8516402) < 1e-6
    assert mk.muon_default_scale(1792, 6144) == 1.0
    assert mk.muon_default_scale(0, 5) == 1.0


def test_argument_errors_are_returned_without_touching_the_gpu(lib):
    c3 = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    # negative sizes, null pointers, bad eps, null coefficients
    assert lib.muon_ns_batched(None, 1, 8, 8, 5, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched(None, -1, 8, 8, 5, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 0, 8, 5, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 8, 8, -1, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 8, 8, 5, None, 1e-7, None) == -1
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 8, 8, 5, c3, -1.0, None) == -1
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 8, 8, 5, c3, float("nan"), None) == -1
    bad = (ctypes.c_float * 3)(float("inf"), 0, 0)
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 8, 8, 5, bad, 1e-7, None) == -1
    # shapes and alignment the tensor-core path does not take
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 12, 16, 5, c3, 1e-7, None) == -2
    assert lib.muon_ns_batched(ctypes.c_void_p(258), 1, 16, 16, 5, c3, 1e-7, None) == -2
    assert lib.muon_ns_batched(ctypes.c_void_p(256), 1, 1 << 21, 8, 5, c3, 1e-7, None) == -2
    # batch 0 is a no-op even with a null pointer
    assert lib.muon_ns_batched(None, 0, 8, 8, 5, c3, 1e-7, None) == 0
    assert lib.muon_ns_batched_f32(None, 0, 3, 5, 5, c3, 1e-7, None) == 0
    # workspace checks of the _ws variant (alignment, size)
    need = lib.muon_ns_workspace_bytes(2, 64, 128)
    assert need > 2 * 2 * 64 * 128 * 2
    assert lib.muon_ns_batched_ws(ctypes.c_void_p(256), 2, 64, 128, 5, c3, 1e-7, ctypes.c_void_p(4096 + 16), need,
                                  None) == -1
    assert lib.muon_ns_batched_ws(ctypes.c_void_p(256), 2, 64, 128, 5, c3, 1e-7, ctypes.c_void_p(4096), need - 1,
                                  None) == -4
    # elementwise calls
    assert lib.muon_momentum_update(None, None, None, -1, 0.9, 1, None) == -1
    assert lib.muon_momentum_update(None, None, None, 10, 0.9, 1, None) == -1
    assert lib.muon_momentum_update(None, None, None, 0, 0.9, 1, None) == 0
    assert lib.muon_apply_update(None, None, 1, 4, -4, 0.02, 0.1, 0.0, None) == -1
    assert lib.muon_apply_update(None, None, 1, 4, 4, 0.02, 0.1, 0.0, None) == -1
    assert lib.muon_apply_update(None, None, 0, 4, 4, 0.02, 0.1, 0.0, None) == 0
    assert lib.muon_selftest_wait_timeout(0, None) == -1


def test_workspace_size_formula(lib):
    # X buffers, A and B, plus small per-matrix scalars; orientation-free
    b, m, n = 96, 1792, 6144
    got = lib.muon_ns_workspace_bytes(b, m, n)
    core = 2 * b * m * n * 2 + b * m * n + 2 * b * m * m * 2   # X ping-pong, X's 8-bit low half, A, B
    assert core <= got <= core + 64 * 1024
    assert lib.muon_ns_workspace_bytes(b, n, m) == got
    assert lib.muon_ns_workspace_bytes(0, m, n) == 0
    core32 = 2 * b * m * n * 4 + 2 * b * m * m * 4     # fp32: X ping-pong, A, B
    assert core32 <= lib.muon_ns_workspace_bytes_f32(b, m, n) <= core32 + 64 * 1024


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(mk, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(mk, "_lib", None)
    with pytest.raises(mk.MuonLibraryMissing):
        mk.lib()


def test_newer_entry_points_reject_bad_arguments_on_the_host(lib):
    c3 = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    # schedules: every coefficient checked, steps bounded
    sched = (ctypes.c_float * 6)(3.4445, -4.775, 2.0315, float("nan"), 0, 0)
    assert lib.muon_ns_batched_schedule(ctypes.c_void_p(256), 1, 8, 8, 2, sched, 1e-7, None) == -1
    assert lib.muon_ns_batched_schedule(ctypes.c_void_p(256), 1, 12, 8, 1, sched, 1e-7, None) == -2
    assert lib.muon_ns_batched_schedule(None, 0, 8, 8, 2, sched, 1e-7, None) == -1
    assert lib.muon_ns_batched_schedule(ctypes.c_void_p(256), 1, 8, 8, 1001, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched_schedule_f32(None, 0, 3, 5, 1, c3, 1e-7, None) == 0
    # AdamW: step >= 1, betas in [0, 1)
    assert lib.muon_adamw_update(None, None, None, None, 0, 1e-3, 0.9, 0.95, 1e-8, 0.1, 0, None) == -1
    assert lib.muon_adamw_update(None, None, None, None, 0, 1e-3, 1.0, 0.95, 1e-8, 0.1, 1, None) == -1
    assert lib.muon_adamw_update(None, None, None, None, 0, 1e-3, 0.9, 0.95, -1.0, 0.1, 1, None) == -1
    assert lib.muon_adamw_update(None, None, None, None, 0, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, None) == 0
    assert lib.muon_adamw_update(None, None, None, None, 16, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, None) == -1
    assert lib.muon_adamw_update_f32(None, None, None, None, -1, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, None) == -1
    # host-resident step: sizes, null pointers, shapes
    assert lib.muon_step_host(None, None, None, 0, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, 0, None) == 0
    assert lib.muon_step_host(None, None, None, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, 0, None) == -1
    assert lib.muon_step_host(None, None, None, -1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, 0, None) == -1
    assert lib.muon_step_host(None, None, None, 1, 8, 8, 0.95, 1, 5, None, 1e-7, 0.02, 0.1, 0.0, 0, None) == -1
    # fused device step: sizes, null pointers, shapes, alignment, workspace
    P = ctypes.c_void_p(256)
    assert lib.muon_step_batched(None, None, None, 0, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == 0
    assert lib.muon_step_batched(None, P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -1
    assert lib.muon_step_batched(P, None, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -1
    assert lib.muon_step_batched(P, P, None, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -1
    assert lib.muon_step_batched(P, P, P, 1, 12, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -2
    assert lib.muon_step_batched(ctypes.c_void_p(264), P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0,
                                 None, 0, None) == -2
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, 0.95, 1, 5, None, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -1
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, float("nan"), 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                 None) == -1
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, float("inf"), 0.1, 0.0, None, 0,
                                 None) == -1
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, 0.95, 1, -1, c3, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -1
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, ctypes.c_void_p(272),
                                 1 << 20, None) == -1      # workspace not 256-byte aligned
    assert lib.muon_step_batched(P, P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, P, 64, None) == -4
    sched2 = (ctypes.c_float * 6)(3.4445, -4.775, 2.0315, 3.0, -3.2, 1.2)
    assert lib.muon_step_batched_schedule(None, None, None, 0, 8, 8, 0.95, 1, 2, sched2, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                          None) == 0
    assert lib.muon_step_batched_schedule(P, P, P, 1, 8, 8, 0.95, 1, 2, None, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                          None) == -1
    assert lib.muon_step_batched_schedule(P, P, P, 1, 8, 8, 0.95, 1, 2, sched, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                          None) == -1      # a NaN coefficient in step 2
    assert lib.muon_step_batched_schedule(P, P, P, 1, 12, 8, 0.95, 1, 2, sched2, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                          None) == -2
    assert lib.muon_step_batched_schedule(P, P, P, 1, 8, 8, 0.95, 1, 2, sched2, 1e-7, 0.02, 0.1, 0.0, P, 64,
                                          None) == -4
    # the same checks, before any CUDA call, with a parameter-free event (any handle; it is not touched)
    E = ctypes.c_void_p(512)
    assert lib.muon_step_batched_after(None, None, None, 0, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                       E, None) == 0
    assert lib.muon_step_batched_after(P, None, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                       E, None) == -1
    assert lib.muon_step_batched_after(P, P, P, 1, 8, 12, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                       E, None) == -2
    assert lib.muon_step_batched_after(P, P, P, 1, 8, 8, 0.95, 1, 5, None, 1e-7, 0.02, 0.1, 0.0, None, 0,
                                       E, None) == -1
    assert lib.muon_step_batched_after(P, P, P, 1, 8, 8, 0.95, 1, 5, c3, 1e-7, 0.02, 0.1, 0.0, P, 64,
                                       E, None) == -4
    assert lib.muon_step_workspace_bytes(96, 6144, 1792) == lib.muon_ns_workspace_bytes(96, 1792, 6144)
    assert lib.muon_step_workspace_bytes(0, 8, 8) == 0


def test_trace_without_gpu_work_is_empty(lib):
    assert lib.muon_trace_begin() == 0
    entries = (mk.TraceEntry * 4)()
    assert lib.muon_trace_end(entries, 4) == 0


def test_static_entry_reports_the_errors_of_muon_ns_batched_first(lib):
    # argument and shape errors come before the size limit, as in muon_ns_batched;
    # none of these calls reaches the GPU
    c3 = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    P = ctypes.c_void_p(256)
    big = 1024   # 1024 expert-sized matrices: far over the static scratch
    assert lib.muon_ns_workspace_bytes(big, 1792, 6144) > mk.NS_STATIC_SCRATCH_BYTES
    assert lib.muon_ns_batched_static(P, big, 1792, 6144, 5, c3, float("nan"), None) == -1
    assert lib.muon_ns_batched_static(P, big, 1792, 6144, 1001, c3, 1e-7, None) == -1
    assert lib.muon_ns_batched_static(P, big, 1792, 6144, 5, None, 1e-7, None) == -1
    assert lib.muon_ns_batched_static(P, big, 7, 6144, 5, c3, 1e-7, None) == -2
    assert lib.muon_ns_batched_static(ctypes.c_void_p(258), big, 1792, 6144, 5, c3, 1e-7, None) == -2
    assert lib.muon_ns_batched_static(P, big, 1792, 6144, 5, c3, 1e-7, None) == -4
    assert lib.muon_ns_batched_static(None, 0, 1792, 6144, 5, c3, 1e-7, None) == 0
    assert lib.muon_ns_batched_static(None, -1, 1792, 6144, 5, c3, 1e-7, None) == -1


def test_coefficients_whose_iterates_leave_the_scaled_fp16_range_are_unsupported(lib):
    # X grows by up to 1e6 per step: after a few steps no power-of-two scale keeps
    # its bound inside fp16, so the tensor-core path refuses before any launch
    grow = (ctypes.c_float * 3)(1e6, 0.0, 0.0)
    P = ctypes.c_void_p(256)
    assert lib.muon_ns_batched(P, 1, 64, 64, 5, grow, 1e-7, None) == -2
    assert lib.muon_ns_batched_static(P, 1, 64, 64, 5, grow, 1e-7, None) == -2
    assert lib.muon_step_batched(P, P, P, 1, 64, 64, 0.95, 1, 5, grow, 1e-7, 0.02, 0.1, 0.0, None, 0, None) == -2
    # the fp32 verification path has no such limit
    assert lib.muon_ns_batched_f32(None, 0, 64, 64, 5, grow, 1e-7, None) == 0


def test_allocation_failure_injection_counts_on_the_host(lib):
    # the hook only sets a counter (no CUDA call); the GPU test checks its effect
    assert lib.muon_inject_alloc_failures(2) == 0
    assert lib.muon_inject_alloc_failures(0) == 2
    assert lib.muon_inject_alloc_failures(-1) == -1        # MUON_ERR_INVALID_ARG
    assert lib.muon_inject_alloc_failures(0) == 0


def test_grouped_host_step_rejects_bad_groups_on_the_host(lib):
    import muon_newton_schulz_expert_gb300 as m
    co = (ctypes.c_float * 3)(3.4445, -4.7750, 2.0315)
    f = lib.muon_step_host_grouped
    assert f(None, 0, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == 0        # nothing to do
    assert f(None, -1, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == -1
    assert f(None, 2, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == -1
    buf = ctypes.create_string_buffer(1024)
    ptr = ctypes.addressof(buf)
    groups = (m.HostGroup * 2)(m.HostGroup(ptr, ptr, ptr, 0, 64, 64, 0.0), m.HostGroup(ptr, ptr, ptr, 2, 64, 60, 0.0))
    g = ctypes.cast(groups, ctypes.c_void_p)
    assert f(g, 2, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == -2         # cols not a multiple of 8
    groups[1] = m.HostGroup(None, ptr, ptr, 2, 64, 64, 0.0)
    assert f(g, 2, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == -1         # null parameter array
    groups[1] = m.HostGroup(ptr, ptr, ptr, -1, 64, 64, 0.0)
    assert f(g, 2, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0, None) == -1         # negative batch
    assert f(g, 2, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, -1, None) == -1        # negative chunk


def test_checked_variant_builds_and_exports_every_symbol():
    # the same sources with -DMUON_DEVICE_CHECKS (its GPU behaviour is checked
    # in tests/test_gpu_checked_build.py)
    path = mkbuild.build(checked=True)
    raw = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(raw, n), n
