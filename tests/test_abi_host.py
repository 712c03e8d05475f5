"""Host-only contract tests of the C ABI (no GPU needed, no compute call made).

Modelled on the hermetic contract tests the vLLM PR #52781 review describes:
they check argument validation, sizing, error codes and the host-side wait,
never values computed on a device.  Every call here returns before the
library touches the CUDA runtime.
"""
import ctypes
import os
import re
import subprocess
import tempfile
import time

import numpy as np
import pytest

from oracle import ep_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def ep():
    import combine_topk_idx_gb300 as ep
    from combine_topk_idx_gb300 import _build_lib
    _build_lib.build()
    ep.load_library()
    return ep


def _declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(ep):
    names = _declared_symbols()
    assert {"ep_layout", "ep_dispatch", "ep_combine", "ep_handle_free"} <= set(names)
    lib = ep.load_library()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ep.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ep_\w+)", out))
    assert set(names) <= exported
    assert exported <= set(names), f"undeclared exports: {exported - set(names)}"
    assert lib.ep_abi_version() == ep.EP_ABI_VERSION


def test_struct_layout_matches_c_header(ep):
    """ctypes mirrors of the ABI structs have the C compiler's sizes and offsets."""
    prog = r'''
#include <stddef.h>
#include <stdio.h>
#include "ep.h"
#define P(T, f) printf(#T " " #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("ep_config size %zu\n", sizeof(ep_config));
  printf("ep_layout_info size %zu\n", sizeof(ep_layout_info));
  printf("ep_layout_buffers size %zu\n", sizeof(ep_layout_buffers));
  P(ep_config, num_tokens) P(ep_config, topk_idx_is_int64) P(ep_config, do_expand)
  P(ep_config, use_tma_aligned_col_major_sf) P(ep_config, num_sms) P(ep_config, cpu_sync_timeout_ms)
  P(ep_config, fixed_capacity) P(ep_config, reserved0)
  P(ep_layout_info, rows_alloc) P(ep_layout_info, topk_idx) P(ep_layout_info, error_word)
  P(ep_layout_info, meta_rows) P(ep_layout_info, expert_capacity)
  P(ep_layout_info, sf_expert_stride) P(ep_layout_info, layout_kernels)
  P(ep_layout_buffers, status)
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        open(c, "w").write(prog)
        exe = os.path.join(d, "t")
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for ln in lines:
        if ln:
            a, b, v = ln.split()
            got[(a, b)] = int(v)
    C, I, B = ep.EpConfigC, ep.EpLayoutInfoC, ep.EpLayoutBuffersC
    assert got[("ep_config", "size")] == ctypes.sizeof(C)
    assert got[("ep_layout_info", "size")] == ctypes.sizeof(I)
    assert got[("ep_layout_buffers", "size")] == ctypes.sizeof(B)
    for f in ("num_tokens", "topk_idx_is_int64", "do_expand", "use_tma_aligned_col_major_sf",
              "num_sms", "cpu_sync_timeout_ms", "fixed_capacity", "reserved0"):
        assert got[("ep_config", f)] == getattr(C, f).offset, f
    for f in ("rows_alloc", "topk_idx", "error_word", "meta_rows", "expert_capacity",
              "sf_expert_stride", "layout_kernels"):
        assert got[("ep_layout_info", f)] == getattr(I, f).offset, f
    assert got[("ep_layout_buffers", "status")] == B.status.offset


def _cfg(ep, **kw):
    base = dict(num_tokens=128, num_topk=2, num_experts=16, num_ranks=4, hidden=256,
                num_max_tokens_per_rank=32, expert_alignment=8, do_expand=True,
                do_zero_padding=True, do_cpu_sync=True, use_fp8=False)
    base.update(kw)
    args = [base.pop(k) for k in ("num_tokens", "num_topk", "num_experts", "num_ranks", "hidden",
                                  "num_max_tokens_per_rank")]
    return ep.make_config(*args, **base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"num_experts": 18}, 1),                       # E % R != 0
    ({"hidden": 250}, 1),                           # H % 8 != 0
    ({"use_fp8": True, "hidden": 264}, 1),          # FP8 needs H % 128 == 0
    ({"use_fp8": True, "hidden": 384}, 0),
    ({"num_tokens": 129}, 1),                       # T > M * R
    ({"num_tokens": -1}, 1),
    ({"num_topk": 0}, 1),
    ({"num_topk": 33}, 2),                          # beyond EP_MAX_TOPK
    ({"num_experts": 4096, "num_ranks": 4}, 2),     # beyond EP_MAX_EXPERTS
    ({"hidden": 65536}, 2),                         # beyond EP_MAX_HIDDEN
    ({"expert_alignment": 0}, 1),
    ({"num_max_tokens_per_rank": 0}, 1),
    ({"num_sms": -3}, 1),
    ({"cpu_sync_timeout_ms": -1}, 1),
    ({"fixed_capacity": True, "do_expand": True, "expert_alignment": 1,
      "do_zero_padding": False}, 0),
    ({"fixed_capacity": True, "do_expand": False, "expert_alignment": 1}, 1),
    ({"fixed_capacity": True, "do_expand": True, "expert_alignment": 8,
      "do_zero_padding": False}, 1),                # no alignment in the fixed layout
    ({"fixed_capacity": True, "do_expand": True, "expert_alignment": 1,
      "do_zero_padding": True}, 1),
    ({"fixed_capacity": True, "do_expand": True, "expert_alignment": 1, "do_zero_padding": False,
      "num_experts": 2048, "num_ranks": 16, "num_tokens": 16384,
      "num_max_tokens_per_rank": 65536}, 2),       # E * M * R rows past int32
])
def test_validate_config(ep, kw, status):
    assert ep.validate_config(_cfg(ep, **kw)) == status


def test_validate_rejects_bad_flags_and_reserved(ep):
    c = _cfg(ep)
    c.do_expand = 2
    assert ep.validate_config(c) == ep.EP_ERR_INVALID_ARG
    c = _cfg(ep)
    c.reserved0[1] = 7
    assert ep.validate_config(c) == ep.EP_ERR_INVALID_ARG
    c = _cfg(ep, do_zero_padding=False, expert_alignment=1)
    c.fixed_capacity = 2
    assert ep.validate_config(c) == ep.EP_ERR_INVALID_ARG
    c = _cfg(ep)
    c.topk_idx_is_int64 = 5
    assert ep.validate_config(c) == ep.EP_ERR_INVALID_ARG
    assert ep.load_library().ep_validate_config(None) == ep.EP_ERR_INVALID_ARG


def test_upper_bound_rows_match_oracle(ep):
    rng = np.random.default_rng(3)
    for _ in range(300):
        R = int(rng.choice([1, 2, 4, 8, 32]))
        E = R * int(rng.integers(1, 9))
        K = int(rng.integers(1, min(E, 32) + 1))
        M = int(rng.integers(1, 3000))
        T = int(rng.integers(0, M * R + 1))
        A = int(rng.choice([1, 2, 8, 128]))
        for de in (False, True):
            c = ep.make_config(T, K, E, R, 128, M, A, de)
            assert ep.upper_bound_rows(c) == O.upper_bound_rows(T, K, E, R, M, A, de)
        c = ep.make_config(T, K, E, R, 128, M, 1, True, fixed_capacity=True)
        assert ep.upper_bound_rows(c) == E * M * R


def test_host_wait_flag_deadline(ep):
    flag = ctypes.c_int32(0)
    t0 = time.perf_counter()
    assert ep.host_wait_flag(flag, 1, 80) == ep.EP_ERR_TIMEOUT      # nothing sets it
    el = time.perf_counter() - t0
    assert 0.07 <= el < 2.0
    flag.value = 9
    assert ep.host_wait_flag(flag, 9, 80) == ep.EP_OK
    assert ep.load_library().ep_host_wait_flag(None, 1, 10) == ep.EP_ERR_INVALID_ARG
    assert ep.host_wait_flag(flag, 9, -1) == ep.EP_ERR_INVALID_ARG


def test_entry_points_reject_bad_arguments_before_any_cuda_call(ep):
    lib = ep.load_library()
    info = ep.EpLayoutInfoC()
    h = ctypes.c_void_p(0)
    # missing outputs, bad config, missing topk_idx: refused on the host
    assert lib.ep_layout(ctypes.byref(_cfg(ep)), None, None, None, ctypes.byref(info)) == 1
    assert lib.ep_layout(ctypes.byref(_cfg(ep, num_experts=18)), None, None, ctypes.byref(h),
                         ctypes.byref(info)) == 1
    assert lib.ep_layout(ctypes.byref(_cfg(ep)), None, None, ctypes.byref(h),
                         ctypes.byref(info)) == 1
    assert lib.ep_layout(ctypes.byref(_cfg(ep)), ctypes.c_void_p(0x1003), None, ctypes.byref(h),
                         ctypes.byref(info)) == 1                  # misaligned int64 topk_idx
    assert h.value is None
    assert lib.ep_dispatch(None, None, None, None, None, None, None, None) == 1
    assert lib.ep_combine(None, None, None, None, None, None, None, None) == 1
    lib.ep_handle_free(None)
    assert lib.ep_dispatch_backward(None, None, None, None, None, None) == 1
    assert lib.ep_combine_backward(None, None, None, None) == 1
    assert lib.ep_dispatch_fp8(None, None, None, 0, 0, None, None, None, None, None, None) == 1
    # allocation-free layout: sync mode, missing buffers, oversized problems
    b = ep.EpLayoutBuffersC()
    fn = lib.ep_layout_noalloc
    fn.argtypes = [ctypes.POINTER(ep.EpConfigC), ctypes.c_void_p,
                   ctypes.POINTER(ep.EpLayoutBuffersC), ctypes.c_void_p]
    assert fn(ctypes.byref(_cfg(ep)), ctypes.c_void_p(0x1000), ctypes.byref(b), None) == 1
    assert fn(ctypes.byref(_cfg(ep, do_cpu_sync=False)), ctypes.c_void_p(0x1000),
              ctypes.byref(b), None) == 1
    for n, _ in ep.EpLayoutBuffersC._fields_:
        setattr(b, n, 0x10000)
    T = 256 * 300
    big = ep.make_config(T, 8, 2048, 16, 128, T // 16 + 1, 1, True, False, False)
    assert fn(ctypes.byref(big), ctypes.c_void_p(0x1000), ctypes.byref(b), None) == 2
    # layout + dispatch in one call: exact allocation, missing outputs, missing
    # or misaligned x and receive buffers are refused on the host
    ld = lib.ep_layout_dispatch
    v = ctypes.c_void_p
    nos = _cfg(ep, do_cpu_sync=False)  # BF16: recv_sf must be NULL

    def call(cfg, x=v(0x1000), w=None, rx=v(0x1000), rsf=None, rw=None, out=True):
        return ld(ctypes.byref(cfg), v(0x1000), x, w, rx, rsf, rw, None, None,
                  ctypes.byref(h) if out else None, ctypes.byref(info))
    assert call(_cfg(ep)) == 1                      # exact allocation (count wait)
    assert call(nos, out=False) == 1                # no handle output
    assert call(nos, x=None) == 1                   # missing x
    assert call(nos, x=v(0x1008)) == 1              # x not 16-byte aligned
    assert call(nos, rx=None) == 1                  # missing recv_x
    assert call(nos, rsf=v(0x1000)) == 1            # scales for a BF16 dispatch
    assert call(nos, rw=v(0x1000)) == 1             # weights out, none in
    assert h.value is None
    # bounded-wait self-test: argument checks happen on the host
    st = lib.ep_selftest_bounded_wait
    st.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    assert st(1000, 0, None, None) == 1
    assert st(0, 0, ctypes.byref(ctypes.c_uint32()), None) == 1


def test_plan_layout_sizes(ep):
    """ep_plan_layout reports, without GPU work, the sizes ep.h states for a
    layout without the count wait: the upper-bound rows and the scale-factor
    layout of each mode."""
    def al4(x):
        return (x + 3) // 4 * 4
    T, K, E, R, M, H = 300, 6, 32, 4, 80, 512
    nb = H // 128
    cases = [  # (expand, fp8, col_major, fixed)
        (False, True, False, False), (False, True, True, False), (True, True, True, False),
        (True, True, False, False), (False, False, False, False), (True, True, True, True),
        (True, True, False, True), (True, False, False, True)]
    for ex, fp8, cm, fixed in cases:
        cfg = ep.make_config(T, K, E, R, H, M, 1 if fixed else 8, ex, False, False, fp8, cm,
                             fixed_capacity=fixed)
        info = ep.plan_layout(cfg)
        rows = ep.upper_bound_rows(cfg)
        cap = M * R if fixed else 0
        assert info.rows_alloc == rows and info.meta_rows == rows
        assert info.expert_capacity == cap
        assert info.num_recv_tokens == -1 and info.num_expanded_tokens == -1
        assert not info.dst_buffer_slot_idx and not info.error_word
        if not fp8:
            want = (0, 0, 0, 0)
        elif fixed and cm:
            want = (1, al4(cap), E * nb * al4(cap), nb * al4(cap))
        elif fixed:
            want = (nb, 1, E * nb * cap, nb * cap)
        elif cm:
            want = (1, al4(rows), nb * al4(rows), 0)
        else:
            want = (nb, 1, nb * rows, 0)
        got = (info.sf_token_stride, info.sf_hidden_stride, info.sf_numel, info.sf_expert_stride)
        assert got == want, (ex, fp8, cm, fixed)
    with pytest.raises(ep.EpError):
        ep.plan_layout(ep.make_config(T, K, E, R, H, M, 8, True, True, True))
    assert ep.load_library().ep_plan_layout(ctypes.byref(_cfg(ep)), None) == 1


def test_status_strings(ep):
    for code in range(8):
        s = ep.status_string(code)
        assert s and s != "unknown status"
    assert ep.status_string(99) == "unknown status"
