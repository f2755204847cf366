"""The C-ABI library loads without a GPU, exports every symbol include/usaf.h declares, and its
host-side argument checks and workspace queries behave as the header states (nothing is launched
in these calls)."""
import ctypes
import math

import pytest
import torch

from sparse_moe_fine_gb300 import binding as B

# The argument-check tests pass fake device addresses that a launch would dereference. They are
# meant for a machine without a GPU, where a check that failed to refuse could not reach a device.
fake_addresses = pytest.mark.skipif(torch.cuda.is_available(),
                                    reason="fake device addresses; run where no GPU is visible")


def test_library_exports_every_header_symbol():
    L = B.lib()
    syms = B.header_symbols()
    assert len(syms) == 43
    for s in syms:
        assert hasattr(L, s), s
    assert L.usaf_abi_version() == 2
    assert L.usaf_status_string(0) == b"ok"
    assert L.usaf_status_string(3) == b"workspace missing or too small"


def _header_arity():
    """Parameter count of every function the header declares (declarations, not comments)."""
    import os
    import re
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "usaf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for name, params in re.findall(r"\b(usaf_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = " ".join(params.split())
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_prototypes_match_the_header():
    """Every ctypes prototype has as many arguments as the header's declaration."""
    arity = _header_arity()
    assert set(arity) == set(B.header_symbols())
    for name, (_, args) in B._SIGS.items():
        assert name in arity, name
        assert len(args) == arity[name], (name, len(args), arity[name])
    assert set(B._SIGS) == set(arity)


@fake_addresses
def test_shard_selection_host_checks():
    L = B.lib()
    fake = ctypes.c_void_p(256)  # never dereferenced: every call below fails on the host
    # digit widths outside 1..11 and digits past bit 30
    assert L.usaf_shard_key_histogram(fake, 10, None, 0, 0, 12, fake, None) == 1
    assert L.usaf_shard_key_histogram(fake, 10, None, 0, 21, 11, fake, None) == 1
    assert L.usaf_shard_key_histogram(fake, 10, None, 0, 0, 0, fake, None) == 1
    assert L.usaf_shard_key_histogram(fake, 1 << 32, None, 0, 0, 7, fake, None) == 1
    assert L.usaf_shard_key_histogram(fake, 10, None, 0, 0, 7, None, None) == 1
    # more ties than entries, a negative base, no workspace
    assert L.usaf_shard_emit(fake, 10, None, 0, 11, 11, 0, fake, None, fake, 1 << 20, None) == 1
    assert L.usaf_shard_emit(fake, 10, None, 0, 1, 1, -1, fake, None, fake, 1 << 20, None) == 1
    assert L.usaf_shard_emit(fake, 10, None, 0, 1, 1, 0, fake, None, None, 0, None) == 3
    assert L.usaf_shard_emit_workspace_size(1 << 32, 1) == 0
    assert L.usaf_active_bitmap(fake, 5, 0, 0, fake, None) == 1
    # K above the entry count, D above K, a missing grow set
    assert L.usaf_rigl_apply(fake, 100, 50, 10, fake, fake, fake, fake, fake, 50, None, 1, fake,
                             fake, fake, fake, fake, None, fake, 1 << 30, None) == 1
    assert L.usaf_rigl_apply(fake, 10, 50, 11, fake, fake, fake, fake, fake, 50, None, 1, fake,
                             fake, fake, fake, fake, None, fake, 1 << 30, None) == 1
    assert L.usaf_rigl_apply(fake, 10, 50, 2, None, fake, fake, fake, fake, 50, None, 1, fake,
                             fake, fake, fake, fake, None, fake, 1 << 30, None) == 1
    # the second weight segment missing while N > n_seg0
    assert L.usaf_reselect_carry(fake, 10, 50, fake, 10, fake, fake, fake, fake, 40, None, 1,
                                 fake, fake, fake, fake, None, fake, 1 << 20, None) == 1
    assert L.usaf_reselect_carry(fake, 10, 50, fake, 10, fake, fake, fake, fake, 50, None, 1,
                                 fake, fake, fake, fake, None, None, 0, None) == 3


@fake_addresses
def test_select_and_swap_host_checks():
    L = B.lib()
    fake = [ctypes.c_void_p(a) for a in range(1 << 20, 12 << 20, 1 << 20)]  # 1 MiB apart
    g, sel, act, p, m, v, w, new, po, mo, vo = fake
    ns, ws = ctypes.c_void_p(256), ctypes.c_void_p(512)

    def call(K_sel, K, D, sel_ptr=sel, new_ptr=new, ws_bytes=1 << 40):
        return L.usaf_select_and_swap(g, 1000, K_sel, sel_ptr, act, K, D, p, m, v, w, 1000, None,
                                      1, new_ptr, po, mo, vo, ns, None, ws, ws_bytes, None)

    assert call(0, 100, 10) == 1     # K_sel < 1
    assert call(1001, 100, 10) == 1  # K_sel > N
    assert call(50, 100, 101) == 1   # D > K
    assert call(50, 100, 10, sel_ptr=None) == 1
    assert call(50, 100, 10, sel_ptr=new) == 1  # the selection overlaps the new active set
    assert call(50, 100, 10, new_ptr=act) == 1  # an output overlaps an input
    assert call(50, 100, 10, ws_bytes=16) == 3


@fake_addresses
def test_forward_stage_and_scan_host_checks():
    L = B.lib()
    s = B.shape(8, 64, 4, 2, 64)
    fake = ctypes.c_void_p(256)  # never dereferenced: every call below fails on the host
    r = B._Routing(*[256] * 7)
    for bad in (0, 8, -1):  # stage sets outside 1..7
        assert L.usaf_moe_fwd_stage(ctypes.byref(s), 1, fake, fake, fake, ctypes.byref(r), fake,
                                    fake, fake, fake, bad, None, fake, 1 << 30, None) == 1
    assert L.usaf_scan_nonfinite(fake, -1, fake, None) == 1
    assert L.usaf_scan_nonfinite(None, 4, fake, None) == 1
    assert L.usaf_scan_nonfinite(fake, 4, None, None) == 1
    assert L.usaf_scan_nonfinite(None, 0, fake, None) == 0  # nothing to scan
    # skip modes beyond 2 are refused
    assert L.usaf_sparse_adam_step(4, None, fake, fake, fake, fake, fake, 4, None, 0, 1e-3, 0.9,
                                   0.999, 1e-8, 1, 3, fake, None) == 1


def test_capacity_and_workspace_queries():
    s = B.shape(4096, 2048, 128, 8, 768)
    cap = B.routed_rows_capacity(s)
    assert cap >= 4096 * 8 + 128 * 15 and cap % 256 == 0
    assert B.route_topk_workspace_size(s) > 4096 * 128 * 4
    assert B.moe_fwd_workspace_size(s, B.BF16) >= 4096 * 2048 * 4
    assert B.moe_bwd_workspace_size(s, B.BF16, 3019899) > 0
    off = B.moe_bwd_dlogit_offset(s, B.BF16, 3019899)
    assert off % 256 == 0 and off + 4096 * 8 * 4 <= B.moe_bwd_workspace_size(s, B.BF16, 3019899)
    N = 603979776
    K = math.ceil(0.005 * N)
    ws = B.importance_select_workspace_size(N, K)
    assert 0 < ws < 0.2 * N * 4  # candidates only, not a copy of g
    assert B.rigl_swap_workspace_size(N, K, int(0.3 * K)) > N // 8  # holds the N-bit bitmap
    bad = B.shape(0, 2048, 128, 8, 768)
    assert B.routed_rows_capacity(bad) == -1
    assert B.importance_select_workspace_size(10, 11) == 0
    assert B.rigl_swap_workspace_size(10, 8, 3) == 0  # D > N - K
    # one pass for both selections: the shared candidates, less than the two calls' workspaces
    D = int(0.3 * K)
    fused = B.select_and_swap_workspace_size(N, K, K, D)
    assert N // 8 < fused < ws + B.rigl_swap_workspace_size(N, K, D)
    assert B.select_and_swap_workspace_size(N, 0, K, D) == 0
    assert B.select_and_swap_workspace_size(10, 11, 2, 1) == 0
    assert B.select_and_swap_workspace_size(10, 5, 8, 3) == 0  # D > N - K
    # where the two selections run one after the other, both calls' workspaces
    assert B.select_and_swap_workspace_size(5000, 700, 700, 200) >= \
        B.importance_select_workspace_size(5000, 700) + B.rigl_swap_workspace_size(5000, 700, 200)


def _call(name, *args):
    return getattr(B.lib(), name)(*args)


@fake_addresses
def test_host_argument_checks_return_codes():
    s = B.shape(8, 64, 4, 2, 64)
    r = B._Routing()
    # null routing arrays
    assert _call("usaf_route_topk", ctypes.byref(s), 1, 0, 1, None, None, 1, ctypes.byref(r),
                 None, 1, 1 << 20, None) == 1
    # k > E
    s2 = B.shape(8, 64, 4, 5, 64)
    assert _call("usaf_routed_rows_capacity", ctypes.byref(s2)) == -1
    # SparseAdam: step 0, skip without a status word, betas out of range
    assert _call("usaf_sparse_adam_step", 4, None, 1, 1, 1, 1, 1, 4, None, 0, 1e-3, 0.9, 0.999,
                 1e-8, 0, 0, None, None) == 1
    assert _call("usaf_sparse_adam_step", 4, None, 1, 1, 1, 1, 1, 4, None, 0, 1e-3, 0.9, 0.999,
                 1e-8, 1, 1, None, None) == 1
    assert _call("usaf_sparse_adam_step", 4, None, 1, 1, 1, 1, 1, 4, None, 0, 1e-3, 1.0, 0.999,
                 1e-8, 1, 0, None, None) == 1
    # dense form needs n <= n_seg0
    assert _call("usaf_sparse_adam_step", 8, None, 1, 1, 1, 1, 1, 4, None, 0, 1e-3, 0.9, 0.999,
                 1e-8, 1, 0, None, None) == 1
    # n = 0 is a no-op
    assert _call("usaf_sparse_adam_step", 0, None, None, None, None, None, None, 0, None, 0, 1e-3,
                 0.9, 0.999, 1e-8, 1, 0, None, None) == 0
    # selection: K > N, workspace too small
    assert _call("usaf_importance_select", 1, 10, 11, 1, None, 1, 1 << 20, None) == 1
    assert _call("usaf_importance_select", 1, 1 << 20, 10, 1, None, 1, 16, None) == 3
    # RigL: overlapping input/output state, D > K
    assert _call("usaf_rigl_swap", 1, 100, 4096, 10, 2, 8192, 16384, 24576, 1, 100, None, 0,
                 40960, 8192, 49152, 57344, 1, None, 1, 1 << 30, None) == 1
    assert _call("usaf_rigl_swap", 1, 100, 4096, 10, 11, 8192, 16384, 24576, 1, 100, None, 0,
                 40960, 65536, 49152, 57344, 1, None, 1, 1 << 30, None) == 1
    # bf16 layers need H and I multiples of 64
    s3 = B.shape(8, 96, 4, 2, 64)
    assert _call("usaf_moe_fwd", ctypes.byref(s3), 1, 1, 1, 1, ctypes.byref(B._Routing(*[1] * 7)),
                 1, 1, 1, 1, None, 1, 1 << 30, None) == 2
    # active-set validation needs a status word and a positive bound
    assert _call("usaf_validate_active", 1, 4, 10, None, None) == 1
    assert _call("usaf_validate_active", 1, 4, 0, 1, None) == 1
    assert _call("usaf_validate_active", None, 4, 10, 1, None) == 1
    # the bounded-wait check: limit in [1, 2^32], status word required
    assert _call("usaf_diag_bounded_wait", 0, 1, None) == 1
    assert _call("usaf_diag_bounded_wait", (1 << 32) + 1, 1, None) == 1
    assert _call("usaf_diag_bounded_wait", 1000, None, None) == 1


@fake_addresses
def test_reselect_full_host_checks():
    L = B.lib()
    N, K = 1 << 20, 5000
    assert L.usaf_reselect_full_workspace_size(N, K) > 0
    assert L.usaf_reselect_full_workspace_size(N, N + 1) == 0
    assert L.usaf_reselect_full_workspace_size(1 << 32, K) == 0
    fake = ctypes.c_void_p(256)  # never dereferenced: every call below fails on the host
    one = ctypes.c_void_p(512)
    # null gradient / null count
    assert L.usaf_reselect_full(None, N, K, fake, K, fake, fake, fake, fake, N, None, 1, fake,
                                fake, fake, fake, fake, None, fake, 1 << 30, None) == 1
    assert L.usaf_reselect_full(fake, N, K, fake, K, fake, fake, fake, fake, N, None, 1, fake,
                                fake, fake, fake, None, None, fake, 1 << 30, None) == 1
    # an output aliasing an input
    assert L.usaf_reselect_full(fake, N, K, fake, K, one, fake, fake, fake, N, None, 1, fake,
                                one, fake, fake, fake, None, fake, 1 << 30, None) == 1
    # workspace too small
    assert L.usaf_reselect_full(fake, N, K, ctypes.c_void_p(1 << 20), K,
                                ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20),
                                ctypes.c_void_p(4 << 20), fake, N, None, 1,
                                ctypes.c_void_p(5 << 20), ctypes.c_void_p(6 << 20),
                                ctypes.c_void_p(7 << 20), ctypes.c_void_p(8 << 20), fake, None,
                                fake, 16, None) == 3



@fake_addresses
def test_layer_call_host_checks():
    """The forward and backward entry points refuse bad arguments on the host, before any launch:
    every pointer below is a fake address that a launch would fault on."""
    s = B.shape(64, 64, 4, 2, 64)
    rt = ctypes.byref(B._Routing(*[4096] * 7))
    f = 8192  # fake device address, 16-byte aligned
    big = 1 << 30
    fwd_ws = B.moe_fwd_workspace_size(s, B.BF16)
    bwd_ws = B.moe_bwd_workspace_size(s, B.BF16, 100)
    assert fwd_ws > 0 and bwd_ws > 0
    fwd = lambda y, ev, ws: _call("usaf_moe_fwd_wait", ctypes.byref(s), B.BF16, f, f, f, rt, f, f,
                                  f, y, ev, None, f, ws, None)
    assert fwd(None, None, big) == 1           # no output buffer
    assert fwd(f, None, fwd_ws - 1) == 3       # workspace one byte short
    assert fwd(f, f, fwd_ws - 1) == 3          # the same with an event to wait for
    assert _call("usaf_moe_fwd_wait", ctypes.byref(s), 7, f, f, f, rt, f, f, f, f, None, None, f,
                 big, None) == 1               # unknown dtype

    def bwd(name, renorm=1, logits=f, K=100, ws=big):
        return _call(name, ctypes.byref(s), B.BF16, renorm, f, f, f, f, rt, logits, f, f, f, f,
                     f, K, f, f, f, None, None, f, ws, None)
    for name in ("usaf_moe_bwd_sparse", "usaf_moe_bwd_sparse_accumulate"):
        assert bwd(name, renorm=2) == 1                 # renorm must be 0 or 1
        assert bwd(name, renorm=0, logits=None) == 1    # the all-E softmax form needs the logits
        assert bwd(name, K=-1) == 1
        assert bwd(name, K=64 * 3 * 64 * 4 + 1) == 1    # K > N
        assert bwd(name, ws=bwd_ws - 1) == 3

    def dense(g, acc=0, ws=big):
        return _call("usaf_moe_bwd_dense", ctypes.byref(s), B.BF16, 1, f, f, f, f, rt, f, f, f,
                     f, f, g, acc, f, f, None, None, f, ws, None)
    assert dense(f + 4) == 1          # the dense gradient must be 16-byte aligned
    assert dense(f, acc=2) == 1       # accumulate must be 0 or 1
    assert dense(None) == 1
    assert dense(f, ws=B.moe_bwd_workspace_size(s, B.BF16, 0) - 1) == 3
