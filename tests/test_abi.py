"""The C-ABI library on the CPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch.

No test here reaches a kernel launch: every call either fails validation or
has nothing to do, so these run without a GPU. Fake pointer values are never
dereferenced on those paths.
"""
import os
import re

import pytest

from gated_deltanet_linear_build_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE = 0, -1, -2, -3, -4
A16 = 0x10000          # a 16-byte-aligned fake device address
A8 = 0x10008           # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("gdn_build_conv_chunks", "gdn_causal_conv1d_fwd", "gdn_causal_conv1d_update",
                 "gdn_delta_rule_decode", "gdn_delta_rule_prefill_chunked"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from gated_deltanet_linear_build_gb300 import gdn
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(gdn.EXPORTED_SYMBOLS) == declared_symbols()


def test_status_strings(lib):
    for s in (OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE, -5, -6):
        assert lib.gdn_status_string(s).startswith(b"GDN")
    assert lib.gdn_last_cuda_error_string() is not None


def test_build_chunks_validation(lib):
    f = lib.gdn_build_conv_chunks
    assert f(None, 2, 8, A16, 10, A16, None, None) == INVALID        # no cu_seqlens
    assert f(A16, -1, 8, A16, 10, A16, None, None) == INVALID        # negative N
    assert f(A16, 2, 2, A16, 10, A16, None, None) == INVALID         # chunk < K - 1
    assert f(A16, 2, 8, None, 10, A16, None, None) == INVALID        # capacity but no array
    assert f(A16, 2, 8, A16, 10, None, None, None) == INVALID        # no count output
    assert f(A16, 2, 8, A8, 10, A16, None, None) == ALIGN


def conv_fwd(lib, **kw):
    args = dict(x=A16, x_stride=64, w=A16, bias=None, state=A16, has=None, cu=A16, chunks=None,
                num=None, max_chunks=0, T=18, C=64, K=4, N=2, silu=1, y=A16)
    args.update(kw)
    return lib.gdn_causal_conv1d_fwd(*args.values(), None)


def test_conv_fwd_validation(lib):
    assert conv_fwd(lib, chunks=A16) == INVALID                 # half-set descriptor pair
    assert conv_fwd(lib, num=A16) == INVALID
    assert conv_fwd(lib, x=None) == INVALID
    assert conv_fwd(lib, cu=None) == INVALID
    assert conv_fwd(lib, T=-1) == INVALID
    assert conv_fwd(lib, x_stride=32) == INVALID                # stride < C
    assert conv_fwd(lib, silu=2) == INVALID
    assert conv_fwd(lib, K=3) == UNSUPPORTED
    assert conv_fwd(lib, C=60, x_stride=64) == UNSUPPORTED      # C % 8
    assert conv_fwd(lib, x_stride=68) == ALIGN
    assert conv_fwd(lib, x=A8) == ALIGN
    assert conv_fwd(lib, bias=A8) == ALIGN
    assert conv_fwd(lib, chunks=A8, num=A16, max_chunks=4) == ALIGN
    assert conv_fwd(lib, T=0) == OK                             # nothing to do
    assert conv_fwd(lib, N=0) == OK


def test_conv_update_validation(lib):
    f = lib.gdn_causal_conv1d_update
    assert f(A16, 64, A16, None, A16, 2, 64, 4, 1, None, None) == INVALID
    assert f(A16, 64, A16, None, A16, 2, 64, 5, 1, A16, None) == UNSUPPORTED
    assert f(A16, 64, A16, None, A8, 2, 64, 4, 1, A16, None) == ALIGN
    assert f(A16, 64, A16, None, A16, 0, 64, 4, 1, A16, None) == OK


def decode(lib, **kw):
    args = dict(q=A16, k=A16, qk_stride=4096, v=A16, v_stride=4096, a=A16, b=A16, S=A16, o=A16,
                N=32, Hk=16, Hv=32, dk=128, dv=128, l2=0)
    args.update(kw)
    return lib.gdn_delta_rule_decode(*args.values(), None)


def test_decode_validation(lib):
    assert decode(lib, S=None) == INVALID
    assert decode(lib, Hk=12) == INVALID                        # Hv % Hk
    assert decode(lib, qk_stride=1024) == INVALID               # stride < Hk * dk
    assert decode(lib, l2=8) == INVALID                         # unknown flag bit
    assert decode(lib, l2=-1) == INVALID
    assert decode(lib, dk=96) == UNSUPPORTED
    assert decode(lib, dv=256, v_stride=8192) == UNSUPPORTED
    assert decode(lib, qk_stride=4100) == ALIGN
    assert decode(lib, S=A8) == ALIGN
    assert decode(lib, N=0) == OK


def prefill(lib, **kw):
    args = dict(q=A16, k=A16, qk_stride=4096, v=A16, v_stride=4096, a=A16, b=A16, cu=A16, N=2,
                T=2048, S=A16, has=None, o=A16, Hk=16, Hv=32, dk=128, dv=128, chunk=64, l2=0,
                ws=A16 * 16, ws_bytes=1 << 40)
    args.update(kw)
    return lib.gdn_delta_rule_prefill_chunked(*args.values(), None)


def test_prefill_validation(lib):
    need = lib.gdn_delta_rule_prefill_workspace_size(2048, 2, 32, 128, 128, 64)
    assert need > 0
    assert lib.gdn_delta_rule_prefill_workspace_size(2048, 2, 32, 128, 128, 32) == 0
    assert prefill(lib, cu=None) == INVALID
    assert prefill(lib, chunk=32) == UNSUPPORTED
    assert prefill(lib, dk=64) == UNSUPPORTED                   # dk != dv
    assert prefill(lib, ws_bytes=need - 1) == WORKSPACE
    assert prefill(lib, ws=None) == WORKSPACE
    assert prefill(lib, ws=A16 * 16 + 16) == ALIGN              # workspace 256-byte rule
    assert prefill(lib, T=0) == OK
    assert prefill(lib, N=0) == OK


def prefill_noalloc(lib, **kw):
    args = dict(q=A16, k=A16, qk_stride=4096, v=A16, v_stride=4096, a=A16, b=A16, cu=A16, N=2,
                T=512, S=A16, has=None, o=A16, Hk=16, Hv=32, dk=128, dv=128, chunk=64, l2=0)
    args.update(kw)
    return lib.gdn_delta_rule_prefill_chunked_noalloc(*args.values(), None)


def test_prefill_noalloc_validation_before_any_cuda_call(lib):
    # Every check of the regular entry point, and the fixed array's size limit,
    # run before the call looks up its scratch (no CUDA call on these paths).
    assert prefill_noalloc(lib, cu=None) == INVALID
    assert prefill_noalloc(lib, q=None) == INVALID
    assert prefill_noalloc(lib, chunk=32) == UNSUPPORTED
    assert prefill_noalloc(lib, dk=64) == UNSUPPORTED
    assert prefill_noalloc(lib, Hv=24) == INVALID                # Hv % Hk != 0
    assert prefill_noalloc(lib, S=A8) == ALIGN
    assert prefill_noalloc(lib, T=2048) == WORKSPACE             # beyond the 64 MiB array
    assert prefill_noalloc(lib, T=0) == OK
    assert lib.gdn_delta_rule_prefill_chunked_noalloc_status(None, None) == INVALID


def test_prefill_plan_validation(lib):
    f = lib.gdn_delta_rule_prefill_plan
    need = lib.gdn_delta_rule_prefill_workspace_size(2048, 2, 32, 128, 128, 64)
    ws = A16 * 16
    assert f(None, 2, 2048, 32, 128, 128, 64, ws, need, None) == INVALID
    assert f(A16, 2, 2048, 32, 128, 128, 32, ws, need, None) == UNSUPPORTED
    assert f(A16, 2, 2048, 32, 128, 64, 64, ws, need, None) == UNSUPPORTED
    assert f(A16, 2, 2048, 32, 128, 128, 64, ws, need - 1, None) == WORKSPACE
    assert f(A16, 2, 2048, 32, 128, 128, 64, ws + 16, need, None) == ALIGN
    assert f(A16, 2, 0, 32, 128, 128, 64, ws, need, None) == OK
    # the planned bit belongs to the prefill only
    assert prefill(lib, l2=8) == INVALID                        # unknown flag bit
    assert decode(lib, l2=4) == INVALID
    assert prefill_noalloc(lib, l2=4) == INVALID


def test_decode_step_fused_validation(lib):
    f = lib.gdn_decode_step_fused
    C = 2 * 16 * 128 + 32 * 128
    N = 4
    sb = N * C * 3 * 2                      # bytes of one conv state buffer
    s_in, s_out = A16, A16 + 0x1000000      # disjoint fake buffers
    args = dict(x=A16, xs=C, w=A16, bias=None, si=s_in, so=s_out, a=A16, b=A16, S=A16, o=A16,
                N=N, Hk=16, Hv=32, dk=128, dv=128, K=4, silu=1, l2=1)

    def call(**kw):
        d = dict(args, **kw)
        return f(d["x"], d["xs"], d["w"], d["bias"], d["si"], d["so"], d["a"], d["b"], d["S"],
                 d["o"], d["N"], d["Hk"], d["Hv"], d["dk"], d["dv"], d["K"], d["silu"], d["l2"],
                 None)

    assert call(N=0) == OK                           # nothing to do, no launch
    assert call(N=-1) == INVALID
    assert call(x=None) == INVALID
    assert call(so=None) == INVALID
    assert call(so=s_in + sb - 16) == INVALID          # output state overlaps the input state
    assert call(si=s_out + 16) == INVALID
    assert call(Hv=24, Hk=16) == INVALID               # Hv % Hk != 0
    assert call(silu=2) == INVALID
    assert call(xs=C - 8) == INVALID                   # row stride shorter than C
    assert call(dk=64, dv=64) == UNSUPPORTED           # the fused path is d = 128 only
    assert call(K=3) == UNSUPPORTED
    assert call(xs=C + 4) == ALIGN
    assert call(x=A8) == ALIGN
    assert call(bias=A8) == ALIGN
    assert call(so=s_out + 8) == ALIGN


def test_state_slot_variants_validation(lib):
    """The *_slots entry points check their slot arguments first, then the
    arguments of the call they extend; nothing launches."""
    conv_args = [A16, 64, A16, None, A16, None, A16, None, None, 0, 18, 64, 4, 2, 1, A16]
    f = lib.gdn_causal_conv1d_fwd_slots
    assert f(*conv_args, None, 4, None) == INVALID                  # no state_indices
    assert f(*conv_args, A16, -1, None) == INVALID                  # negative slot count
    assert f(*conv_args, A16 + 2, 4, None) == ALIGN                 # int32 alignment
    bad = list(conv_args)
    bad[0] = A8
    assert f(*bad, A16, 4, None) == ALIGN                           # the base check still runs
    bad = list(conv_args)
    bad[10] = 0
    assert f(*bad, A16, 4, None) == OK                              # T == 0: nothing to do

    g = lib.gdn_causal_conv1d_update_slots
    assert g(A16, 64, A16, None, A16, 2, 64, 4, 1, A16, None, 4, None) == INVALID
    assert g(A16, 64, A16, None, A16, 2, 64, 5, 1, A16, A16, 4, None) == UNSUPPORTED
    assert g(A16, 64, A16, None, A16, 0, 64, 4, 1, A16, A16, 0, None) == OK

    dec = [A16, A16, 4096, A16, 4096, A16, A16, A16, A16, 32, 16, 32, 128, 128, 0]
    h = lib.gdn_delta_rule_decode_slots
    assert h(*dec, None, 32, None) == INVALID
    assert h(*dec, A16 + 1, 32, None) == ALIGN
    bad = list(dec)
    bad[12] = 96
    assert h(*bad, A16, 32, None) == UNSUPPORTED
    bad = list(dec)
    bad[9] = 0
    assert h(*bad, A16, 32, None) == OK

    pre = [A16, A16, 4096, A16, 4096, A16, A16, A16, 2, 2048, A16, None, A16, 16, 32, 128, 128,
           64, 0, A16 * 16, 1 << 40]
    p = lib.gdn_delta_rule_prefill_chunked_slots
    assert p(*pre, None, 8, None) == INVALID
    assert p(*pre, A16, -3, None) == INVALID
    bad = list(pre)
    bad[20] = 16
    assert p(*bad, A16, 8, None) == WORKSPACE
    bad = list(pre)
    bad[9] = 0
    assert p(*bad, A16, 8, None) == OK


def test_device_status_validation(lib):
    f = lib.gdn_device_status
    assert f(None, 0, None) == INVALID
    assert f(A16, 2, None) == INVALID
    assert f(A16 + 2, 0, None) == ALIGN


def test_selftest_bounded_wait_validation(lib):
    f = lib.gdn_selftest_bounded_wait
    assert f(None, 1000, None) == INVALID
    assert f(A16, 0, None) == INVALID
    assert f(A16, 5000000000, None) == INVALID
