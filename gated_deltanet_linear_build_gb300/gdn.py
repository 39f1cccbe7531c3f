"""Python binding of the GDN C ABI (``include/gdn.h``), via ctypes.

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream of PyTorch to the library entry point of the same name
and raises ``GdnError`` on a non-zero status. No arithmetic of the method
happens here, and there is no fallback: if ``libgdn_gb300.so`` is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_ALIGNMENT = -3
GDN_ERR_WORKSPACE = -4
GDN_ERR_CUDA = -5
GDN_ERR_TIMEOUT = -6

# Option bits of the delta-rule calls' flags argument (GDN_FLAG_* in gdn.h).
GDN_FLAG_QK_L2NORM = 1
GDN_FLAG_GATE_LOGITS = 2
GDN_FLAG_PLANNED = 4

# Every symbol that include/gdn.h declares.
EXPORTED_SYMBOLS = (
    "gdn_build_conv_chunks",
    "gdn_causal_conv1d_fwd",
    "gdn_causal_conv1d_update",
    "gdn_delta_rule_decode",
    "gdn_decode_step_fused",
    "gdn_delta_rule_prefill_workspace_size",
    "gdn_delta_rule_prefill_chunked",
    "gdn_delta_rule_prefill_plan",
    "gdn_delta_rule_prefill_chunked_noalloc",
    "gdn_delta_rule_prefill_chunked_noalloc_status",
    "gdn_causal_conv1d_fwd_slots",
    "gdn_causal_conv1d_update_slots",
    "gdn_delta_rule_decode_slots",
    "gdn_delta_rule_prefill_chunked_slots",
    "gdn_selftest_bounded_wait",
    "gdn_device_status",
    "gdn_status_string",
    "gdn_last_cuda_error_string",
)


class GdnError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        text = _LIB.gdn_status_string(status).decode() if _LIB is not None else str(status)
        if status == GDN_ERR_CUDA and _LIB is not None:
            text += " (" + _LIB.gdn_last_cuda_error_string().decode() + ")"
        super().__init__(f"{fn}: {text}")


_LIB = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64

_SIGNATURES = {
    "gdn_build_conv_chunks": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _P]),
    "gdn_causal_conv1d_fwd": (ctypes.c_int, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _I32,
                                             _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "gdn_causal_conv1d_update": (ctypes.c_int, [_P, _I64, _P, _P, _P, _I32, _I32, _I32, _I32,
                                                _P, _P]),
    "gdn_delta_rule_decode": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P, _P, _I32, _I32,
                                             _I32, _I32, _I32, _I32, _P]),
    "gdn_decode_step_fused": (ctypes.c_int, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                             _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "gdn_delta_rule_prefill_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32, _I32, _I32,
                                                                _I32]),
    "gdn_delta_rule_prefill_chunked": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P, _I32,
                                                      _I32, _P, _P, _P, _I32, _I32, _I32, _I32,
                                                      _I32, _I32, _P, ctypes.c_size_t, _P]),
    "gdn_delta_rule_prefill_plan": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                                   ctypes.c_size_t, _P]),
    "gdn_delta_rule_prefill_chunked_noalloc": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P,
                                                              _I32, _I32, _P, _P, _P, _I32, _I32,
                                                              _I32, _I32, _I32, _I32, _P]),
    "gdn_delta_rule_prefill_chunked_noalloc_status": (ctypes.c_int, [_P, _P]),
    "gdn_causal_conv1d_fwd_slots": (ctypes.c_int, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _I32,
                                                   _I32, _I32, _I32, _I32, _I32, _P, _P, _I32,
                                                   _P]),
    "gdn_causal_conv1d_update_slots": (ctypes.c_int, [_P, _I64, _P, _P, _P, _I32, _I32, _I32,
                                                      _I32, _P, _P, _I32, _P]),
    "gdn_delta_rule_decode_slots": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P, _P, _I32,
                                                   _I32, _I32, _I32, _I32, _I32, _P, _I32, _P]),
    "gdn_delta_rule_prefill_chunked_slots": (ctypes.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P,
                                                            _I32, _I32, _P, _P, _P, _I32, _I32,
                                                            _I32, _I32, _I32, _I32, _P,
                                                            ctypes.c_size_t, _P, _I32, _P]),
    "gdn_selftest_bounded_wait": (ctypes.c_int, [_P, _I64, _P]),
    "gdn_device_status": (ctypes.c_int, [_P, _I32, _P]),
    "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_last_cuda_error_string": (ctypes.c_char_p, []),
}


def load_library(path: str = LIB_PATH):
    """Load the shared library (once) and declare its signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"GDN CUDA library not built: {path} is missing "
                           "(run __graft_entry__.build() or python -m "
                           "gated_deltanet_linear_build_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _lib():
    return _LIB if _LIB is not None else load_library()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _flags(qk_l2norm: bool, gate_logits: bool, planned: bool = False) -> int:
    return ((GDN_FLAG_QK_L2NORM if qk_l2norm else 0) | (GDN_FLAG_GATE_LOGITS if gate_logits else 0)
            | (GDN_FLAG_PLANNED if planned else 0))


def _check(rc: int, fn: str):
    if rc != GDN_OK:
        raise GdnError(rc, fn)


# ----------------------------------------------------------------------------
# Entry points (same names as the C ABI, without the gdn_ prefix)
# ----------------------------------------------------------------------------

def build_conv_chunks(cu_seqlens, chunks, num_chunks, *, chunk_tokens: int = 8,
                      device_status=None, stream=None):
    """Descriptors of the exact (sequence, chunk) dispatch.

    cu_seqlens int32 [N+1]; chunks int32 [capacity, 4] (output); num_chunks
    int32 [1] (output); device_status int32 [1] or None.
    """
    n = cu_seqlens.numel() - 1
    rc = _lib().gdn_build_conv_chunks(_ptr(cu_seqlens), n, chunk_tokens, _ptr(chunks),
                                      chunks.shape[0] if chunks is not None else 0,
                                      _ptr(num_chunks), _ptr(device_status), _stream(stream))
    _check(rc, "gdn_build_conv_chunks")


def causal_conv1d_fwd(x, w, bias, conv_state, has_initial_state, cu_seqlens, y, *,
                      chunks=None, num_chunks=None, silu: bool = True, stream=None):
    """Varlen causal conv prefill. x [T, C] (row stride x.stride(0)), w [C, 4],
    bias [C] or None, conv_state [N, C, 3], has_initial_state uint8 [N] or None,
    y [T, C]. chunks/num_chunks as built by build_conv_chunks, or both None for
    whole-sequence dispatch."""
    T, C = x.shape
    N = cu_seqlens.numel() - 1
    rc = _lib().gdn_causal_conv1d_fwd(
        _ptr(x), x.stride(0), _ptr(w), _ptr(bias), _ptr(conv_state), _ptr(has_initial_state),
        _ptr(cu_seqlens), _ptr(chunks), _ptr(num_chunks),
        chunks.shape[0] if chunks is not None else 0, T, C, w.shape[1], N, int(silu), _ptr(y),
        _stream(stream))
    _check(rc, "gdn_causal_conv1d_fwd")


def causal_conv1d_update(x, w, bias, conv_state, y, *, silu: bool = True, stream=None):
    """One decode token per sequence: x [N, C], conv_state [N, C, 3], y [N, C]."""
    N, C = x.shape
    rc = _lib().gdn_causal_conv1d_update(_ptr(x), x.stride(0), _ptr(w), _ptr(bias),
                                         _ptr(conv_state), N, C, w.shape[1], int(silu),
                                         _ptr(y), _stream(stream))
    _check(rc, "gdn_causal_conv1d_update")


def delta_rule_decode(q, k, v, a, b, S, o, *, qk_l2norm: bool = False, gate_logits: bool = False, stream=None):
    """Decode update. q, k [N, Hk, dk] (token stride q.stride(0), heads
    contiguous), v [N, Hv, dv], a, b [N, Hv] float32 (activated gates, or their
    logits with gate_logits=True: the kernel then computes a = exp(-softplus(a)),
    b = sigmoid(b)), S [N, Hv, dv, dk] float32 (in place), o [N, Hv, dv]."""
    N, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert k.stride(0) == q.stride(0), "q and k share one token stride"
    rc = _lib().gdn_delta_rule_decode(_ptr(q), _ptr(k), q.stride(0), _ptr(v), v.stride(0),
                                      _ptr(a), _ptr(b), _ptr(S), _ptr(o), N, Hk, Hv, dk, dv,
                                      _flags(qk_l2norm, gate_logits), _stream(stream))
    _check(rc, "gdn_delta_rule_decode")


def decode_step_fused(x, w, bias, conv_state_in, conv_state_out, a, b, S, o, *, Hk: int,
                      silu: bool = True, qk_l2norm: bool = False, gate_logits: bool = False, stream=None):
    """Conv update and delta-rule decode in one launch. x [N, C] conv inputs
    (C = 2 Hk d + Hv d), conv_state_in / conv_state_out [N, C, 3] (distinct
    buffers), a, b [N, Hv], S [N, Hv, d, d] (in place), o [N, Hv, d]."""
    N = x.shape[0]
    Hv, dv, dk = S.shape[1], S.shape[2], S.shape[3]
    rc = _lib().gdn_decode_step_fused(_ptr(x), x.stride(0), _ptr(w), _ptr(bias),
                                      _ptr(conv_state_in), _ptr(conv_state_out), _ptr(a),
                                      _ptr(b), _ptr(S), _ptr(o), N, Hk, Hv, dk, dv, w.shape[1],
                                      int(silu), _flags(qk_l2norm, gate_logits), _stream(stream))
    _check(rc, "gdn_decode_step_fused")


def delta_rule_prefill_workspace_size(T: int, N: int, Hv: int, dk: int, dv: int,
                                      chunk: int = 64) -> int:
    return int(_lib().gdn_delta_rule_prefill_workspace_size(T, N, Hv, dk, dv, chunk))


def delta_rule_prefill_plan(cu_seqlens, T: int, Hv: int, dk: int, dv: int, workspace, *,
                            chunk: int = 64, stream=None):
    """Build the chunk plan of cu_seqlens into ``workspace`` once per engine
    step; the step's prefill calls then pass planned=True and reuse it."""
    N = cu_seqlens.numel() - 1
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib().gdn_delta_rule_prefill_plan(_ptr(cu_seqlens), N, T, Hv, dk, dv, chunk,
                                            _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "gdn_delta_rule_prefill_plan")


def delta_rule_prefill_chunked(q, k, v, a, b, cu_seqlens, S, has_initial_state, o, workspace,
                               *, chunk: int = 64, qk_l2norm: bool = False,
                               gate_logits: bool = False, planned: bool = False, stream=None):
    """Chunked prefill over packed sequences. q, k [T, Hk, dk]; v [T, Hv, dv];
    a, b [T, Hv]; cu_seqlens [N+1]; S [N, Hv, dv, dk] (initial in, final out);
    has_initial_state uint8 [N] or None; o [T, Hv, dv]; workspace uint8 tensor
    of at least delta_rule_prefill_workspace_size(...) bytes."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    assert k.stride(0) == q.stride(0), "q and k share one token stride"
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib().gdn_delta_rule_prefill_chunked(
        _ptr(q), _ptr(k), q.stride(0), _ptr(v), v.stride(0), _ptr(a), _ptr(b),
        _ptr(cu_seqlens), N, T, _ptr(S), _ptr(has_initial_state), _ptr(o), Hk, Hv, dk, dv,
        chunk, _flags(qk_l2norm, gate_logits, planned), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "gdn_delta_rule_prefill_chunked")


def delta_rule_prefill_chunked_noalloc(q, k, v, a, b, cu_seqlens, S, has_initial_state, o, *,
                                       chunk: int = 64, qk_l2norm: bool = False, gate_logits: bool = False, stream=None):
    """The chunked prefill without a workspace argument, for callers that may
    not allocate device memory: scratch is the library's fixed 64 MiB device
    array. Same arguments and results as delta_rule_prefill_chunked. Calls
    that overlap on the GPU share that array and must be serialised."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    assert k.stride(0) == q.stride(0), "q and k share one token stride"
    rc = _lib().gdn_delta_rule_prefill_chunked_noalloc(
        _ptr(q), _ptr(k), q.stride(0), _ptr(v), v.stride(0), _ptr(a), _ptr(b),
        _ptr(cu_seqlens), N, T, _ptr(S), _ptr(has_initial_state), _ptr(o), Hk, Hv, dk, dv,
        chunk, _flags(qk_l2norm, gate_logits), _stream(stream))
    _check(rc, "gdn_delta_rule_prefill_chunked_noalloc")


def delta_rule_prefill_chunked_noalloc_status(status, *, stream=None):
    """Copy the two device-side status words of the last allocation-free
    prefill (descriptor builder, state pass) into ``status`` (int32 [2], on
    the device or in host memory), on the stream."""
    rc = _lib().gdn_delta_rule_prefill_chunked_noalloc_status(_ptr(status), _stream(stream))
    _check(rc, "gdn_delta_rule_prefill_chunked_noalloc_status")


# ----------------------------------------------------------------------------
# State-slot variants: conv_state [num_slots, C, 3] and S [num_slots, Hv, dv, dk]
# form a cache; sequence n of the batch uses slot state_indices[n] (device
# int32 [N]); an index outside [0, num_slots) is a padding entry whose state
# and outputs are left untouched. num_slots defaults to the cache's first
# dimension.
# ----------------------------------------------------------------------------

def causal_conv1d_fwd_slots(x, w, bias, conv_state, has_initial_state, cu_seqlens, y,
                            state_indices, *, num_slots=None, chunks=None, num_chunks=None,
                            silu: bool = True, stream=None):
    T, C = x.shape
    N = cu_seqlens.numel() - 1
    ns = conv_state.shape[0] if num_slots is None else num_slots
    rc = _lib().gdn_causal_conv1d_fwd_slots(
        _ptr(x), x.stride(0), _ptr(w), _ptr(bias), _ptr(conv_state), _ptr(has_initial_state),
        _ptr(cu_seqlens), _ptr(chunks), _ptr(num_chunks),
        chunks.shape[0] if chunks is not None else 0, T, C, w.shape[1], N, int(silu), _ptr(y),
        _ptr(state_indices), ns, _stream(stream))
    _check(rc, "gdn_causal_conv1d_fwd_slots")


def causal_conv1d_update_slots(x, w, bias, conv_state, y, state_indices, *, num_slots=None,
                               silu: bool = True, stream=None):
    N, C = x.shape
    ns = conv_state.shape[0] if num_slots is None else num_slots
    rc = _lib().gdn_causal_conv1d_update_slots(_ptr(x), x.stride(0), _ptr(w), _ptr(bias),
                                               _ptr(conv_state), N, C, w.shape[1], int(silu),
                                               _ptr(y), _ptr(state_indices), ns, _stream(stream))
    _check(rc, "gdn_causal_conv1d_update_slots")


def delta_rule_decode_slots(q, k, v, a, b, S, o, state_indices, *, num_slots=None,
                            qk_l2norm: bool = False, gate_logits: bool = False, stream=None):
    N, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert k.stride(0) == q.stride(0), "q and k share one token stride"
    ns = S.shape[0] if num_slots is None else num_slots
    rc = _lib().gdn_delta_rule_decode_slots(_ptr(q), _ptr(k), q.stride(0), _ptr(v), v.stride(0),
                                            _ptr(a), _ptr(b), _ptr(S), _ptr(o), N, Hk, Hv, dk,
                                            dv, _flags(qk_l2norm, gate_logits), _ptr(state_indices), ns,
                                            _stream(stream))
    _check(rc, "gdn_delta_rule_decode_slots")


def delta_rule_prefill_chunked_slots(q, k, v, a, b, cu_seqlens, S, has_initial_state, o,
                                     workspace, state_indices, *, num_slots=None,
                                     chunk: int = 64, qk_l2norm: bool = False, gate_logits: bool = False, stream=None):
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    assert k.stride(0) == q.stride(0), "q and k share one token stride"
    ns = S.shape[0] if num_slots is None else num_slots
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib().gdn_delta_rule_prefill_chunked_slots(
        _ptr(q), _ptr(k), q.stride(0), _ptr(v), v.stride(0), _ptr(a), _ptr(b),
        _ptr(cu_seqlens), N, T, _ptr(S), _ptr(has_initial_state), _ptr(o), Hk, Hv, dk, dv,
        chunk, _flags(qk_l2norm, gate_logits), _ptr(workspace), nbytes, _ptr(state_indices), ns, _stream(stream))
    _check(rc, "gdn_delta_rule_prefill_chunked_slots")


def selftest_bounded_wait(device_status, *, max_cycles: int = 2_000_000, stream=None):
    """One CTA waits for an mbarrier phase that nothing completes, with the
    library's bounded wait; device_status int32 [1] becomes GDN_ERR_TIMEOUT."""
    rc = _lib().gdn_selftest_bounded_wait(_ptr(device_status), int(max_cycles), _stream(stream))
    _check(rc, "gdn_selftest_bounded_wait")


def device_status(status, *, clear: bool = False, stream=None):
    """Enqueue the read of the library's sticky device status into ``status``
    (device int32 [1]): GDN_OK, or the first failure a kernel recorded
    (GDN_ERR_TIMEOUT) since the last clear; ``clear`` resets it."""
    rc = _lib().gdn_device_status(_ptr(status), int(clear), _stream(stream))
    _check(rc, "gdn_device_status")


def prefill_workspace_status(workspace):
    """(descriptor builder status, state pass status) from a prefill workspace
    once the call has completed (words 1 and 2)."""
    w = workspace[:12].view(torch.int32).cpu()
    return int(w[1]), int(w[2])


def status_string(status: int) -> str:
    return _lib().gdn_status_string(status).decode()
