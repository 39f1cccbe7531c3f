"""Parity bars of the GPU tests against the oracle, in one place.

The bars the workloads fix: BF16 outputs within 2e-2 relative error, the
float32 recurrent state within 1e-4, descriptors and conv-state bytes exact.
Relative error is max |x - ref| / max |ref| (``oracle.rel_err``), applied
three ways so that a small head or row cannot hide behind a large one:

* delta-rule outputs o [T, Hv, dv]: over the whole tensor, over each v-head
  (all its tokens), and over each (token, v-head) row of dv values, the row's
  scale floored at 1/16 of the tensor's (a row of a token that the gates
  nearly silence is measured against that floor instead of its own tiny
  maximum: its absolute error stays below 2e-2 / 16 of the tensor scale);
* states S [N, Hv, dv, dk]: over each (sequence, v-head) state, its scale
  floored at 1e-30 of the tensor's (the kernels treat decays below 1e-30 as
  1e-30, and float32 flushes values below 2^-126: gates that saturate can
  leave a state of magnitude 1e-39, whose digits lie outside that contract);
* conv outputs: elementwise, one BF16 rounding of a float32 value
  (|y - ref| <= 2^-8 |ref| + 1e-6), as before.
"""
import numpy as np

from oracle import gdn_oracle as O

TOL_BF16 = 2e-2
TOL_STATE = 1e-4
ROW_FLOOR = 1.0 / 16.0
STATE_FLOOR = 1e-30


def o_errors(o, ref):
    """(tensor, worst head, worst row) relative errors of a [T, H, dv] output."""
    o = np.asarray(o, np.float64)
    ref = np.asarray(ref, np.float64)
    tensor = O.rel_err(o, ref)
    per_head = O.rel_err_slices(np.swapaxes(o, 0, 1), np.swapaxes(ref, 0, 1), 2)
    per_row = O.rel_err_slices(o, ref, 1, floor=ROW_FLOOR)
    return tensor, per_head, per_row


def assert_o(o, ref, tol=TOL_BF16):
    errs = o_errors(o, ref)
    assert max(errs) < tol, ("o (tensor, head, row)", errs)
    return errs


def assert_S(S, ref, tol=TOL_STATE):
    """Each (sequence, head) state [dv, dk] against its own scale."""
    e = O.rel_err_slices(np.asarray(S, np.float64), np.asarray(ref, np.float64), 2,
                         floor=STATE_FLOOR)
    assert e < tol, ("S per (sequence, head)", e)
    return e


def assert_conv_y(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert O.rel_err(y, ref) < TOL_BF16
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
