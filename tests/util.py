"""Shared test helpers: the GEMM / MoE output tolerance, written out here.

Outputs are bf16, which keeps 8 significant bits: rounding even the exact
result to bf16 moves it by up to 2^-8 (3.9e-3) relative, so an elementwise
2e-3 relative bound cannot hold for any bf16 output.  The criterion used
instead is stricter where it can be:
  1. elementwise, the GPU value g must be the bf16 rounding of some value
     within tau of the exact result r:  bf16(r - tau) <= g <= bf16(r + tau),
     tau = 2^-18 * alpha * sum_k |deqA deqB| + 2^-22 * |r|.  The first term
     bounds the fp32 accumulation-order error of the tensor cores (its typical
     size is ~2^-24 of that magnitude sum), the second the fp32 alpha /
     epilogue multiplies.  Away from bf16 rounding boundaries this demands the
     correctly rounded bf16 result.
  2. norm-wise, ||g - r|| / ||r|| <= 2e-3.
"""
import numpy as np

import oracle as O

REL = 2e-3
ACC_FLOOR = 2.0 ** -18
MUL_SLACK = 2.0 ** -22


def check_close(got, ref, mag, rel=REL, floor=ACC_FLOOR, what="output", extra_tau=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "%s has non-finite values" % what
    tau = floor * mag + MUL_SLACK * np.abs(ref)
    if extra_tau is not None:
        tau = tau + extra_tau
    lo = O.bf16_round(ref - tau)
    hi = O.bf16_round(ref + tau)
    bad = (got < lo) | (got > hi)
    if bad.any():
        err = np.abs(got - ref)
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        raise AssertionError("%s: %d / %d elements are not a bf16 rounding of the reference within tau; e.g. at %s:"
                             " got %r ref %r tau %r" % (what, bad.sum(), bad.size, i, got[i], ref[i], tau[i]))
    nref = np.linalg.norm(ref)
    if nref > 0:
        nerr = np.linalg.norm(got - ref) / nref
        assert nerr <= rel, "%s: norm-wise relative error %g > %g" % (what, nerr, rel)


def bf16_to_np(t):
    """bf16 torch tensor (any device) -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)
