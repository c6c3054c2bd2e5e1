"""Parity gates shared by the GPU tests (tolerances of the method's accept rule)."""

import numpy as np

from oracle import vq3_oracle as O

REL_MAX_ERR = 2e-3      # max|gpu - ref| / max|ref|
MIN_ROW_COSINE = 0.9999  # per output row


def assert_parity(got, ref, what="", rel=REL_MAX_ERR, cos=MIN_ROW_COSINE):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    e = O.rel_max_err(got, ref)
    c = O.row_cosine(got, ref).min() if ref.size else 1.0
    assert e <= rel and c >= cos, f"{what}: rel_max_err={e:.3e} (<= {rel}) min_row_cos={c:.7f} (>= {cos})"
    return e, c
