"""The test helper that reads blocked workspace matrices back agrees with the
per-element layout formula documented in include/mfsdp.h."""
import numpy as np

from tests import helpers as H


def test_unblock_matches_documented_formula():
    rng = np.random.default_rng(0)
    rows_pad, cols_pad = 16, 128
    dense = rng.standard_normal((rows_pad, cols_pad)).astype(np.float32)
    bits = (dense.view(np.uint32) >> 16).astype(np.uint16)
    buf = np.zeros(rows_pad * cols_pad * 2 + 64, np.uint8)
    off = 64
    for r in range(rows_pad):
        for c in range(cols_pad):
            atom = ((c // 64) * (rows_pad // 8) + r // 8) * 1024
            inner = (r % 8) * 128 + ((((c % 64) // 8) ^ (r % 8)) * 16) + (c % 8) * 2
            buf[off + atom + inner: off + atom + inner + 2] = np.frombuffer(bits[r, c].tobytes(), np.uint8)
    out = H.unblock(buf, off, rows_pad, cols_pad)
    assert np.array_equal(out, H.bf16_bits_to_f32(bits))


def test_symmetric_from_upper_restores_lower_blocks():
    rng = np.random.default_rng(5)
    full = rng.standard_normal((768, 768)).astype(np.float32)
    full = full + full.T
    kept = full.copy()
    for i in range(3):
        for j in range(i):
            kept[i * 256:(i + 1) * 256, j * 256:(j + 1) * 256] = np.nan   # never stored
    assert np.array_equal(H.symmetric_from_upper(kept), full)
    # the diagonal 256 x 256 blocks are kept whole, including their lower halves
    assert np.array_equal(H.symmetric_from_upper(kept)[300:400, 260:290], full[300:400, 260:290])
