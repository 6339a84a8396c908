"""Pins for the oracle's TensorScatter step (CPU only).

"Skill: Attention Optimization", "In-place KV for ONNX Attention via
TensorScatter (static cache)": new rows are written into the preallocated
buffer at write_indices, in place; nothing else changes.  The pins are the
identity of a copy: written rows equal the update byte for byte, every other
slot keeps its canary, an empty update changes nothing.
"""
import numpy as np
import pytest

import oracle


def _canary(shape, dt, seed):
    rng = np.random.default_rng(seed)
    if dt == "f32":
        return rng.standard_normal(shape).astype(np.float32)
    return rng.integers(0, 2 ** 16, size=shape, dtype=np.uint16)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_rows_land_at_write_idx_and_nothing_else_moves(dt):
    B, H, L, D, S = 3, 2, 40, 16, 5
    kc, vc = _canary((B, H, L, D), dt, 1), _canary((B, H, L, D), dt, 2)
    k0, v0 = kc.copy(), vc.copy()
    kn, vn = _canary((B, H, S, D), dt, 3), _canary((B, H, S, D), dt, 4)
    w = np.array([0, 17, L - S], np.int64)
    assert oracle.scatter(kc, vc, kn, vn, w) == 0
    for b in range(B):
        sl = slice(w[b], w[b] + S)
        assert kc[b, :, sl].tobytes() == kn[b].tobytes()
        assert vc[b, :, sl].tobytes() == vn[b].tobytes()
        keep = np.ones(L, bool)
        keep[sl] = False
        assert kc[b, :, keep].tobytes() == k0[b, :, keep].tobytes()
        assert vc[b, :, keep].tobytes() == v0[b, :, keep].tobytes()


def test_empty_update_is_a_no_op():
    kc, vc = _canary((2, 2, 8, 8), "bf16", 5), _canary((2, 2, 8, 8), "bf16", 6)
    k0, v0 = kc.copy(), vc.copy()
    e = np.zeros((2, 2, 0, 8), np.uint16)
    assert oracle.scatter(kc, vc, e, e, [3, 8]) == 0
    assert (kc == k0).all() and (vc == v0).all()


def test_out_of_range_batches_are_skipped_and_counted():
    kc, vc = _canary((3, 1, 8, 4), "f32", 7), _canary((3, 1, 8, 4), "f32", 8)
    k0 = kc.copy()
    kn, vn = _canary((3, 1, 3, 4), "f32", 9), _canary((3, 1, 3, 4), "f32", 10)
    assert oracle.scatter(kc, vc, kn, vn, [-1, 6, 5]) == 2
    assert (kc[0] == k0[0]).all() and (kc[1] == k0[1]).all()
    assert (kc[2, :, 5:8] == kn[2]).all()
