"""The test-side NVFP4 layout helpers (code packing, block-scale atoms) on the CPU: packing
round-trips, and the atom offsets are a one-to-one map into the buffer, in pair order too."""
import numpy as np

import oracle as O
from tests import nvfp4_layout as L


def test_pack_unpack_round_trip_and_nibble_order():
    rng = np.random.default_rng(3)
    q = O.e2m1_decode(rng.integers(0, 16, size=(5, 64)))
    b = L.pack_codes(q)
    assert b.shape == (5, 32)
    np.testing.assert_array_equal(O.e2m1_decode(L.unpack_codes(b)), q)
    assert b[0, 0] == (O.e2m1_encode(q[0, 0]) | (O.e2m1_encode(q[0, 1]) << 4))


def test_atom_offsets_are_one_to_one():
    for R, K, pair in [(300, 512, 0), (256, 192, 128), (128, 64, 0)]:
        off = L.atom_offsets(R, K, pair)
        assert off.shape == (R, K // 16)
        assert len(np.unique(off)) == off.size
        assert off.max() < L.scale_bytes(R, K)
        sf = np.arange(off.size, dtype=np.uint64).reshape(off.shape).astype(np.uint8)
        np.testing.assert_array_equal(L.from_atoms(L.to_atoms(sf, R, K, pair), R, K, pair), sf)


def test_pair_order_puts_gate_and_up_rows_of_a_group_in_one_block():
    off = L.atom_offsets(256, 64, pair_half=128)
    # gate row 3 and up row 128 + 3 share scale block 0, at scale rows 3 and 64 + 3
    assert off[3, 0] == 16 * 3 and off[131, 0] == 16 * 3 + 4 * 2
    assert off[64, 0] == 512 and off[192, 0] == 512 + 4 * 2   # the next group: the next 128-row block
