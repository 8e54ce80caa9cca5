"""The test-side NVFP4 layout helpers (code packing, block-scale atoms) on the CPU: packing
round-trips, the atom offsets are a one-to-one map into the buffer, and each row's scales sit
where the MMA reads them."""
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
    for R, K in [(300, 512), (256, 192), (128, 64)]:
        off = L.atom_offsets(R, K)
        assert off.shape == (R, K // 16)
        assert len(np.unique(off)) == off.size
        assert off.max() < L.scale_bytes(R, K)
        sf = np.arange(off.size, dtype=np.uint64).reshape(off.shape).astype(np.uint8)
        np.testing.assert_array_equal(L.from_atoms(L.to_atoms(sf, R, K), R, K), sf)


def test_atom_rows_match_the_mma_reading_order():
    # a 32-lane copy of an atom puts its 16-byte row i in lanes i, 32 + i, 64 + i, 96 + i,
    # four bytes per column; the MMA reads row m in lane m, column (m % 128) / 32: so row m's
    # four scales must be bytes 4 ((m % 128) / 32) of the atom's row m % 32
    off = L.atom_offsets(256, 64)
    for m in (0, 5, 37, 70, 127, 200):
        assert list(off[m]) == [(m // 128) * 512 + 16 * (m % 32) + 4 * ((m % 128) // 32) + i for i in range(4)]
