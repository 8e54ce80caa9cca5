"""Host-side layout of NVFP4 tensors for the tests: packing of the oracle's e2m1 codes two per
byte, and the block-scale atom layout the library reads and writes (include/coda.h, at
coda_quantize_nvfp4).  Pure data movement: no rounding or arithmetic of the method."""
import numpy as np
import torch

import oracle as O


def pack_codes(q: np.ndarray) -> np.ndarray:
    """uint8 [R, K / 2] from e2m1 values [R, K]: element 2j in the low nibble of byte j."""
    c = O.e2m1_encode(q).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(b: np.ndarray) -> np.ndarray:
    """4-bit codes [R, K] from packed bytes [R, K / 2]."""
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def atom_offsets(R: int, K: int) -> np.ndarray:
    """Byte offset [R, K / 16] of each row's block scales in the atom layout."""
    kc = K // 64
    r = np.arange(R)[:, None]
    kb = np.arange(K // 16)[None, :]
    return ((r // 128) * kc + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + kb % 4


def scale_bytes(R: int, K: int) -> int:
    return -(-R // 128) * (K // 64) * 512


def to_atoms(sf_codes: np.ndarray, R: int, K: int) -> np.ndarray:
    """Atom-layout byte buffer (zeros elsewhere) from e4m3 scale bytes [R, K / 16]."""
    buf = np.zeros(scale_bytes(R, K), dtype=np.uint8)
    buf[atom_offsets(R, K)] = sf_codes
    return buf


def from_atoms(buf: np.ndarray, R: int, K: int) -> np.ndarray:
    return np.asarray(buf, dtype=np.uint8)[atom_offsets(R, K)]


def oracle_nvfp4(x: np.ndarray, s: float, device="cuda"):
    """The oracle's NVFP4 quantisation of x, as device tensors the library reads
    (codes, atom-layout scales) plus the oracle's own values (q, sf)."""
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    q, sf = O.nvfp4_quantize(x, s)
    R, K = q.shape
    codes = torch.from_numpy(pack_codes(q)).to(device)
    scales = torch.from_numpy(to_atoms(O.e4m3_encode(sf), R, K)).to(device)
    return C.Nvfp4(codes, scales, s), q, sf


def nvfp4_values(t, R: int, K: int) -> np.ndarray:
    """float64 values s * sf * q of a device Nvfp4 tensor."""
    q = O.e2m1_decode(unpack_codes(t.codes.cpu().numpy()))
    sf = O.e4m3_decode(from_atoms(t.scales.cpu().numpy(), R, K))
    return O.nvfp4_dequantize(q, sf, t.s)
