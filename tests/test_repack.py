"""Host-side conversion of a plainly packed int4 checkpoint into the library's
code layout (spec_repack_w4_codes; no GPU).  Pinned against the oracle's
independent nibble decoder and the input generator's packer."""
import numpy as np
import pytest

import oracle
import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import inputs


def _plain_pack(codes: np.ndarray) -> np.ndarray:
    # byte i of a row: k = 2i in the low nibble, k = 2i + 1 in the high one
    c = codes.astype(np.uint8)
    return np.ascontiguousarray(c[:, 0::2] | (c[:, 1::2] << 4))


@pytest.mark.parametrize("N,K", [(1, 8), (3, 64), (64, 4096)])
def test_repack_matches_oracle_decoder_and_packer(N, K):
    rng = np.random.default_rng(N * 131 + K)
    codes = rng.integers(0, 16, size=(N, K))
    src = _plain_pack(codes)
    dst = np.empty_like(src)
    sv.spec_repack_w4_codes(src, dst, N, K)
    np.testing.assert_array_equal(oracle.unpack_w4_codes(dst, N, K), codes)
    np.testing.assert_array_equal(dst, inputs.pack_w4_codes(codes))


def test_repack_hand_example():
    # k = 0..7 carry codes 1..8: plain bytes 0x21 0x43 0x65 0x87 become
    # (k0|k2<<4, k4|k6<<4, k1|k3<<4, k5|k7<<4) = 0x31 0x75 0x42 0x86
    src = np.array([[0x21, 0x43, 0x65, 0x87]], dtype=np.uint8)
    dst = np.empty_like(src)
    sv.spec_repack_w4_codes(src, dst, 1, 8)
    assert dst.tolist() == [[0x31, 0x75, 0x42, 0x86]]


def test_repack_in_place_and_rejects_bad_shapes():
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 16, size=(5, 128))
    buf = _plain_pack(codes)
    sv.spec_repack_w4_codes(buf, buf, 5, 128)
    np.testing.assert_array_equal(oracle.unpack_w4_codes(buf, 5, 128), codes)
    small = np.zeros((1, 2), dtype=np.uint8)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_repack_w4_codes(small, small, 1, 4)
    assert e.value.status == -2
