"""Pins of the packed-cache byte layout and its bytes-per-token formula."""
import numpy as np
import pytest

from oracle import qwm_oracle as O


@pytest.mark.parametrize("d,r,C,bpt", [(128, 16, 256, 129), (128, 0, 256, 97), (128, 8, 256, 113),
                                       (128, 32, 256, 161), (64, 4, 16, 57), (128, 16, 1024, 130)])
def test_bytes_per_token(d, r, C, bpt):
    # index + K codes + V codes + fp16 (zero, scale) for K and V per group + r fp16
    assert O.bytes_per_token(d, r, C) == bpt
    assert O.tile_layout(d, r, C)["tile_bytes"] == 128 * bpt


def test_sections_are_16_byte_aligned():
    for d, r, C in [(128, 16, 256), (64, 4, 16), (128, 5, 1024), (128, 0, 64)]:
        L = O.tile_layout(d, r, C)
        for k, v in L.items():
            assert v % 16 == 0, (k, v)


def test_encode_decode_roundtrip():
    rng = np.random.default_rng(0)
    d, r, nC = 128, 16, 256
    C = rng.standard_normal((nC, d)).astype(np.float32)
    k = (C[rng.integers(0, nC, 300)] + 0.3 * rng.standard_normal((300, d))).astype(np.float32)
    v = rng.standard_normal((300, d)).astype(np.float32)
    U, _, _ = O.psac_basis(rng.standard_normal((200, d)), r)
    seg = O.append_head(k, v, C, O.group_weights(np.ones(d, np.float32)), U, version=3)
    raw = O.encode_segment(seg, d, r, nC)
    L = O.tile_layout(d, r, nC)
    assert len(raw) == 3 * L["tile_bytes"]
    for t in range(3):
        cnt = min(128, 300 - 128 * t)
        back = O.decode_tile(raw[t * L["tile_bytes"]:(t + 1) * L["tile_bytes"]], cnt, d, r, nC, C, 3)
        sl = slice(128 * t, 128 * t + cnt)
        assert (back.idx == seg.idx[sl]).all()
        assert (back.kcodes == seg.kcodes[sl]).all()
        assert (back.vcodes == seg.vcodes[sl]).all()
        assert np.array_equal(back.e16, seg.e16[sl])
        assert np.array_equal(back.khat, seg.khat[sl])
        assert np.array_equal(back.vhat, seg.vhat[sl])
    # pad slots of the last tile are zero
    last = np.frombuffer(raw[2 * L["tile_bytes"]:], np.uint8)
    assert not last[L["idx"] + 44:L["kcode"]].any()


def test_hand_built_token_bytes():
    """One token, d = 64, r = 1, C = 4: every section's first bytes by hand."""
    d, r, nC = 64, 1, 4
    seg = O.Segment(idx=np.array([2]), kzero=np.array([[1.0, -2.0]], np.float16),
                    kscale=np.array([[0.5, 0.25]], np.float16),
                    kcodes=np.array([[1, 2, 3, 0] * 16], np.uint8),
                    e16=np.array([[1.5]], np.float16),
                    vzero=np.array([[0.0, 1.0]], np.float16), vscale=np.array([[2.0, 4.0]], np.float16),
                    vcodes=np.array([[3] * 64], np.uint8), version=0)
    raw = np.frombuffer(O.encode_segment(seg, d, r, nC), np.uint8)
    L = O.tile_layout(d, r, nC)
    assert raw[L["idx"]] == 2
    assert raw[L["kcode"]] == 0b00111001                       # codes 1,2,3,0
    # (zero, scale) pairs, little-endian fp16: 1.0 = 0x3C00, 0.5 = 0x3800
    assert raw[L["kqp"]:L["kqp"] + 8].tobytes().hex() == "003c0038 00c00034".replace(" ", "")
    assert raw[L["e"]:L["e"] + 2].tobytes().hex() == "003e"  # 1.5 = 0x3E00
    assert raw[L["vcode"]] == 0xFF
    assert raw[L["vqp"]:L["vqp"] + 8].tobytes().hex() == "00000040003c0044"
