"""The KV cache page layouts that include/nvfp4.h documents, checked on the
CPU against the test helpers that build the GPU tests' caches (the GPU tests
then check the kernels against the same helpers): every byte offset of a
key code, key scale, value code and value scale, the key-slot formulas, and
the property the slot order exists for (the 8 keys of one score n-tile of
the attention are 8 consecutive slots)."""
import numpy as np

from helpers import kv_pack_fp8, kv_pack_nvfp4, kv_unpack_fp8, kv_unpack_nvfp4


def slot4(k):   # NVFP4: token k of a half page -> key slot (nvfp4.h)
    return 8 * ((k >> 1) & 3) + 2 * (k >> 3) + (k & 1)


def slot8(k):   # FP8
    return (k & 16) | ((k & 2) << 2) | ((k >> 1) & 6) | (k & 1)


def test_slot_orders_are_permutations_that_group_score_tiles():
    assert sorted(slot4(k) for k in range(32)) == list(range(32))
    assert sorted(slot8(k) for k in range(32)) == list(range(32))
    for j in range(4):
        for n in range(8):
            # keys of column n of score n-tile j (NVFP4: four 8-key groups
            # interleaved two by two; FP8: the same within 16-key halves)
            k4 = 8 * (n >> 1) + (n & 1) + 2 * j
            k8 = 16 * (j >> 1) + 4 * (n >> 1) + (n & 1) + 2 * (j & 1)
            assert slot4(k4) == 8 * j + n
            assert slot8(k8) == 8 * j + n


def test_nvfp4_page_block_offsets():
    rng = np.random.default_rng(7)
    kc, vc = (rng.integers(0, 256, (2, 64, 64)).astype(np.uint8) for _ in range(2))
    ks, vs = (rng.integers(0, 256, (2, 64, 8)).astype(np.uint8) for _ in range(2))
    b = kv_pack_nvfp4(kc, ks, vc, vs)
    assert b.shape == (2, 9216)
    for p in range(2):
        for tok in range(64):
            h, k = divmod(tok, 32)
            base = 4608 * h
            for q in range(4):          # key codes: [4 dim chunks][32 slots][16 B]
                off = base + (q * 32 + slot4(k)) * 16
                assert np.array_equal(b[p, off:off + 16], kc[p, tok, 16 * q:16 * q + 16])
            off = base + 2048 + slot4(k) * 8
            assert np.array_equal(b[p, off:off + 8], ks[p, tok])
            for d in range(128):        # value codes: [128 dims][16 B], tokens 2j, 2j+1 in byte j
                nib = (vc[p, tok, d // 2] >> (4 * (d & 1))) & 15
                byte = b[p, base + 2304 + d * 16 + k // 2]
                assert (byte >> (4 * (k & 1))) & 15 == nib
            for blk in range(8):        # value scales: [8 blocks][32 tokens]
                assert b[p, base + 4352 + blk * 32 + k] == vs[p, tok, blk]
    back = kv_unpack_nvfp4(b)
    for x, y in zip(back, (kc, ks, vc, vs)):
        assert np.array_equal(x, y)


def test_fp8_page_block_offsets():
    rng = np.random.default_rng(8)
    k, v = (rng.integers(0, 256, (2, 64, 128)).astype(np.uint8) for _ in range(2))
    b = kv_pack_fp8(k, v)
    assert b.shape == (2, 16384)
    for p in range(2):
        for tok in range(64):
            h, t = divmod(tok, 32)
            base = 8192 * h
            for q in range(8):          # keys: [8 dim chunks][32 slots][16 B]
                off = base + (q * 32 + slot8(t)) * 16
                assert np.array_equal(b[p, off:off + 16], k[p, tok, 16 * q:16 * q + 16])
            u, j = divmod(t, 16)        # values: [2 token groups][128 dims][16 B]
            rows = base + 4096 + (u * 128 + np.arange(128)) * 16 + j
            assert np.array_equal(b[p, rows], v[p, tok])
    kk, vv = kv_unpack_fp8(b)
    assert np.array_equal(kk, k) and np.array_equal(vv, v)
