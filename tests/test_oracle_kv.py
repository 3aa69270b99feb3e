"""Pins for the oracle's NVFP4 KV cache and decode attention.

Encode: the cache encode is the given-scale block encode of the BF16 values
(checked against the tensor-mode encoder at the tensor's own scale, whose
pins are in test_oracle_encode.py).  Attention: a single cached token
returns its value vector; equal keys give the mean of the values; a
hand-evaluated two-token case with exactly decodable keys and values;
invariance under page placement and token order; doubling the values
doubles the output, while the tensor scale alone does not change it; grouped
query heads sharing a KV head; an empty context."""
import math

import numpy as np
import pytest

import synth

P = 64


def paged(orc, rows_bf16, s, pages_of_seq, n_pages, H_kv, D, seq_heads):
    """Encode vectors into a page pool: rows_bf16[b][hk] is [n_b, D] BF16."""
    codes = np.zeros((n_pages, H_kv, P, D // 2), np.uint8)
    scales = np.zeros((n_pages, H_kv, P, D // 16), np.uint8)
    for b, per_head in enumerate(rows_bf16):
        for hk in range(H_kv):
            c, sc = orc.kv_encode(per_head[hk], s)
            for t in range(c.shape[0]):
                pg = pages_of_seq[b][t // P]
                codes[pg, hk, t % P] = c[t]
                scales[pg, hk, t % P] = sc[t]
    return codes, scales


def test_kv_encode_is_the_tensor_encoder_at_its_own_scale(orc):
    x = synth.activations(9, 90, 40, 128, 0.02, 30.0)
    c, s_, sg = orc.nvfp4_encode(x)
    c2, s2 = orc.kv_encode(x, sg)
    np.testing.assert_array_equal(c, c2)
    np.testing.assert_array_equal(s_, s2)


def _single_seq(orc, K_bf16, V_bf16, s_k=0.01, s_v=0.01, table=None):
    n, D = K_bf16.shape
    npg = -(-n // P)
    table = list(range(npg)) if table is None else table
    kc = paged(orc, [[K_bf16]], s_k, [table], max(table) + 1, 1, D, None)
    vc = paged(orc, [[V_bf16]], s_v, [table], max(table) + 1, 1, D, None)
    return kc, vc, np.array([table + [0]]), np.array([n])


def test_single_token_returns_its_value(orc):
    rng = np.random.default_rng(1)
    D = 128
    K = synth.bf16_bits(rng.standard_normal((1, D)).astype(np.float32))
    V = synth.bf16_bits(rng.standard_normal((1, D)).astype(np.float32))
    kc, vc, bt, cl = _single_seq(orc, K, V)
    q = rng.standard_normal((1, 1, D))
    o = orc.decode_attention(q, kc, vc, 0.01, 0.01, bt, cl, 1 / math.sqrt(D))
    vdq = orc.nvfp4_dequant(*orc.kv_encode(V, 0.01), 0.01)
    np.testing.assert_allclose(o[0, 0], vdq[0], rtol=1e-15, atol=0)


def test_equal_keys_average_the_values(orc):
    rng = np.random.default_rng(2)
    D, n = 128, 70
    K = np.tile(synth.bf16_bits(rng.standard_normal((1, D)).astype(np.float32)), (n, 1))
    V = synth.bf16_bits(rng.standard_normal((n, D)).astype(np.float32))
    kc, vc, bt, cl = _single_seq(orc, K, V)
    o = orc.decode_attention(rng.standard_normal((1, 1, D)), kc, vc, 0.01, 0.01, bt, cl, 0.1)
    vdq = orc.nvfp4_dequant(*orc.kv_encode(V, 0.01), 0.01)
    np.testing.assert_allclose(o[0, 0], vdq.mean(axis=0), rtol=1e-12, atol=1e-15)


def test_two_tokens_by_hand(orc):
    # D = 16, tensor scale 2^-10.  Keys 0.375 e0 and 0.75 e0: each block's
    # maximum is 6 * 2^k, so t = amax/6, u = t/s and the block scale are exact
    # powers of two and the keys decode exactly; values +-0.375 e3 likewise.
    # Query 1.5 e0, softmax scale 0.5: scores 0.28125 and 0.5625.
    D = 16
    s = 2.0 ** -10
    K = synth.bf16_bits(np.array([[0.375] + [0.0] * 15, [0.75] + [0.0] * 15], np.float32))
    V = synth.bf16_bits(np.array([[0, 0, 0, 0.375] + [0.0] * 12, [0, 0, 0, -0.375] + [0.0] * 12], np.float32))
    kc, vc, bt, cl = _single_seq(orc, K, V, s, s)
    kd = orc.nvfp4_dequant(*orc.kv_encode(K, s), s)
    vd = orc.nvfp4_dequant(*orc.kv_encode(V, s), s)
    assert kd[0, 0] == 0.375 and kd[1, 0] == 0.75 and vd[0, 3] == 0.375 and vd[1, 3] == -0.375
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.5
    o = orc.decode_attention(q, kc, vc, s, s, bt, cl, 0.5)
    w1, w2 = math.exp(0.28125), math.exp(0.5625)
    assert o[0, 0, 3] == pytest.approx(0.375 * (w1 - w2) / (w1 + w2), rel=1e-14)
    assert np.count_nonzero(o) == 1


def test_page_placement_token_order_and_linearity(orc):
    rng = np.random.default_rng(3)
    D, n = 128, 150
    K = synth.bf16_bits(rng.standard_normal((n, D)).astype(np.float32))
    V = synth.bf16_bits(rng.standard_normal((n, D)).astype(np.float32))
    q = rng.standard_normal((1, 1, D))
    a = orc.decode_attention(q, *_single_seq(orc, K, V)[:2], 0.01, 0.01, *_single_seq(orc, K, V)[2:], 0.09)
    kc, vc, bt, cl = _single_seq(orc, K, V, table=[5, 1, 3])
    b = orc.decode_attention(q, kc, vc, 0.01, 0.01, bt, cl, 0.09)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
    perm = rng.permutation(n)
    kc, vc, bt, cl = _single_seq(orc, K[perm], V[perm])
    c = orc.decode_attention(q, kc, vc, 0.01, 0.01, bt, cl, 0.09)
    np.testing.assert_allclose(a, c, rtol=1e-12, atol=1e-14)
    # doubling the values (exact in BF16) doubles every block scale and the
    # output; the tensor scale itself only moves the split between the block
    # scale and itself, so the decoded values stay the same
    V2 = synth.bf16_bits(2 * orc.bf16_to_f32(V))
    kc, vc, bt, cl = _single_seq(orc, K, V2)
    d = orc.decode_attention(q, kc, vc, 0.01, 0.01, bt, cl, 0.09)
    np.testing.assert_allclose(d, 2 * a, rtol=1e-13, atol=1e-15)
    kc, vc, bt, cl = _single_seq(orc, K, V, s_v=0.02)
    e = orc.decode_attention(q, kc, vc, 0.01, 0.02, bt, cl, 0.09)
    np.testing.assert_allclose(e, a, rtol=1e-13, atol=1e-15)


def test_grouped_query_heads_share_a_kv_head(orc):
    rng = np.random.default_rng(4)
    D, n, H_kv, G = 64, 90, 2, 3
    Ks = [synth.bf16_bits(rng.standard_normal((n, D)).astype(np.float32)) for _ in range(H_kv)]
    Vs = [synth.bf16_bits(rng.standard_normal((n, D)).astype(np.float32)) for _ in range(H_kv)]
    table = [[0, 1]]
    kc = paged(orc, [Ks], 0.01, table, 2, H_kv, D, None)
    vc = paged(orc, [Vs], 0.01, table, 2, H_kv, D, None)
    q = rng.standard_normal((1, H_kv * G, D))
    o = orc.decode_attention(q, kc, vc, 0.01, 0.01, np.array(table), np.array([n]), 0.125)
    for h in range(H_kv * G):
        hk = h // G
        kcs, vcs, bt, cl = _single_seq(orc, Ks[hk], Vs[hk])
        ref = orc.decode_attention(q[:, h:h + 1], kcs, vcs, 0.01, 0.01, bt, cl, 0.125)
        np.testing.assert_allclose(o[0, h], ref[0, 0], rtol=1e-13, atol=1e-15)
    # an empty context gives zeros
    z = orc.decode_attention(q, kc, vc, 0.01, 0.01, np.array(table), np.array([0]), 0.125)
    assert not z.any()


def test_fp8_encode_matches_the_token_quantiser_and_torch(orc):
    # one row at its own amax / 448 scale is exactly the per-token FP8 encode
    x = synth.activations(9, 91, 1, 128, 0.02, 30.0)
    a, st = orc.fp8_token_encode(x)
    np.testing.assert_array_equal(orc.kv_encode_fp8(x, st[0]), a)
    # in-range products round like torch's E4M3 cast (an independent library)
    import torch
    xs = synth.activations(9, 92, 16, 128, 0.0, 1.0)
    s = np.float32(0.01)
    c = orc.kv_encode_fp8(xs, s)
    prod = (orc.bf16_to_f32(xs) * (np.float32(1) / s)).astype(np.float32)
    assert np.abs(prod).max() < 448
    ref = torch.from_numpy(prod).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(c, ref)
    # saturation at +-448 and exact decoding of E4M3 multiples of s
    big = synth.bf16_bits(np.array([[1e4, -1e4, 2.0, 0.0]], np.float32))
    np.testing.assert_array_equal(orc.kv_encode_fp8(big, 1.0), [[0x7E, 0xFE, 0x40, 0x00]])


def test_fp8_attention_matches_the_fp4_formula_on_decoded_values(orc):
    # the same attention definition over FP8 codes: single token and a
    # hand-built two-token case with exactly representable values
    D = 16
    K = synth.bf16_bits(np.array([[0.375] + [0.0] * 15, [0.75] + [0.0] * 15], np.float32))
    V = synth.bf16_bits(np.array([[0, 0, 0, 0.375] + [0.0] * 12, [0, 0, 0, -0.375] + [0.0] * 12], np.float32))
    s = 2.0 ** -6
    kc = np.zeros((1, 1, P, D), np.uint8)
    vc = np.zeros((1, 1, P, D), np.uint8)
    kc[0, 0, :2] = orc.kv_encode_fp8(K, s)
    vc[0, 0, :2] = orc.kv_encode_fp8(V, s)
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.5
    o = orc.decode_attention(q, kc, vc, s, s, np.array([[0]]), np.array([2]), 0.5, fmt="fp8")
    w1, w2 = math.exp(0.28125), math.exp(0.5625)
    assert o[0, 0, 3] == pytest.approx(0.375 * (w1 - w2) / (w1 + w2), rel=1e-14)
    o1 = orc.decode_attention(q, kc, vc, s, s, np.array([[0]]), np.array([1]), 0.5, fmt="fp8")
    assert o1[0, 0, 3] == 0.375 and np.count_nonzero(o1) == 1
