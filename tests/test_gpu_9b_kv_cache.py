"""NVFP4 paged KV cache against the oracle: the append kernel's page bytes
bit for bit (neighbouring slots untouched), and decode attention over
caches the oracle builds (ragged and empty contexts, page boundaries,
shuffled page placement, several context splits, 1 / 8 / 16 query heads
per KV head, BF16 and FP32 outputs).

Tolerance, from the arithmetic: the keys and values decode exactly in FP16,
scores and sums accumulate in FP32, and the probabilities enter the value
product rounded to FP16 (relative 2^-11), so per (sequence, head)
max_d |o - o_ref| <= 1e-3 * max_t,d |v_t,d| (twice that bound), plus half a
BF16 ulp of o_ref for BF16 outputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import host, nv
from helpers import bf16_half_ulp, kv_pack_fp8, kv_pack_nvfp4, kv_unpack_fp8, kv_unpack_nvfp4

pytestmark = pytest.mark.gpu

P, D = 64, 128


def build_cache(rng, ctx_lens, H_kv, s_k, s_v, spare_pages=3, shuffle=True):
    """Oracle-encoded paged cache for sequences of the given lengths: returns
    (device KvCache, oracle (codes, scales) of K and V in the natural
    layout, block table, max_pages)."""
    B = len(ctx_lens)
    pages_per = [max(1, -(-n // P)) for n in ctx_lens]
    max_pages = max(pages_per)
    n_pages = sum(pages_per) + spare_pages
    order = rng.permutation(n_pages) if shuffle else np.arange(n_pages)
    table = np.zeros((B, max_pages), np.int32)
    k_c = rng.integers(0, 256, (n_pages, H_kv, P, D // 2)).astype(np.uint8)   # stale bytes in unused slots
    k_s = rng.integers(0, 256, (n_pages, H_kv, P, D // 16)).astype(np.uint8)
    v_c = rng.integers(0, 256, (n_pages, H_kv, P, D // 2)).astype(np.uint8)
    v_s = rng.integers(0, 256, (n_pages, H_kv, P, D // 16)).astype(np.uint8)
    nxt = 0
    for b, n in enumerate(ctx_lens):
        for i in range(pages_per[b]):
            table[b, i] = order[nxt]
            nxt += 1
        for hk in range(H_kv):
            kb = synth.activations(9, 100 + 7 * b + hk, n, D, 0.02, 8.0)
            vb = synth.activations(9, 200 + 7 * b + hk, n, D, 0.0, 1.0)
            kc, ks = oracle.kv_encode(kb, s_k)
            vc, vs = oracle.kv_encode(vb, s_v)
            for tkn in range(n):
                pg = table[b, tkn // P]
                k_c[pg, hk, tkn % P], k_s[pg, hk, tkn % P] = kc[tkn], ks[tkn]
                v_c[pg, hk, tkn % P], v_s[pg, hk, tkn % P] = vc[tkn], vs[tkn]
    cache = nv.KvCache(torch.from_numpy(kv_pack_nvfp4(k_c, k_s, v_c, v_s)).cuda(),
                       torch.tensor([s_k], dtype=torch.float32, device="cuda"),
                       torch.tensor([s_v], dtype=torch.float32, device="cuda"))
    return cache, (k_c, k_s), (v_c, v_s), table, max_pages


def check_attention(out, ref, v_nat, s_v, table, ctx_lens, H_kv, G, bf16):
    B = ref.shape[0]
    for b in range(B):
        n = int(ctx_lens[b])
        for h in range(ref.shape[1]):
            if n == 0:
                assert not out[b, h].any()
                continue
            V = oracle.kv_gather(v_nat[0], v_nat[1], s_v, table[b], n, h // G)
            tol = 1e-3 * np.abs(V).max()
            err = np.abs(out[b, h] - ref[b, h])
            if bf16:
                err = np.maximum(err - bf16_half_ulp(ref[b, h]), 0.0)
            assert err.max() <= tol, f"seq {b} head {h}: {err.max():.3e} > {tol:.3e}"


@pytest.mark.parametrize("ctx_lens,H_kv,G,out_dtype", [
    ([1, 63, 64, 65, 200, 0], 2, 8, nv.OUT_FP32),       # page boundaries, an empty context
    ([3000, 17, 1100], 1, 8, nv.OUT_FP32),              # several context splits
    ([700, 128, 5], 2, 16, nv.OUT_BF16),               # 16 query heads per KV head
    ([513, 64, 1], 4, 1, nv.OUT_BF16),                 # one query head per KV head
])
def test_decode_attention_against_oracle(ctx_lens, H_kv, G, out_dtype):
    rng = np.random.default_rng(sum(ctx_lens) + 31 * G)
    s_k, s_v = 8.0 / 2688, 4.0 / 2688
    cache, k_nat, v_nat, table, max_pages = build_cache(rng, ctx_lens, H_kv, s_k, s_v)
    H = H_kv * G
    B = len(ctx_lens)
    qb = synth.activations(9, 300 + G, B * H, D, 0.0, 1.0).reshape(B, H, D)
    max_ctx = max(ctx_lens)
    sm = 1.0 / math.sqrt(D)
    q = torch.from_numpy(qb.view(np.int16)).cuda().view(torch.bfloat16)
    out = nv.kv_decode_attention(cache, q, torch.tensor(ctx_lens, dtype=torch.int32, device="cuda"),
                                 torch.from_numpy(table).cuda(), max_ctx, sm, out_dtype=out_dtype)
    on = host(out.float()).astype(np.float64)
    ref = oracle.decode_attention(oracle.bf16_to_f32(qb).astype(np.float64), k_nat, v_nat, s_k, s_v, table,
                                  np.array(ctx_lens), sm)
    check_attention(on, ref, v_nat, s_v, table, ctx_lens, H_kv, G, out_dtype == nv.OUT_BF16)


def test_append_bytes_bit_exact_and_neighbours_untouched():
    rng = np.random.default_rng(7)
    H_kv, B = 3, 5
    s_k, s_v = 6.0 / 2688, 3.0 / 2688
    n_pages, max_pages = 16, 3
    blocks0 = rng.integers(0, 256, (n_pages, H_kv, 9216)).astype(np.uint8)
    cache = nv.KvCache(torch.from_numpy(blocks0.copy()).cuda(), torch.tensor([s_k], device="cuda"),
                       torch.tensor([s_v], device="cuda"))
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    positions = np.array([0, 1, 63, 64, 130], np.int32)     # first, odd, last slot, next page, page 3
    kb = synth.activations(9, 400, B * H_kv, D, 0.02, 8.0).reshape(B, H_kv, D)
    vb = synth.activations(9, 401, B * H_kv, D, 0.0, 1.0).reshape(B, H_kv, D)
    to_dev = lambda x: torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    nv.kv_append(cache, to_dev(kb), to_dev(vb), torch.from_numpy(positions).cuda(), torch.from_numpy(table).cuda())
    k_c, k_s, v_c, v_s = kv_unpack_nvfp4(host(cache.pages))
    ek_c, ek_s, ev_c, ev_s = [x.copy() for x in kv_unpack_nvfp4(blocks0)]
    for b in range(B):
        pg, sl = table[b, positions[b] // P], positions[b] % P
        for hk in range(H_kv):
            c, sc = oracle.kv_encode(kb[b, hk:hk + 1], s_k)
            ek_c[pg, hk, sl], ek_s[pg, hk, sl] = c[0], sc[0]
            c, sc = oracle.kv_encode(vb[b, hk:hk + 1], s_v)
            ev_c[pg, hk, sl], ev_s[pg, hk, sl] = c[0], sc[0]
    np.testing.assert_array_equal(k_c, ek_c)
    np.testing.assert_array_equal(k_s, ek_s)
    np.testing.assert_array_equal(v_c, ev_c)
    np.testing.assert_array_equal(v_s, ev_s)


def test_append_then_attend():
    # a cache filled token by token through the append kernel attends like the
    # oracle's cache of the same tokens (whose bytes it must equal first)
    rng = np.random.default_rng(9)
    H_kv, G, B, n = 2, 4, 2, 70
    s_k, s_v = 8.0 / 2688, 4.0 / 2688
    n_pages, max_pages = 4, 2
    cache = nv.KvCache.empty(n_pages, H_kv, torch.tensor([s_k], device="cuda"),
                             torch.tensor([s_v], device="cuda"))
    table = np.array([[2, 0], [1, 3]], np.int32)
    tdev = torch.from_numpy(table).cuda()
    kb = synth.activations(9, 500, n * B * H_kv, D, 0.02, 8.0).reshape(n, B, H_kv, D)
    vb = synth.activations(9, 501, n * B * H_kv, D, 0.0, 1.0).reshape(n, B, H_kv, D)
    to_dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    for tkn in range(n):
        nv.kv_append(cache, to_dev(kb[tkn]), to_dev(vb[tkn]), torch.full((B,), tkn, dtype=torch.int32,
                                                                          device="cuda"), tdev)
    k_c, k_s, v_c, v_s = kv_unpack_nvfp4(host(cache.pages))
    k_nat, v_nat = (k_c, k_s), (v_c, v_s)
    for b in range(B):
        for hk in range(H_kv):
            c, sc = oracle.kv_encode(kb[:, b, hk], s_k)
            got = np.stack([k_nat[0][table[b, t // P], hk, t % P] for t in range(n)])
            np.testing.assert_array_equal(got, c)
            c, sc = oracle.kv_encode(vb[:, b, hk], s_v)
            got = np.stack([v_nat[0][table[b, t // P], hk, t % P] for t in range(n)])
            np.testing.assert_array_equal(got, c)
    qb = synth.activations(9, 502, B * H_kv * G, D, 0.0, 1.0).reshape(B, H_kv * G, D)
    q = torch.from_numpy(qb.view(np.int16)).cuda().view(torch.bfloat16)
    ctx = [n, n - 9]
    out = host(nv.kv_decode_attention(cache, q, torch.tensor(ctx, dtype=torch.int32, device="cuda"), tdev, n,
                                      0.0884, out_dtype=nv.OUT_FP32)).astype(np.float64)
    ref = oracle.decode_attention(oracle.bf16_to_f32(qb).astype(np.float64), k_nat, v_nat, s_k, s_v, table,
                                  np.array(ctx), 0.0884)
    check_attention(out, ref, v_nat, s_v, table, ctx, H_kv, G, False)


# ---- FP8 cache ---------------------------------------------------------------------------

def build_cache_fp8(rng, ctx_lens, H_kv, s_k, s_v):
    B = len(ctx_lens)
    pages_per = [max(1, -(-n // P)) for n in ctx_lens]
    n_pages = sum(pages_per) + 2
    order = rng.permutation(n_pages)
    table = np.zeros((B, max(pages_per)), np.int32)
    k = rng.integers(0, 256, (n_pages, H_kv, P, D)).astype(np.uint8)     # stale bytes (NaN codes too)
    v = rng.integers(0, 256, (n_pages, H_kv, P, D)).astype(np.uint8)
    nxt = 0
    for b, n in enumerate(ctx_lens):
        for i in range(pages_per[b]):
            table[b, i] = order[nxt]
            nxt += 1
        for hk in range(H_kv):
            kc = oracle.kv_encode_fp8(synth.activations(9, 600 + 7 * b + hk, n, D, 0.02, 8.0), s_k)
            vc = oracle.kv_encode_fp8(synth.activations(9, 700 + 7 * b + hk, n, D, 0.0, 1.0), s_v)
            for tkn in range(n):
                k[table[b, tkn // P], hk, tkn % P] = kc[tkn]
                v[table[b, tkn // P], hk, tkn % P] = vc[tkn]
    cache = nv.KvCache(torch.from_numpy(kv_pack_fp8(k, v)).cuda(),
                       torch.tensor([s_k], dtype=torch.float32, device="cuda"),
                       torch.tensor([s_v], dtype=torch.float32, device="cuda"), nv.KV_FP8)
    return cache, k, v, table


@pytest.mark.parametrize("ctx_lens,H_kv,G,out_dtype", [
    ([1, 31, 32, 33, 64, 65, 200, 0], 2, 8, nv.OUT_FP32),  # half-page and page boundaries, empty
    ([3000, 17, 1100], 1, 8, nv.OUT_BF16),                 # several context splits
    ([700, 96, 5], 2, 16, nv.OUT_FP32),
])
def test_fp8_decode_attention_against_oracle(ctx_lens, H_kv, G, out_dtype):
    rng = np.random.default_rng(sum(ctx_lens) + 7 * G)
    s_k, s_v = 8.0 / 448, 4.0 / 448
    cache, k, v, table = build_cache_fp8(rng, ctx_lens, H_kv, s_k, s_v)
    H, B = H_kv * G, len(ctx_lens)
    qb = synth.activations(9, 800 + G, B * H, D, 0.0, 1.0).reshape(B, H, D)
    q = torch.from_numpy(qb.view(np.int16)).cuda().view(torch.bfloat16)
    sm = 1.0 / math.sqrt(D)
    out = nv.kv_decode_attention(cache, q, torch.tensor(ctx_lens, dtype=torch.int32, device="cuda"),
                                 torch.from_numpy(table).cuda(), max(ctx_lens), sm, out_dtype=out_dtype)
    on = host(out.float()).astype(np.float64)
    ref = oracle.decode_attention(oracle.bf16_to_f32(qb).astype(np.float64), k, v, s_k, s_v, table,
                                  np.array(ctx_lens), sm, fmt="fp8")
    for b in range(B):
        n = ctx_lens[b]
        for h in range(H):
            if n == 0:
                assert not on[b, h].any()
                continue
            V = oracle.kv_gather_fp8(v, s_v, table[b], n, h // G)
            err = np.abs(on[b, h] - ref[b, h])
            if out_dtype == nv.OUT_BF16:
                err = np.maximum(err - bf16_half_ulp(ref[b, h]), 0.0)
            assert err.max() <= 1e-3 * np.abs(V).max(), f"seq {b} head {h}"


def test_fp8_append_bit_exact():
    rng = np.random.default_rng(17)
    H_kv, B, n_pages, max_pages = 2, 4, 10, 2
    s_k, s_v = 6.0 / 448, 3.0 / 448
    blocks0 = rng.integers(0, 256, (n_pages, H_kv, 16384)).astype(np.uint8)
    cache = nv.KvCache(torch.from_numpy(blocks0.copy()).cuda(), torch.tensor([s_k], device="cuda"),
                       torch.tensor([s_v], device="cuda"), nv.KV_FP8)
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    positions = np.array([0, 31, 32, 127], np.int32)
    kb = synth.activations(9, 900, B * H_kv, D, 0.02, 8.0).reshape(B, H_kv, D)
    vb = synth.activations(9, 901, B * H_kv, D, 0.0, 1.0).reshape(B, H_kv, D)
    to_dev = lambda x: torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    nv.kv_append(cache, to_dev(kb), to_dev(vb), torch.from_numpy(positions).cuda(), torch.from_numpy(table).cuda())
    ek, ev = kv_unpack_fp8(blocks0)
    for b in range(B):
        pg, sl = table[b, positions[b] // P], positions[b] % P
        for hk in range(H_kv):
            ek[pg, hk, sl] = oracle.kv_encode_fp8(kb[b, hk:hk + 1], s_k)[0]
            ev[pg, hk, sl] = oracle.kv_encode_fp8(vb[b, hk:hk + 1], s_v)[0]
    gk, gv = kv_unpack_fp8(host(cache.pages))
    np.testing.assert_array_equal(gk, ek)
    np.testing.assert_array_equal(gv, ev)
