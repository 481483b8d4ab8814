"""Pins of the oracle's paged-cache attention and of the commit of the accepted
path (CPU only).

* Paged attention equals contiguous attention on the same context gathered
  page by page with numpy indexing (a different formulation of the page walk).
* The commit writes, at context positions C..C+a, the K/V that belong to the
  prefixes of the best beam (K/V defined per prefix tuple, independent of the
  packing), leaves every other cache row untouched and returns C + a + 1.
"""
import numpy as np
import pytest

import oracle
from tests.pins import bf16_round


def _paged_case(seed, B, page_size, Hq, Hkv, D, max_ctx):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_ctx + 1, size=B).astype(np.int32)
    max_pages = int(np.ceil(max_ctx / page_size)) + 1
    n_pages = int(sum(-(-l // page_size) for l in lens)) + 3
    perm = rng.permutation(n_pages)                      # pages in shuffled order
    bt = np.full((B, max_pages), -7, np.int32)           # unused slots hold junk
    k = 0
    for b in range(B):
        need = -(-int(lens[b]) // page_size)
        bt[b, :need] = perm[k:k + need]
        k += need
    k_pool = bf16_round(rng.standard_normal((n_pages, page_size, Hkv, D)).astype(np.float32))
    v_pool = bf16_round(rng.standard_normal((n_pages, page_size, Hkv, D)).astype(np.float32))
    return rng, lens, bt, k_pool, v_pool


@pytest.mark.parametrize("seed,page_size,Hq,Hkv,D", [(0, 16, 4, 2, 16), (1, 64, 2, 2, 8),
                                                     (2, 8, 3, 1, 8)])
def test_paged_equals_contiguous_on_gathered_context(seed, page_size, Hq, Hkv, D):
    B, W, L, P = 3, 3, 3, 9
    rng, lens, bt, k_pool, v_pool = _paged_case(seed, B, page_size, Hq, Hkv, D, max_ctx=70)
    beams = rng.integers(0, 3, size=(B, W, L)).astype(np.int32)
    pk = oracle.oracle_pack(beams, P)
    q = bf16_round(rng.standard_normal((B, P, Hq, D)).astype(np.float32))
    kn = bf16_round(rng.standard_normal((B, P, Hkv, D)).astype(np.float32))
    vn = bf16_round(rng.standard_normal((B, P, Hkv, D)).astype(np.float32))
    got = oracle.oracle_tree_attention_paged(q, kn, vn, k_pool, v_pool, bt, lens,
                                             pk["packed_len"], pk["mask"], n_threads=2)
    # gather each request's context: flat pool row = page * page_size + offset
    flat_k = k_pool.reshape(-1, Hkv, D)
    flat_v = v_pool.reshape(-1, Hkv, D)
    rows = [bt[b, np.arange(lens[b]) // page_size] * page_size + np.arange(lens[b]) % page_size
            for b in range(B)]
    rows = np.concatenate(rows).astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ref = oracle.oracle_tree_attention(q, kn, vn, flat_k[rows], flat_v[rows], offs,
                                       pk["packed_len"], pk["mask"], n_threads=2)
    np.testing.assert_array_equal(got, ref)


def test_paged_rejects_a_page_outside_the_pool():
    B, page_size, Hq, Hkv, D = 1, 16, 1, 1, 8
    rng, lens, bt, k_pool, v_pool = _paged_case(3, B, page_size, Hq, Hkv, D, max_ctx=40)
    lens[:] = 40
    bt[0, :3] = [0, 1, k_pool.shape[0]]
    z = np.zeros((1, 4, 1, D), np.uint16)
    with pytest.raises(ValueError):
        oracle.oracle_tree_attention_paged(z, z, z, k_pool, v_pool, bt, lens,
                                           np.array([1], np.int32), np.ones((1, 4, 1), np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_commit_writes_the_accepted_path(seed):
    rng = np.random.default_rng(seed)
    B, W, L, Hkv, D, page_size = 3, 4, 5, 2, 8, 4
    beams = rng.integers(0, 3, size=(B, W, L)).astype(np.int32)
    beams[:, :, 0] = beams[:, :1, 0]
    P = W * L
    pk = oracle.oracle_pack(beams, P)
    vec = {}

    def kv_of(b, pre, which):
        key = (b, which) + pre
        if key not in vec:
            h = hash(key) & 0xFFFFFFFF
            vec[key] = bf16_round(np.random.default_rng(h).standard_normal((Hkv, D)).astype(
                np.float32))
        return vec[key]

    kn = np.zeros((B, P, Hkv, D), np.uint16)
    vn = np.zeros((B, P, Hkv, D), np.uint16)
    for b in range(B):
        for p in range(pk["packed_len"][b]):
            f = pk["packer"][b, p]
            pre = tuple(int(x) for x in beams[b, f // L, : f % L + 1])
            kn[b, p], vn[b, p] = kv_of(b, pre, 0), kv_of(b, pre, 1)
    lens = rng.integers(0, 9, size=B).astype(np.int32)
    max_pages = 5
    n_pages = B * max_pages
    bt = rng.permutation(n_pages).astype(np.int32).reshape(B, max_pages)
    k_pool = bf16_round(rng.standard_normal((n_pages, page_size, Hkv, D)).astype(np.float32))
    v_pool = bf16_round(rng.standard_normal((n_pages, page_size, Hkv, D)).astype(np.float32))
    best = rng.integers(0, W, size=B).astype(np.int32)
    n_acc = rng.integers(0, L, size=B).astype(np.int32)
    k2, v2, new_lens = oracle.oracle_commit_accepted(kn, vn, pk["unpacker"], best, n_acc, k_pool,
                                                     v_pool, bt, lens)
    np.testing.assert_array_equal(new_lens, lens + n_acc + 1)
    touched = np.zeros((n_pages, page_size), bool)
    for b in range(B):
        for i in range(n_acc[b] + 1):
            pos = lens[b] + i
            pg, off = bt[b, pos // page_size], pos % page_size
            pre = tuple(int(x) for x in beams[b, best[b], : i + 1])
            np.testing.assert_array_equal(k2[pg, off], kv_of(b, pre, 0))
            np.testing.assert_array_equal(v2[pg, off], kv_of(b, pre, 1))
            touched[pg, off] = True
    np.testing.assert_array_equal(k2[~touched], k_pool[~touched])
    np.testing.assert_array_equal(v2[~touched], v_pool[~touched])
