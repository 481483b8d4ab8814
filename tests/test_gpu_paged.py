"""Parity of the paged-cache attention and of the commit of the accepted path
(through the C ABI) against the fp64 CPU oracle.  Attention within
|gpu - oracle| <= 2e-2 + 1e-2 |oracle|; the commit (a copy) bit-exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _rd():
    import tree_attention_verify_gb300 as rd
    return rd


def _close(got, ref, what):
    err = np.abs(got - ref)
    bad = err > 2e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside tolerance, max err {err.max():.4g}"


def _paged_inputs(cfg, ctx, page_size, seed=0):
    inp = workloads.make_verify_inputs(cfg, device=DEV, ctx_override=ctx)
    rng = np.random.default_rng(seed + 77)
    pg = workloads.make_paged(inp["k_cache"], inp["v_cache"], inp["ctx_lens"], page_size, rng)
    return inp, pg


@pytest.mark.parametrize("page_size,ctx,Hq,Hkv,D", [
    (64, ("uniform", 0, 700), 8, 2, 128), (128, ("uniform", 1, 900), 4, 4, 128),
    (256, ("uniform", 100, 1000), 8, 1, 64), (64, ("fixed", 0), 2, 2, 128)])
def test_paged_attention_matches_oracle(page_size, ctx, Hq, Hkv, D):
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=5, vocab=50, Hq=Hq, Hkv=Hkv,
                              D=D, share=("p", 0.4))
    inp, pg = _paged_inputs(cfg, ctx, page_size)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    o = rd.rd_tree_attention_paged(inp["q"], inp["k_draft"], inp["v_draft"], pg["k_pool"],
                                   pg["v_pool"], pg["block_table"], pg["ctx_lens"],
                                   pk["packed_len"], pk["mask"],
                                   max_ctx=max(1, int(inp["ctx_lens"].max())), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    pk_ref = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    ref = oracle.oracle_tree_attention_paged(
        bf16_bits(inp["q"]), bf16_bits(inp["k_draft"]), bf16_bits(inp["v_draft"]),
        bf16_bits(pg["k_pool"]), bf16_bits(pg["v_pool"]), pg["block_table"].cpu().numpy(),
        pg["ctx_lens"].cpu().numpy(), pk_ref["packed_len"], pk_ref["mask"])
    _close(o.float().cpu().numpy(), ref, "paged")


def test_paged_with_identity_table_equals_contiguous_kernel():
    # pages laid out in order over the contiguous cache: the same bits
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["13b_b64"], B=6, Hq=8, Hkv=8)
    inp = workloads.make_verify_inputs(cfg, device=DEV, ctx_override=("fixed", 1024))
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max)
    ps = 64
    n_pages = inp["k_cache"].shape[0] // ps
    table = torch.arange(n_pages, dtype=torch.int32, device=DEV).view(cfg.B, -1).contiguous()
    k_pool = inp["k_cache"].view(n_pages, ps, cfg.Hkv, cfg.D)
    v_pool = inp["v_cache"].view(n_pages, ps, cfg.Hkv, cfg.D)
    lens = torch.full((cfg.B,), 1024, dtype=torch.int32, device=DEV)
    a = rd.rd_tree_attention(inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"],
                             inp["v_cache"], inp["ctx_offsets"], pk["packed_len"], pk["mask"],
                             max_ctx=1024)
    b = rd.rd_tree_attention_paged(inp["q"], inp["k_draft"], inp["v_draft"], k_pool, v_pool,
                                   table, lens, pk["packed_len"], pk["mask"], max_ctx=1024)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_paged_bad_page_sets_status():
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=2, D=128, ties=False)
    inp, pg = _paged_inputs(cfg, ("fixed", 200), 64)
    table = pg["block_table"].clone()
    table[1, 1] = pg["k_pool"].shape[0] + 3
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max)
    rd.rd_tree_attention_paged(inp["q"], inp["k_draft"], inp["v_draft"], pg["k_pool"],
                               pg["v_pool"], table, pg["ctx_lens"], pk["packed_len"], pk["mask"],
                               max_ctx=200, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_BAD_INDEX


@pytest.mark.parametrize("name", ["8b_gqa_b16", "13b_b64"])
def test_commit_accepted_matches_oracle(name):
    rd = _rd()
    cfg = workloads.CONFIGS[name]
    inp, pg = _paged_inputs(cfg, ("uniform", 0, 300), 64, seed=5)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    acc = rd.rd_greedy_accept(inp["logits"], inp["beams"], pk["unpacker"], pk["packed_len"],
                              dev_status=st)
    k0, v0 = bf16_bits(pg["k_pool"]), bf16_bits(pg["v_pool"])
    new_lens = rd.rd_commit_accepted(inp["k_draft"], inp["v_draft"], pk["unpacker"],
                                     acc["best_beam"], acc["n_accepted"], pg["k_pool"],
                                     pg["v_pool"], pg["block_table"], pg["ctx_lens"],
                                     dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    k_ref, v_ref, lens_ref = oracle.oracle_commit_accepted(
        bf16_bits(inp["k_draft"]), bf16_bits(inp["v_draft"]), pk["unpacker"].cpu().numpy(),
        acc["best_beam"].cpu().numpy(), acc["n_accepted"].cpu().numpy(), k0, v0,
        pg["block_table"].cpu().numpy(), pg["ctx_lens"].cpu().numpy())
    np.testing.assert_array_equal(new_lens.cpu().numpy(), lens_ref)
    np.testing.assert_array_equal(bf16_bits(pg["k_pool"]), k_ref)
    np.testing.assert_array_equal(bf16_bits(pg["v_pool"]), v_ref)


def test_paged_attention_13b_full_size_sampled():
    # The 13B-shaped batch at full size (64 requests, 40 heads, 8192-position
    # contexts) in 256-position pages of a shuffled pool; sampled (request, kv
    # head) pairs against the oracle, each given the request's own pages (in a
    # shuffled sub-pool with a renumbered block table) and that head.
    rd = _rd()
    cfg = workloads.CONFIGS["13b_b64"]
    inp, pg = _paged_inputs(cfg, None, 256, seed=3)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    o = rd.rd_tree_attention_paged(inp["q"], inp["k_draft"], inp["v_draft"], pg["k_pool"],
                                   pg["v_pool"], pg["block_table"], pg["ctx_lens"],
                                   pk["packed_len"], pk["mask"], max_ctx=8192, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    pk_ref = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    got = o.float().cpu().numpy()
    table = pg["block_table"].cpu().numpy()
    lens = pg["ctx_lens"].cpu().numpy()
    rng = np.random.default_rng(23)
    sample = [(0, 0), (63, 39)] + [(int(rng.integers(64)), int(rng.integers(40)))
                                   for _ in range(6)]
    for b, h in sample:
        n_b = -(-int(lens[b]) // 256)
        pages = table[b, :n_b].astype(np.int64)
        perm = rng.permutation(n_b)                      # sub-pool slot of each page
        sub_k = torch.empty((n_b, 256, 1, cfg.D), dtype=torch.bfloat16, device=DEV)
        sub_v = torch.empty_like(sub_k)
        idx = torch.from_numpy(pages).to(DEV)
        sub_k[torch.from_numpy(perm).to(DEV)] = pg["k_pool"][idx, :, h:h + 1]
        sub_v[torch.from_numpy(perm).to(DEV)] = pg["v_pool"][idx, :, h:h + 1]
        sub_table = perm.astype(np.int32)[None, :]
        ref = oracle.oracle_tree_attention_paged(
            bf16_bits(inp["q"][b:b + 1, :, h:h + 1]), bf16_bits(inp["k_draft"][b:b + 1, :, h:h + 1]),
            bf16_bits(inp["v_draft"][b:b + 1, :, h:h + 1]), bf16_bits(sub_k), bf16_bits(sub_v),
            sub_table, lens[b:b + 1], pk_ref["packed_len"][b:b + 1], pk_ref["mask"][b:b + 1])
        _close(got[b:b + 1, :, h:h + 1], ref, f"paged 13B b={b} h={h}")
