"""Parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Integers (packing, index maps, masks, argmax, acceptance) and unpack must be
bit-exact.  bf16 attention outputs must satisfy
|gpu - oracle| <= 2e-2 + 1e-2 * |oracle| element by element (fp32 accumulation
on the GPU, fp64 in the oracle; inputs are identical bf16 values).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2
DEV = torch.device("cuda:0")


def _rd():
    import tree_attention_verify_gb300 as rd
    return rd


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _to_dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _close(got: np.ndarray, ref: np.ndarray, what: str):
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, "
                           f"max err {float(err.max()):.4g}")


def _pack_check(beams_np, pk, P_cap):
    ref = oracle.oracle_pack(beams_np, P_cap)
    for k in ("tokens", "packer", "unpacker", "depth", "packed_len"):
        np.testing.assert_array_equal(pk[k].cpu().numpy(), ref[k], err_msg=k)
    np.testing.assert_array_equal(pk["mask"].cpu().numpy().view(np.uint32), ref["mask"])
    return ref


# ------------------------------------------------------------------------------
# rd_pack_beams
# ------------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_pack_configs(name):
    rd = _rd()
    cfg = workloads.CONFIGS[name]
    rng = np.random.default_rng(cfg.seed)
    trees = workloads.draft_trees(cfg.B, cfg.W, cfg.L, cfg.vocab, cfg.share, rng)
    st = _status()
    pk = rd.rd_pack_beams(torch.from_numpy(trees.beams).to(DEV), cfg.P_max, dev_status=st)
    _pack_check(trees.beams, pk, cfg.P_max)
    assert st.item() == 0


@pytest.mark.parametrize("seed,W,L,vocab,P_cap", [
    (0, 32, 8, 2, 256), (1, 1, 1, 5, 1), (2, 7, 9, 3, 70), (3, 32, 7, 1000, 224),
    (4, 5, 40, 2, 200), (5, 16, 16, 4, 256)])
def test_pack_random_and_extremes(seed, W, L, vocab, P_cap):
    rd = _rd()
    rng = np.random.default_rng(seed)
    beams = rng.integers(0, vocab, size=(9, W, L)).astype(np.int32)
    beams[3] = beams[3, :1]                     # identical beams
    beams[4, :, 0] = np.arange(W) + 5000        # distinct anchors
    ref_need = max(int(oracle.oracle_pack(beams[b:b + 1], W * L)["packed_len"][0])
                   for b in range(9))
    if ref_need > P_cap:
        pytest.skip("capacity case covered by test_pack_overflow_flag")
    st = _status()
    pk = rd.rd_pack_beams(torch.from_numpy(beams).to(DEV), P_cap, dev_status=st)
    ref = _pack_check(beams, pk, P_cap)
    assert ref["packed_len"][3] == L and ref["packed_len"][4] == W * L
    assert st.item() == 0


def test_pack_golden_examples():
    import json, os
    rd = _rd()
    with open(os.path.join(os.path.dirname(__file__), "golden", "pack_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        beams = np.array(c["beams"], np.int32)
        pk = rd.rd_pack_beams(torch.from_numpy(beams).to(DEV))
        np.testing.assert_array_equal(pk["packed_len"].cpu().numpy(), c["packed_len"])
        np.testing.assert_array_equal(pk["unpacker"].cpu().numpy(), c["unpacker"])
        np.testing.assert_array_equal(pk["mask"].cpu().numpy().view(np.uint32),
                                      np.array(c["mask"], np.uint32))


def test_pack_overflow_flag():
    rd = _rd()
    beams = np.arange(2 * 3 * 4, dtype=np.int32).reshape(2, 3, 4)   # 12 distinct nodes each
    st = _status()
    pk = rd.rd_pack_beams(torch.from_numpy(beams).to(DEV), 8, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_OVERFLOW
    assert (pk["packed_len"].cpu().numpy() == 12).all()


def test_empty_batch_everywhere():
    rd = _rd()
    st = _status()
    e = torch.zeros((0, 4, 4), dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(e, 16, dev_status=st)
    lg = torch.zeros((0, 16, 100), dtype=torch.bfloat16, device=DEV)
    rd.rd_greedy_accept(lg, e, pk["unpacker"], pk["packed_len"], dev_status=st)
    q = torch.zeros((0, 16, 4, 64), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((0, 16, 2, 64), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    rd.rd_tree_attention(q, kv, kv, kc, kc, torch.zeros(1, dtype=torch.int64, device=DEV),
                         pk["packed_len"], pk["mask"], max_ctx=0, dev_status=st)
    rd.rd_causal_attention(torch.zeros((0, 4, 64), dtype=torch.bfloat16, device=DEV), kc, kc,
                           torch.zeros(1, dtype=torch.int32, device=DEV), max_seqlen=0,
                           dev_status=st)
    rd.rd_unpack(torch.zeros((0, 16, 8), dtype=torch.bfloat16, device=DEV), e, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0


# ------------------------------------------------------------------------------
# rd_unpack
# ------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,Dh", [(torch.bfloat16, 4096), (torch.float16, 100),
                                      (torch.float32, 7), (torch.int32, 5120),
                                      (torch.bfloat16, 3)])
def test_unpack_exact(dtype, Dh):
    rd = _rd()
    g = torch.Generator(device="cpu").manual_seed(Dh)
    B, P, W, L = 3, 20, 5, 4
    if dtype.is_floating_point:
        packed = torch.randn(B, P, Dh, generator=g).to(dtype)
    else:
        packed = torch.randint(-2**31, 2**31 - 1, (B, P, Dh), generator=g, dtype=torch.int64).to(dtype)
    unp = torch.randint(0, P, (B, W, L), generator=g, dtype=torch.int32)
    out = rd.rd_unpack(packed.to(DEV), unp.to(DEV))
    ref = torch.gather(packed, 1, unp.long().view(B, W * L, 1).expand(-1, -1, Dh)).reshape(
        B, W, L, Dh)
    assert torch.equal(out.cpu().view(torch.int16 if packed.element_size() == 2 else torch.int32),
                       ref.view(torch.int16 if packed.element_size() == 2 else torch.int32))


def test_unpack_bad_index_sets_status():
    rd = _rd()
    packed = torch.ones(1, 4, 16, dtype=torch.bfloat16, device=DEV)
    unp = torch.tensor([[[0, 1], [4, -1]]], dtype=torch.int32, device=DEV)
    st = _status()
    out = rd.rd_unpack(packed, unp, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_BAD_INDEX
    assert (out[0, 1].float() == 0).all() and (out[0, 0].float() == 1).all()


# ------------------------------------------------------------------------------
# rd_greedy_accept
# ------------------------------------------------------------------------------
def _accept_check(inp, pk_ref, acc):
    ref = oracle.oracle_greedy_accept(bf16_bits(inp["logits"]), inp["beams"].cpu().numpy(),
                                      pk_ref["unpacker"], pk_ref["packed_len"])
    for k in ref:
        np.testing.assert_array_equal(acc[k].cpu().numpy(), ref[k], err_msg=k)
    return ref


@pytest.mark.parametrize("name", ["tiny", "7b_b1", "8b_gqa_b16", "13b_b64"])
def test_greedy_accept_configs(name):
    rd = _rd()
    cfg = workloads.CONFIGS[name]
    rng = np.random.default_rng(cfg.seed)
    gen = torch.Generator(device=DEV).manual_seed(cfg.seed)
    trees = workloads.draft_trees(cfg.B, cfg.W, cfg.L, cfg.vocab, cfg.share, rng)
    logits = workloads.make_logits(trees, cfg.P_max, cfg.vocab, cfg.plant, rng, gen, DEV,
                                   ties=cfg.ties)
    beams = torch.from_numpy(trees.beams).to(DEV)
    st = _status()
    pk = rd.rd_pack_beams(beams, cfg.P_max, dev_status=st)
    ws = torch.zeros(rd.rd_greedy_accept_workspace_size(cfg.B, cfg.P_max, cfg.vocab),
                     dtype=torch.uint8, device=DEV)
    for _ in range(2):                         # the workspace must come back zeroed
        acc = rd.rd_greedy_accept(logits, beams, pk["unpacker"], pk["packed_len"],
                                  workspace=ws, dev_status=st)
        pk_ref = oracle.oracle_pack(trees.beams, cfg.P_max)
        _accept_check(dict(logits=logits, beams=beams), pk_ref, acc)
    assert int(ws.count_nonzero()) == 0
    assert st.item() == 0


def test_greedy_accept_golden_and_unaligned_vocab():
    import json, os
    rd = _rd()
    with open(os.path.join(os.path.dirname(__file__), "golden", "accept_examples.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        for V in (g["vocab"], 16):             # V=10 takes the scalar path, 16 the vector path
            logits = torch.full((1, g["P_max"], V), -1.0)
            for row, entries in case["rows"].items():
                for col, val in entries.items():
                    logits[0, int(row), int(col)] = val
            acc = rd.rd_greedy_accept(logits.to(torch.bfloat16).to(DEV),
                                      torch.tensor(g["beams"], dtype=torch.int32, device=DEV),
                                      torch.tensor(g["unpacker"], dtype=torch.int32, device=DEV),
                                      torch.tensor(g["packed_len"], dtype=torch.int32, device=DEV))
            for k in ("argmax", "accept_len", "best_beam", "n_accepted", "out_tokens"):
                np.testing.assert_array_equal(acc[k].cpu().numpy(), np.array(case[k]),
                                              err_msg=f"{case['name']} {k} V={V}")


def test_greedy_accept_ties_across_chunks():
    rd = _rd()
    B, P, V = 2, 3, 128256
    logits = torch.zeros(B, P, V, dtype=torch.bfloat16)
    logits[0, 0, [5, 70000, 128255]] = 3.0       # ties in different vocab chunks
    logits[0, 1, [128255]] = 3.0
    logits[1, 2, [64128, 64127]] = -0.0          # all zeros incl. -0: lowest index 0
    logits[1, 0] = -float("inf")                 # all -inf: index 0
    beams = torch.zeros(B, 1, 1, dtype=torch.int32)
    unp = torch.zeros(B, 1, 1, dtype=torch.int32)
    plen = torch.tensor([3, 3], dtype=torch.int32)
    acc = rd.rd_greedy_accept(logits.to(DEV), beams.to(DEV), unp.to(DEV), plen.to(DEV))
    ref = oracle.oracle_greedy_accept(bf16_bits(logits), beams.numpy(), unp.numpy(), plen.numpy())
    np.testing.assert_array_equal(acc["argmax"].cpu().numpy(), ref["argmax"])
    assert acc["argmax"][0, 0].item() == 5 and acc["argmax"][1, 0].item() == 0


def test_greedy_accept_context_requests():
    # context-phase requests: W = L = 1, the greedy token of the last prompt row
    rd = _rd()
    gen = torch.Generator(device=DEV).manual_seed(7)
    logits = (torch.randn(5, 1, 128256, generator=gen, device=DEV) * 2).to(torch.bfloat16)
    beams = torch.zeros(5, 1, 1, dtype=torch.int32, device=DEV)
    unp = torch.zeros(5, 1, 1, dtype=torch.int32, device=DEV)
    plen = torch.ones(5, dtype=torch.int32, device=DEV)
    acc = rd.rd_greedy_accept(logits, beams, unp, plen)
    ref = oracle.oracle_greedy_accept(bf16_bits(logits), beams.cpu().numpy(), unp.cpu().numpy(),
                                      plen.cpu().numpy())
    np.testing.assert_array_equal(acc["out_tokens"].cpu().numpy(), ref["out_tokens"])
    assert (acc["n_accepted"].cpu().numpy() == 0).all()


def test_greedy_accept_bad_inputs_set_status():
    rd = _rd()
    logits = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device=DEV)
    beams = torch.tensor([[[1, 2, 99]]], dtype=torch.int32, device=DEV)
    unp = torch.tensor([[[7, 0, 1]]], dtype=torch.int32, device=DEV)   # 7 >= packed_len
    st = _status()
    rd.rd_greedy_accept(logits, beams, unp, torch.tensor([4], dtype=torch.int32, device=DEV),
                        dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_BAD_INDEX
    st.zero_()
    rd.rd_greedy_accept(logits, beams, unp, torch.tensor([9], dtype=torch.int32, device=DEV),
                        dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_BAD_LENGTH


# ------------------------------------------------------------------------------
# rd_tree_attention
# ------------------------------------------------------------------------------
def _attention_case(inp, sample_bh=None):
    """Run pack + tree attention on device; compare with the oracle (all rows, or the
    sampled (b, kv head) pairs as independent sub-problems)."""
    rd = _rd()
    cfg = inp["cfg"]
    d = _to_dev(inp) if inp["q"].device.type == "cpu" else inp
    st = _status()
    pk = rd.rd_pack_beams(d["beams"], cfg.P_max, dev_status=st)
    o = rd.rd_tree_attention(d["q"], d["k_draft"], d["v_draft"], d["k_cache"], d["v_cache"],
                             d["ctx_offsets"], pk["packed_len"], pk["mask"],
                             max_ctx=int(inp["ctx_lens"].max()), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    pk_ref = oracle.oracle_pack(d["beams"].cpu().numpy(), cfg.P_max)
    got = o.float().cpu().numpy()
    offs = d["ctx_offsets"].cpu().numpy()
    G = cfg.Hq // cfg.Hkv
    if sample_bh is None:
        ref = oracle.oracle_tree_attention(bf16_bits(d["q"]), bf16_bits(d["k_draft"]),
                                           bf16_bits(d["v_draft"]), bf16_bits(d["k_cache"]),
                                           bf16_bits(d["v_cache"]), offs, pk_ref["packed_len"],
                                           pk_ref["mask"])
        _close(got, ref, cfg.name)
        return got
    for b, h in sample_bh:
        sl = slice(int(offs[b]), int(offs[b + 1]))
        hs = slice(h * G, (h + 1) * G)
        ref = oracle.oracle_tree_attention(
            bf16_bits(d["q"][b:b + 1, :, hs]), bf16_bits(d["k_draft"][b:b + 1, :, h:h + 1]),
            bf16_bits(d["v_draft"][b:b + 1, :, h:h + 1]), bf16_bits(d["k_cache"][sl, h:h + 1]),
            bf16_bits(d["v_cache"][sl, h:h + 1]),
            np.array([0, offs[b + 1] - offs[b]], np.int64), pk_ref["packed_len"][b:b + 1],
            pk_ref["mask"][b:b + 1])
        _close(got[b:b + 1, :, hs], ref, f"{cfg.name} b={b} h={h}")
    return got


@pytest.mark.parametrize("name", ["tiny", "7b_b1", "8b_gqa_b16"])
def test_tree_attention_configs(name):
    _attention_case(workloads.make_verify_inputs(workloads.CONFIGS[name], device="cpu"))


@pytest.mark.parametrize("ctx", [("fixed", 0), ("uniform", 0, 70), ("uniform", 1, 300)])
def test_tree_attention_ragged_and_empty_context(ctx):
    import dataclasses
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=5, vocab=50, Hq=8, Hkv=2,
                              share=("p", 0.3))
    _attention_case(workloads.make_verify_inputs(cfg, device="cpu", ctx_override=ctx))


def test_tree_attention_zero_and_bad_packed_lengths():
    # a small batch runs on chunk ranges: a request with no packed nodes owns no
    # chunks, and one with packed_len > P_max is flagged and skipped; both must
    # still come out as zero rows (the output starts as garbage), and every other
    # request must match the oracle
    import dataclasses
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=6, vocab=50,
                              ctx=("uniform", 100, 1500))
    inp = _to_dev(workloads.make_verify_inputs(cfg, device="cpu"))
    st = _status()
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    plen = pk["packed_len"].clone()
    plen[1] = 0
    plen[3] = cfg.P_max + 5
    max_ctx = int(inp["ctx_lens"].max())
    assert rd.rd_tree_attention_workspace_size(cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D,
                                               max_ctx) > 0      # chunk ranges
    o = torch.full_like(inp["q"], 7.0)
    rd.rd_tree_attention(inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"],
                         inp["v_cache"], inp["ctx_offsets"], plen, pk["mask"],
                         max_ctx=max_ctx, out=o, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & rd.DEV_BAD_LENGTH
    got = o.float().cpu().numpy()
    assert not got[1].any() and not got[3].any()
    pk_ref = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    plen_ref = pk_ref["packed_len"].copy()
    plen_ref[1] = 0
    plen_ref[3] = 0
    ref = oracle.oracle_tree_attention(bf16_bits(inp["q"]), bf16_bits(inp["k_draft"]),
                                       bf16_bits(inp["v_draft"]), bf16_bits(inp["k_cache"]),
                                       bf16_bits(inp["v_cache"]), inp["ctx_offsets"].cpu().numpy(),
                                       plen_ref, pk_ref["mask"])
    _close(got, ref, "zero and bad packed lengths")


def test_tree_attention_deep_trees_span_draft_chunks():
    # W*L up to 160 packed nodes: the draft segment crosses 64-position chunks
    import dataclasses
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=3, W=8, L=20, Hq=4, Hkv=2, D=128,
                              share=("p", 0.2), ctx=("uniform", 30, 200), ties=False)
    _attention_case(workloads.make_verify_inputs(cfg, device="cpu"))


def test_tree_attention_13b_full_size_sampled():
    cfg = workloads.CONFIGS["13b_b64"]
    inp = workloads.make_verify_inputs(cfg, device=DEV)
    rng = np.random.default_rng(11)
    sample = [(0, 0), (63, 39)] + [(int(rng.integers(64)), int(rng.integers(40))) for _ in range(6)]
    _attention_case(inp, sample_bh=sample)


# ------------------------------------------------------------------------------
# rd_causal_attention (context-phase requests of the in-flight batch)
# ------------------------------------------------------------------------------
@pytest.mark.parametrize("lens,Hq,Hkv,D", [([512, 512, 512], 32, 8, 128), ([1, 37, 200, 64], 8, 2, 64),
                                           ([130], 4, 4, 128), ([300, 17], 6, 2, 128),
                                           ([777, 5, 256], 16, 1, 64), ([1000, 0, 129], 8, 1, 128),
                                           ([200, 9], 128, 1, 64), ([150, 301], 4, 2, 128)])
def test_causal_attention(lens, Hq, Hkv, D):
    rd = _rd()
    gen = torch.Generator(device="cpu").manual_seed(sum(lens))
    inp = workloads.make_context_inputs(len(lens), 0, Hq, Hkv, D, 100, gen, "cpu",
                                        lens=np.array(lens, np.int64))
    st = _status()
    o = rd.rd_causal_attention(inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV),
                               inp["cu_seqlens"].to(DEV), max_seqlen=max(lens), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.oracle_causal_attention(bf16_bits(inp["q"]), bf16_bits(inp["k"]),
                                         bf16_bits(inp["v"]), inp["cu_seqlens"].numpy())
    _close(o.float().cpu().numpy(), ref, "causal")


def test_causal_attention_many_units_sampled():
    """48 sequences of 1-1024 tokens on 8B shapes (32 query / 8 kv heads x 128):
    about 40 units per CTA, whole and partial 128-row tiles, pairs with one or
    two live tiles, output tiles both by TMA stores and by row stores.  Sampled
    (sequence, kv head) slices are compared with the oracle run on that slice
    alone (causal attention is independent per sequence and kv head)."""
    rd = _rd()
    rng = np.random.default_rng(2026)
    lens = rng.integers(1, 1025, size=48).astype(np.int64)
    lens[:4] = (1024, 1, 257, 32)
    Hq, Hkv, D = 32, 8, 128
    G = Hq // Hkv
    gen = torch.Generator(device="cpu").manual_seed(7)
    inp = workloads.make_context_inputs(len(lens), 0, Hq, Hkv, D, 100, gen, "cpu", lens=lens)
    st = _status()
    o = rd.rd_causal_attention(inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV),
                               inp["cu_seqlens"].to(DEV), max_seqlen=int(lens.max()), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = o.float().cpu().numpy()
    cu = inp["cu_seqlens"].numpy()
    q16, k16, v16 = bf16_bits(inp["q"]), bf16_bits(inp["k"]), bf16_bits(inp["v"])
    samples = [(0, 0), (1, 7), (2, 3), (3, 5)] + [(int(rng.integers(48)), int(rng.integers(Hkv)))
                                                  for _ in range(6)]
    for b, h in samples:
        s0, s1 = int(cu[b]), int(cu[b + 1])
        ref = oracle.oracle_causal_attention(q16[s0:s1, h * G:(h + 1) * G], k16[s0:s1, h:h + 1],
                                             v16[s0:s1, h:h + 1], np.array([0, s1 - s0], np.int32))
        _close(o[s0:s1, h * G:(h + 1) * G], ref, f"causal b={b} h={h}")


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([3000, 1500, 77], 32, 8, 128), ([2500, 640], 8, 8, 64)])
def test_causal_attention_long_sampled(lens, Hq, Hkv, D):
    """Long sequences: up to 47 chunks per unit, the K/V ring wrapping many times
    within a unit.  Sampled (sequence, kv head) slices against the oracle."""
    rd = _rd()
    G = Hq // Hkv
    gen = torch.Generator(device="cpu").manual_seed(len(lens) * 1000 + D)
    inp = workloads.make_context_inputs(len(lens), 0, Hq, Hkv, D, 100, gen, "cpu",
                                        lens=np.array(lens, np.int64))
    st = _status()
    o = rd.rd_causal_attention(inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV),
                               inp["cu_seqlens"].to(DEV), max_seqlen=max(lens), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = o.float().cpu().numpy()
    cu = inp["cu_seqlens"].numpy()
    q16, k16, v16 = bf16_bits(inp["q"]), bf16_bits(inp["k"]), bf16_bits(inp["v"])
    for b, h in [(0, 0), (0, Hkv - 1), (1, Hkv // 2), (len(lens) - 1, 1)]:
        s0, s1 = int(cu[b]), int(cu[b + 1])
        ref = oracle.oracle_causal_attention(q16[s0:s1, h * G:(h + 1) * G], k16[s0:s1, h:h + 1],
                                             v16[s0:s1, h:h + 1], np.array([0, s1 - s0], np.int32))
        _close(o[s0:s1, h * G:(h + 1) * G], ref, f"causal long b={b} h={h}")


def test_wrong_out_buffers_are_rejected_before_launch():
    """A caller-supplied output of the wrong shape or dtype raises before any
    kernel runs (it would otherwise be written out of bounds)."""
    rd = _rd()
    q = torch.zeros(64, 8, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(64, 2, 128, dtype=torch.bfloat16, device=DEV)
    cu = torch.tensor([0, 64], dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        rd.rd_causal_attention(q, k, k, cu, max_seqlen=64, out=torch.empty(63, 8, 128, dtype=torch.bfloat16,
                                                                            device=DEV))
    with pytest.raises(TypeError):
        rd.rd_causal_attention(q, k, k, cu, max_seqlen=64, out=torch.empty(64, 8, 128, dtype=torch.float16,
                                                                            device=DEV))
    packed = torch.zeros(2, 6, 16, dtype=torch.bfloat16, device=DEV)
    unp = torch.zeros(2, 2, 3, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        rd.rd_unpack(packed, unp, out=torch.empty(2, 2, 3, 15, dtype=torch.bfloat16, device=DEV))
    beams = torch.zeros(2, 2, 3, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        rd.rd_pack_beams(beams, 6, out=dict(tokens=torch.empty(2, 5, dtype=torch.int32, device=DEV)))
    torch.cuda.synchronize()


# ------------------------------------------------------------------------------
# the whole verification step, and the in-flight mixed batch
# ------------------------------------------------------------------------------
@pytest.mark.parametrize("split", ["mixed", "all_ctx", "all_gen"])
def test_mixed_batch(split):
    rd = _rd()
    m = workloads.make_mixed_inputs(split, device="cpu", scale=0.25)
    st = _status()
    # context half: causal prefill + greedy token of its last row
    c = m["ctx"]
    n_ctx = m["n_ctx"]
    oc = rd.rd_causal_attention(c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV),
                                c["cu_seqlens"].to(DEV), max_seqlen=m["prefill_len"],
                                dev_status=st)
    one = torch.zeros((n_ctx, 1, 1), dtype=torch.int32, device=DEV)
    acc_c = rd.rd_greedy_accept(c["logits"].to(DEV), one, one,
                                torch.ones(n_ctx, dtype=torch.int32, device=DEV), dev_status=st)
    # generation half: the verification step
    if m["n_gen"] > 0:
        _attention_case(m["gen"])
    torch.cuda.synchronize()
    assert st.item() == 0
    if n_ctx:
        ref = oracle.oracle_causal_attention(bf16_bits(c["q"]), bf16_bits(c["k"]),
                                             bf16_bits(c["v"]), c["cu_seqlens"].numpy())
        _close(oc.float().cpu().numpy(), ref, "context half")
        g = np.argmax((bf16_bits(c["logits"]).astype(np.uint32) << 16).view(np.float32), -1)
        np.testing.assert_array_equal(acc_c["out_tokens"].cpu().numpy()[:, 0], g[:, 0])


@pytest.mark.parametrize("name", ["tiny", "7b_b1", "8b_gqa_b16"])
def test_verify_step_unpack_hidden(name):
    rd = _rd()
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_verify_inputs(cfg, device="cpu")
    d = _to_dev(inp)
    pk = rd.rd_pack_beams(d["beams"], cfg.P_max)
    acc = rd.rd_greedy_accept(d["logits"], d["beams"], pk["unpacker"], pk["packed_len"])
    hid = rd.rd_unpack(d["hidden"], pk["unpacker"])
    pk_ref = oracle.oracle_pack(inp["beams"].numpy(), cfg.P_max)
    _accept_check(inp, pk_ref, acc)
    np.testing.assert_array_equal(bf16_bits(hid), oracle.oracle_unpack(bf16_bits(inp["hidden"]),
                                                                       pk_ref["unpacker"]))


def test_tree_attention_growing_scores_rescale():
    # Scores that grow along the context force the online softmax to move its
    # running maximum many times (and to rescale the partial output).
    import dataclasses
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=2, W=3, L=3, Hq=2, Hkv=1, D=128,
                              ties=False)
    inp = workloads.make_verify_inputs(cfg, device="cpu", ctx_override=("fixed", 700))
    C = 700
    ramp = torch.linspace(-4.0, 6.0, C).repeat(cfg.B)[:, None, None]
    inp["k_cache"] = (ramp * torch.ones(1, 1, cfg.D)).to(torch.bfloat16).contiguous()
    inp["q"] = torch.full_like(inp["q"], 1.0)
    _attention_case(inp)


def test_tree_attention_maximum_packed_length():
    # W*L = 256 packed nodes (the largest P_max), 8 mask words, 4 draft chunks,
    # G = 2 -> 512 stacked rows = 4 tiles per (request, kv head)
    import dataclasses
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=2, W=32, L=8, vocab=100000, Hq=4,
                              Hkv=2, D=128, share=("p", 0.05), ctx=("uniform", 1, 300),
                              ties=False)
    inp = workloads.make_verify_inputs(cfg, device="cpu")
    pk = oracle.oracle_pack(inp["beams"].numpy(), cfg.P_max)
    assert pk["packed_len"].max() > 192              # the last draft chunk is used
    _attention_case(inp)


def test_tree_attention_reused_workspace_split_launches():
    # the pieces of units cut by CTA boundaries go through the workspace; the
    # merge reads only slots this call wrote, so a workspace full of NaN bit
    # patterns (0xff bytes) gives the same result as a fresh one, call after call
    rd = _rd()
    cfg = workloads.CONFIGS["8b_gqa_b16"]
    inp = workloads.make_verify_inputs(cfg, device=DEV)
    st = _status()
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    max_ctx = int(inp["ctx_lens"].max())
    n_ws = rd.rd_tree_attention_workspace_size(cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D, max_ctx)
    assert n_ws > 0                                      # this workload cuts units
    G = cfg.Hq // cfg.Hkv
    outs = []
    for fill in (0, 255, 255):
        ws = torch.full((n_ws,), fill, dtype=torch.uint8, device=DEV)
        o = rd.rd_tree_attention(inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"],
                                 inp["v_cache"], inp["ctx_offsets"], pk["packed_len"], pk["mask"],
                                 max_ctx=max_ctx, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert not torch.isnan(o.float()).any()
        outs.append(o.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    rng = np.random.default_rng(5)
    sample = [(int(rng.integers(cfg.B)), int(rng.integers(cfg.Hkv))) for _ in range(3)]
    offs = inp["ctx_offsets"].cpu().numpy()
    pk_ref = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    got = outs[2].float().cpu().numpy()
    for b, h in sample:
        sl = slice(int(offs[b]), int(offs[b + 1]))
        hs = slice(h * G, (h + 1) * G)
        ref = oracle.oracle_tree_attention(
            bf16_bits(inp["q"][b:b + 1, :, hs]), bf16_bits(inp["k_draft"][b:b + 1, :, h:h + 1]),
            bf16_bits(inp["v_draft"][b:b + 1, :, h:h + 1]), bf16_bits(inp["k_cache"][sl, h:h + 1]),
            bf16_bits(inp["v_cache"][sl, h:h + 1]), np.array([0, offs[b + 1] - offs[b]], np.int64),
            pk_ref["packed_len"][b:b + 1], pk_ref["mask"][b:b + 1])
        _close(got[b:b + 1, :, hs], ref, f"{cfg.name} b={b} h={h}")


@pytest.mark.parametrize("split", ["mixed", "all_ctx", "all_gen"])
def test_mixed_batch_full_size(split):
    # The in-flight batch at its stated size: 32 requests on 8B-GQA shapes, each a
    # 512-token causal prefill chunk or a W=8, L=5 verification over a context of
    # 512..8192 positions (G = 4).  Context half: every sequence against the oracle
    # and its greedy token bit-exact.  Generation half: pack and greedy acceptance
    # bit-exact for every request; attention on sampled (request, kv head) pairs
    # that include the longest context; unpack bit-exact.
    rd = _rd()
    m = workloads.make_mixed_inputs(split, device=DEV)
    st = _status()
    c, n_ctx = m["ctx"], m["n_ctx"]
    if n_ctx:
        oc = rd.rd_causal_attention(c["q"], c["k"], c["v"], c["cu_seqlens"],
                                    max_seqlen=m["prefill_len"], dev_status=st)
        one = torch.zeros((n_ctx, 1, 1), dtype=torch.int32, device=DEV)
        acc_c = rd.rd_greedy_accept(c["logits"], one, one,
                                    torch.ones(n_ctx, dtype=torch.int32, device=DEV),
                                    dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        ref = oracle.oracle_causal_attention(bf16_bits(c["q"]), bf16_bits(c["k"]),
                                             bf16_bits(c["v"]), c["cu_seqlens"].cpu().numpy())
        _close(oc.float().cpu().numpy(), ref, f"{split}: context half")
        lg = bf16_bits(c["logits"])
        g = np.argmax((lg.astype(np.uint32) << 16).view(np.float32), -1)
        np.testing.assert_array_equal(acc_c["out_tokens"].cpu().numpy()[:, 0], g[:, 0])
    if m["n_gen"]:
        g_inp = m["gen"]
        cfg = g_inp["cfg"]
        lens = np.asarray(g_inp["ctx_lens"])
        rng = np.random.default_rng(17)
        longest = int(np.argmax(lens))
        sample = [(longest, 0), (longest, cfg.Hkv - 1), (int(np.argmin(lens)), 3)]
        sample += [(int(rng.integers(cfg.B)), int(rng.integers(cfg.Hkv))) for _ in range(6)]
        _attention_case(g_inp, sample_bh=sample)
        assert lens.max() > 7000
        pk = rd.rd_pack_beams(g_inp["beams"], cfg.P_max, dev_status=st)
        acc = rd.rd_greedy_accept(g_inp["logits"], g_inp["beams"], pk["unpacker"],
                                  pk["packed_len"], dev_status=st)
        hid = rd.rd_unpack(g_inp["hidden"], pk["unpacker"], dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        pk_ref = oracle.oracle_pack(g_inp["beams"].cpu().numpy(), cfg.P_max)
        _accept_check(g_inp, pk_ref, acc)
        np.testing.assert_array_equal(bf16_bits(hid), oracle.oracle_unpack(
            bf16_bits(g_inp["hidden"]), pk_ref["unpacker"]))
