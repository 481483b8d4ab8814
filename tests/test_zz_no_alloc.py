"""rd_greedy_accept_noalloc, the greedy-verification entry point that allocates
nothing (for callers that cannot allocate device memory on the serving path),
against rd_greedy_accept with a caller-owned workspace.

Runs last (file name) so that a stop at the first failure has already run every
other test.  It must pass both alone in a fresh process and after the others.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(name, seed_offset=0, cfg=None):
    import tree_attention_verify_gb300 as rd
    cfg = workloads.CONFIGS[name] if cfg is None else cfg
    rng = np.random.default_rng(cfg.seed + seed_offset)
    gen = torch.Generator(device=DEV).manual_seed(cfg.seed + seed_offset)
    trees = workloads.draft_trees(cfg.B, cfg.W, cfg.L, cfg.vocab, cfg.share, rng)
    logits = workloads.make_logits(trees, cfg.P_max, cfg.vocab, cfg.plant, rng, gen, DEV,
                                   ties=cfg.ties)
    beams = torch.from_numpy(trees.beams).to(DEV)
    pk = rd.rd_pack_beams(beams, cfg.P_max)
    return logits, beams, pk["unpacker"], pk["packed_len"]


def _call_noalloc(logits, beams, unpacker, packed_len):
    import tree_attention_verify_gb300 as rd
    fn = rd._lib.rd_greedy_accept_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, I, I, I, P, P, P, I, I, P, P, P, P, P, P, P]
    fn.restype = I
    B, P_max, V = logits.shape
    W, L = beams.shape[1], beams.shape[2]
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(argmax=torch.full((B, P_max), 7, **i32), accept_len=torch.full((B, W), 7, **i32),
               best_beam=torch.full((B,), 7, **i32), n_accepted=torch.full((B,), 7, **i32),
               out_tokens=torch.full((B, L), 7, **i32))
    st = torch.zeros(1, **i32)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = fn(ptr(logits), B, P_max, V, ptr(beams), ptr(unpacker), ptr(packed_len), W, L,
            ptr(out["argmax"]), ptr(out["accept_len"]), ptr(out["best_beam"]),
            ptr(out["n_accepted"]), ptr(out["out_tokens"]), ptr(st),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, f"rd_greedy_accept_noalloc returned {rc}"
    torch.cuda.synchronize()
    assert st.item() == 0
    return out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import tree_attention_verify_gb300 as rd
    # three calls in a row: the same large batch twice, then a smaller one, so a
    # call that saw the previous call's scratch contents would disagree
    for name, off in (("8b_gqa_b16", 0), ("8b_gqa_b16", 0), ("tiny", 5)):
        logits, beams, unpacker, packed_len = _inputs(name, off)
        ref = rd.rd_greedy_accept(logits, beams, unpacker, packed_len)
        got = _call_noalloc(logits, beams, unpacker, packed_len)
        for k in ref:
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(),
                                          err_msg=f"{name}: {k}")
        _check_oracle(got, logits, beams, unpacker, packed_len, name)


def _check_oracle(got, logits, beams, unpacker, packed_len, what):
    # the fp64 oracle of greedy verification decides the same integers
    ref = oracle.oracle_greedy_accept(bf16_bits(logits), beams.cpu().numpy(),
                                      unpacker.cpu().numpy(), packed_len.cpu().numpy())
    for k in ref:
        np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k], err_msg=f"{what}: {k}")


def test_noalloc_wrapper_at_the_scratch_limit():
    # B * P_max == 65536 keys: the whole key array and the tickets behind it are
    # used; two calls in a row through the Python binding, each against the
    # workspace entry point and the oracle
    import tree_attention_verify_gb300 as rd
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=1024, W=8, L=8, vocab=512,
                              name="noalloc_limit")
    assert cfg.B * cfg.P_max == 65536
    for off in (0, 1):
        logits, beams, unpacker, packed_len = _inputs(None, off, cfg)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        got = rd.rd_greedy_accept_noalloc(logits, beams, unpacker, packed_len, dev_status=st)
        ref = rd.rd_greedy_accept(logits, beams, unpacker, packed_len)
        torch.cuda.synchronize()
        assert st.item() == 0
        for k in ref:
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(),
                                          err_msg=f"limit call {off}: {k}")
        _check_oracle(got, logits, beams, unpacker, packed_len, f"limit call {off}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import tree_attention_verify_gb300 as rd
    fn = rd._lib.rd_greedy_accept_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, I, I, I, P, P, P, I, I, P, P, P, P, P, P, P]
    fn.restype = I
    one = ctypes.c_void_p(256)
    # 300 requests x 256 packed rows = 76800 keys > 65536
    assert fn(one, 300, 256, 1000, one, one, one, 4, 4, one, one, one, one, one, None,
              None) == rd.RD_ERR_UNSUPPORTED
    # one key past the array: 1025 x 64 = 65600, and 65537 requests of one row
    assert fn(one, 1025, 64, 1000, one, one, one, 8, 8, one, one, one, one, one, None,
              None) == rd.RD_ERR_UNSUPPORTED
    assert fn(one, 65537, 1, 1000, one, one, one, 1, 1, one, one, one, one, one, None,
              None) == rd.RD_ERR_UNSUPPORTED
