"""Parity of stochastic verification (rd_sample_accept, through the C ABI)
against the fp64 oracle: accepted lengths, best beam, accepted count and
emitted tokens bit-exact.

The kernel decides in fp32, the oracle in fp64.  Uniforms of a request whose
oracle decisions are closer than 1e-3 (relative: the two sides of a ratio test,
or the two best keys of the draw) are re-drawn before the comparison, so every
compared decision is one that both precisions take the same way.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
MARGIN = 1e-3


def _rd():
    import tree_attention_verify_gb300 as rd
    return rd


def _well_conditioned(inp, pk_ref, seed):
    cfg = inp["cfg"]
    rng = np.random.default_rng(seed + 77)
    ua, us = inp["u_accept"].cpu().numpy().copy(), inp["u_sample"].cpu().numpy().copy()
    tb, db = bf16_bits(inp["target"]), bf16_bits(inp["draft"])
    beams = inp["beams"].cpu().numpy()
    for _ in range(20):
        ref = oracle.oracle_sample_accept(tb, db, inp["temperature"], beams, pk_ref["packer"],
                                          pk_ref["unpacker"], pk_ref["packed_len"], ua, us)
        bad = ref["margin"] < MARGIN
        if not bad.any():
            return ua, us, ref
        ua[bad] = rng.random((int(bad.sum()), ua.shape[1]), dtype=np.float32)
        us[bad] = rng.random((int(bad.sum()), us.shape[1]), dtype=np.float32)
    raise AssertionError("could not draw well-conditioned uniforms")


def _sample_case(cfg, T, seed=None):
    rd = _rd()
    seed = cfg.seed if seed is None else seed
    inp = workloads.make_sample_inputs(cfg, T, device="cpu", seed=seed)
    pk_ref = oracle.oracle_pack(inp["beams"].numpy(), cfg.P_max)
    ua, us, ref = _well_conditioned(inp, pk_ref, seed)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    beams = inp["beams"].to(DEV)
    pk = rd.rd_pack_beams(beams, cfg.P_max, dev_status=st)
    out = rd.rd_sample_accept(inp["target"].to(DEV), inp["draft"].to(DEV), T, beams,
                              pk["packer"], pk["unpacker"], pk["packed_len"],
                              torch.from_numpy(ua).to(DEV), torch.from_numpy(us).to(DEV),
                              dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for k in ("n_accepted", "out_tokens", "best_beam", "accept_len"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), ref[k], err_msg=f"{cfg.name} {k}")
    return ref


@pytest.mark.parametrize("name,T", [("tiny", 1.0), ("7b_b1", 0.7), ("8b_gqa_b16", 1.0),
                                    ("13b_b64", 1.0), ("13b_b64", 0.5)])
def test_sample_accept_configs(name, T):
    ref = _sample_case(workloads.CONFIGS[name], T)
    assert ref["n_accepted"].max() >= 1


@pytest.mark.parametrize("V", [1001, 37, 8])
def test_sample_accept_unaligned_and_small_vocab(V):
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=12, W=6, L=5, vocab=V,
                              share=("p", 0.5))
    _sample_case(cfg, 1.2, seed=21 + V)


def test_sample_accept_deep_and_wide_trees():
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=6, W=32, L=8, vocab=500,
                              share=("p", 0.7), ties=False)
    _sample_case(cfg, 0.9, seed=5)


def test_sample_accept_low_temperature():
    cfg = dataclasses.replace(workloads.CONFIGS["7b_b1"], B=8, vocab=4000)
    _sample_case(cfg, 0.05, seed=9)


def test_sample_accept_bad_length_sets_status():
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=2)
    inp = workloads.make_sample_inputs(cfg, 1.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    plen = pk["packed_len"].clone()
    plen[1] = cfg.P_max + 5
    out = rd.rd_sample_accept(inp["target"], inp["draft"], 1.0, inp["beams"], pk["packer"],
                              pk["unpacker"], plen, inp["u_accept"], inp["u_sample"],
                              dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 8                       # RD_DEV_BAD_LENGTH
    assert out["n_accepted"][1].item() == 0
    assert (out["out_tokens"][1] == -1).all()
