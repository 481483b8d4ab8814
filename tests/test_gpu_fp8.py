"""Parity of the FP8 (e4m3) context-cache tree attention (through the C ABI)
against the fp64 CPU oracle on the same e4m3 codes and scales.

The GPU contracts in f16 with fp32 accumulation; the only roundings beyond the
bf16 path's are draft K/V divided by the scales (f16, relative 2^-11) and the
attention weights stored as f16 (relative 2^-11), so the bf16 path's bound
|gpu - oracle| <= 2e-2 + 1e-2 |oracle| is kept.
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


def _rd():
    import tree_attention_verify_gb300 as rd
    return rd


def _close(got, ref, what):
    err = np.abs(got - ref)
    bad = err > 2e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside tolerance, max err {err.max():.4g}"


def _fp8_case(cfg, ctx=None, sample_bh=None, seed=None):
    rd = _rd()
    inp = workloads.make_verify_inputs(cfg, device=DEV, ctx_override=ctx, seed=seed)
    kc, ks = workloads.make_fp8_cache(inp["k_cache"])
    vc, vs = workloads.make_fp8_cache(inp["v_cache"])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
    o = rd.rd_tree_attention_fp8(inp["q"], inp["k_draft"], inp["v_draft"], kc, vc, ks, vs,
                                 inp["ctx_offsets"], pk["packed_len"], pk["mask"],
                                 max_ctx=max(1, int(inp["ctx_lens"].max())), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = o.float().cpu().numpy()
    pk_ref = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    offs = inp["ctx_offsets"].cpu().numpy()
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    if sample_bh is None:
        ref = oracle.oracle_tree_attention_fp8(
            bf16_bits(inp["q"]), bf16_bits(inp["k_draft"]), bf16_bits(inp["v_draft"]), kc_np,
            vc_np, ks, vs, offs, pk_ref["packed_len"], pk_ref["mask"])
        _close(got, ref, cfg.name)
        return
    G = cfg.Hq // cfg.Hkv
    for b, h in sample_bh:
        sl = slice(int(offs[b]), int(offs[b + 1]))
        hs = slice(h * G, (h + 1) * G)
        ref = oracle.oracle_tree_attention_fp8(
            bf16_bits(inp["q"][b:b + 1, :, hs]), bf16_bits(inp["k_draft"][b:b + 1, :, h:h + 1]),
            bf16_bits(inp["v_draft"][b:b + 1, :, h:h + 1]), kc_np[sl, h:h + 1],
            vc_np[sl, h:h + 1], ks, vs, np.array([0, offs[b + 1] - offs[b]], np.int64),
            pk_ref["packed_len"][b:b + 1], pk_ref["mask"][b:b + 1])
        _close(got[b:b + 1, :, hs], ref, f"{cfg.name} b={b} h={h}")


@pytest.mark.parametrize("name", ["7b_b1", "8b_gqa_b16"])
def test_fp8_configs(name):
    _fp8_case(workloads.CONFIGS[name])


@pytest.mark.parametrize("ctx,Hq,Hkv", [(("uniform", 1, 300), 8, 2), (("uniform", 0, 700), 4, 4),
                                         (("fixed", 65), 8, 1)])
def test_fp8_ragged_context(ctx, Hq, Hkv):
    cfg = dataclasses.replace(workloads.CONFIGS["8b_gqa_b16"], B=5, vocab=50, Hq=Hq, Hkv=Hkv,
                              share=("p", 0.3))
    _fp8_case(cfg, ctx=ctx)


def test_fp8_deep_trees_span_draft_chunks():
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=3, W=8, L=20, Hq=4, Hkv=2, D=128,
                              share=("p", 0.2), ctx=("uniform", 30, 200), ties=False)
    _fp8_case(cfg)


def test_fp8_13b_full_size_sampled():
    cfg = workloads.CONFIGS["13b_b64"]
    rng = np.random.default_rng(12)
    sample = [(0, 0), (63, 39)] + [(int(rng.integers(64)), int(rng.integers(40))) for _ in range(4)]
    _fp8_case(cfg, sample_bh=sample)


def test_fp8_unsupported_shapes_are_rejected():
    rd = _rd()
    q = torch.zeros((1, 4, 2, 64), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((8, 2, 64), dtype=torch.uint8, device=DEV)
    pl = torch.full((1,), 4, dtype=torch.int32, device=DEV)
    mask = torch.zeros((1, 4, 1), dtype=torch.int32, device=DEV)
    offs = torch.tensor([0, 8], dtype=torch.int64, device=DEV)
    with pytest.raises(RuntimeError, match="UNSUPPORTED|unsupported"):
        rd.rd_tree_attention_fp8(q, q[:, :, :2], q[:, :, :2], kc, kc, 1.0, 1.0, offs, pl, mask,
                                 max_ctx=8)
    with pytest.raises(RuntimeError, match="INVALID|invalid"):
        q2 = torch.zeros((1, 4, 2, 128), dtype=torch.bfloat16, device=DEV)
        kc2 = torch.zeros((8, 2, 128), dtype=torch.uint8, device=DEV)
        rd.rd_tree_attention_fp8(q2, q2, q2, kc2, kc2, 0.0, 1.0, offs, pl, mask, max_ctx=8)


def test_fp8_maximum_packed_length():
    cfg = dataclasses.replace(workloads.CONFIGS["tiny"], B=2, W=32, L=8, vocab=100000, Hq=4,
                              Hkv=2, D=128, share=("p", 0.05), ctx=("uniform", 1, 300),
                              ties=False)
    _fp8_case(cfg)
