"""Failure detection without a GPU fault: every wait inside the attention kernel
is bounded.  The test hook rd_debug_stall_attention makes each CTA's MMA issuer
wait on a barrier that nothing completes, with a short clock budget (about a
millisecond); the wait must run out, the kernel must record DEV_TIMEOUT, stop
its other roles, drain what it issued and return, and the next ordinary call on
the same context must again match the oracle."""
import dataclasses
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BUDGET = 2_000_000            # SM clock cycles: about 1 ms at 2 GHz


def _rd():
    import tree_attention_verify_gb300 as rd
    return rd


def _close(got, ref, what):
    err = np.abs(got - ref)
    bad = err > 2e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside tolerance, max err {err.max():.4g}"


def _stalled(fn):
    """Run fn with the stall armed; return (device status, seconds to finish)."""
    rd = _rd()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    rd.rd_debug_stall_attention(BUDGET)
    try:
        t0 = time.perf_counter()
        fn(st)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        rd.rd_debug_stall_attention(0)
    return int(st.item()), dt


@pytest.mark.parametrize("name,B,Hq,Hkv", [("tiny", None, None, None),
                                           ("8b_gqa_b16", 4, 8, 2)])
def test_tree_attention_wait_runs_out_then_next_call_is_correct(name, B, Hq, Hkv):
    rd = _rd()
    cfg = workloads.CONFIGS[name]
    if B is not None:
        cfg = dataclasses.replace(cfg, B=B, Hq=Hq, Hkv=Hkv, vocab=100)
    inp = workloads.make_verify_inputs(cfg, device=DEV)
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max)
    max_ctx = int(inp["ctx_lens"].max())

    def call(st, ws=None):
        return rd.rd_tree_attention(inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"],
                                    inp["v_cache"], inp["ctx_offsets"], pk["packed_len"],
                                    pk["mask"], max_ctx=max_ctx, workspace=ws, dev_status=st)

    status, dt = _stalled(call)
    assert status & rd.DEV_TIMEOUT, f"status {status}: the planted wait did not run out"
    assert dt < 30.0
    # the next ordinary call (fresh workspace) on the same context is correct
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = call(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pk = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    ref = oracle.oracle_tree_attention(bf16_bits(inp["q"]), bf16_bits(inp["k_draft"]),
                                       bf16_bits(inp["v_draft"]), bf16_bits(inp["k_cache"]),
                                       bf16_bits(inp["v_cache"]),
                                       inp["ctx_offsets"].cpu().numpy(),
                                       ref_pk["packed_len"], ref_pk["mask"])
    _close(o.float().cpu().numpy(), ref, f"{name} after the timeout")


def test_causal_attention_wait_runs_out_then_next_call_is_correct():
    rd = _rd()
    gen = torch.Generator(device="cpu").manual_seed(3)
    lens = np.array([200, 64, 131], np.int64)
    c = workloads.make_context_inputs(3, 0, 8, 2, 128, 10, gen, "cpu", lens=lens)
    q, k, v, cu = (c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV), c["cu_seqlens"].to(DEV))

    def call(st):
        return rd.rd_causal_attention(q, k, v, cu, max_seqlen=int(lens.max()), dev_status=st)

    status, _ = _stalled(call)
    assert status & rd.DEV_TIMEOUT
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = call(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.oracle_causal_attention(bf16_bits(c["q"]), bf16_bits(c["k"]), bf16_bits(c["v"]),
                                         c["cu_seqlens"].numpy())
    _close(o.float().cpu().numpy(), ref, "causal after the timeout")


def test_fp8_attention_wait_runs_out_then_next_call_is_correct():
    rd = _rd()
    cfg = dataclasses.replace(workloads.CONFIGS["13b_b64"], B=3, Hq=4, Hkv=4, vocab=100)
    inp = workloads.make_verify_inputs(cfg, device=DEV, ctx_override=("uniform", 1, 400))
    kc, ks = workloads.make_fp8_cache(inp["k_cache"])
    vc, vs = workloads.make_fp8_cache(inp["v_cache"])
    pk = rd.rd_pack_beams(inp["beams"], cfg.P_max)
    max_ctx = int(inp["ctx_lens"].max())

    def call(st):
        return rd.rd_tree_attention_fp8(inp["q"], inp["k_draft"], inp["v_draft"], kc, vc, ks, vs,
                                        inp["ctx_offsets"], pk["packed_len"], pk["mask"],
                                        max_ctx=max_ctx, dev_status=st)

    status, _ = _stalled(call)
    assert status & rd.DEV_TIMEOUT
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = call(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pk = oracle.oracle_pack(inp["beams"].cpu().numpy(), cfg.P_max)
    ref = oracle.oracle_tree_attention_fp8(bf16_bits(inp["q"]), bf16_bits(inp["k_draft"]),
                                           bf16_bits(inp["v_draft"]), kc.cpu().numpy(),
                                           vc.cpu().numpy(), ks, vs,
                                           inp["ctx_offsets"].cpu().numpy(),
                                           ref_pk["packed_len"], ref_pk["mask"])
    _close(o.float().cpu().numpy(), ref, "fp8 after the timeout")
