"""Parity of rd_beam_search_step (through the C ABI) against the fp64 oracle.

The kernel ranks candidates by fp32 scores, the oracle by fp64 scores; they
must select the same candidates wherever the oracle's ranking is decided by
more than fp32 rounding.  Where two candidates are closer than that, either
order is correct: the test then checks that the GPU's selection is a valid
top-W (every selected candidate at least as good, within the rounding, as
every one left out).  Scores within 1e-4 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
EPS = 1e-4


def _check(lg, s_in, beams_in, got):
    ref = oracle.oracle_beam_search_step(bf16_bits(lg), s_in.double().cpu().numpy(),
                                         beams_in.cpu().numpy())
    x = (bf16_bits(lg).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    B, W, V = lg.shape
    t = beams_in.shape[2]
    gp = got["parent"].cpu().numpy()
    gb = got["beams"].cpu().numpy()
    gs = got["scores"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(gs, ref["scores"], atol=EPS, rtol=0)
    for b in range(B):
        s = s_in[b].double().cpu().numpy()
        lse = np.log(np.exp(x[b] - x[b].max(1, keepdims=True)).sum(1)) + x[b].max(1)
        cand = (s[:, None] + x[b] - lse[:, None]).reshape(-1)
        sel = gp[b] * V + gb[b, :, t]
        if np.array_equal(sel, ref["parent"][b] * V + ref["beams"][b, :, t]):
            continue
        # a near-tie: the GPU's set must be a valid top-W within the rounding
        assert len(set(sel.tolist())) == W
        rest = np.ones(W * V, bool)
        rest[sel] = False
        assert cand[sel].min() >= cand[rest].max() - EPS
        assert np.all(np.diff(cand[sel]) <= EPS)
    np.testing.assert_array_equal(gb[:, :, :t],
                                  beams_in.cpu().numpy()[np.arange(B)[:, None], gp])


# rows of up to 32768 tokens are held in registers, longer ones streamed; a
# batch of 40 requests at W = 8 takes clusters of four CTAs (two rows each),
# smaller ones one row per CTA; t = 0 is the first step (no beam prefix yet);
# 64 requests at W = 5 take clusters of four whose second rows mostly run past W
@pytest.mark.parametrize("B,W,V,t,ties", [(16, 8, 32000, 3, False), (4, 5, 1000, 1, True),
                                          (2, 16, 128256, 4, False), (3, 1, 77, 2, False),
                                          (2, 8, 32768, 2, False), (2, 8, 32776, 2, False),
                                          (40, 8, 1000, 2, True), (3, 16, 32000, 1, False),
                                          (3, 4, 1000, 0, False), (64, 5, 1000, 1, False)])
def test_beam_search_step(B, W, V, t, ties):
    import tree_attention_verify_gb300 as rd
    g = torch.Generator(device=DEV).manual_seed(W * V + t)
    x = torch.randn(B, W, V, generator=g, device=DEV) * 2
    if ties:
        x = torch.round(x)
    lg = x.to(torch.bfloat16)
    s_in = torch.randn(B, W, generator=g, device=DEV) * 3
    s_in[0, 1:] = -float("inf")
    beams_in = torch.randint(0, 1000, (B, W, t), generator=g, device=DEV, dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = rd.rd_beam_search_step(lg, s_in, beams_in, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check(lg, s_in, beams_in, got)


def test_beam_search_drafts_then_pack():
    # L-1 steps from the anchor produce W beams; they pack like any beam set
    import tree_attention_verify_gb300 as rd
    B, W, L, V = 4, 8, 5, 32000
    g = torch.Generator(device=DEV).manual_seed(3)
    beams = torch.randint(0, V, (B, 1, 1), generator=g, device=DEV, dtype=torch.int32)
    beams = beams.expand(B, W, 1).contiguous()
    scores = torch.full((B, W), -float("inf"), device=DEV)
    scores[:, 0] = 0.0
    for _ in range(L - 1):
        lg = (torch.randn(B, W, V, generator=g, device=DEV) * 2).to(torch.bfloat16)
        out = rd.rd_beam_search_step(lg, scores, beams)
        _check(lg, scores, beams, out)
        beams, scores = out["beams"], out["scores"]
    assert beams.shape == (B, W, L)
    for b in range(B):                             # beam search keeps distinct sequences
        assert len({tuple(r) for r in beams[b].cpu().numpy().tolist()}) == W
    pk = rd.rd_pack_beams(beams.contiguous(), W * L)
    ref = oracle.oracle_pack(beams.cpu().numpy(), W * L)
    np.testing.assert_array_equal(pk["packed_len"].cpu().numpy(), ref["packed_len"])


def test_beam_search_step_all_tied_rows():
    # every logit of a row equal: more tied candidates than the kernel's
    # candidate slots, which exercises its exact fallback selection
    import tree_attention_verify_gb300 as rd
    B, W, V, t = 3, 4, 5000, 2
    lg = torch.zeros((B, W, V), dtype=torch.bfloat16, device=DEV)
    lg[1, 2, 4000:] = 1.0                        # one row with a tied block at the top
    g = torch.Generator(device=DEV).manual_seed(7)
    s_in = torch.randn(B, W, generator=g, device=DEV)
    beams_in = torch.randint(0, 1000, (B, W, t), generator=g, device=DEV, dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = rd.rd_beam_search_step(lg, s_in, beams_in, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check(lg, s_in, beams_in, got)
