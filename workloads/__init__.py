"""Seeded synthetic inputs for the ReDrafter verification step.

This module only draws random inputs. It holds none of the arithmetic of the
method (no packing, no attention, no argmax, no acceptance): both the CUDA path
and the CPU oracle consume what it produces, and neither is imported here.

Workload shapes follow the pages' workloads, restated as five named configs:
Vicuna-7B/13B-class attention (32x128 and 40x128 heads, vocab 32000), an
8B-class GQA shape (32 query / 8 KV heads, vocab 128256), a tiny case, and an
in-flight batch mixing context-phase and generation-phase requests
("Recurrent Drafter for Fast Speculative Decoding in LLMs", abstract: beam
search drafts conditioned on the initial token; NVIDIA blog "ReDrafter in
TensorRT-LLM", section "Inflight-batching Compatible Engine": context and
generation sub-batches, either of which may be empty).

Draft trees. Each request's W beams of L tokens are drawn as a random trie:
position 0 of every beam is the anchor (the token the LLM already emitted);
beam 0 is the anchor followed by uniform tokens; beam w >= 1 copies the first
d tokens of beam w-1 and draws the rest, where d >= 1 is a random depth.  The
token drawn at the divergence point differs from every token already hanging
below the shared prefix, so beam w really leaves the trie there.  The
generator numbers trie nodes in the order it creates them; it uses that
numbering only to decide which logit rows to plant (so that a configured
fraction of drafts is accepted).  Whether the numbering equals the packed order
of the method does not affect parity, which always compares the CUDA path and
the oracle on the same inputs.

Logits.  bf16 N(0, std=2).  For each trie node that has a child, with the
configured probability, the first child's token gets the value 40.0 in that
node's row, which is above any N(0, 2) sample, so the greedy choice at that node
is the drafted token.  The tiny config also plants exact ties: 40.0 at a lower
index than the child token in some rows (so the lowest-index rule rejects the
draft), and 30.0 at two indices in some unplanted rows.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

PLANT_VALUE = 40.0
TIE_VALUE = 30.0


@dataclasses.dataclass(frozen=True)
class GenConfig:
    name: str
    B: int
    W: int
    L: int
    vocab: int
    Hq: int
    Hkv: int
    D: int
    Dh: int              # hidden size of the shape class (input of unpack)
    share: tuple         # ("depth",) | ("p", p) | ("p_range", lo, hi)
    ctx: tuple           # ("fixed", n) | ("uniform", lo, hi)
    plant: float         # probability that a node's first child is the greedy choice
    seed: int
    ties: bool = False   # plant exact bf16 ties (tiny config)

    @property
    def P_max(self) -> int:
        """Row stride of every packed tensor: the worst case W*L."""
        return self.W * self.L


CONFIGS = {
    "tiny": GenConfig("tiny", B=1, W=4, L=4, vocab=1000, Hq=1, Hkv=1, D=64, Dh=64,
                      share=("depth",), ctx=("fixed", 128), plant=0.6, seed=0,
                      ties=True),
    "7b_b1": GenConfig("7b_b1", B=1, W=5, L=4, vocab=32000, Hq=32, Hkv=32, D=128,
                       Dh=4096, share=("p", 0.5), ctx=("fixed", 2048), plant=0.7,
                       seed=1),
    "8b_gqa_b16": GenConfig("8b_gqa_b16", B=16, W=8, L=5, vocab=128256, Hq=32, Hkv=8,
                            D=128, Dh=4096, share=("p_range", 0.2, 0.8),
                            ctx=("uniform", 1024, 4096), plant=0.6, seed=2),
    "13b_b64": GenConfig("13b_b64", B=64, W=8, L=6, vocab=32000, Hq=40, Hkv=40, D=128,
                         Dh=5120, share=("p", 0.5), ctx=("fixed", 8192), plant=0.5,
                         seed=3),
}

# The in-flight mixed batch: 32 requests on the 8B GQA shapes.
MIXED = dict(n_requests=32, p_context=0.5, prefill_len=512, W=8, L=5,
             ctx=("uniform", 512, 8192), share=("p_range", 0.2, 0.8), plant=0.6,
             Hq=32, Hkv=8, D=128, Dh=4096, vocab=128256, seed=4)


# ----------------------------------------------------------------------------
# draft trees
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DraftTrees:
    beams: np.ndarray          # int32 [B, W, L]
    n_nodes: np.ndarray        # int32 [B]   generator's node count per request
    first_child: list          # per request: list (per generator node) of first child token or -1


def _share_depth(rng: np.random.Generator, share: tuple, L: int, p_req: float) -> int:
    if share[0] == "depth":
        return int(rng.integers(1, L + 1))
    d = 1
    while d < L and rng.random() < p_req:
        d += 1
    return d


def draft_trees(B: int, W: int, L: int, vocab: int, share: tuple,
                rng: np.random.Generator) -> DraftTrees:
    beams = np.zeros((B, W, L), dtype=np.int32)
    n_nodes = np.zeros(B, dtype=np.int32)
    first_child = []
    for b in range(B):
        if share[0] == "p_range":
            p_req = float(rng.uniform(share[1], share[2]))
        elif share[0] == "p":
            p_req = float(share[1])
        else:
            p_req = 0.0
        node_of = np.full((W, L), -1, dtype=np.int64)
        children: list = []      # per node: list of (token, child node)
        nn = 0
        for w in range(W):
            d = 0 if w == 0 else _share_depth(rng, share, L, p_req)
            for i in range(L):
                if i < d:
                    beams[b, w, i] = beams[b, w - 1, i]
                    node_of[w, i] = node_of[w - 1, i]
                    continue
                if w == 0 and i == 0:
                    tok = int(rng.integers(0, vocab))
                else:
                    parent = node_of[w, i - 1]
                    taken = {t for t, _ in children[parent]}
                    tok = int(rng.integers(0, vocab))
                    while tok in taken:
                        tok = int(rng.integers(0, vocab))
                beams[b, w, i] = tok
                node_of[w, i] = nn
                children.append([])
                if i > 0:
                    children[node_of[w, i - 1]].append((tok, nn))
                nn += 1
        n_nodes[b] = nn
        first_child.append([c[0][0] if c else -1 for c in children])
    return DraftTrees(beams=beams, n_nodes=n_nodes, first_child=first_child)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------
def _randn_bf16(shape, gen: torch.Generator, device, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def _ctx_lengths(ctx: tuple, B: int, rng: np.random.Generator) -> np.ndarray:
    if ctx[0] == "fixed":
        return np.full(B, ctx[1], dtype=np.int64)
    return rng.integers(ctx[1], ctx[2] + 1, size=B).astype(np.int64)


def make_logits(trees: DraftTrees, P_max: int, vocab: int, plant: float,
                rng: np.random.Generator, gen: torch.Generator, device,
                ties: bool = False) -> torch.Tensor:
    """bf16 [B, P_max, vocab] ~ N(0, 2) with planted greedy choices (see module doc)."""
    B = trees.beams.shape[0]
    logits = _randn_bf16((B, P_max, vocab), gen, device, std=2.0)
    rows, cols, vals = [], [], []
    for b in range(B):
        nn = int(trees.n_nodes[b])
        if nn < P_max:
            logits[b, nn:].zero_()
        for node in range(nn):
            child = trees.first_child[b][node]
            if child >= 0 and rng.random() < plant:
                rows.append(b * P_max + node); cols.append(child); vals.append(PLANT_VALUE)
                if ties and child > 0 and rng.random() < 0.3:
                    lower = int(rng.integers(0, child))
                    rows.append(b * P_max + node); cols.append(lower); vals.append(PLANT_VALUE)
            elif ties and rng.random() < 0.5:
                i1, i2 = rng.choice(vocab, size=2, replace=False)
                for c in (i1, i2):
                    rows.append(b * P_max + node); cols.append(int(c)); vals.append(TIE_VALUE)
    if rows:
        flat = logits.view(B * P_max, vocab)
        r = torch.tensor(rows, dtype=torch.long, device=logits.device)
        c = torch.tensor(cols, dtype=torch.long, device=logits.device)
        flat[r, c] = torch.tensor(vals, dtype=torch.bfloat16, device=logits.device)
    return logits


def make_verify_inputs(cfg: GenConfig, device="cpu", seed: Optional[int] = None,
                       ctx_override: Optional[tuple] = None) -> dict:
    """All inputs of one verification step for a generation sub-batch.

    Returns a dict of tensors on `device` (beams, q, k_draft, v_draft, k_cache,
    v_cache, ctx_offsets, logits, hidden) plus host metadata.  Packed tensors have
    row stride P_max = W*L; rows beyond a request's packed length are random
    (q, k_draft, v_draft, hidden) or zero (logits) and must be ignored.
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    trees = draft_trees(cfg.B, cfg.W, cfg.L, cfg.vocab, cfg.share, rng)
    ctx = ctx_override if ctx_override is not None else cfg.ctx
    lens = _ctx_lengths(ctx, cfg.B, rng)
    offsets = np.zeros(cfg.B + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(lens)
    total = int(offsets[-1])
    P = cfg.P_max
    out = dict(
        cfg=cfg, P_max=P, ctx_lens=lens, trees=trees,
        beams=torch.from_numpy(trees.beams.copy()).to(device),
        q=_randn_bf16((cfg.B, P, cfg.Hq, cfg.D), gen, device),
        k_draft=_randn_bf16((cfg.B, P, cfg.Hkv, cfg.D), gen, device),
        v_draft=_randn_bf16((cfg.B, P, cfg.Hkv, cfg.D), gen, device),
        k_cache=_randn_bf16((total, cfg.Hkv, cfg.D), gen, device),
        v_cache=_randn_bf16((total, cfg.Hkv, cfg.D), gen, device),
        ctx_offsets=torch.from_numpy(offsets).to(device),
        hidden=_randn_bf16((cfg.B, P, cfg.Dh), gen, device),
    )
    out["logits"] = make_logits(trees, P, cfg.vocab, cfg.plant, rng, gen, device,
                                ties=cfg.ties)
    return out


def make_context_inputs(n_req: int, T: int, Hq: int, Hkv: int, D: int, vocab: int,
                        gen: torch.Generator, device, lens: Optional[np.ndarray] = None
                        ) -> dict:
    """Inputs of a context-phase (prefill chunk) sub-batch: ragged q/k/v + last-row logits."""
    if lens is None:
        lens = np.full(n_req, T, dtype=np.int64)
    cu = np.zeros(n_req + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    tot = int(cu[-1])
    return dict(
        cu_seqlens=torch.from_numpy(cu).to(device),
        seq_lens=lens,
        q=_randn_bf16((tot, Hq, D), gen, device),
        k=_randn_bf16((tot, Hkv, D), gen, device),
        v=_randn_bf16((tot, Hkv, D), gen, device),
        logits=_randn_bf16((n_req, 1, vocab), gen, device, std=2.0),
    )


def make_mixed_inputs(split: str = "mixed", device="cpu", scale: float = 1.0,
                      seed: Optional[int] = None) -> dict:
    """The in-flight batch: 32 requests, each a context request with prob 0.5.

    split: "mixed" (the drawn mix), "all_ctx" or "all_gen" (one half empty).
    scale < 1 shrinks context and prefill lengths for quick tests.
    """
    m = MIXED
    seed = m["seed"] if seed is None else seed
    rng = np.random.default_rng(seed)
    is_ctx = rng.random(m["n_requests"]) < m["p_context"]
    if split == "all_ctx":
        is_ctx[:] = True
    elif split == "all_gen":
        is_ctx[:] = False
    n_ctx = int(is_ctx.sum())
    n_gen = m["n_requests"] - n_ctx
    T = max(1, int(m["prefill_len"] * scale))
    lo, hi = m["ctx"][1], m["ctx"][2]
    ctx = ("uniform", max(0, int(lo * scale)), max(0, int(hi * scale)))
    gen_cfg = GenConfig("mixed_gen", B=n_gen, W=m["W"], L=m["L"], vocab=m["vocab"],
                        Hq=m["Hq"], Hkv=m["Hkv"], D=m["D"], Dh=m["Dh"], share=m["share"],
                        ctx=ctx, plant=m["plant"], seed=seed + 100)
    gen_inp = make_verify_inputs(gen_cfg, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed + 200)
    ctx_inp = make_context_inputs(n_ctx, T, m["Hq"], m["Hkv"], m["D"], m["vocab"], g, device)
    return dict(is_context=is_ctx, n_ctx=n_ctx, n_gen=n_gen, gen=gen_inp, ctx=ctx_inp,
                prefill_len=T)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array (no rounding)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def make_paged(k_cache: torch.Tensor, v_cache: torch.Tensor, ctx_lens, page_size: int,
               rng: np.random.Generator, spare_pages: int = 2, spare_slots: int = 1) -> dict:
    """Scatter a contiguous ragged cache [sum C, Hkv, D] into a paged pool
    [num_pages, page_size, Hkv, D] whose pages are assigned in a random order.
    Each request gets `spare_slots` extra pages in its block table (room to append)
    and the pool holds `spare_pages` pages nobody uses; unused pool rows and
    table slots hold random junk."""
    lens = np.asarray(ctx_lens, np.int64)
    B = len(lens)
    need = [int(-(-int(c) // page_size)) + spare_slots for c in lens]
    max_pages = max(need) if B else 1
    n_pages = int(sum(need)) + spare_pages
    perm = rng.permutation(n_pages).astype(np.int32)
    table = rng.integers(-5, n_pages + 5, size=(B, max_pages)).astype(np.int32)
    Hkv, D = k_cache.shape[1], k_cache.shape[2]
    dev = k_cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(rng.integers(1 << 31)))
    k_pool = _randn_bf16((n_pages, page_size, Hkv, D), gen, dev)
    v_pool = _randn_bf16((n_pages, page_size, Hkv, D), gen, dev)
    off, k = 0, 0
    for b in range(B):
        table[b, :need[b]] = perm[k:k + need[b]]
        k += need[b]
        C = int(lens[b])
        for slot in range(-(-C // page_size)):
            n = min(page_size, C - slot * page_size)
            pg = int(table[b, slot])
            k_pool[pg, :n] = k_cache[off + slot * page_size: off + slot * page_size + n]
            v_pool[pg, :n] = v_cache[off + slot * page_size: off + slot * page_size + n]
        off += C
    return dict(k_pool=k_pool, v_pool=v_pool, block_table=torch.from_numpy(table).to(dev),
                ctx_lens=torch.from_numpy(lens.astype(np.int32)).to(dev), page_size=page_size)


def make_fp8_cache(cache: torch.Tensor) -> tuple:
    """Quantise a bf16 cache [rows, Hkv, D] to e4m3 with one scale per tensor
    (amax / 448, the largest finite e4m3 value).  Returns (uint8 codes, scale)."""
    amax = float(cache.float().abs().max()) if cache.numel() else 1.0
    scale = max(amax, 1e-30) / 448.0
    codes = (cache.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, scale


def make_draft_logits(target: torch.Tensor, gen: torch.Generator, mix: float = 0.7,
                      noise: float = 1.0) -> torch.Tensor:
    """Drafter logits correlated with the target's: bf16(mix * target + N(0, noise))."""
    n = torch.randn(target.shape, generator=gen, device=target.device, dtype=torch.float32)
    return (mix * target.float() + noise * n).to(torch.bfloat16)


def make_uniforms(B: int, P_max: int, V: int, rng: np.random.Generator) -> tuple:
    """The random numbers of stochastic verification: u_accept [B, P_max] and
    u_sample [B, V], float32 uniforms in [0, 1)."""
    return (torch.from_numpy(rng.random((B, P_max), dtype=np.float32)),
            torch.from_numpy(rng.random((B, V), dtype=np.float32)))


def make_sample_inputs(cfg: GenConfig, temperature: float = 1.0, device="cpu",
                       seed: Optional[int] = None) -> dict:
    """Inputs of stochastic verification for a generation sub-batch: beams, target
    logits (as make_logits), drafter logits correlated with them, and uniforms."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed + 1000)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1000)
    trees = draft_trees(cfg.B, cfg.W, cfg.L, cfg.vocab, cfg.share, rng)
    target = make_logits(trees, cfg.P_max, cfg.vocab, cfg.plant, rng, gen, device,
                         ties=cfg.ties)
    draft = make_draft_logits(target, gen)
    u_accept, u_sample = make_uniforms(cfg.B, cfg.P_max, cfg.vocab, rng)
    return dict(cfg=cfg, temperature=temperature, trees=trees,
                beams=torch.from_numpy(trees.beams.copy()).to(device), target=target,
                draft=draft, u_accept=u_accept.to(device), u_sample=u_sample.to(device))
