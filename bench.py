#!/usr/bin/env python
"""Benchmark of the ReDrafter verification step on GB300.

One step = rd_pack_beams + rd_tree_attention + rd_greedy_accept + rd_unpack over
one batch of the 13B-shaped workload (B=64 requests, W=8 beams x L=6 tokens,
40/40 heads x 128, context 8192, vocab 32000, hidden 5120), seeded synthetic
inputs resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (test infrastructure) on the host
cores, one whole step of the same workload per timed step.
For N > 1 (torchrun, one rank per GPU) every rank verifies its own batch
(weak scaling, no collective on the data path); the step time is the maximum
over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verify_steps_per_s"
UNIT = "steps/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0          # GB300 HBM3e, nominal (context for the measured peak)
# the sources the tree-attention kernel is compiled from (the ncu traffic figure
# in profiles/ holds only while their combined hash is the one recorded there)
ATTN_SRCS = [os.path.join(ROOT, "tree_attention_verify_gb300", "csrc", f)
             for f in ("attention_tc.cu", "attn_common.cuh", "tc_ptx.cuh")]


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="13b_b64", choices=list(workloads.CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip timing the calls beyond the verification step")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's request count (small profiling runs)")
    ap.add_argument("--profile-case", default="",
                    choices=["", "attention", "attention_fp8", "causal_all_ctx", "greedy_accept"],
                    help="run only this call (warmup + steps launches, no JSON contract line): "
                         "the commands the ncu summaries are taken with")
    return ap.parse_args()


def _config(args):
    import dataclasses
    cfg = workloads.CONFIGS[args.workload]
    if args.batch > 0:
        cfg = dataclasses.replace(cfg, B=args.batch, name=f"{cfg.name}_B{args.batch}")
    return cfg


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(cfg, rank: int) -> int:
    """Each rank verifies its own batch (weak scaling): its inputs use this seed."""
    return cfg.seed + 1000 * rank


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's value (the only collective besides the barrier)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _sha256(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _profile_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary,
    or None if there is none or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"tree_attention_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m2 = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not m1 or not m2 or m2.group(1) != _sha256(ATTN_SRCS):
        return None
    return float(m1.group(1))


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = [r.split(", ") for r in open(self.file.name).read().strip().splitlines()]
        os.unlink(self.file.name)
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                mhz.append(float(r[2]))
                mx.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(mhz)}


def attention_bytes(cfg, ctx_lens, packed_len) -> float:
    """Algorithmic HBM bytes of one rd_tree_attention launch: per (request, kv head)
    4*D*(C_b + P_b) bytes of K/V (context and drafts) plus 4*G*D*P_b bytes of q and o,
    plus the mask rows, offsets and lengths."""
    G = cfg.Hq // cfg.Hkv
    NW = (cfg.P_max + 31) // 32
    C = np.asarray(ctx_lens, np.float64)
    P = np.asarray(packed_len, np.float64)
    per_b = cfg.Hkv * (4.0 * cfg.D * (C + P) + 4.0 * G * cfg.D * P) + 4.0 * NW * P
    return float(per_b.sum() + cfg.B * 12 + 8)


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
def oracle_host_inputs(inp, n_req=None) -> dict:
    """Host copies (bf16 bit patterns) of the first n_req requests of one step's
    inputs (all requests if None), made once, outside any timed region."""
    bits = workloads.bf16_bits
    cfg = inp["cfg"]
    n_req = cfg.B if n_req is None else max(1, min(n_req, cfg.B))
    offs = inp["ctx_offsets"].cpu().numpy()[: n_req + 1]
    end = int(offs[-1])
    return dict(cfg=cfg, n_req=n_req, offs=offs, beams=inp["beams"][:n_req].cpu().numpy(),
                q=bits(inp["q"][:n_req]), kd=bits(inp["k_draft"][:n_req]),
                vd=bits(inp["v_draft"][:n_req]), kc=bits(inp["k_cache"][:end]),
                vc=bits(inp["v_cache"][:end]), logits=bits(inp["logits"][:n_req]),
                hidden=bits(inp["hidden"][:n_req]))


def oracle_step_time(h: dict, threads: int) -> float:
    """Seconds of one oracle verification step over the requests in h: pack,
    tree attention, greedy accept and unpack, as the GPU step runs them."""
    import oracle
    t0 = time.perf_counter()
    pk = oracle.oracle_pack(h["beams"], h["cfg"].P_max)
    oracle.oracle_tree_attention(h["q"], h["kd"], h["vd"], h["kc"], h["vc"], h["offs"],
                                 pk["packed_len"], pk["mask"], n_threads=threads)
    oracle.oracle_greedy_accept(h["logits"], h["beams"], pk["unpacker"], pk["packed_len"])
    oracle.oracle_unpack(h["hidden"], pk["unpacker"])
    return time.perf_counter() - t0


def run_reference(args):
    """The oracle timed on the host cores: every timed step is one whole
    verification step of the workload (all requests, all heads); each warm-up
    step runs the first request only (it loads the library and touches the code;
    a whole step there would only add minutes)."""
    import oracle
    world, rank, _ = _dist()
    if rank != 0:
        return
    cfg = _config(args)
    inp = workloads.make_verify_inputs(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
    oracle.build()
    threads = oracle.n_threads_default()
    h_full = oracle_host_inputs(inp)
    h_warm = oracle_host_inputs(inp, 1)
    del inp
    for _ in range(args.warmup):
        oracle_step_time(h_warm, threads)
    times = [oracle_step_time(h_full, threads) for _ in range(args.steps)]
    step_s = statistics.mean(times)
    value = 1.0 / step_s
    sample = (f"every timed step is one whole {cfg.B}-request step (pack, tree attention, greedy "
              f"accept, unpack) of the fp64 oracle on {threads} threads; warm-up steps run "
              f"request 0 only")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": cfg.name, "B": cfg.B, "W": cfg.W, "L": cfg.L, "Hq": cfg.Hq,
                       "Hkv": cfg.Hkv, "D": cfg.D, "context": cfg.ctx[1], "vocab": cfg.vocab,
                       "Dh": cfg.Dh},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                             "host_cpus": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our CUDA path
# ----------------------------------------------------------------------------
# A spin kernel of this many SM clocks (about 100 us) per call is queued ahead of
# the timed calls, so that the host has enqueued them before the device reaches
# them: the events then time the calls' device work, not the host's call overhead.
_HOST_AHEAD_CYCLES = 200_000


def _time_us(fn, n: int = 20) -> float:
    """Mean device time of one call, n calls back to back on the current stream
    (CUDA events, after three warm-up calls)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(_HOST_AHEAD_CYCLES * n)     # the device idles while the host enqueues
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n * 1e3


def _time_us_cold(fn, flush: torch.Tensor, n: int = 30) -> float:
    """Mean device time of one call with L2 flushed before each call: the flush
    (a write of a buffer larger than L2) runs outside the events around the call."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for e0, e1 in evs:
        torch.cuda._sleep(_HOST_AHEAD_CYCLES)
        flush.zero_()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3


def measure_other_configs(dev, peak: float) -> dict:
    """rd_tree_attention and rd_greedy_accept on the 8B-GQA serving batch and the
    7B batch-1 workloads, each call timed with L2 flushed before it (their inputs
    are smaller than or close to L2)."""
    import tree_attention_verify_gb300 as rd
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)     # 256 MB
    rows = {}
    for name in ("8b_gqa_b16", "7b_b1"):
        cfg = workloads.CONFIGS[name]
        inp = workloads.make_verify_inputs(cfg, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
        max_ctx = int(inp["ctx_lens"].max())
        n_ws = rd.rd_tree_attention_workspace_size(cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D,
                                                   max_ctx, dev)
        ws = torch.zeros(max(16, n_ws), dtype=torch.uint8, device=dev)
        o = torch.empty_like(inp["q"])
        us = _time_us_cold(lambda: rd.rd_tree_attention(
            inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"], inp["v_cache"],
            inp["ctx_offsets"], pk["packed_len"], pk["mask"], max_ctx=max_ctx, out=o,
            workspace=ws, dev_status=st), flush)
        plen = pk["packed_len"].cpu().numpy()
        nb = attention_bytes(cfg, inp["ctx_lens"], plen)
        wsa = torch.zeros(max(8, rd.rd_greedy_accept_workspace_size(cfg.B, cfg.P_max,
                                                                    cfg.vocab)),
                          dtype=torch.uint8, device=dev)
        acc = rd.rd_greedy_accept(inp["logits"], inp["beams"], pk["unpacker"], pk["packed_len"],
                                  workspace=wsa, dev_status=st)
        us_acc = _time_us_cold(lambda: rd.rd_greedy_accept(
            inp["logits"], inp["beams"], pk["unpacker"], pk["packed_len"], out=acc,
            workspace=wsa, dev_status=st), flush)
        acc_bytes = float(plen.sum()) * cfg.vocab * 2
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise SystemExit(f"device status {int(st.item())} on {name}")
        rows[name] = {
            "rd_tree_attention": {"us": us, "gbs": nb / us / 1e3, "frac": nb / us / 1e3 / peak,
                                  "algorithmic_bytes": nb, "workspace_bytes": n_ws},
            "rd_greedy_accept": {"us": us_acc, "gbs": acc_bytes / us_acc / 1e3,
                                 "frac": acc_bytes / us_acc / 1e3 / peak},
            "l2": "flushed before every timed call"}
        del inp, o, ws
    return rows


def measure_next_rows(cfg, inp, step, dev, peak: float) -> dict:
    """The calls beyond the verification step, timed on the same workload's
    tensors after the timed region: FP8 and paged-cache attention, stochastic
    verification, commit of the accepted path, and one drafter beam-search step."""
    import tree_attention_verify_gb300 as rd
    rows = {}
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pk, acc = step.pk, step.acc
    max_ctx = max(1, int(inp["ctx_lens"].max()))
    ws = torch.zeros(max(16, rd.rd_tree_attention_workspace_size(
        cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D, max_ctx, dev)), dtype=torch.uint8, device=dev)
    o = torch.empty_like(inp["q"])
    plen = pk["packed_len"].cpu().numpy()
    bf16_bytes = attention_bytes(cfg, inp["ctx_lens"], plen)
    ctx_kv = cfg.Hkv * 4.0 * cfg.D * float(np.asarray(inp["ctx_lens"], np.float64).sum())
    # FP8 (e4m3) context cache: context K/V bytes halve
    kc, ks = workloads.make_fp8_cache(inp["k_cache"])
    vc, vs = workloads.make_fp8_cache(inp["v_cache"])
    us = _time_us(lambda: rd.rd_tree_attention_fp8(
        inp["q"], inp["k_draft"], inp["v_draft"], kc, vc, ks, vs, inp["ctx_offsets"],
        pk["packed_len"], pk["mask"], max_ctx=max_ctx, out=o, workspace=ws, dev_status=st))
    b8 = bf16_bytes - ctx_kv / 2
    rows["rd_tree_attention_fp8"] = {"us": us, "gbs": b8 / us / 1e3, "frac": b8 / us / 1e3 / peak,
                                     "algorithmic_bytes": b8}
    del kc, vc
    # paged cache (256-position pages in a shuffled pool)
    pg = workloads.make_paged(inp["k_cache"], inp["v_cache"], inp["ctx_lens"], 256,
                              np.random.default_rng(cfg.seed + 5))
    us = _time_us(lambda: rd.rd_tree_attention_paged(
        inp["q"], inp["k_draft"], inp["v_draft"], pg["k_pool"], pg["v_pool"], pg["block_table"],
        pg["ctx_lens"], pk["packed_len"], pk["mask"], max_ctx=max_ctx, out=o, workspace=ws,
        dev_status=st))
    rows["rd_tree_attention_paged"] = {"us": us, "gbs": bf16_bytes / us / 1e3,
                                       "frac": bf16_bytes / us / 1e3 / peak, "page_size": 256}
    # commit of the accepted path into the paged cache (idempotent: lengths not advanced)
    new_lens = torch.empty_like(pg["ctx_lens"])
    us = _time_us(lambda: rd.rd_commit_accepted(
        inp["k_draft"], inp["v_draft"], pk["unpacker"], acc["best_beam"], acc["n_accepted"],
        pg["k_pool"], pg["v_pool"], pg["block_table"], pg["ctx_lens"], new_ctx_lens=new_lens,
        dev_status=st))
    rows["rd_commit_accepted"] = {"us": us}
    del pg
    # stochastic verification with drafter logits correlated with the target's
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed + 6)
    draft = workloads.make_draft_logits(inp["logits"], gen)
    ua, usm = workloads.make_uniforms(cfg.B, cfg.P_max, cfg.vocab, np.random.default_rng(cfg.seed + 6))
    ua, usm = ua.to(dev), usm.to(dev)
    sout = rd.rd_sample_accept(inp["logits"], draft, 1.0, inp["beams"], pk["packer"],
                               pk["unpacker"], pk["packed_len"], ua, usm, dev_status=st)
    us = _time_us(lambda: rd.rd_sample_accept(
        inp["logits"], draft, 1.0, inp["beams"], pk["packer"], pk["unpacker"], pk["packed_len"],
        ua, usm, out=sout, dev_status=st))
    rows["rd_sample_accept"] = {"us": us, "temperature": 1.0,
                                "mean_accepted": float(sout["n_accepted"].float().mean())}
    # one drafter beam-search step (W x V candidates per request)
    lg = (torch.randn((cfg.B, cfg.W, cfg.vocab), generator=gen, device=dev) * 2).to(torch.bfloat16)
    sc = torch.zeros((cfg.B, cfg.W), dtype=torch.float32, device=dev)
    bi = inp["beams"][:, :, :cfg.L - 1].contiguous()
    bout = rd.rd_beam_search_step(lg, sc, bi, dev_status=st)
    us = _time_us(lambda: rd.rd_beam_search_step(lg, sc, bi, out=bout, dev_status=st))
    nb = lg.numel() * 2                        # the drafter logits, read once
    rows["rd_beam_search_step"] = {"us": us, "gbs": nb / us / 1e3, "frac": nb / us / 1e3 / peak,
                                   "algorithmic_bytes": float(nb)}
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise SystemExit(f"device status {int(st.item())} in the next-row calls")
    return rows


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measure_mixed(dev) -> dict:
    """The in-flight batch on 8B-GQA shapes (32 requests, each a 512-token causal
    prefill chunk with probability 0.5, else a W=8, L=5 verification over a
    512-8192 context) and its all-context / all-generation splits: one in-flight
    step = causal attention + next-token argmax of the context half, and
    pack + tree attention + greedy accept + unpack of the generation half."""
    import tree_attention_verify_gb300 as rd
    from tree_attention_verify_gb300.step import VerifyStep
    peak_tf, _ = _peak_tflops()
    peak_gbs, _ = _peak_hbm()
    out = {}
    for split in ("mixed", "all_ctx", "all_gen"):
        m = workloads.make_mixed_inputs(split, device=dev)
        c, g = m["ctx"], m["gen"]
        n_ctx, n_gen, T = m["n_ctx"], m["n_gen"], m["prefill_len"]
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        parts = []
        row = {"n_context": n_ctx, "n_generation": n_gen}
        if n_ctx:
            oc = torch.empty_like(c["q"])
            one = torch.zeros((n_ctx, 1, 1), dtype=torch.int32, device=dev)
            plen1 = torch.ones(n_ctx, dtype=torch.int32, device=dev)
            V = c["logits"].shape[2]
            wsc = torch.zeros(max(8, rd.rd_greedy_accept_workspace_size(n_ctx, 1, V)),
                              dtype=torch.uint8, device=dev)
            accc = rd.rd_greedy_accept(c["logits"], one, one, plen1, workspace=wsc, dev_status=st)
            causal = lambda: rd.rd_causal_attention(c["q"], c["k"], c["v"], c["cu_seqlens"],  # noqa
                                                    max_seqlen=T, out=oc, dev_status=st)
            parts.append(causal)
            parts.append(lambda: rd.rd_greedy_accept(c["logits"], one, one, plen1, out=accc,
                                                     workspace=wsc, dev_status=st))
            Hq, D = c["q"].shape[1], c["q"].shape[2]
            flops = float(sum(4.0 * Hq * D * t * (t + 1) / 2 for t in c["seq_lens"]))
            # algorithmic bytes: q, k, v read once, o written once
            nbytes = float(2 * c["q"].numel() + c["k"].numel() + c["v"].numel()) * 2.0
            us = _time_us(causal)
            # the binding roof is the one with the longer minimum time
            hbm_bound = nbytes / (peak_gbs * 1e3) >= flops / (peak_tf * 1e6)
            row["rd_causal_attention"] = {"us": us, "tflops": flops / us / 1e6,
                                          "tensor_frac": flops / us / 1e6 / peak_tf,
                                          "gbs": nbytes / us / 1e3,
                                          "hbm_frac": nbytes / us / 1e3 / peak_gbs,
                                          "algorithmic_bytes": nbytes,
                                          "bound": "hbm" if hbm_bound else "tensor",
                                          "frac": (nbytes / us / 1e3 / peak_gbs) if hbm_bound
                                          else flops / us / 1e6 / peak_tf}
        if n_gen:
            gc = g["cfg"]
            step = VerifyStep(gc.B, gc.W, gc.L, gc.Hq, gc.Hkv, gc.D, gc.vocab, gc.Dh,
                              max(1, int(g["ctx_lens"].max())), dev)
            parts.append(lambda: step(g["beams"], g["q"], g["k_draft"], g["v_draft"],
                                      g["k_cache"], g["v_cache"], g["ctx_offsets"], g["logits"],
                                      g["hidden"]))
        us = _time_us(lambda: [f() for f in parts])
        row["step_us"] = us
        row["requests_per_s"] = (n_ctx + n_gen) / us * 1e6
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise SystemExit(f"device status {int(st.item())} in the in-flight batch")
        out[split] = row
    return out


def run_ours(args):
    import tree_attention_verify_gb300 as rd
    from tree_attention_verify_gb300.step import VerifyStep

    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist

    cfg = _config(args)
    inp = workloads.make_verify_inputs(cfg, device=dev, seed=rank_seed(cfg, rank))
    max_ctx = int(inp["ctx_lens"].max())
    step = VerifyStep(cfg.B, cfg.W, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab, cfg.Dh, max_ctx,
                      dev)
    call = lambda ev=None: step(inp["beams"], inp["q"], inp["k_draft"], inp["v_draft"],  # noqa
                                inp["k_cache"], inp["v_cache"], inp["ctx_offsets"],
                                inp["logits"], inp["hidden"], events=ev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local).start()
    time.sleep(0.3)
    t0.record(stream)
    for k in range(K):
        call(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), pg, dev)
    ms_step = ms / K
    kern_us = {name: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K)) * 1e3
               for i, name in enumerate(("rd_pack_beams", "rd_tree_attention", "rd_greedy_accept",
                                          "rd_unpack"))}
    status = int(step.status.item())
    if status != 0:
        raise SystemExit(f"device status {status} after the timed steps")

    packed_len = step.pk["packed_len"].cpu().numpy()
    n_acc = step.acc["n_accepted"].cpu().numpy()
    draft_tokens = cfg.B * cfg.W * cfg.L
    value = world * 1e3 / ms_step
    attn_bytes = attention_bytes(cfg, inp["ctx_lens"], packed_len)
    attn_s = kern_us["rd_tree_attention"] * 1e-6
    peak, peak_kind = _peak_hbm()
    achieved = attn_bytes / attn_s / 1e9
    roofline = {"bound": "hbm", "kernel": "rd_tree_attention", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "traffic": _profile_traffic(cfg.name),
                "algorithmic_bytes_per_launch": attn_bytes,
                "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "nominal_peak": NOMINAL_HBM_GBS}

    next_rows = None
    if rank == 0 and not args.no_next_rows:
        next_rows = measure_next_rows(cfg, inp, step, dev, peak)
        next_rows["inflight_batch_8b"] = measure_mixed(dev)
        next_rows["other_configs"] = measure_other_configs(dev, peak)

    # ---- end to end through the public API, host buffers ----------------------
    # Every step copies its inputs from pinned host memory and reads its accepted
    # tokens back.  Two device buffer sets and a copy stream let the copies of
    # step k+1 run while step k computes (at most two steps in flight).
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        names = ("beams", "q", "k_draft", "v_draft", "logits", "hidden")
        host = {n: torch.empty_like(inp[n], device="cpu").pin_memory() for n in names}
        for n in names:
            host[n].copy_(inp[n])
        devbuf = [{n: torch.empty_like(inp[n]) for n in names} for _ in range(2)]
        outs = ("out_tokens", "n_accepted", "best_beam")
        host_out = [{n: torch.empty_like(step.acc[n], device="cpu").pin_memory() for n in outs}
                    for _ in range(2)]
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = sum(host_out[0][n].numel() * host_out[0][n].element_size() for n in outs)
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n_steps):
            # iteration k: enqueue step k-1 first (its inputs were copied in
            # iteration k-1), so the compute stream never waits for the host;
            # then wait until step k-2 has finished (its buffers are free) and
            # enqueue the copies of step k
            for k in range(n_steps + 1):
                if k >= 1:
                    j = k - 1
                    sb = j % 2
                    stream.wait_event(copied[sb])
                    d = devbuf[sb]
                    step(d["beams"], d["q"], d["k_draft"], d["v_draft"], inp["k_cache"],
                         inp["v_cache"], inp["ctx_offsets"], d["logits"], d["hidden"])
                    consumed[sb].record(stream)
                    for n in outs:
                        host_out[sb][n].copy_(step.acc[n], non_blocking=True)
                    done[sb].record(stream)
                if k < n_steps:
                    sb = k % 2
                    if k >= 2:
                        done[sb].synchronize()            # result k-2 read back, buffers free
                    copy_stream.wait_event(consumed[sb])
                    with torch.cuda.stream(copy_stream):
                        for n in names:
                            devbuf[sb][n].copy_(host[n], non_blocking=True)
                        copied[sb].record(copy_stream)
            for e in done:
                e.synchronize()

        e2e_run(3)
        if pg:
            pg.barrier()
        w0 = time.perf_counter()
        e2e_run(args.e2e_steps)
        wall = max_over_ranks(time.perf_counter() - w0, pg, dev)
        e2e = {"value": world * args.e2e_steps / wall, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "note": "per-step inputs (beams, q/k/v of the drafts, logits, hidden) copied from "
                       "pinned host memory and accepted tokens read back every step, copies of "
                       "step k+1 overlapped with step k; the KV cache is resident state"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.n_threads_default()
        h = oracle_host_inputs(inp)
        dt = oracle_step_time(h, threads)
        del h
        cpu = {"value": 1.0 / dt, "unit": UNIT, "cores": threads, "host_cpus": os.cpu_count(),
               "kind": "oracle",
               "sample": f"one whole step of the workload ({cfg.B} requests: pack, tree "
                         f"attention, greedy accept, unpack) of the fp64 oracle, {dt:.1f} s, "
                         f"not scaled"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "B": cfg.B, "W": cfg.W, "L": cfg.L, "Hq": cfg.Hq,
                       "Hkv": cfg.Hkv, "D": cfg.D, "context": max_ctx, "vocab": cfg.vocab,
                       "Dh": cfg.Dh, "l2": "inputs larger than L2 (KV cache "
                       f"{inp['k_cache'].numel() * 4 / 1e9:.1f} GB)",
                       "parallelism": f"replicas x{world}"},
            "draft_tokens_per_s": value * draft_tokens,
            "packed_tokens_per_s": world * 1e3 / ms_step * float(packed_len.sum()),
            "dedup_pct": 100.0 * (1.0 - packed_len.sum() / draft_tokens),
            "mean_accepted": float(n_acc.mean()),
            "kernel_us": kern_us,
            "tree_attention_gbs": achieved,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "next_rows": next_rows,
            # per step: pack, attention (+ the merge launch when the batch takes
            # chunk ranges), greedy accept (argmax, then acceptance), unpack
            "gpu_launches": (1 + (2 if rd.rd_tree_attention_workspace_size(
                cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D, max_ctx, dev) > 0 else 1) + 2 + 1) * K,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def run_profile_case(args):
    """One call of the path, repeated: --warmup untimed launches, then --steps more,
    on the workload (--workload, --batch).  A profiler skips the warm-up launches
    and captures the next one; the printed time is only a sanity figure."""
    import tree_attention_verify_gb300 as rd
    dev = torch.device("cuda", 0)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    case = args.profile_case
    if case == "causal_all_ctx":
        m = workloads.make_mixed_inputs("all_ctx", device=dev)
        c = m["ctx"]
        o = torch.empty_like(c["q"])
        fn = lambda: rd.rd_causal_attention(c["q"], c["k"], c["v"], c["cu_seqlens"],  # noqa
                                            max_seqlen=m["prefill_len"], out=o, dev_status=st)
        name = f"in-flight batch, all context ({m['n_ctx']} x {m['prefill_len']} tokens)"
    else:
        cfg = _config(args)
        inp = workloads.make_verify_inputs(cfg, device=dev)
        pk = rd.rd_pack_beams(inp["beams"], cfg.P_max, dev_status=st)
        max_ctx = max(1, int(inp["ctx_lens"].max()))
        name = cfg.name
        if case == "greedy_accept":
            ws = torch.zeros(max(8, rd.rd_greedy_accept_workspace_size(cfg.B, cfg.P_max, cfg.vocab)),
                             dtype=torch.uint8, device=dev)
            acc = rd.rd_greedy_accept(inp["logits"], inp["beams"], pk["unpacker"], pk["packed_len"],
                                      workspace=ws, dev_status=st)
            fn = lambda: rd.rd_greedy_accept(inp["logits"], inp["beams"], pk["unpacker"],  # noqa
                                             pk["packed_len"], out=acc, workspace=ws, dev_status=st)
        else:
            ws = torch.zeros(max(16, rd.rd_tree_attention_workspace_size(
                cfg.B, cfg.P_max, cfg.Hq, cfg.Hkv, cfg.D, max_ctx, dev)), dtype=torch.uint8, device=dev)
            o = torch.empty_like(inp["q"])
            if case == "attention_fp8":
                kc, ks = workloads.make_fp8_cache(inp["k_cache"])
                vc, vs = workloads.make_fp8_cache(inp["v_cache"])
                del inp["k_cache"], inp["v_cache"]
                fn = lambda: rd.rd_tree_attention_fp8(  # noqa
                    inp["q"], inp["k_draft"], inp["v_draft"], kc, vc, ks, vs, inp["ctx_offsets"],
                    pk["packed_len"], pk["mask"], max_ctx=max_ctx, out=o, workspace=ws, dev_status=st)
            else:
                fn = lambda: rd.rd_tree_attention(  # noqa
                    inp["q"], inp["k_draft"], inp["v_draft"], inp["k_cache"], inp["v_cache"],
                    inp["ctx_offsets"], pk["packed_len"], pk["mask"], max_ctx=max_ctx, out=o,
                    workspace=ws, dev_status=st)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise SystemExit(f"device status {int(st.item())}")
    us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
    print(json.dumps({"profile_case": case, "workload": name, "launches": args.warmup + args.steps,
                      "us_per_launch_warm": us}), flush=True)


def main():
    args = _args()
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
