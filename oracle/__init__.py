"""fp64 CPU oracle of the ReDrafter verification step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA library and never
imports it.  The arithmetic lives in ``rd_oracle.c`` (plain C, fp64); this
module compiles it with gcc, marshals numpy arrays into it, and adds
``oracle_unpack``, the gather written as plain numpy indexing.

Each function states the passage it follows in the C source; the unpack gather
follows the PyTorch listing in the NVIDIA blog "ReDrafter in TensorRT-LLM",
section "Implementing in-Engine Validation and Drafting" (gather along the
packed dimension with the unpacker as index, reshaped to [B, W, L, D]).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rd_oracle.c")
_LIB = os.path.join(_HERE, "librd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile rd_oracle.c into librd_oracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
               "-lpthread"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_pack.argtypes = [P, I, I, I, I, P, P, P, P, P, P]
            lib.oracle_tree_attention.argtypes = [I, I, I, I, I, ctypes.c_double, P, P, P, P,
                                                  P, P, P, P, I, P, I]
            lib.oracle_causal_attention.argtypes = [I, I, I, I, ctypes.c_double, P, P, P, P,
                                                    P, I]
            lib.oracle_tree_attention_paged.argtypes = [I, I, I, I, I, ctypes.c_double, P, P, P,
                                                        P, P, I, I, P, I, P, P, P, I, P, I]
            lib.oracle_greedy_accept.argtypes = [P, I, I, I, P, P, P, I, I, P, P, P, P, P]
            lib.oracle_beam_search_step.argtypes = [P, P, P, I, I, I, I, P, P, P]
            lib.oracle_tree_attention_fp8.argtypes = [I, I, I, I, I, ctypes.c_double, P, P, P, P,
                                                      P, ctypes.c_double, ctypes.c_double, P, P,
                                                      P, I, P]
            lib.oracle_sample_accept.argtypes = [P, P, I, I, I, ctypes.c_double, P, P, P, P, I,
                                                 I, P, P, P, P, P, P, P]
            lib.oracle_e4m3_value.argtypes = [I]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            for f in (lib.oracle_pack, lib.oracle_tree_attention,
                      lib.oracle_tree_attention_paged, lib.oracle_causal_attention,
                      lib.oracle_greedy_accept, lib.oracle_beam_search_step,
                      lib.oracle_tree_attention_fp8, lib.oracle_sample_accept):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


def oracle_pack(beams: np.ndarray, P_cap: int | None = None) -> dict:
    """Prefix dedup of [B, W, L] beams (see oracle_pack in rd_oracle.c)."""
    beams = _c(beams, np.int32)
    B, W, L = beams.shape
    P_cap = W * L if P_cap is None else P_cap
    NW = (P_cap + 31) // 32
    out = dict(tokens=np.zeros((B, P_cap), np.int32), packer=np.zeros((B, P_cap), np.int32),
               unpacker=np.zeros((B, W, L), np.int32),
               mask=np.zeros((B, P_cap, NW), np.uint32), depth=np.zeros((B, P_cap), np.int32),
               packed_len=np.zeros(B, np.int32))
    rc = _load().oracle_pack(_ptr(beams), B, W, L, P_cap, _ptr(out["tokens"]),
                             _ptr(out["packer"]), _ptr(out["unpacker"]), _ptr(out["mask"]),
                             _ptr(out["depth"]), _ptr(out["packed_len"]))
    if rc != 0:
        raise ValueError(f"oracle_pack rejected the input (rc={rc})")
    return out


def oracle_tree_attention(q, k_new, v_new, k_cache, v_cache, ctx_offsets, packed_len,
                          mask, scale: float = 0.0, n_threads: int | None = None
                          ) -> np.ndarray:
    """Tree-masked attention in fp64.  bf16 inputs as uint16 bit arrays:
    q [B,P,Hq,D], k_new/v_new [B,P,Hkv,D], k_cache/v_cache [sum C, Hkv, D],
    ctx_offsets int64 [B+1], packed_len int32 [B], mask uint32 [B,P,NW].
    Returns float64 [B,P,Hq,D]."""
    q = _c(q, np.uint16); k_new = _c(k_new, np.uint16); v_new = _c(v_new, np.uint16)
    k_cache = _c(k_cache, np.uint16); v_cache = _c(v_cache, np.uint16)
    ctx_offsets = _c(ctx_offsets, np.int64); packed_len = _c(packed_len, np.int32)
    mask = _c(mask, np.uint32)
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    o = np.zeros((B, P, Hq, D), np.float64)
    rc = _load().oracle_tree_attention(B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new),
                                       _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(ctx_offsets), _ptr(packed_len), _ptr(mask),
                                       mask.shape[2], _ptr(o),
                                       n_threads or n_threads_default())
    if rc != 0:
        raise ValueError(f"oracle_tree_attention rejected the input (rc={rc})")
    return o


def oracle_tree_attention_paged(q, k_new, v_new, k_pool, v_pool, block_table, ctx_lens,
                                packed_len, mask, scale: float = 0.0,
                                n_threads: int | None = None) -> np.ndarray:
    """Tree-masked attention with the context in a paged cache (see
    oracle_tree_attention_paged in rd_oracle.c): k_pool/v_pool [pages, page_size,
    Hkv, D] (uint16 bf16 bits), block_table int32 [B, max_pages], ctx_lens int32 [B]."""
    q = _c(q, np.uint16); k_new = _c(k_new, np.uint16); v_new = _c(v_new, np.uint16)
    k_pool = _c(k_pool, np.uint16); v_pool = _c(v_pool, np.uint16)
    block_table = _c(block_table, np.int32); ctx_lens = _c(ctx_lens, np.int32)
    packed_len = _c(packed_len, np.int32); mask = _c(mask, np.uint32)
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    num_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    o = np.zeros((B, P, Hq, D), np.float64)
    rc = _load().oracle_tree_attention_paged(
        B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
        _ptr(v_pool), num_pages, page_size, _ptr(block_table), block_table.shape[1],
        _ptr(ctx_lens), _ptr(packed_len), _ptr(mask), mask.shape[2], _ptr(o),
        n_threads or n_threads_default())
    if rc != 0:
        raise ValueError(f"oracle_tree_attention_paged rejected the input (rc={rc})")
    return o


def oracle_e4m3_value(code: int) -> float:
    """The value of an e4m3 bit pattern (see e4m3_to_f64 in rd_oracle.c)."""
    return float(_load().oracle_e4m3_value(int(code)))


def oracle_tree_attention_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, ctx_offsets,
                              packed_len, mask, scale: float = 0.0) -> np.ndarray:
    """Tree-masked attention with e4m3 context K/V (uint8 bit patterns
    [sum C, Hkv, D]) and per-tensor scales; q/k_new/v_new bf16 bits as in
    oracle_tree_attention.  Returns float64 [B, P, Hq, D]."""
    q = _c(q, np.uint16); k_new = _c(k_new, np.uint16); v_new = _c(v_new, np.uint16)
    k_cache = _c(k_cache, np.uint8); v_cache = _c(v_cache, np.uint8)
    ctx_offsets = _c(ctx_offsets, np.int64); packed_len = _c(packed_len, np.int32)
    mask = _c(mask, np.uint32)
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    o = np.zeros((B, P, Hq, D), np.float64)
    rc = _load().oracle_tree_attention_fp8(B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new),
                                           _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                           float(k_scale), float(v_scale), _ptr(ctx_offsets),
                                           _ptr(packed_len), _ptr(mask), mask.shape[2], _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle_tree_attention_fp8 rejected the input (rc={rc})")
    return o


def oracle_commit_accepted(k_new, v_new, unpacker, best_beam, n_accepted, k_pool, v_pool,
                           block_table, ctx_lens):
    """Append the K/V of each request's accepted path to its paged cache.

    The accepted path of request b is its best beam's anchor and accepted drafts,
    nodes (w*, 0..a) with a = n_accepted[b]; their K/V rows k_new[b, unpacker[b, w*, i]]
    go to context positions ctx_lens[b] + i of the paged cache (the tokens the
    verification step has confirmed; NVIDIA blog introduction: accept the best
    path before drafting the next tokens).  Returns (k_pool, v_pool, new_ctx_lens)
    as new arrays; the inputs are not modified."""
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    new_lens = np.array(ctx_lens, dtype=np.int32, copy=True)
    page_size = k_pool.shape[1]
    for b in range(unpacker.shape[0]):
        w, a, C = int(best_beam[b]), int(n_accepted[b]), int(ctx_lens[b])
        for i in range(a + 1):
            pos = C + i
            page = int(block_table[b, pos // page_size])
            node = int(unpacker[b, w, i])
            k_pool[page, pos % page_size] = k_new[b, node]
            v_pool[page, pos % page_size] = v_new[b, node]
        new_lens[b] = C + a + 1
    return k_pool, v_pool, new_lens


def oracle_causal_attention(q, k, v, cu_seqlens, scale: float = 0.0,
                            n_threads: int | None = None) -> np.ndarray:
    """Causal attention per sequence in fp64: q [T,Hq,D], k/v [T,Hkv,D] (uint16 bf16 bits),
    cu_seqlens int32 [Bc+1].  Returns float64 [T,Hq,D]."""
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    o = np.zeros((T, Hq, D), np.float64)
    rc = _load().oracle_causal_attention(len(cu) - 1, Hq, Hkv, D, float(scale), _ptr(q),
                                         _ptr(k), _ptr(v), _ptr(cu), _ptr(o),
                                         n_threads or n_threads_default())
    if rc != 0:
        raise ValueError(f"oracle_causal_attention rejected the input (rc={rc})")
    return o


def oracle_sample_accept(target, draft, temperature, beams, packer, unpacker, packed_len,
                         u_accept, u_sample) -> dict:
    """Stochastic verification by multi-step speculative sampling (see
    oracle_sample_accept in rd_oracle.c).  target/draft logits [B,P,V] (uint16
    bf16 bits), beams/unpacker [B,W,L], packer [B,P], u_accept float32 [B,P],
    u_sample float32 [B,V].  Returns accept_len, best_beam, n_accepted,
    out_tokens and margin (the smallest relative gap of a decision taken)."""
    target = _c(target, np.uint16); draft = _c(draft, np.uint16)
    beams = _c(beams, np.int32); packer = _c(packer, np.int32)
    unpacker = _c(unpacker, np.int32); packed_len = _c(packed_len, np.int32)
    u_accept = _c(u_accept, np.float32); u_sample = _c(u_sample, np.float32)
    B, P, V = target.shape
    W, L = beams.shape[1], beams.shape[2]
    out = dict(accept_len=np.zeros((B, W), np.int32), best_beam=np.zeros(B, np.int32),
               n_accepted=np.zeros(B, np.int32), out_tokens=np.zeros((B, L), np.int32),
               margin=np.zeros(B, np.float64))
    rc = _load().oracle_sample_accept(_ptr(target), _ptr(draft), B, P, V, float(temperature),
                                      _ptr(beams), _ptr(packer), _ptr(unpacker),
                                      _ptr(packed_len), W, L, _ptr(u_accept), _ptr(u_sample),
                                      _ptr(out["accept_len"]), _ptr(out["best_beam"]),
                                      _ptr(out["n_accepted"]), _ptr(out["out_tokens"]),
                                      _ptr(out["margin"]))
    if rc != 0:
        raise ValueError(f"oracle_sample_accept rejected the input (rc={rc})")
    return out


def oracle_greedy_accept(logits, beams, unpacker, packed_len) -> dict:
    """Greedy verification: logits [B,P,V] (uint16 bf16 bits), beams/unpacker [B,W,L]."""
    logits = _c(logits, np.uint16); beams = _c(beams, np.int32)
    unpacker = _c(unpacker, np.int32); packed_len = _c(packed_len, np.int32)
    B, P, V = logits.shape
    W, L = beams.shape[1], beams.shape[2]
    out = dict(argmax=np.zeros((B, P), np.int32), accept_len=np.zeros((B, W), np.int32),
               best_beam=np.zeros(B, np.int32), n_accepted=np.zeros(B, np.int32),
               out_tokens=np.zeros((B, L), np.int32))
    rc = _load().oracle_greedy_accept(_ptr(logits), B, P, V, _ptr(beams), _ptr(unpacker),
                                      _ptr(packed_len), W, L, _ptr(out["argmax"]),
                                      _ptr(out["accept_len"]), _ptr(out["best_beam"]),
                                      _ptr(out["n_accepted"]), _ptr(out["out_tokens"]))
    if rc != 0:
        raise ValueError(f"oracle_greedy_accept rejected the input (rc={rc})")
    return out


def oracle_beam_search_step(logits, scores_in, beams_in) -> dict:
    """One beam-search step in fp64: logits [B, W, V] (uint16 bf16 bits),
    scores_in [B, W] (cumulative log-probabilities; -inf = beam not live),
    beams_in int32 [B, W, t].  Returns beams [B, W, t+1], scores [B, W], parent [B, W]."""
    logits = _c(logits, np.uint16)
    scores_in = _c(scores_in, np.float64)
    beams_in = _c(beams_in, np.int32)
    B, W, V = logits.shape
    t = beams_in.shape[2]
    out = dict(beams=np.zeros((B, W, t + 1), np.int32), scores=np.zeros((B, W), np.float64),
               parent=np.zeros((B, W), np.int32))
    rc = _load().oracle_beam_search_step(_ptr(logits), _ptr(scores_in), _ptr(beams_in), B, W, V,
                                         t, _ptr(out["beams"]), _ptr(out["scores"]),
                                         _ptr(out["parent"]))
    if rc != 0:
        raise ValueError(f"oracle_beam_search_step rejected the input (rc={rc})")
    return out


def oracle_unpack(packed: np.ndarray, unpacker: np.ndarray) -> np.ndarray:
    """out[b, w, i, :] = packed[b, unpacker[b, w, i], :] (any dtype, exact copy)."""
    B, W, L = unpacker.shape
    assert packed.ndim == 3 and packed.shape[0] == B
    bidx = np.arange(B)[:, None, None]
    return packed[bidx, unpacker]
