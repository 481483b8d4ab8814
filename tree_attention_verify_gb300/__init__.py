"""Python binding of librd, the GB300 verification step of ReDrafter-style
speculative decoding (prefix-trie packing, tree attention, greedy acceptance,
unpack).

The binding only marshals arguments: it checks tensor shapes, dtypes, devices
and contiguity, allocates outputs with torch when the caller passes none, and
calls the C ABI declared in include/rd.h with the tensors' device current, on
that device's current CUDA stream (or the stream passed).  Every step
of the computation runs in the CUDA kernels of librd.so.  There is no CPU path:
if the library cannot be loaded, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "rd_pack_beams", "rd_tree_attention", "rd_tree_attention_workspace_size",
    "rd_causal_attention", "rd_unpack", "rd_greedy_accept",
    "rd_greedy_accept_workspace_size", "rd_greedy_accept_noalloc",
    "rd_tree_attention_paged", "rd_commit_accepted", "rd_beam_search_step",
    "rd_tree_attention_fp8", "rd_sample_accept", "rd_debug_stall_attention", "RdError",
    "DEV_BAD_INDEX", "DEV_BAD_TOKEN", "DEV_OVERFLOW", "DEV_BAD_LENGTH", "DEV_TIMEOUT",
    "lib_path",
]

DEV_BAD_INDEX, DEV_BAD_TOKEN, DEV_OVERFLOW, DEV_BAD_LENGTH, DEV_TIMEOUT = 1, 2, 4, 8, 16
RD_OK, RD_ERR_INVALID_ARG, RD_ERR_UNSUPPORTED, RD_ERR_CUDA = 0, 1, 2, 3
_DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2, torch.int32: 3}


class RdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_lib.rd_status_string(status).decode()} ({status})")


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if _build.needs_build():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"librd.so missing at {path}; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, I64, F, S = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                       ctypes.c_size_t)
    sig = {
        "rd_pack_beams": [P, I, I, I, I, P, P, P, P, P, P, P, P],
        "rd_tree_attention_workspace_size": [I, I, I, I, I, I],
        "rd_tree_attention": [I, I, I, I, I, F, P, P, P, P, P, P, I64, I, P, P, I, P, P, S,
                              P, P],
        "rd_causal_attention": [I, I, I, I, F, P, P, P, P, I64, I, P, P, P],
        "rd_unpack": [P, I, I, I, I, P, I, I, P, P, P],
        "rd_greedy_accept_workspace_size": [I, I, I],
        "rd_greedy_accept": [P, I, I, I, P, P, P, I, I, P, P, P, P, P, P, S, P, P],
        "rd_greedy_accept_noalloc": [P, I, I, I, P, P, P, I, I, P, P, P, P, P, P, P],
        "rd_tree_attention_paged": [I, I, I, I, I, F, P, P, P, P, P, I, I, P, I, P, I, P, P, I,
                                    P, P, S, P, P],
        "rd_commit_accepted": [I, I, I, I, I, I, P, P, P, P, P, P, P, I, I, P, I, P, P, P, P],
        "rd_beam_search_step": [P, P, P, I, I, I, I, P, P, P, P, P],
        "rd_tree_attention_fp8": [I, I, I, I, I, F, P, P, P, P, P, F, F, P, I64, I, P, P, I, P, P,
                                  S, P, P],
        "rd_sample_accept": [P, P, I, I, I, F, P, P, P, P, I, I, P, P, P, P, P, P, P, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = S if name.endswith("workspace_size") else I
    lib.rd_status_string.argtypes = [I]
    lib.rd_status_string.restype = ctypes.c_char_p
    lib.rd_debug_stall_attention.argtypes = [ctypes.c_longlong]
    lib.rd_debug_stall_attention.restype = None
    return lib


_lib = _load()


def lib_path() -> str:
    return _build.LIB


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _check(fn: str, status: int):
    if status != RD_OK:
        raise RdError(fn, status)


def _run(name: str, like: torch.Tensor, *args, stream=None):
    """Call librd's `name` with `like`'s device current and that device's
    stream (or `stream`) as the last argument; raise RdError on a bad status."""
    with torch.cuda.device(like.device):
        _check(name, getattr(_lib, name)(*args, _stream(stream, like.device)))


def _empty(shape, dtype, like: torch.Tensor):
    return torch.empty(shape, dtype=dtype, device=like.device)


def _out(t, name: str, shape, dtype, like: torch.Tensor) -> torch.Tensor:
    """A caller-supplied output: allocated if None, else checked (shape, dtype,
    device, contiguity) before anything is launched, so that a kernel never
    writes outside it."""
    if t is None:
        return _empty(shape, dtype, like)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {tuple(shape)}, got {tuple(t.shape)}")
    _need(t, name, dtype, like.device)
    return t


def _out_dict(out, shapes: dict, dtypes: dict, like: torch.Tensor) -> dict:
    if out is None:
        return {k: _empty(shapes[k], dtypes[k], like) for k in shapes}
    if not isinstance(out, dict):
        raise TypeError("out must be a dict of tensors")
    return {k: _out(out.get(k), f"out[{k!r}]", shapes[k], dtypes[k], like) if k in out
            else _empty(shapes[k], dtypes[k], like) for k in shapes}


_ACCEPT_OUTS = ("argmax", "accept_len", "best_beam", "n_accepted", "out_tokens")


def _accept_shapes(logits, beams, unpacker, packed_len, out=None) -> dict:
    """Shapes of the greedy-verification arguments, checked against each other
    before anything is launched: a batch or beam count that disagrees between
    logits, beams, unpacker, packed_len and the outputs would make the kernel
    index outside those tensors.  Returns the expected output shapes."""
    if logits.dim() != 3:
        raise ValueError(f"logits must be [B, P_max, V], got {tuple(logits.shape)}")
    B, P, _ = logits.shape
    if beams.dim() != 3 or beams.shape[0] != B:
        raise ValueError(f"beams must be [B={B}, W, L], got {tuple(beams.shape)}")
    W, L = beams.shape[1], beams.shape[2]
    if tuple(unpacker.shape) != tuple(beams.shape):
        raise ValueError(f"unpacker must have the shape of beams {tuple(beams.shape)}, "
                         f"got {tuple(unpacker.shape)}")
    if packed_len.dim() != 1 or packed_len.numel() != B:
        raise ValueError(f"packed_len must be [B={B}], got {tuple(packed_len.shape)}")
    shapes = dict(argmax=(B, P), accept_len=(B, W), best_beam=(B,), n_accepted=(B,),
                  out_tokens=(B, L))
    if out is not None:
        for k in _ACCEPT_OUTS:
            t = out.get(k)
            if not isinstance(t, torch.Tensor):
                raise TypeError(f"out[{k!r}] must be a tensor")
            if tuple(t.shape) != shapes[k]:
                raise ValueError(f"out[{k!r}] must be {shapes[k]}, got {tuple(t.shape)}")
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(f"out[{k!r}] must be a contiguous int32 tensor")
            if t.device != logits.device:
                raise ValueError(f"out[{k!r}] is on {t.device}, expected {logits.device}")
    return shapes


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------
def rd_pack_beams(beams: torch.Tensor, P_cap: Optional[int] = None, *, out: Optional[dict] = None,
                  dev_status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Prefix dedup of int32 beams [B, W, L].  Returns dict(tokens, packer, unpacker,
    mask, depth, packed_len) of device tensors (see rd_pack_beams in rd.h)."""
    _need(beams, "beams", torch.int32, ndim=3)
    B, W, L = beams.shape
    P_cap = W * L if P_cap is None else int(P_cap)
    NW = (P_cap + 31) // 32
    # mask: uint32 bit rows held as int32
    out = _out_dict(out, dict(tokens=(B, P_cap), packer=(B, P_cap), unpacker=(B, W, L),
                              mask=(B, P_cap, NW), depth=(B, P_cap), packed_len=(B,)),
                    dict.fromkeys(("tokens", "packer", "unpacker", "mask", "depth", "packed_len"),
                                  torch.int32), beams)
    _run("rd_pack_beams", beams,
        _ptr(beams), B, W, L, P_cap, _ptr(out["tokens"]), _ptr(out["packer"]),
        _ptr(out["unpacker"]), _ptr(out["mask"]), _ptr(out.get("depth")),
        _ptr(out["packed_len"]), _ptr(dev_status), stream=stream)
    return out


def rd_tree_attention_workspace_size(B: int, P_max: int, Hq: int, Hkv: int, D: int,
                                     max_ctx: int, device=None) -> int:
    """Bytes of attention workspace (partials of units cut by the CTAs' chunk
    ranges, and the request table); it depends on the SM count of the device the
    call will run on (`device`, else the current device)."""
    if device is not None and torch.device(device).type == "cuda":
        with torch.cuda.device(device):
            return int(_lib.rd_tree_attention_workspace_size(B, P_max, Hq, Hkv, D, max_ctx))
    return int(_lib.rd_tree_attention_workspace_size(B, P_max, Hq, Hkv, D, max_ctx))


def rd_tree_attention(q, k_new, v_new, k_cache, v_cache, ctx_offsets, packed_len, mask, *,
                      max_ctx: int, scale: float = 0.0, out=None, workspace=None,
                      dev_status=None, stream=None) -> torch.Tensor:
    """Tree-masked attention of packed drafts (see rd_tree_attention in rd.h).
    q [B,P,Hq,D], k_new/v_new [B,P,Hkv,D], k_cache/v_cache [sum C,Hkv,D] bf16;
    ctx_offsets int64 [B+1]; packed_len int32 [B]; mask uint32/int32 [B,P,NW].
    The workspace (if the plan needs one) needs no initial contents; pass the
    same workspace again to reuse it."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
        _need(t, n, torch.bfloat16, q.device, ndim=4)
    _need(k_cache, "k_cache", torch.bfloat16, q.device, ndim=3)
    _need(v_cache, "v_cache", torch.bfloat16, q.device, ndim=3)
    _need(ctx_offsets, "ctx_offsets", torch.int64, q.device, ndim=1)
    _need(packed_len, "packed_len", torch.int32, q.device, ndim=1)
    if (mask.dim() != 3 or not mask.is_contiguous() or mask.element_size() != 4
            or mask.device != q.device):
        raise ValueError("mask must be a contiguous 32-bit [B, P_max, NW] tensor on q's device")
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    if k_new.shape != (B, P, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, P_max, Hkv, D]")
    if k_cache.shape[1:] != (Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [total_ctx, Hkv, D]")
    if ctx_offsets.numel() != B + 1 or packed_len.numel() != B or mask.shape[:2] != (B, P):
        raise ValueError("ctx_offsets/packed_len/mask shapes do not match q")
    out = _out(out, "out", q.shape, torch.bfloat16, q)
    ws_need = rd_tree_attention_workspace_size(B, P, Hq, Hkv, D, max_ctx, q.device)
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    _run("rd_tree_attention", q,
        B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
        _ptr(v_cache), _ptr(ctx_offsets), int(k_cache.shape[0]), int(max_ctx), _ptr(packed_len),
        _ptr(mask), int(mask.shape[2]), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(dev_status), stream=stream)
    return out


def rd_tree_attention_fp8(q, k_new, v_new, k_cache, v_cache, k_scale: float, v_scale: float,
                          ctx_offsets, packed_len, mask, *, max_ctx: int, scale: float = 0.0,
                          out=None, workspace=None, dev_status=None, stream=None) -> torch.Tensor:
    """rd_tree_attention with an e4m3 context cache: k_cache/v_cache uint8 (or
    float8_e4m3fn) [total_ctx, Hkv, D] holding e4m3 bit patterns, per-tensor
    scales k_scale/v_scale (see rd_tree_attention_fp8 in rd.h)."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
        _need(t, n, torch.bfloat16, q.device, ndim=4)
    if k_cache.dtype != torch.uint8:
        k_cache = k_cache.view(torch.uint8)
    if v_cache.dtype != torch.uint8:
        v_cache = v_cache.view(torch.uint8)
    _need(k_cache, "k_cache", torch.uint8, q.device, ndim=3)
    _need(v_cache, "v_cache", torch.uint8, q.device, ndim=3)
    _need(ctx_offsets, "ctx_offsets", torch.int64, q.device, ndim=1)
    _need(packed_len, "packed_len", torch.int32, q.device, ndim=1)
    if (mask.dim() != 3 or not mask.is_contiguous() or mask.element_size() != 4
            or mask.device != q.device):
        raise ValueError("mask must be a contiguous 32-bit [B, P_max, NW] tensor on q's device")
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    if k_new.shape != (B, P, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, P_max, Hkv, D]")
    if k_cache.shape[1:] != (Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [total_ctx, Hkv, D]")
    if ctx_offsets.numel() != B + 1 or packed_len.numel() != B or mask.shape[:2] != (B, P):
        raise ValueError("ctx_offsets/packed_len/mask shapes do not match q")
    out = _out(out, "out", q.shape, torch.bfloat16, q)
    ws_need = rd_tree_attention_workspace_size(B, P, Hq, Hkv, D, max_ctx, q.device)
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    _run("rd_tree_attention_fp8", q,
        B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
        _ptr(v_cache), float(k_scale), float(v_scale), _ptr(ctx_offsets),
        int(k_cache.shape[0]), int(max_ctx), _ptr(packed_len), _ptr(mask), int(mask.shape[2]),
        _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(dev_status), stream=stream)
    return out


def rd_tree_attention_paged(q, k_new, v_new, k_pool, v_pool, block_table, ctx_lens, packed_len,
                            mask, *, max_ctx: int, scale: float = 0.0, out=None, workspace=None,
                            dev_status=None, stream=None) -> torch.Tensor:
    """rd_tree_attention with the context in a paged cache: k_pool/v_pool
    [num_pages, page_size, Hkv, D] bf16, block_table int32 [B, max_pages],
    ctx_lens int32 [B] (see rd_tree_attention_paged in rd.h)."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
        _need(t, n, torch.bfloat16, q.device, ndim=4)
    _need(k_pool, "k_pool", torch.bfloat16, q.device, ndim=4)
    _need(v_pool, "v_pool", torch.bfloat16, q.device, ndim=4)
    _need(block_table, "block_table", torch.int32, q.device, ndim=2)
    _need(ctx_lens, "ctx_lens", torch.int32, q.device, ndim=1)
    _need(packed_len, "packed_len", torch.int32, q.device, ndim=1)
    if (mask.dim() != 3 or not mask.is_contiguous() or mask.element_size() != 4
            or mask.device != q.device):
        raise ValueError("mask must be a contiguous 32-bit [B, P_max, NW] tensor on q's device")
    B, P, Hq, D = q.shape
    Hkv = k_new.shape[2]
    n_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    if k_pool.shape[2:] != (Hkv, D) or v_pool.shape != k_pool.shape:
        raise ValueError("k_pool/v_pool must be [num_pages, page_size, Hkv, D]")
    if block_table.shape[0] != B or ctx_lens.numel() != B or packed_len.numel() != B:
        raise ValueError("block_table/ctx_lens/packed_len do not match the batch")
    out = _out(out, "out", q.shape, torch.bfloat16, q)
    ws_need = rd_tree_attention_workspace_size(B, P, Hq, Hkv, D, max_ctx, q.device)
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    _run("rd_tree_attention_paged", q,
        B, P, Hq, Hkv, D, float(scale), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
        _ptr(v_pool), n_pages, page_size, _ptr(block_table), block_table.shape[1],
        _ptr(ctx_lens), int(max_ctx), _ptr(packed_len), _ptr(mask), int(mask.shape[2]),
        _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(dev_status), stream=stream)
    return out


def rd_commit_accepted(k_new, v_new, unpacker, best_beam, n_accepted, k_pool, v_pool,
                       block_table, ctx_lens, *, new_ctx_lens=None, dev_status=None,
                       stream=None) -> torch.Tensor:
    """Append the accepted path's K/V to the paged cache (k_pool/v_pool modified in
    place).  Returns new_ctx_lens = ctx_lens + n_accepted + 1 (see rd.h)."""
    _need(k_new, "k_new", torch.bfloat16, ndim=4)
    _need(v_new, "v_new", torch.bfloat16, k_new.device, ndim=4)
    _need(k_pool, "k_pool", torch.bfloat16, k_new.device, ndim=4)
    _need(v_pool, "v_pool", torch.bfloat16, k_new.device, ndim=4)
    for n, t in (("unpacker", unpacker), ("best_beam", best_beam), ("n_accepted", n_accepted),
                 ("block_table", block_table), ("ctx_lens", ctx_lens)):
        _need(t, n, torch.int32, k_new.device)
    B, P, Hkv, D = k_new.shape
    _, W, L = unpacker.shape
    if new_ctx_lens is None:
        new_ctx_lens = torch.empty_like(ctx_lens)
    _run("rd_commit_accepted", k_new,
        B, W, L, P, Hkv, D, _ptr(k_new), _ptr(v_new), _ptr(unpacker), _ptr(best_beam),
        _ptr(n_accepted), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], k_pool.shape[1],
        _ptr(block_table), block_table.shape[1], _ptr(ctx_lens), _ptr(new_ctx_lens),
        _ptr(dev_status), stream=stream)
    return new_ctx_lens


def rd_causal_attention(q, k, v, cu_seqlens, *, max_seqlen: int, scale: float = 0.0,
                        out=None, dev_status=None, stream=None) -> torch.Tensor:
    """Causal prefill attention: q [T,Hq,D], k/v [T,Hkv,D] bf16, cu_seqlens int32 [B+1]."""
    _need(q, "q", torch.bfloat16, ndim=3)
    _need(k, "k", torch.bfloat16, q.device, ndim=3)
    _need(v, "v", torch.bfloat16, q.device, ndim=3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, q.device, ndim=1)
    T, Hq, D = q.shape
    if k.shape[0] != T or v.shape != k.shape or k.shape[2] != D:
        raise ValueError("k/v must be [T, Hkv, D] with the rows of q")
    out = _out(out, "out", q.shape, torch.bfloat16, q)
    _run("rd_causal_attention", q,
        cu_seqlens.numel() - 1, Hq, k.shape[1], D, float(scale), _ptr(q), _ptr(k), _ptr(v),
        _ptr(cu_seqlens), T, int(max_seqlen), _ptr(out), _ptr(dev_status), stream=stream)
    return out


def rd_unpack(packed: torch.Tensor, unpacker: torch.Tensor, *, out=None, dev_status=None,
              stream=None) -> torch.Tensor:
    """out[b,w,i,:] = packed[b, unpacker[b,w,i], :] (exact copy)."""
    if packed.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {packed.dtype}")
    _need(packed, "packed", packed.dtype, ndim=3)
    _need(unpacker, "unpacker", torch.int32, packed.device, ndim=3)
    B, P, Dh = packed.shape
    _, W, L = unpacker.shape
    if unpacker.shape[0] != B:
        raise ValueError("unpacker batch does not match packed")
    out = _out(out, "out", (B, W, L, Dh), packed.dtype, packed)
    _run("rd_unpack", packed, _ptr(packed), _DTYPES[packed.dtype], B, P, Dh, _ptr(unpacker), W,
         L, _ptr(out), _ptr(dev_status), stream=stream)
    return out


def rd_greedy_accept_workspace_size(B: int, P_max: int, V: int) -> int:
    return int(_lib.rd_greedy_accept_workspace_size(B, P_max, V))


def rd_greedy_accept(logits, beams, unpacker, packed_len, *, out=None, workspace=None,
                     dev_status=None, stream=None) -> dict:
    """Greedy verification (see rd_greedy_accept in rd.h).  Returns dict(argmax,
    accept_len, best_beam, n_accepted, out_tokens).  The workspace must start
    zero-filled; every call leaves it zeroed."""
    shapes = _accept_shapes(logits, beams, unpacker, packed_len, out)
    dev = logits.device
    _need(logits, "logits", torch.bfloat16, ndim=3)
    _need(beams, "beams", torch.int32, dev, ndim=3)
    _need(unpacker, "unpacker", torch.int32, dev, ndim=3)
    _need(packed_len, "packed_len", torch.int32, dev, ndim=1)
    B, P, V = logits.shape
    _, W, L = beams.shape
    if out is None:
        out = {k: _empty(shapes[k], torch.int32, logits) for k in _ACCEPT_OUTS}
    if workspace is None:
        workspace = torch.zeros(max(8, rd_greedy_accept_workspace_size(B, P, V)),
                                dtype=torch.uint8, device=dev)
    elif workspace.device != dev or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {dev}")
    _run("rd_greedy_accept", logits,
         _ptr(logits), B, P, V, _ptr(beams), _ptr(unpacker), _ptr(packed_len), W, L,
         _ptr(out["argmax"]), _ptr(out["accept_len"]), _ptr(out["best_beam"]),
         _ptr(out["n_accepted"]), _ptr(out["out_tokens"]), _ptr(workspace),
         workspace.numel() * workspace.element_size(), _ptr(dev_status), stream=stream)
    return out


def rd_sample_accept(target_logits, draft_logits, temperature: float, beams, packer, unpacker,
                     packed_len, u_accept, u_sample, *, out=None, dev_status=None,
                     stream=None) -> dict:
    """Stochastic verification by multi-step speculative sampling (see
    rd_sample_accept in rd.h).  Returns dict(accept_len, best_beam, n_accepted,
    out_tokens)."""
    _need(target_logits, "target_logits", torch.bfloat16, ndim=3)
    _need(draft_logits, "draft_logits", torch.bfloat16, target_logits.device, ndim=3)
    _need(beams, "beams", torch.int32, target_logits.device, ndim=3)
    _need(packer, "packer", torch.int32, target_logits.device, ndim=2)
    _need(unpacker, "unpacker", torch.int32, target_logits.device, ndim=3)
    _need(packed_len, "packed_len", torch.int32, target_logits.device, ndim=1)
    _need(u_accept, "u_accept", torch.float32, target_logits.device, ndim=2)
    _need(u_sample, "u_sample", torch.float32, target_logits.device, ndim=2)
    B, P, V = target_logits.shape
    _, W, L = beams.shape
    if draft_logits.shape != target_logits.shape or packer.shape != (B, P):
        raise ValueError("draft_logits / packer shapes do not match target_logits")
    if u_accept.shape != (B, P) or u_sample.shape != (B, V):
        raise ValueError("u_accept must be [B, P_max] and u_sample [B, V]")
    out = _out_dict(out, dict(accept_len=(B, W), best_beam=(B,), n_accepted=(B,), out_tokens=(B, L)),
                    dict.fromkeys(("accept_len", "best_beam", "n_accepted", "out_tokens"), torch.int32),
                    target_logits)
    _run("rd_sample_accept", target_logits,
        _ptr(target_logits), _ptr(draft_logits), B, P, V, float(temperature), _ptr(beams),
        _ptr(packer), _ptr(unpacker), _ptr(packed_len), W, L, _ptr(u_accept), _ptr(u_sample),
        _ptr(out["accept_len"]), _ptr(out["best_beam"]), _ptr(out["n_accepted"]),
        _ptr(out["out_tokens"]), _ptr(dev_status), stream=stream)
    return out


def rd_greedy_accept_noalloc(logits, beams, unpacker, packed_len, *, out=None, dev_status=None,
                             stream=None) -> dict:
    """rd_greedy_accept without a caller workspace, for callers that cannot allocate
    device memory: the scratch is a fixed array inside librd shared by every call
    on the device, so calls must not overlap on the GPU.  Limits: B * P_max <= 65536
    and B <= 65535.  (The outputs are allocated here only when `out` is not given:
    a caller that cannot allocate passes them.)"""
    shapes = _accept_shapes(logits, beams, unpacker, packed_len, out)
    dev = logits.device
    _need(logits, "logits", torch.bfloat16, ndim=3)
    _need(beams, "beams", torch.int32, dev, ndim=3)
    _need(unpacker, "unpacker", torch.int32, dev, ndim=3)
    _need(packed_len, "packed_len", torch.int32, dev, ndim=1)
    B, P, V = logits.shape
    _, W, L = beams.shape
    if out is None:
        out = {k: _empty(shapes[k], torch.int32, logits) for k in _ACCEPT_OUTS}
    _run("rd_greedy_accept_noalloc", logits,
         _ptr(logits), B, P, V, _ptr(beams), _ptr(unpacker), _ptr(packed_len), W, L,
         _ptr(out["argmax"]), _ptr(out["accept_len"]), _ptr(out["best_beam"]),
         _ptr(out["n_accepted"]), _ptr(out["out_tokens"]), _ptr(dev_status), stream=stream)
    return out


def rd_beam_search_step(logits, scores_in, beams_in, *, out=None, dev_status=None,
                        stream=None) -> dict:
    """One beam-search step of the drafter (see rd_beam_search_step in rd.h):
    logits bf16 [B, W, V], scores_in fp32 [B, W], beams_in int32 [B, W, t].
    Returns dict(beams [B, W, t+1], scores [B, W], parent [B, W])."""
    _need(logits, "logits", torch.bfloat16, ndim=3)
    _need(scores_in, "scores_in", torch.float32, logits.device, ndim=2)
    _need(beams_in, "beams_in", torch.int32, logits.device, ndim=3)
    B, W, V = logits.shape
    t = beams_in.shape[2]
    out = _out_dict(out, dict(beams=(B, W, t + 1), scores=(B, W), parent=(B, W)),
                    dict(beams=torch.int32, scores=torch.float32, parent=torch.int32), logits)
    _run("rd_beam_search_step", logits,
        _ptr(logits), _ptr(scores_in), _ptr(beams_in) if t > 0 else None, B, W, V, t,
        _ptr(out["beams"]), _ptr(out["scores"]), _ptr(out["parent"]), _ptr(dev_status),
        stream=stream)
    return out


def rd_debug_stall_attention(budget_cycles: int) -> None:
    """Failure-detection test hook (see rd_debug_stall_attention in rd.h): with
    budget_cycles > 0, every later attention launch first waits, for at most that
    many SM clock cycles, on a barrier that nothing completes, so its bounded
    wait runs out and the kernel reports DEV_TIMEOUT and returns.  0 disarms it."""
    _lib.rd_debug_stall_attention(int(budget_cycles))
