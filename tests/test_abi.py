"""The C ABI boundary, without a GPU: librd.so loads, exports every function that
include/rd.h declares, and rejects bad host-side arguments (or accepts empty
batches) before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rd.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rd_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("rd_pack_beams", "rd_tree_attention", "rd_tree_attention_workspace_size",
              "rd_causal_attention", "rd_unpack", "rd_greedy_accept",
              "rd_greedy_accept_workspace_size", "rd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import tree_attention_verify_gb300 as rd
    lib = ctypes.CDLL(rd.lib_path())
    for n in _declared():
        assert hasattr(lib, n), f"librd.so does not export {n}"


def test_status_strings():
    import tree_attention_verify_gb300 as rd
    assert rd._lib.rd_status_string(0) == b"ok"
    assert rd._lib.rd_status_string(2) == b"unsupported configuration"


def test_host_validation_without_device():
    import tree_attention_verify_gb300 as rd
    lib = rd._lib
    N = None
    # pack: W < 1, P_cap too large, W too large
    assert lib.rd_pack_beams(N, 1, 0, 4, 4, N, N, N, N, N, N, N, N) == rd.RD_ERR_INVALID_ARG
    assert lib.rd_pack_beams(N, 1, 4, 4, 257, N, N, N, N, N, N, N, N) == rd.RD_ERR_UNSUPPORTED
    assert lib.rd_pack_beams(N, 1, 33, 2, 64, N, N, N, N, N, N, N, N) == rd.RD_ERR_UNSUPPORTED
    # empty batch: OK, nothing launched (works without a device)
    assert lib.rd_pack_beams(N, 0, 4, 4, 16, N, N, N, N, N, N, N, N) == rd.RD_OK
    assert lib.rd_tree_attention(0, 16, 32, 8, 128, 0.0, N, N, N, N, N, N, 0, 0, N, N, 1, N, N,
                                 0, N, N) == rd.RD_OK
    assert lib.rd_causal_attention(0, 32, 8, 128, 0.0, N, N, N, N, 0, 0, N, N, N) == rd.RD_OK
    assert lib.rd_unpack(N, 0, 0, 16, 4096, N, 4, 4, N, N, N) == rd.RD_OK
    assert lib.rd_greedy_accept(N, 0, 16, 1000, N, N, N, 4, 4, N, N, N, N, N, N, 0, N,
                                N) == rd.RD_OK
    # attention: bad head split, unsupported head dim, wrong mask words, null pointers
    assert lib.rd_tree_attention(1, 16, 32, 5, 128, 0.0, N, N, N, N, N, N, 0, 0, N, N, 1, N,
                                 N, 0, N, N) == rd.RD_ERR_INVALID_ARG
    assert lib.rd_tree_attention(1, 16, 32, 8, 96, 0.0, N, N, N, N, N, N, 0, 0, N, N, 1, N, N,
                                 0, N, N) == rd.RD_ERR_UNSUPPORTED
    assert lib.rd_tree_attention(1, 40, 32, 8, 128, 0.0, N, N, N, N, N, N, 0, 0, N, N, 1, N,
                                 N, 0, N, N) == rd.RD_ERR_INVALID_ARG
    assert lib.rd_tree_attention(1, 16, 32, 8, 128, 0.0, N, N, N, N, N, N, 0, 0, N, N, 1, N,
                                 N, 0, N, N) == rd.RD_ERR_INVALID_ARG
    # greedy accept: workspace missing / too small
    assert lib.rd_greedy_accept(ctypes.c_void_p(16), 1, 16, 1000, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 4,
                                ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                8, N, N) == rd.RD_ERR_INVALID_ARG
    # unpack: bad dtype
    assert lib.rd_unpack(N, 9, 1, 16, 64, N, 4, 4, N, N, N) == rd.RD_ERR_INVALID_ARG


def test_workspace_queries():
    import tree_attention_verify_gb300 as rd
    assert rd.rd_greedy_accept_workspace_size(64, 48, 32000) >= 64 * 48 * 8
    assert rd.rd_greedy_accept_workspace_size(0, 48, 32000) == 0
    # chunk-range division: per CTA two 128-row fp32 slots (O, m, l) for the pieces
    # of cut units and a 16-byte merge descriptor
    for B, P, Hq, Hkv, D, C in ((1, 20, 32, 32, 128, 2048), (16, 40, 32, 8, 128, 4096)):
        n = rd.rd_tree_attention_workspace_size(B, P, Hq, Hkv, D, C)
        per_cta = 2 * 128 * (D * 4 + 8) + 16
        assert n > 0 and n % per_cta == 0
    # a batch with at least two units (request, kv head, tile) per CTA runs whole
    # units round-robin: no workspace
    assert rd.rd_tree_attention_workspace_size(64, 48, 40, 40, 128, 8192) == 0
    # too many requests for the per-request table in shared memory: whole units
    # round-robin, no workspace
    assert rd.rd_tree_attention_workspace_size(481, 20, 32, 32, 128, 2048) == 0


def test_product_path_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "tree_attention_verify_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower().replace("oracles", ""), f


def test_sample_accept_host_validation():
    import tree_attention_verify_gb300 as rd
    lib = rd._lib
    N = None
    # empty batch: OK without a device; bad temperature; too many beams / packed nodes
    assert lib.rd_sample_accept(N, N, 0, 48, 32000, 1.0, N, N, N, N, 8, 6, N, N, N, N, N, N, N,
                                N) == rd.RD_OK
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.rd_sample_accept(N, N, 1, 48, 32000, T, N, N, N, N, 8, 6, N, N, N, N, N, N,
                                    N, N) == rd.RD_ERR_INVALID_ARG
    assert lib.rd_sample_accept(N, N, 1, 48, 32000, 1.0, N, N, N, N, 33, 6, N, N, N, N, N, N, N,
                                N) == rd.RD_ERR_UNSUPPORTED
    assert lib.rd_sample_accept(N, N, 1, 300, 32000, 1.0, N, N, N, N, 8, 6, N, N, N, N, N, N, N,
                                N) == rd.RD_ERR_UNSUPPORTED
    # null pointers with a non-empty batch
    assert lib.rd_sample_accept(N, N, 1, 48, 32000, 1.0, N, N, N, N, 8, 6, N, N, N, N, N, N, N,
                                N) == rd.RD_ERR_INVALID_ARG
