"""Host-side argument checks of the Python binding, without a GPU: arguments
whose shapes disagree are rejected before anything is launched (a batch or beam
count that differs between tensors would make a kernel index outside them)."""
import pytest
import torch


def _accept_args(B=4, P=8, V=100, W=2, L=4):
    return (torch.zeros(B, P, V, dtype=torch.bfloat16), torch.zeros(B, W, L, dtype=torch.int32),
            torch.zeros(B, W, L, dtype=torch.int32), torch.zeros(B, dtype=torch.int32))


def _outs(B=4, P=8, W=2, L=4):
    i32 = dict(dtype=torch.int32)
    return dict(argmax=torch.zeros(B, P, **i32), accept_len=torch.zeros(B, W, **i32),
                best_beam=torch.zeros(B, **i32), n_accepted=torch.zeros(B, **i32),
                out_tokens=torch.zeros(B, L, **i32))


def test_accept_shapes_accepts_consistent_arguments():
    import tree_attention_verify_gb300 as rd
    shapes = rd._accept_shapes(*_accept_args(), out=_outs())
    assert shapes == dict(argmax=(4, 8), accept_len=(4, 2), best_beam=(4,), n_accepted=(4,),
                          out_tokens=(4, 4))


@pytest.mark.parametrize("case", ["beams_batch", "unpacker_shape", "packed_len", "logits_rank"])
def test_accept_shapes_reject_mismatched_inputs(case):
    import tree_attention_verify_gb300 as rd
    lg, beams, unp, plen = _accept_args()
    if case == "beams_batch":
        beams, unp = beams[:3], unp[:3]
    elif case == "unpacker_shape":
        unp = torch.zeros(4, 2, 5, dtype=torch.int32)
    elif case == "packed_len":
        plen = torch.zeros(5, dtype=torch.int32)
    else:
        lg = lg[0]
    with pytest.raises(ValueError):
        rd._accept_shapes(lg, beams, unp, plen)
    # the public entry points run the same check first, before any device check
    for fn in (rd.rd_greedy_accept, rd.rd_greedy_accept_noalloc):
        with pytest.raises(ValueError):
            fn(lg, beams, unp, plen)


@pytest.mark.parametrize("key,bad", [("argmax", (4, 7)), ("accept_len", (4, 3)),
                                     ("best_beam", (5,)), ("out_tokens", (4, 5))])
def test_accept_shapes_reject_mismatched_outputs(key, bad):
    import tree_attention_verify_gb300 as rd
    out = _outs()
    out[key] = torch.zeros(bad, dtype=torch.int32)
    with pytest.raises(ValueError):
        rd._accept_shapes(*_accept_args(), out=out)
    out = _outs()
    out[key] = out[key].to(torch.int64)
    with pytest.raises(ValueError):
        rd._accept_shapes(*_accept_args(), out=out)
    out = _outs()
    del out[key]
    with pytest.raises(TypeError):
        rd._accept_shapes(*_accept_args(), out=out)


def test_out_helper_rejects_wrong_shape_and_dtype():
    """Caller-supplied outputs of every other entry point go through _out: the
    shape and dtype are checked before anything is launched."""
    import tree_attention_verify_gb300 as rd
    like = torch.zeros(3, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rd._out(torch.zeros(3, 4, 7, dtype=torch.bfloat16), "out", like.shape, torch.bfloat16, like)
    with pytest.raises(TypeError):
        rd._out(torch.zeros(3, 4, 8, dtype=torch.float32), "out", like.shape, torch.bfloat16, like)
    with pytest.raises(TypeError):
        rd._out([1, 2], "out", like.shape, torch.bfloat16, like)
    # a dict of outputs: a wrong entry is rejected, a missing one is allocated
    shapes = dict(a=(2, 3), b=(2,))
    dtypes = dict(a=torch.int32, b=torch.int32)
    with pytest.raises(ValueError):
        rd._out_dict(dict(a=torch.zeros(2, 4, dtype=torch.int32)), shapes, dtypes, like)
    got = rd._out_dict(None, shapes, dtypes, like)
    assert tuple(got["a"].shape) == (2, 3) and tuple(got["b"].shape) == (2,)
