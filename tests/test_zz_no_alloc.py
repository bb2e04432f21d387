"""dsa_select_noalloc: the select call for callers that cannot allocate.

Callers inside a CUDA stream capture, plugins whose host framework owns all
device memory, and serving loops that forbid allocation cannot hand dsa_select
a workspace; dsa_select_noalloc keeps that scratch in a static device array.
Its outputs must match dsa_select's on the same inputs, call after call (the
array is shared and reused, so a second call must not see the first call's
leftovers).  This file is collected last on purpose.
"""
import pytest
import torch

from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
from sparse_attention_indexer_kpool_gb300.synth import Geometry

pytestmark = pytest.mark.gpu


def _batch(seed):
    geo = Geometry(D=128, H=32, kpool=4, select_k=64, out_width=320, Hm=64, L=512, dtype="bf16")
    return synth.make_batch(geo, [3001, 40, 1203, 9000], [2, 0, 5, 1], device="cuda", seed=seed)


def _noalloc(bt, buf):
    scores = torch.full_like(buf.scores, 7.0)
    ids = torch.full_like(buf.pool_ids, 0x7F7F7F7F)
    tok = torch.full_like(buf.token_ids, 0x7F7F7F7F)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.dsa_select_noalloc(bt.q, bt.weights, bt.scale, buf.pool_keys, buf.pool_start,
                           buf.pool_valid, buf.n_pools, bt.cu_pool_cap, bt.q_seq, bt.q_pos,
                           bt.geo.kpool, scores, ids, tok, st)
    return scores, ids, tok, st


def test_noalloc_matches_select_on_two_calls_in_a_row():
    for call, seed in enumerate((101, 202)):       # two different inputs, back to back
        bt = _batch(seed)
        buf = pipeline.LayerBuffers.alloc(bt)
        pipeline.compress(bt, buf)
        pipeline.select(bt, buf)                    # the existing entry point
        scores, ids, tok, st = _noalloc(bt, buf)
        torch.cuda.synchronize()
        fin = torch.isfinite(buf.scores)
        assert torch.equal(torch.isfinite(scores), fin), call
        assert torch.allclose(scores[fin], buf.scores[fin], rtol=0, atol=0), call
        assert torch.equal(ids, buf.pool_ids), call
        assert torch.equal(tok, buf.token_ids), call
        assert int(st.item()) == int(buf.status.item()) == 0, call


def test_noalloc_matches_select_where_no_scratch_is_used():
    """fp32 at a small geometry: the scoring kernel keeps no histogram, the
    selection builds its own on chip, and the static array is not touched."""
    for call, seed in enumerate((7, 8)):
        bt = synth.tiny(device="cuda", seed=seed)
        buf = pipeline.LayerBuffers.alloc(bt)
        pipeline.compress(bt, buf)
        pipeline.select(bt, buf)
        scores, ids, tok, st = _noalloc(bt, buf)
        torch.cuda.synchronize()
        assert torch.equal(scores, buf.scores), call
        assert torch.equal(ids, buf.pool_ids), call
        assert torch.equal(tok, buf.token_ids), call
        assert int(st.item()) == int(buf.status.item()) == 0, call


def test_noalloc_refuses_more_queries_than_its_scratch():
    geo = Geometry(D=128, H=32, kpool=4, select_k=8, out_width=32, Hm=64, L=512, dtype="bf16")
    bt = synth.make_batch(geo, [64] * 65, [0] * 65, device="cuda", seed=3)
    buf = pipeline.LayerBuffers.alloc(bt)
    with pytest.raises(ops.DsaError) as e:
        _noalloc(bt, buf)
    assert e.value.code == 3        # DSA_ERR_UNSUPPORTED
