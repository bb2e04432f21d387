"""Failure detection on the GPU without a fault: the give-up path of the
tensor-core kernels.

Their waits on their own copies and MMAs are bounded.  The failure drill makes
each of those kernels skip arming the barrier its first wait needs, so that
wait runs out (after 1 ms) with no copy or MMA in flight.  Each test checks
that the call returns, that the device status carries DSA_DEV_TIMEOUT, that
the CUDA context is still usable, and that the same call made normally
afterwards gives the same outputs as before the drill.
"""
import pytest
import torch

from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
from sparse_attention_indexer_kpool_gb300.synth import Geometry

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 64  # DSA_DEV_TIMEOUT


def decode_batch(n_seq=4, seed=21, select_k=64):
    geo = Geometry(D=128, H=32, kpool=4, select_k=select_k, out_width=4 * select_k, Hm=64, L=512,
                   dtype="bf16")
    return synth.make_batch(geo, [3000 + 517 * i for i in range(n_seq)], [i for i in range(n_seq)],
                            device=DEV, seed=seed)


class drill:
    def __init__(self, mode=ops.DSA_DRILL_SKIP_ARM):
        self.mode = mode

    def __enter__(self):
        ops.dsa_set_failure_drill(self.mode)

    def __exit__(self, *exc):
        ops.dsa_set_failure_drill(0)
        return False


def snapshot(buf):
    return {n: getattr(buf, n).clone() for n in ("scores", "pool_ids", "token_ids", "out", "lse")}


def assert_same(buf, ref, names):
    for n in names:
        assert torch.equal(getattr(buf, n), ref[n]), n


def test_scoring_kernel_gives_up_and_recovers():
    bt = decode_batch()
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, buf)
    pipeline.select(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    ref = snapshot(buf)
    with drill():
        buf.scores.fill_(0.0)
        pipeline.select(bt, buf)
        torch.cuda.synchronize()
    assert int(buf.status.item()) & TIMEOUT
    buf.status.zero_()
    pipeline.select(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert_same(buf, ref, ("scores", "pool_ids", "token_ids"))


@pytest.mark.parametrize("n_seq,select_k", [(4, 64), (64, 512)])
def test_attention_kernels_give_up_and_recover(n_seq, select_k):
    # 4 queries x 256 rows: the one-tile attention kernel + merge; 64 queries x
    # 2048 rows: the streaming kernel + merge
    bt = decode_batch(n_seq=n_seq, seed=22 + n_seq, select_k=select_k)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    ref = snapshot(buf)
    with drill():
        pipeline.attend(bt, buf)
        torch.cuda.synchronize()
    assert int(buf.status.item()) & TIMEOUT
    # the give-up path reports "nothing selected" for the CTAs that gave up
    assert torch.isinf(buf.lse).all() and (buf.out == 0).all()
    buf.status.zero_()
    pipeline.attend(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert_same(buf, ref, ("out", "lse"))


@pytest.mark.parametrize("case", ["eight_tiles_per_cta", "one_tile_per_cta"])
def test_streaming_attention_gives_up_with_mmas_in_flight(case):
    """The drill that lets the streaming attention kernel issue its MMAs but arm
    none of its PV chunk barriers: those waits run out with MMAs in flight (64
    queries x 2048 rows: eight 128-row tiles per CTA, two splits; 320 queries
    x 128 rows: one tile per CTA).  The kernel issues nothing more, drains
    through one more commit, frees its tensor memory and returns: the call is
    flagged, its outputs read "nothing selected", and the same call afterwards
    gives the outputs it gave before."""
    if case == "eight_tiles_per_cta":
        bt = decode_batch(n_seq=64, seed=24, select_k=512)
    else:
        geo = Geometry(D=128, H=32, kpool=4, select_k=32, out_width=128, Hm=64, L=512,
                       dtype="bf16")
        bt = synth.make_batch(geo, [600 + 3 * i for i in range(320)], [0] * 320, device=DEV,
                              seed=25)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    ref = snapshot(buf)
    with drill(ops.DSA_DRILL_SKIP_PV_COMMIT):
        pipeline.attend(bt, buf)
        torch.cuda.synchronize()
    assert int(buf.status.item()) & TIMEOUT
    assert torch.isinf(buf.lse).all() and (buf.out == 0).all()
    buf.status.zero_()
    pipeline.attend(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert_same(buf, ref, ("out", "lse"))


def test_fused_decode_layer_gives_up_and_recovers():
    bt = decode_batch(seed=31)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, buf)
    torch.cuda.synchronize()
    begin = (buf.n_pools - 1).clamp(min=0).to(torch.int32)
    pipeline.decode_layer(bt, buf, pool_begin=begin, max_pools=1)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    ref = snapshot(buf)
    with drill():
        pipeline.decode_layer(bt, buf, pool_begin=begin, max_pools=1)
        torch.cuda.synchronize()
    assert int(buf.status.item()) & TIMEOUT
    buf.status.zero_()
    pipeline.decode_layer(bt, buf, pool_begin=begin, max_pools=1)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert_same(buf, ref, ("scores", "pool_ids", "token_ids", "out", "lse"))
