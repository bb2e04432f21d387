"""Full-size workloads on the GPU vs the CPU oracle.

* ragged64: 64 sequences of 4 096..65 536 tokens with 0..7 tokens of left
  padding - every stage checked element by element.
* long262k: one DSA layer of 4 x 262 144 tokens in the bench's launch shape -
  sampled pool keys (first, last and random pools of every sequence), full score
  rows, selection and attention for all four queries.
* prefill: 4 096 queries appended to a 131 072-token context at kpool 8 with the
  causal rule - sampled queries around the causal edges, full rows each.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_kpool_gb300 import pipeline, synth
from tests import _parity as par
from tests._util import npf, npi, oracle_inputs, ulp_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_ragged64_all_stages():
    bt = synth.ragged64(device=DEV)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    par.check_compress(o, buf)
    par.check_scores(o, buf)
    par.check_topk(buf, bt.geo.select_k)
    par.check_expand(o, buf)
    par.check_mla(o, buf)
    assert int(buf.status.item()) == 0


def _sampled_pool_keys(bt, buf, pools_per_seq=48, seed=0):
    """Oracle pool keys for sampled pools, computed from just their tokens."""
    rng = np.random.default_rng(seed)
    kp, D = bt.geo.kpool, bt.geo.D
    cu = bt.cu_seqlens.cpu().numpy()
    cap = bt.cu_pool_cap.cpu().numpy()
    n = buf.n_pools.cpu().numpy()
    gam, bet = npf(bt.ln_gamma), npf(bt.ln_beta)
    ape = npf(bt.ape)
    for b in range(bt.B):
        t0 = bt.pads[b]
        P = (bt.lengths[b] - t0) // kp
        assert n[b] == P
        pools = np.unique(np.r_[0, P - 1, rng.integers(0, P, pools_per_seq)])
        toks = cu[b] + t0 + pools[:, None] * kp + np.arange(kp)[None, :]
        idx = torch.as_tensor(toks.reshape(-1), device=DEV)
        k = npf(bt.k[idx]).reshape(len(pools), kp, D)
        g = npf(bt.gate[idx]).reshape(len(pools), kp, D)
        # each sampled pool as its own one-pool sequence of kp valid tokens
        kk = k.reshape(-1, D)
        gg = g.reshape(-1, D)
        m = len(pools)
        ref, ps, pv, _, st = oracle.kpool_compress(
            kk, gg, np.ones(m * kp, np.uint8), ape, gam, bet, bt.geo.ln_eps,
            np.arange(m + 1) * kp, np.arange(m + 1), kp, bt.geo.dtype)
        got = npf(buf.pool_keys[torch.as_tensor(cap[b] + pools, device=DEV)])
        kn = oracle.round_store(oracle.layernorm(kk, gam, bet, bt.geo.ln_eps), bt.geo.dtype)
        knmax = np.abs(kn).reshape(m, kp, D).max(axis=1)
        tol = par.pool_key_tol(ref, knmax, bt.geo.dtype)
        assert np.all(np.abs(got - ref) <= tol), f"seq {b}: pool keys out of tolerance"
        starts = buf.pool_start[torch.as_tensor(cap[b] + pools, device=DEV)].cpu().numpy()
        assert np.array_equal(starts, t0 + pools * kp)


def _mla_rows(bt, buf, rows):
    """Oracle attention for query rows, gathering only the selected latent rows."""
    o = dict(q_lat=npf(bt.q_lat), sm_scale=bt.sm_scale, dtype=bt.geo.dtype)
    cu = bt.cu_seqlens.cpu().numpy()
    for i in rows:
        b = i if bt.q_seq is not None else 0
        tok = buf.token_ids[i].cpu().numpy()
        sel = tok[tok >= 0]
        C = npf(bt.kv[torch.as_tensor(cu[b] + sel, device=DEV)])
        out, lse, st = oracle.mla_selected_decode(o["q_lat"][i:i + 1], C, [0, len(sel)], None,
                                                  np.arange(len(sel))[None, :], bt.sm_scale,
                                                  bt.geo.dtype)
        got = buf.out[i].cpu().double().numpy()
        assert np.all(np.abs(got - out[0]) <= par.mla_tol(out[0], bt.geo.dtype))
        if bt.geo.dtype == "bf16":  # against the value before its storage rounding
            o32, _, _ = oracle.mla_selected_decode(o["q_lat"][i:i + 1], C, [0, len(sel)], None,
                                                   np.arange(len(sel))[None, :], bt.sm_scale,
                                                   "f32")
            tol = 1e-2 + 0.5 * np.maximum(ulp_bf16(o32[0]), ulp_bf16(got))
            assert np.all(np.abs(got - o32[0]) <= tol)
        gl = buf.lse[i].cpu().double().numpy()
        assert np.allclose(gl, lse[0], rtol=1e-3, atol=1e-3)


def _oracle_row_scores(bt, buf, i, base, P, q_pos=None):
    keys = npf(buf.pool_keys[base:base + P])
    starts = buf.pool_start[base:base + P].cpu().numpy()
    valid = buf.pool_valid[base:base + P].cpu().numpy()
    ref, _ = oracle.index_scores(npf(bt.q[i:i + 1]), npf(bt.weights[i:i + 1]), bt.scale, keys,
                                 starts, valid, [P], [0, P], None,
                                 None if q_pos is None else [q_pos], bt.geo.kpool, bt.P_ld)
    return ref[0]


def _check_row(got, ref):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    r = ref[fin]
    rms = np.sqrt(np.mean(r ** 2))
    assert np.all(np.abs(got[fin] - r) <= 2e-3 * np.abs(r) + 2e-3 * rms)


@pytest.mark.slow
def test_long262k_one_layer_sampled():
    bt = synth.long262k(device=DEV, layer=0)
    bt.q_pos = None                         # the bench's decode form: every complete pool
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    _sampled_pool_keys(bt, buf)
    cap = bt.cu_pool_cap.cpu().numpy()
    for i in range(4):
        ref = _oracle_row_scores(bt, buf, i, cap[i], cap[i + 1] - cap[i])
        _check_row(buf.scores[i].cpu().double().numpy(), ref)
    par.check_topk(buf, bt.geo.select_k)
    o = dict(q_seq=npi(bt.q_seq), cu_pool_cap=cap, kpool=bt.geo.kpool,
             out_width=bt.geo.out_width)
    par.check_expand(o, buf)
    _mla_rows(bt, buf, range(4))


@pytest.mark.slow
def test_prefill_chunk_sampled():
    bt = synth.prefill(device=DEV)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    _sampled_pool_keys(bt, buf, pools_per_seq=64)
    P = int(buf.n_pools[0].item())
    assert P == 135168 // 8
    q_pos = bt.q_pos.cpu().numpy()
    # first query, the queries where a new pool becomes visible, the last ones
    rows = [0, 1, 6, 7, 8, 15, 2047, 2048, 4094, 4095]
    for i in rows:
        ref = _oracle_row_scores(bt, buf, i, 0, P, q_pos=int(q_pos[i]))
        got = buf.scores[i].cpu().double().numpy()
        _check_row(got, ref)
        assert np.isfinite(got).sum() == 16384 + (i + 1) // 8    # causal count
    par.check_topk(buf, bt.geo.select_k, rows=rows)
    o = dict(q_seq=None, cu_pool_cap=bt.cu_pool_cap.cpu().numpy(), kpool=bt.geo.kpool,
             out_width=bt.geo.out_width)
    par.check_expand(o, buf, rows=rows)
    _mla_rows(bt, buf, rows)


@pytest.mark.slow
def test_long262k_decode_steps_repeated():
    """The bench's decode step, called again and again on one 262k layer (top-k
    clusters of 16, the compress inside the scoring kernel): no status bit is
    ever set, and every call gives what compress -> select -> attend gives."""
    bt = synth.long262k(device=DEV, layer=1)
    bt.q_pos = None
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, a)
    pipeline.compress(bt, b)
    torch.cuda.synchronize()
    begin = (a.n_pools - 1).clamp(min=0).to(torch.int32)
    for step in range(24):
        bt.q, bt.weights, bt.q_lat = synth.query_set(bt.geo, bt.Q, device=DEV, seed=700 + step)
        pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=1)
        torch.cuda.synchronize()
        assert int(a.status.item()) == 0, step
        if step % 8 == 0:
            pipeline.run_layer(bt, b, pool_begin=begin, max_pools=1)
            torch.cuda.synchronize()
            assert int(b.status.item()) == 0, step
            for n in ("scores", "pool_ids", "token_ids", "out", "lse"):
                assert torch.equal(getattr(a, n), getattr(b, n)), (step, n)
