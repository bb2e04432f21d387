"""The indexer projections (hidden state / query latent -> k, gate, weights,
q, q_nope, q_lat) on the tensor cores against the oracle's exact sums.

Tolerance, from the arithmetic: both operands are bf16, so every product is
exact in fp32 and the kernel's only error before storage is the fp32
accumulation, at most K * 2^-24 * sum_k |x_k w_k| in any order (plus 2^-24 of
the value for the fp32 scale multiply).  The stored bf16 value is one
rounding of that sum and the oracle's is one rounding of the exact sum, so the
two differ by at most that bound plus one bf16 spacing (fp32 weights: one fp32
spacing).  q_lat is checked on the kernel's own q_nope (the tensor the latent
projection reads), so a one-spacing difference in q_nope does not carry over.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
from tests._util import npf, ulp_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS32 = 2.0 ** -24


def host(t):
    return t.double().cpu().numpy()


def check(name, gpu, ref, abs_sum, K, alpha=1.0, f32=False):
    spacing = (np.abs(ref) * 2.0 ** -23 * 2) if f32 else \
        np.maximum(ulp_bf16(ref), ulp_bf16(gpu))
    tol = spacing + abs(alpha) * (K * EPS32 * abs_sum + EPS32 * abs_sum) + 1e-30
    bad = np.abs(gpu - ref) > tol
    assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} out of tolerance, worst excess " \
                          f"{np.max(np.abs(gpu - ref) - tol):.3g}"


def run(pi, weights_scale, kv_rows=None, rows=None):
    buf = pipeline.ProjectionBuffers.alloc(pi, rows=rows)
    pipeline.project(pi, buf, weights_scale, kv_rows=kv_rows)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    return buf


def check_all(pi, buf, weights_scale, tokens=None, kv_rows=None):
    """Compare every output of the listed tokens with the oracle."""
    T = pi.x.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    x, cq = host(pi.x)[tok], host(pi.cq)[tok]
    w_kgw, w_q, w_uk_t = host(pi.w_kgw), host(pi.w_q), host(pi.w_uk_t)
    H, D, Hm, nope = pi.H, pi.D, pi.Hm, pi.nope
    ref = oracle.indexer_project(x, w_kgw, cq, w_q, w_uk_t, H, D, Hm, nope, weights_scale)
    s_hid = oracle.linear(np.abs(x), np.abs(w_kgw))
    s_q = oracle.linear(np.abs(cq), np.abs(w_q))
    rows = tok if kv_rows is None else kv_rows.cpu().numpy()[tok]
    check("k", host(buf.k)[rows], ref["k"], s_hid[:, :D], x.shape[1])
    check("gate", host(buf.gate)[rows], ref["gate"], s_hid[:, D:2 * D], x.shape[1])
    check("weights", host(buf.weights)[tok], ref["weights"], s_hid[:, 2 * D:], x.shape[1],
          alpha=weights_scale, f32=True)
    check("q", host(buf.q)[tok].reshape(len(tok), -1), ref["q"].reshape(len(tok), -1),
          s_q[:, :H * D], cq.shape[1])
    check("q_nope", host(buf.q_nope)[tok].reshape(len(tok), -1),
          ref["q_nope"].reshape(len(tok), -1), s_q[:, H * D:], cq.shape[1])
    qn = host(buf.q_nope)[tok]
    lat = oracle.round_bf16(oracle.absorb_query(qn, w_uk_t))
    s_lat = oracle.absorb_query(np.abs(qn), np.abs(w_uk_t))
    check("q_lat", host(buf.q_lat)[tok], lat, s_lat, nope)


# small shapes that span several tiles and leave ragged edges everywhere:
# hidden 328 and q_rank 200 end inside a 64-wide stage, 2D + H = 68 and L = 72
# fill part of a 128-feature tile, and the token counts cover the 16-, 64- and
# 128-token tile widths with partial last tiles
SMALL = dict(hidden=328, q_rank=200, H=4, D=32, Hm=3, nope=64, L=72)


@pytest.mark.parametrize("T", [1, 5, 37, 130, 300])
def test_projections_small_ragged(T):
    pi = synth.projection_inputs(T, **SMALL, device=DEV, seed=100 + T)
    buf = run(pi, 0.125)
    check_all(pi, buf, 0.125)


def test_projection_rows_go_to_the_cache_rows_named():
    """k and gate land in the rows kv_rows names (a negative entry drops the
    token); every other row of the cache keeps its contents."""
    T, rows = 9, 40
    pi = synth.projection_inputs(T, **SMALL, device=DEV, seed=7)
    kv_rows = torch.tensor([3, 39, -1, 0, 17, 18, -1, 25, 11], dtype=torch.int32, device=DEV)
    buf = pipeline.ProjectionBuffers.alloc(pi, rows=rows)
    buf.k.fill_(5.0)
    buf.gate.fill_(-5.0)
    pipeline.project(pi, buf, 1.0, kv_rows=kv_rows)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    keep = [t for t in range(T) if kv_rows[t] >= 0]
    check_all(pi, buf, 1.0, tokens=keep, kv_rows=kv_rows)
    untouched = sorted(set(range(rows)) - set(kv_rows[kv_rows >= 0].tolist()))
    assert torch.all(buf.k[untouched] == 5.0) and torch.all(buf.gate[untouched] == -5.0)


def test_projections_are_deterministic():
    """Split contractions are added in split order: two calls on one workspace
    agree bit for bit (the second also shows that the first left the split
    counters re-armed: a counter left off zero would pick the wrong split to
    add the partials)."""
    pi = synth.projection_inputs(4, **synth.PROJ_MAIN, device=DEV, seed=8)
    a = run(pi, 0.5)
    b = pipeline.ProjectionBuffers.alloc(pi)
    b.ws = a.ws                     # the same (re-armed) workspace
    pipeline.project(pi, b, 0.5)
    torch.cuda.synchronize()
    assert a.ws is not None          # 4 tokens: the contractions are split
    for n in ("k", "gate", "weights", "q", "q_nope", "q_lat"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("T", [4, 64])
def test_projections_full_size_decode(T):
    """The full-size shapes in decode (a handful of tokens: the weights stream)."""
    pi = synth.projection_inputs(T, **synth.PROJ_MAIN, device=DEV, seed=9 + T)
    buf = run(pi, synth.PROJ_MAIN["H"] ** -0.5)
    check_all(pi, buf, synth.PROJ_MAIN["H"] ** -0.5)


def test_projections_full_size_prefill_sampled():
    """A prefill chunk (4000 tokens, a ragged last 128-token tile) on sampled
    tokens from every tile position."""
    T = 4000
    pi = synth.projection_inputs(T, **synth.PROJ_MAIN, device=DEV, seed=10)
    buf = run(pi, synth.PROJ_MAIN["H"] ** -0.5)
    tokens = [0, 1, 127, 128, 1000, 2047, 2048, 3071, 3839, 3840, 3900, 3998, 3999]
    check_all(pi, buf, synth.PROJ_MAIN["H"] ** -0.5, tokens=tokens)
