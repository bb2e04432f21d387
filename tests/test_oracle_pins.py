"""Pins for the CPU oracle: values fixed by the pages and by mathematics.

Each test ties one oracle function to something other than itself: a hand-worked
value (tests/golden/hand_cases.json, each with its citation), a closed form, an
invariant, a textbook library routine, or brute force on a tiny input.  Each is
chosen so that a plausible slip (RMSNorm for LayerNorm, softmax over the wrong
axis, relu after the weight, reversed tie order, a dropped -1 tail, an
off-by-one in the causal rule, a wrong row base) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_kpool_gb300 import synth
from tests._util import oracle_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "hand_cases.json")))


# ---------------------------------------------------------------- roundings
def test_round_bf16_hand_ties():
    r = oracle.round_bf16
    assert r(1 + 2 ** -8) == 1.0                      # tie -> even (mantissa 0)
    assert r(1 + 3 * 2 ** -8) == 1 + 2 ** -6          # tie -> even (mantissa 2)
    assert r(1 + 2 ** -8 + 2 ** -20) == 1 + 2 ** -7   # just above the tie
    assert r(-(1 + 2 ** -8 + 2 ** -20)) == -(1 + 2 ** -7)
    assert r(255.5) == 256.0 and r(0.0) == 0.0
    assert np.signbit(r(-0.0))


def test_round_bf16_matches_torch_on_fp32_values():
    # torch's float32 -> bfloat16 conversion rounds to nearest even; on values
    # that are exactly fp32 there is no double rounding to worry about.
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)
    x = torch.cat([x, torch.tensor([1e-39, -3e-40, 3.3e38, 1.0 + 2 ** -8])])
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.to(torch.float64).numpy())
    assert np.array_equal(got, ref)


def test_round_f32_is_nearest():
    x = np.array([1 + 2 ** -24, 1 + 3 * 2 ** -24, 0.1])
    assert oracle.round_f32(x)[0] == 1.0
    assert oracle.round_f32(x)[1] == 1 + 2 ** -22
    assert oracle.round_f32(x)[2] == float(np.float32(0.1))


# ---------------------------------------------------------------- a1 LayerNorm
def test_layernorm_hand_case_and_not_rmsnorm():
    c = GOLD["layernorm_1234"]
    y = oracle.layernorm(np.array(c["x"], float), c["gamma"], c["beta"], c["eps"])
    assert np.allclose(y, c["expect"], rtol=0, atol=1e-15)
    assert not np.allclose(y, c["rmsnorm_would_give"], atol=1e-2)


def test_layernorm_eps_and_bias():
    c = GOLD["layernorm_eps_bias"]
    y = oracle.layernorm(np.array(c["x"], float), c["gamma"], c["beta"], c["eps"])
    assert np.allclose(y, c["expect"], rtol=0, atol=1e-15)


def test_layernorm_invariants_and_torch():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(7, 128))
    gam, bet = rng.normal(size=128), rng.normal(size=128)
    y = oracle.layernorm(x, gam, bet, 1e-5)
    assert np.allclose(oracle.layernorm(x + 3.7, gam, bet, 1e-5), y, atol=1e-12)   # shift invariant
    y0 = oracle.layernorm(x, gam, np.zeros(128), 1e-5)
    assert np.allclose(y - y0, bet[None, :], atol=1e-14)                            # bias adds
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(gam),
                                         torch.from_numpy(bet), 1e-5).numpy()
    assert np.allclose(y, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- a2 kpool_compress
def _one_seq(k, gate, valid, ape, kpool, gamma=None, beta=None, eps=1e-5, dtype="f32", cap=None,
             **kw):
    T, D = k.shape
    gamma = np.ones(D) if gamma is None else gamma
    beta = np.zeros(D) if beta is None else beta
    cap = T // kpool if cap is None else cap
    return oracle.kpool_compress(k, gate, valid, ape, gamma, beta, eps, [0, T], [0, cap], kpool,
                                 dtype, **kw)


def test_compress_kpool1_is_layernorm():
    rng = np.random.default_rng(2)
    k = rng.normal(size=(9, 16))
    gate = rng.normal(size=(9, 16))
    valid = np.ones(9, np.uint8)
    valid[:2] = 0
    pk, ps, pv, n, st = _one_seq(k, gate, valid, np.zeros((1, 16)), 1, dtype="bf16")
    assert n[0] == 7 and st == 0
    assert np.array_equal(pk[:7], oracle.round_bf16(oracle.layernorm(k[2:], 1, 0, 1e-5)))
    assert list(ps[:7]) == list(range(2, 9)) and pv[:7].all()


def test_compress_equal_logits_is_slot_mean():
    rng = np.random.default_rng(3)
    k = rng.normal(size=(8, 16))
    gate = np.tile(rng.normal(size=(1, 16)), (8, 1))     # same logit in every slot
    pk, ps, pv, n, _ = _one_seq(k, gate, np.ones(8, np.uint8), np.zeros((4, 16)), 4)
    kn = oracle.round_f32(oracle.layernorm(k, 1, 0, 1e-5))
    assert np.allclose(pk[:2], oracle.round_f32(kn.reshape(2, 4, 16).mean(axis=1)), atol=1e-7)


def test_compress_ape_enters_the_logits():
    c = GOLD["pool_softmax_ln3"]
    rng = np.random.default_rng(4)
    k = rng.normal(size=(2, 2))
    k[:, 0], k[:, 1] = [1.0, 3.0], [5.0, 2.0]           # LN over D=2 gives +-1 per token
    pk, *_ = _one_seq(k, np.array(c["gate"], float), np.ones(2, np.uint8), np.array(c["ape"]), 2,
                      eps=0.0, dtype="f32")
    kn = oracle.layernorm(k, 1, 0, 0.0)                 # [[-1, 1], [1, -1]]
    w = np.array(c["expect_weights"])
    assert np.allclose(pk[0], oracle.round_f32((w * kn).sum(axis=0)), atol=1e-7)
    assert np.allclose(pk[0], [0.5, 0.0], atol=1e-7)    # 1/4*(-1)+3/4*(1) ; 1/2*1+1/2*(-1)


def test_compress_softmax_is_per_channel_over_slots():
    rng = np.random.default_rng(5)
    k = rng.normal(size=(4, 8))
    gate = np.zeros((4, 8))
    gate[0, 0] = 40.0          # channel 0 takes slot 0
    gate[3, 1] = 40.0          # channel 1 takes slot 3
    pk, *_ = _one_seq(k, gate, np.ones(4, np.uint8), np.zeros((4, 8)), 4, dtype="f32")
    kn = oracle.round_f32(oracle.layernorm(k, 1, 0, 1e-5))
    assert abs(pk[0, 0] - kn[0, 0]) < 1e-12 * 0 + 1e-6
    assert abs(pk[0, 1] - kn[3, 1]) < 1e-6
    assert np.allclose(pk[0, 2:], oracle.round_f32(kn[:, 2:].mean(axis=0)), atol=1e-7)


def test_compress_pools_do_not_mix():
    rng = np.random.default_rng(6)
    k = rng.normal(size=(8, 8))
    gate = rng.normal(size=(8, 8))
    a = _one_seq(k, gate, np.ones(8, np.uint8), np.zeros((4, 8)), 4)[0]
    gate2 = gate.copy()
    gate2[4:] = rng.normal(size=(4, 8)) * 5            # change only pool 1's gates
    b = _one_seq(k, gate2, np.ones(8, np.uint8), np.zeros((4, 8)), 4)[0]
    assert np.array_equal(a[0], b[0]) and not np.array_equal(a[1], b[1])


def test_compress_padding_shift_and_partial_pool():
    rng = np.random.default_rng(7)
    T, D, kp = 23, 16, 4
    k = rng.normal(size=(T, D))
    gate = rng.normal(size=(T, D))
    ape = rng.normal(size=(kp, D)) * 0.1
    base = _one_seq(k, gate, np.ones(T, np.uint8), ape, kp, cap=8)
    m = 3                                              # prepend 3 invalid garbage tokens
    k2 = np.vstack([rng.normal(size=(m, D)) * 9, k])
    g2 = np.vstack([rng.normal(size=(m, D)) * 9, gate])
    v2 = np.r_[np.zeros(m, np.uint8), np.ones(T, np.uint8)]
    sh = _one_seq(k2, g2, v2, ape, kp, cap=8)
    assert base[3][0] == sh[3][0] == T // kp            # 5 full pools, the 3-token tail dropped
    assert np.array_equal(base[0][:5], sh[0][:5])
    assert np.array_equal(base[1][:5] + m, sh[1][:5])
    k3 = np.vstack([k, rng.normal(size=(2, D))])        # 23 + 2 = 25 tokens: still 6? no, 25//4 = 6
    g3 = np.vstack([gate, rng.normal(size=(2, D))])
    more = _one_seq(k3, g3, np.ones(T + 2, np.uint8), ape, kp, cap=8)
    assert more[3][0] == 6 and np.array_equal(more[0][:5], base[0][:5])
    assert list(base[1][5:]) == [-1, -1, -1] and not base[2][5:].any()


def test_compress_holes_invalidate_only_their_pool():
    rng = np.random.default_rng(8)
    T, D, kp = 20, 8, 4
    k, gate = rng.normal(size=(T, D)), rng.normal(size=(T, D))
    valid = np.ones(T, np.uint8)
    valid[0] = 0          # padding: t0 = 1, pools at 1,5,9,13 (4 pools, token 17..19 partial)
    valid[10] = 0         # hole inside pool 2 (tokens 9..12)
    _, ps, pv, n, _ = _one_seq(k, gate, valid, np.zeros((kp, D)), kp)
    assert n[0] == 4 and list(ps[:4]) == [1, 5, 9, 13] and list(pv[:4]) == [1, 1, 0, 1]


def test_compress_tiny_workload_geometry():
    bt = synth.tiny()
    o = oracle_inputs(bt)
    pk, ps, pv, n, st = oracle.kpool_compress(
        o["k"], o["gate"], o["valid"], o["ape"], o["ln_gamma"], o["ln_beta"], o["ln_eps"],
        o["cu_seqlens"], o["cu_pool_cap"], 4, "f32")
    assert n[0] == 63 and st == 0 and bt.P_ld == 64
    assert list(ps[:63]) == [3 + 4 * p for p in range(63)] and ps[63] == -1
    assert ps[62] + 3 == 254 and pv[:63].all() and pv[63] == 0


def test_compress_multi_sequence_and_ranges():
    rng = np.random.default_rng(9)
    D, kp = 8, 2
    L = [7, 0, 10]
    T = sum(L)
    k, gate = rng.normal(size=(T, D)), rng.normal(size=(T, D))
    valid = np.ones(T, np.uint8)
    valid[7] = 0 if T > 7 else 1        # sequence 2 starts at 7; pad one token
    ape = rng.normal(size=(kp, D))
    cu, cap = [0, 7, 7, 17], [0, 3, 3, 8]
    pk, ps, pv, n, st = oracle.kpool_compress(k, gate, valid, ape, np.ones(D), np.zeros(D), 1e-5,
                                              cu, cap, kp, "f32")
    assert list(n) == [3, 0, 4] and st == 0
    solo = _one_seq(k[7:], gate[7:], valid[7:], ape, kp, cap=5)
    assert np.array_equal(pk[3:7], solo[0][:4]) and list(ps[3:8]) == [1, 3, 5, 7, -1]
    # range semantics: pool_begin / max_pools, sentinel, statuses
    pk2, ps2, pv2, n2, st2 = oracle.kpool_compress(
        k, gate, valid, ape, np.ones(D), np.zeros(D), 1e-5, cu, cap, kp, "f32",
        pool_begin=[2, 0, 1], max_pools=2, pool_keys=np.full((8, D), 9.0),
        pool_start=np.full(8, 99), pool_valid=np.full(8, 7, np.uint8))
    assert st2 == oracle.ST_POOL_UNCOVERED                 # seq 2 has pool 3 beyond 1+2
    assert list(ps2) == [99, 99, 4, 99, 3, 5, 99, 99]
    assert np.array_equal(pk2[4:6], pk[4:6]) and (pk2[0] == 9).all()
    _, _, _, n3, st3 = oracle.kpool_compress(k, gate, valid, ape, np.ones(D), np.zeros(D), 1e-5,
                                             cu, [0, 2, 2, 7], kp, "f32")
    assert st3 == oracle.ST_POOL_OVERFLOW and list(n3) == [2, 0, 4]


def test_compress_kpool_bound():
    with pytest.raises(ValueError):
        _one_seq(np.zeros((18, 4)), np.zeros((18, 4)), np.ones(18, np.uint8), np.zeros((9, 4)), 9)


# ---------------------------------------------------------------- a3 index_scores
def _score_one(qh, key, w, scale):
    qh = np.array(qh, float)
    out, st = oracle.index_scores(qh[None], np.array([w], float), scale, np.array([key], float),
                                  np.array([0]), np.array([1], np.uint8), np.array([1]), [0, 1],
                                  None, None, 1, 1)
    return out[0, 0]


def test_scores_closed_forms():
    for name in ("score_closed_form", "score_scale_inside_relu"):
        c = GOLD[name]
        assert _score_one(c["q"], c["key"], c["weights"], c["scale"]) == c["expect"]


def test_scores_all_negative_is_plus_zero():
    s = _score_one([[1, 1], [2, 0]], [-1, -3], [0.7, -0.2], 0.5)
    assert s == 0.0 and not np.signbit(s)
    s = _score_one([[1, 1], [2, 0]], [-1, -3], [-0.7, -0.2], 0.5)   # 0 * negative weight = -0
    assert s == 0.0 and not np.signbit(s)


def test_scores_linear_in_weights_and_fp32():
    rng = np.random.default_rng(10)
    q, key, w = rng.normal(size=(4, 8)), rng.normal(size=8), rng.normal(size=4)
    a = _score_one(q, key, w, 0.3)
    assert a == float(np.float32(a))
    assert abs(_score_one(q, key, 2 * w, 0.3) - 2 * a) <= 4 * abs(a) * 2 ** -24


def test_scores_candidates_and_causal_count():
    kp, D, H = 4, 4, 2
    rng = np.random.default_rng(11)
    t0, P, cap = 3, 12, 14
    keys = np.abs(rng.normal(size=(cap, D))) + 0.1
    starts = np.r_[t0 + kp * np.arange(P), [-1, -1]]
    pv = np.r_[np.ones(P, np.uint8), [0, 0]]
    pv[5] = 0
    q = np.abs(rng.normal(size=(1, H, D)))
    w = np.ones((1, H))
    for pos in range(0, t0 + kp * P + 3):
        out, st = oracle.index_scores(q, w, 1.0, keys, starts, pv, [P], [0, cap], [0], [pos],
                                      kp, 16)
        n_vis = max(0, (pos - t0 + 1) // kp)           # pools whose last token <= pos
        expect = [p for p in range(min(P, n_vis)) if p != 5]
        assert list(np.flatnonzero(np.isfinite(out[0]))) == expect, pos
        assert np.all(out[0, P:] == -np.inf) and st == 0


def test_scores_bad_sequence_and_range_status():
    out, st = oracle.index_scores(np.ones((1, 1, 2)), np.ones((1, 1)), 1.0, np.ones((2, 2)),
                                  np.array([0, 1]), np.ones(2, np.uint8), [2], [0, 2], [1], None,
                                  1, 2)
    assert st == oracle.ST_BAD_QSEQ and np.all(out == -np.inf)
    out, st = oracle.index_scores(np.ones((1, 1, 2)), np.ones((1, 1)), 1.0, np.ones((2, 2)),
                                  np.array([0, 1]), np.ones(2, np.uint8), [3], [0, 2], [0], None,
                                  1, 2)
    assert st == oracle.ST_POOL_RANGE and np.all(out == 2.0)


# ---------------------------------------------------------------- a4 topk_pools
def test_topk_hand_tie_order():
    c = GOLD["topk_tie_order"]
    s = np.array([float(x) for x in c["scores"]])
    assert list(oracle.topk_pools(s[None], c["select_k"])[0]) == c["expect"]


def _is_valid_selection(s, sel, K):
    """Brute-force check of the order: a selected pool beats every later or
    unselected candidate (higher score, or equal score and smaller index)."""
    cand = [i for i in range(len(s)) if s[i] > -np.inf]
    n = min(K, len(cand))
    chosen = [int(x) for x in sel[:n]]
    if any(x != -1 for x in sel[n:]) or len(set(chosen)) != n:
        return False
    beats = lambda a, b: s[a] > s[b] or (s[a] == s[b] and a < b)
    if any(not beats(chosen[i], chosen[i + 1]) for i in range(n - 1)):
        return False
    rest = set(cand) - set(chosen)
    return all(beats(a, b) for a in chosen for b in rest)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(12)
    vals = [-1.0, 0.0, -0.0, 0.5, 2.0, -np.inf]
    for trial in range(400):
        P = int(rng.integers(1, 9))
        s = np.array([vals[i] for i in rng.integers(0, len(vals), P)])
        for K in (1, 3, 8, 10):
            sel = oracle.topk_pools(s[None], K)[0]
            assert _is_valid_selection(s, sel, K), (s, K, sel)
    # exhaustively: every ordering of a small multiset yields the rule's answer
    base = np.array([1.0, 1.0, 0.0, 2.0, 1.0])
    for perm in itertools.permutations(range(5)):
        s = base[list(perm)]
        assert _is_valid_selection(s, oracle.topk_pools(s[None], 3)[0], 3)


def test_topk_special_cases():
    s = np.zeros((1, 10))
    assert list(oracle.topk_pools(s, 4)[0]) == [0, 1, 2, 3]                 # all equal
    s = np.full((1, 6), -np.inf)
    s[0, [1, 4]] = [3.0, 5.0]
    assert list(oracle.topk_pools(s, 5)[0]) == [4, 1, -1, -1, -1]           # -1 tail
    s = np.array([[np.nan, 1.0, np.inf, -np.inf]])
    assert list(oracle.topk_pools(s, 4)[0]) == [2, 1, -1, -1]               # NaN excluded
    rng = np.random.default_rng(13)                                          # stable sort
    s = rng.integers(-3, 4, size=(1, 300)).astype(float)
    stable = sorted(range(300), key=lambda i: -s[0, i])
    assert list(oracle.topk_pools(s, 50)[0]) == stable[:50]


def test_topk_tiny_workload_has_tie_at_cutoff():
    """The tiny workload is built so that equal scores straddle the cutoff."""
    bt = synth.tiny()
    r = oracle.run_path(oracle_inputs(bt))
    s = r["scores"][0]
    order = r["pool_ids"][0]
    K = bt.geo.select_k
    kth = s[order[K - 1]]
    outside = [p for p in range(len(s)) if np.isfinite(s[p]) and p not in set(order)]
    assert any(s[p] == kth for p in outside), "no tie straddles the cutoff"


# ---------------------------------------------------------------- a5 expand_selection
def test_expand_closed_form():
    c = GOLD["expand_closed_form"]
    tok, st = oracle.expand_selection(np.array(c["pool_ids"]), np.array(c["pool_start"]), [0, 4],
                                      None, c["kpool"], c["out_width"])
    assert tok.tolist() == c["expect"] and st == 0


def test_expand_sequence_bases_and_bad_ids():
    pool_start = np.array([0, 4, 10, 12, 14])      # seq0 cap 2, seq1 cap 3
    tok, st = oracle.expand_selection(np.array([[1, -1], [2, 0], [3, 1]]), pool_start,
                                      [0, 2, 5], [0, 1, 1], 2, 5)
    assert tok.tolist() == [[4, 5, -1, -1, -1], [14, 15, 10, 11, -1], [-1, -1, 12, 13, -1]]
    assert st == oracle.ST_BAD_POOL_ID
    tok, st = oracle.expand_selection(np.array([[1, 0]]), np.array([5, -1]), [0, 2], None, 2, 4)
    assert tok.tolist() == [[-1, -1, 5, 6]] and st == 0            # sentinel entry -> -1
    with pytest.raises(ValueError):
        oracle.expand_selection(np.zeros((1, 2), int), pool_start, [0, 5], None, 2, 3)


# ---------------------------------------------------------------- a6 MLA
def _mla(q_lat, kv, tok, sm_scale, cu=None, q_seq=None, dtype="f32"):
    kv = np.asarray(kv, float)
    cu = [0, len(kv)] if cu is None else cu
    return oracle.mla_selected_decode(np.asarray(q_lat, float), kv, cu, q_seq,
                                      np.asarray(tok), sm_scale, dtype)


def test_mla_hand_two_rows():
    c = GOLD["mla_two_rows"]
    out, lse, st = _mla(c["q_lat"], c["rows"], [[0, 1]], c["sm_scale"])
    assert np.allclose(out[0, 0], c["expect_out"], atol=1e-6)
    assert abs(lse[0, 0] - c["expect_lse"]) < 1e-12 and st == 0


def test_mla_single_row_equal_logits_empty():
    rng = np.random.default_rng(14)
    kv = rng.normal(size=(10, 16))
    q = rng.normal(size=(1, 3, 16))
    out, lse, _ = _mla(q, kv, [[-1, 7, -1]], 0.25)
    assert np.allclose(out[0], oracle.round_f32(np.tile(kv[7], (3, 1))), atol=0)
    assert np.allclose(lse[0], 0.25 * q[0] @ kv[7], atol=1e-12)
    out, lse, _ = _mla(np.zeros((1, 2, 16)), kv, [[1, 2, 5, -1]], 1.0)
    assert np.allclose(out[0, 0], oracle.round_f32(kv[[1, 2, 5]].mean(axis=0)), atol=1e-7)
    assert np.allclose(lse[0], math.log(3), atol=1e-15)
    out, lse, _ = _mla(q, kv, [[-1, -1]], 1.0)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_mla_matches_torch_sdpa_and_masked_dense():
    rng = np.random.default_rng(15)
    n, L, Hm = 37, 24, 5
    kv = rng.normal(size=(n, L))
    q = rng.normal(size=(1, Hm, L))
    out, lse, _ = _mla(q, kv, [list(range(n))], 0.3, dtype="f32")
    t = torch.from_numpy
    ref = torch.nn.functional.scaled_dot_product_attention(
        t(q)[:, :, None, :].transpose(0, 1), t(kv)[None, None], t(kv)[None, None],
        scale=0.3)[:, 0, 0, :].numpy()
    assert np.allclose(out[0], oracle.round_f32(ref), atol=1e-6)
    sel = sorted(rng.choice(n, 11, replace=False).tolist())
    out_s, lse_s, _ = _mla(q, kv, [sel + [-1] * 3], 0.3)
    mask = np.full((Hm, n), -np.inf)
    mask[:, sel] = 0.0
    ref2 = torch.nn.functional.scaled_dot_product_attention(
        t(q)[:, :, None, :].transpose(0, 1), t(kv)[None, None], t(kv)[None, None],
        attn_mask=t(mask)[:, None, None, :], scale=0.3)[:, 0, 0, :].numpy()
    assert np.allclose(out_s[0], oracle.round_f32(ref2), atol=1e-6)
    z = 0.3 * q[0] @ kv[sel].T
    assert np.allclose(lse_s[0], np.log(np.exp(z).sum(axis=1)), atol=1e-12)


def test_mla_row_addressing_and_bad_token():
    rng = np.random.default_rng(16)
    kv = rng.normal(size=(9, 4))
    q = rng.normal(size=(2, 1, 4))
    out, lse, st = _mla(q, kv, [[1, -1], [0, 6]], 1.0, cu=[0, 4, 9], q_seq=[1, 1])
    assert np.allclose(out[0, 0], oracle.round_f32(kv[5]), atol=0)   # seq 1 row 1 -> global 5
    assert st == oracle.ST_BAD_TOKEN                                  # token 6 >= T_1 = 5
    assert np.allclose(out[1, 0], oracle.round_f32(kv[4]), atol=0)


def test_mla_bf16_output_rounding():
    kv = np.array([[1.0 + 2 ** -9, 3.0]])
    out, _, _ = _mla(np.ones((1, 1, 2)), kv, [[0]], 1.0, dtype="bf16")
    assert out[0, 0, 0] == 1.0 and out[0, 0, 1] == 3.0


# ---------------------------------------------------------------- a6 on a paged cache, fp8 rows
E4M3_HAND = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9}


def test_fp8_e4m3_hand_values():
    # 1.0 = exponent 7 (the bias), mantissa 0; 448 = the largest finite value;
    # 2^-6 = the smallest normal, 2^-9 = the smallest subnormal
    codes = np.array(sorted(E4M3_HAND), np.uint8)
    got = oracle.fp8_e4m3_decode(codes)
    assert np.array_equal(got, np.array([E4M3_HAND[c] for c in sorted(E4M3_HAND)]))
    neg0 = oracle.fp8_e4m3_decode(np.array([0x80], np.uint8))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) < 0
    nan = np.isnan(oracle.fp8_e4m3_decode(np.arange(256, dtype=np.uint8)))
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]           # no infinities, two NaNs


def test_fp8_e4m3_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.fp8_e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def _paged_layout(rng, lengths, page_size, n_extra=3, fill=None):
    """Scatter a contiguous cache (rows of sequence b at cu[b] + t) into shuffled
    pages of page_size rows; unused rows and pages hold other values."""
    B = len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    blocks = [-(-T // page_size) for T in lengths]
    n_pages = sum(blocks) + n_extra
    perm = rng.permutation(n_pages)
    table = np.full((B, max(blocks) + 1), -1, np.int64)
    rows = np.zeros(n_pages * page_size, np.int64) - 1      # physical row -> contiguous row
    k = 0
    for b, T in enumerate(lengths):
        for blk in range(blocks[b]):
            g = int(perm[k])
            k += 1
            table[b, blk] = g
            for s in range(page_size):
                if blk * page_size + s < T:
                    rows[g * page_size + s] = cu[b] + blk * page_size + s
    return cu, table, rows


def _paged_query(rng, lengths, Q=4, W=12):
    q_seq = rng.integers(0, len(lengths), Q)
    tok = np.full((Q, W), -1, np.int64)
    for i in range(Q):
        T = lengths[q_seq[i]]
        n = rng.integers(1, min(W, T) + 1)
        tok[i, :n] = rng.choice(T, n, replace=False)
    return q_seq, tok


def test_mla_paged_is_the_contiguous_attention_under_any_paging():
    rng = np.random.default_rng(40)
    lengths, L, Hm = [13, 5, 30], 8, 3
    kv = rng.normal(size=(sum(lengths), L))
    q = rng.normal(size=(4, Hm, L))
    q_seq, tok = _paged_query(rng, lengths)
    ref = _mla(q, kv, tok, 0.3, cu=np.concatenate([[0], np.cumsum(lengths)]), q_seq=q_seq)
    for page_size in (1, 4, 7, 64):
        cu, table, rows = _paged_layout(rng, lengths, page_size)
        pages = rng.normal(size=(len(rows), L))
        pages[rows >= 0] = kv[rows[rows >= 0]]
        got = oracle.mla_paged_decode(q, pages, None, "bf16", table, lengths, page_size, q_seq,
                                      tok, 0.3, "f32")
        assert got[2] == ref[2] == 0
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), page_size


def test_mla_paged_fp8_rows_are_code_times_row_scale():
    rng = np.random.default_rng(41)
    lengths, L, Hm, page_size = [20, 9], 16, 2, 4
    cu, table, rows = _paged_layout(rng, lengths, page_size)
    codes = rng.integers(0, 256, size=(len(rows), L)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                       # no NaN codes
    scale = rng.uniform(0.01, 3.0, size=len(rows))
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    kv = np.zeros((sum(lengths), L))
    kv[rows[rows >= 0]] = dec[rows >= 0] * scale[rows >= 0][:, None]
    q = rng.normal(size=(3, Hm, L))
    q_seq, tok = _paged_query(rng, lengths, Q=3)
    ref = _mla(q, kv, tok, 0.25, cu=cu, q_seq=q_seq)
    got = oracle.mla_paged_decode(q, codes, scale, "fp8_e4m3", table, lengths, page_size, q_seq,
                                  tok, 0.25, "f32")
    assert np.allclose(got[0], ref[0], rtol=1e-12, atol=1e-12)
    assert np.allclose(got[1], ref[1], rtol=1e-12, atol=1e-12)


def test_mla_paged_bad_page_and_bad_token_skip_the_row():
    rng = np.random.default_rng(42)
    lengths, L, page_size = [10, 6], 4, 4
    cu, table, rows = _paged_layout(rng, lengths, page_size)
    pages = rng.normal(size=(len(rows), L))
    q = rng.normal(size=(1, 2, L))
    tok = np.array([[0, 5, 9, -1]])
    want = oracle.mla_paged_decode(q, pages, None, "bf16", table, lengths, page_size, [0],
                                   np.array([[0, 5, -1, -1]]), 1.0, "f32")
    bad = table.copy()
    bad[0, 2] = -1                                          # block of token 9: no page
    got = oracle.mla_paged_decode(q, pages, None, "bf16", bad, lengths, page_size, [0], tok, 1.0,
                                  "f32")
    assert got[2] == oracle.ST_BAD_PAGE and np.array_equal(got[0], want[0])
    bad[0, 2] = len(rows) // page_size                      # page past the cache
    got = oracle.mla_paged_decode(q, pages, None, "bf16", bad, lengths, page_size, [0], tok, 1.0,
                                  "f32")
    assert got[2] == oracle.ST_BAD_PAGE and np.array_equal(got[0], want[0])
    narrow = table[:, :2]                                   # table too short for token 9
    got = oracle.mla_paged_decode(q, pages, None, "bf16", narrow, lengths, page_size, [0], tok,
                                  1.0, "f32")
    assert got[2] == oracle.ST_BAD_PAGE and np.array_equal(got[0], want[0])
    got = oracle.mla_paged_decode(q, pages, None, "bf16", table, lengths, page_size, [0],
                                  np.array([[0, 5, 10, -1]]), 1.0, "f32")   # 10 >= seq_lens[0]
    assert got[2] == oracle.ST_BAD_TOKEN and np.array_equal(got[0], want[0])


# ---------------------------------------------------------------- projections
def _proj_case(rng, T=3, hidden=12, q_rank=10, H=2, D=4, Hm=3, nope=5, L=5):
    g = lambda *s: oracle.round_bf16(rng.standard_normal(s))  # bf16-exact values
    return dict(x=g(T, hidden), w_kgw=g(2 * D + H, hidden), cq=g(T, q_rank),
                w_q=g(H * D + Hm * nope, q_rank), w_uk_t=g(Hm, L, nope), H=H, D=D, Hm=Hm,
                nope=nope)


def test_projection_of_unit_vectors_reads_weight_columns():
    """A one-hot token selects one input column: the outputs are that column of
    each weight block, exactly (bf16 values store unchanged), and the row blocks
    land in k, gate, weights, q (head by head) and q_nope in that order."""
    rng = np.random.default_rng(11)
    c = _proj_case(rng)
    T, hidden = c["x"].shape
    cols = [0, 7, hidden - 1]
    x = np.zeros((T, hidden))
    x[np.arange(T), cols] = 1.0
    qcols = [4, 0, 9]
    cq = np.zeros_like(c["cq"])
    cq[np.arange(T), qcols] = 1.0
    H, D, Hm, nope = c["H"], c["D"], c["Hm"], c["nope"]
    o = oracle.indexer_project(x, c["w_kgw"], cq, c["w_q"], c["w_uk_t"], H, D, Hm, nope, 0.25)
    for t in range(T):
        col = c["w_kgw"][:, cols[t]]
        assert np.array_equal(o["k"][t], col[:D])
        assert np.array_equal(o["gate"][t], col[D:2 * D])
        assert np.array_equal(o["weights"][t], 0.25 * col[2 * D:])   # a power of two: exact
        qc = c["w_q"][:, qcols[t]]
        for h in range(H):
            assert np.array_equal(o["q"][t, h], qc[h * D:(h + 1) * D])
        assert np.array_equal(o["q_nope"][t].ravel(), qc[H * D:])


def test_projection_against_brute_force_sums():
    """Every output element as an explicit sum of products (math.fsum, exact
    rounding of the float64 sum), before the storage rounding."""
    rng = np.random.default_rng(12)
    c = _proj_case(rng)
    H, D, Hm, nope = c["H"], c["D"], c["Hm"], c["nope"]
    o = oracle.indexer_project(c["x"], c["w_kgw"], c["cq"], c["w_q"], c["w_uk_t"], H, D, Hm,
                               nope, 0.5, rounded=False)
    T = c["x"].shape[0]
    for t in range(T):
        for f in range(2 * D + H):
            v = math.fsum(float(c["w_kgw"][f, k]) * float(c["x"][t, k])
                          for k in range(c["x"].shape[1]))
            got = o["k"][t, f] if f < D else o["gate"][t, f - D] if f < 2 * D else \
                o["weights"][t, f - 2 * D] / 0.5
            assert got == pytest.approx(v, rel=1e-12, abs=1e-12)
        for f in range(H * D + Hm * nope):
            v = math.fsum(float(c["w_q"][f, k]) * float(c["cq"][t, k])
                          for k in range(c["cq"].shape[1]))
            got = o["q"][t].ravel()[f] if f < H * D else o["q_nope"][t].ravel()[f - H * D]
            assert got == pytest.approx(v, rel=1e-12, abs=1e-12)
        for h in range(Hm):
            for l in range(c["w_uk_t"].shape[1]):
                v = math.fsum(float(o["q_nope"][t, h, n]) * float(c["w_uk_t"][h, l, n])
                              for n in range(nope))
                assert o["q_lat"][t, h, l] == pytest.approx(v, rel=1e-12, abs=1e-12)


def test_absorbed_query_scores_a_latent_row_like_its_up_projected_key():
    """The reason for the latent-space query: for any latent cache row c,
    <q_lat_h, c> = <q_nope_h, W_uk_h c> with W_uk_h = w_uk_t[h]^T.  L == nope
    here, so reading w_uk_t[h] untransposed has the right shape and must fail."""
    rng = np.random.default_rng(13)
    c = _proj_case(rng, nope=5, L=5)
    Hm = c["Hm"]
    q_nope = rng.standard_normal((2, Hm, 5))
    q_lat = oracle.absorb_query(q_nope, c["w_uk_t"])
    cvec = rng.standard_normal(5)
    for h in range(Hm):
        key = c["w_uk_t"][h].T @ cvec                  # W_uk_h c
        for t in range(2):
            assert q_lat[t, h] @ cvec == pytest.approx(q_nope[t, h] @ key, rel=1e-12)
            wrong = q_nope[t, h] @ (c["w_uk_t"][h] @ cvec)
            assert abs(q_lat[t, h] @ cvec - wrong) > 1e-6


def test_projection_storage_roundings():
    """k, gate, q, q_nope, q_lat are stored in bf16 (to nearest even), the
    weights in fp32, and q_lat is formed from the stored q_nope."""
    rng = np.random.default_rng(14)
    c = _proj_case(rng)
    args = (c["x"], c["w_kgw"], c["cq"], c["w_q"], c["w_uk_t"], c["H"], c["D"], c["Hm"],
            c["nope"], 0.3)
    ex = oracle.indexer_project(*args, rounded=False)
    st = oracle.indexer_project(*args)
    for n in ("k", "gate", "q", "q_nope"):
        assert np.array_equal(st[n], oracle.round_bf16(ex[n]))
    assert np.array_equal(st["weights"], ex["weights"].astype(np.float32).astype(np.float64))
    assert np.array_equal(st["q_lat"],
                          oracle.round_bf16(oracle.absorb_query(st["q_nope"], c["w_uk_t"])))
