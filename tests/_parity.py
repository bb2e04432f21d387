"""Stage-wise comparison of the CUDA path against the CPU oracle.

Each GPU stage is checked on the GPU's own inputs for that stage (the previous
stage's GPU output, copied to the host), so selection can be compared bit for
bit: the oracle's top-k runs on the GPU's score tensor and the oracle's expand
on the GPU's pool ids.

Tolerances, each with the arithmetic that sets it:
* pool keys: |gpu - ref| <= 2e-3*|ref| + ulp(ref) + ulp(max_s |kn_s|) + 1e-6*max_s |kn_s|
  - the LayerNorm output is rounded to the activation dtype on both sides
  from fp32 (GPU) and fp64 (oracle) values, so one slot may land one ulp
  apart; it enters the pool with a weight <= 1; the pooled key is rounded once
  more.  fp32 storage uses a few fp32 ulps instead of bf16 ulps.
* scores: |gpu - ref| <= 2e-3*|ref| + 2e-3*rms(ref row); -inf exactly where
  the oracle has -inf.
* selection (pool ids, token ids): bit-exact.
* attention out: 1e-2 absolute against the oracle's output before its storage
  rounding, plus half a bf16 spacing for the GPU's own rounding of its bf16
  output (the oracle's fp32-rounded value stands in for the unrounded one: fp32
  rounding is 2^-16 of a bf16 spacing); and 1e-2 plus one bf16 spacing against
  the oracle's bf16-rounded output.  lse: 1e-3 * max(1, |ref|).
"""
import numpy as np
import torch

import oracle
from tests._util import npf, npi, ulp_bf16


def kn_absmax(o, pool_start, n_pools):
    """max over slots of |round(LN(k))| per (pool, channel), oracle arithmetic."""
    cu, cap, kp = o["cu_seqlens"], o["cu_pool_cap"], o["kpool"]
    D = o["k"].shape[1]
    out = np.zeros((int(cap[-1]), D))
    for b in range(len(cu) - 1):
        P = int(n_pools[b])
        if P == 0:
            continue
        base = int(cap[b])
        starts = np.asarray(pool_start[base:base + P], np.int64)
        toks = int(cu[b]) + starts[:, None] + np.arange(kp)[None, :]        # [P, kp]
        k = np.asarray(o["k"][toks.reshape(-1)], np.float64)
        kn = oracle.round_store(oracle.layernorm(k, o["ln_gamma"], o["ln_beta"], o["ln_eps"]),
                                o["dtype"])
        out[base:base + P] = np.abs(kn).reshape(P, kp, D).max(axis=1)
    return out


def pool_key_tol(ref, knmax, dtype):
    if dtype == "bf16":
        return 2e-3 * np.abs(ref) + ulp_bf16(ref) + ulp_bf16(knmax) + 1e-6 * knmax
    return 2e-3 * np.abs(ref) + 8 * 2.0 ** -24 * (np.abs(ref) + knmax) + 1e-7


def check_compress(o, buf, pool_begin=None, max_pools=None, cache=None):
    pk, ps, pv, n, st = oracle.kpool_compress(
        o["k"], o["gate"], o["valid"], o["ape"], o["ln_gamma"], o["ln_beta"], o["ln_eps"],
        o["cu_seqlens"], o["cu_pool_cap"], o["kpool"], o["dtype"], pool_begin=pool_begin,
        max_pools=max_pools, **(cache or {}))
    g_n = npi(buf.n_pools)
    g_ps = npi(buf.pool_start)[:len(ps)]
    g_pv = buf.pool_valid.cpu().numpy()[:len(pv)]
    g_pk = npf(buf.pool_keys)[:len(pk)]
    assert np.array_equal(g_n, n), (g_n, n)
    assert np.array_equal(g_ps, ps)
    assert np.array_equal(g_pv, pv)
    tol = pool_key_tol(pk, kn_absmax(o, ps, n), o["dtype"])
    bad = np.abs(g_pk - pk) > tol
    assert not bad.any(), f"{bad.sum()} pool-key elements out of tolerance, worst " \
                          f"{np.max(np.abs(g_pk - pk) - tol):.3g}"
    return st


def check_scores(o, buf, rows=None):
    """Oracle scores on the GPU's pool cache; returns (gpu, ref) for the rows."""
    Q = o["q"].shape[0]
    rows = list(range(Q)) if rows is None else list(rows)
    qsel = np.array(rows)
    ref, st = oracle.index_scores(
        o["q"][qsel], o["weights"][qsel], o["scale"], npf(buf.pool_keys), npi(buf.pool_start),
        buf.pool_valid.cpu().numpy(), npi(buf.n_pools), o["cu_pool_cap"],
        None if o["q_seq"] is None else o["q_seq"][qsel],
        None if o["q_pos"] is None else o["q_pos"][qsel], o["kpool"], o["P_ld"])
    gpu = buf.scores[torch.as_tensor(rows, device=buf.scores.device)].cpu().double().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(gpu), fin), "candidate sets differ"
    assert np.all(gpu[~fin] == -np.inf)
    for i in range(len(rows)):
        r = ref[i][fin[i]]
        if r.size == 0:
            continue
        rms = np.sqrt(np.mean(r ** 2))
        err = np.abs(gpu[i][fin[i]] - r)
        tol = 2e-3 * np.abs(r) + 2e-3 * rms
        assert np.all(err <= tol), f"row {rows[i]}: worst excess {np.max(err - tol):.3g}"
    assert not np.any(np.signbit(gpu[np.isfinite(gpu) & (gpu == 0)])), "-0 in scores"
    return gpu, st


def check_topk(buf, select_k, rows=None):
    Q = buf.scores.shape[0]
    rows = list(range(Q)) if rows is None else list(rows)
    idx = torch.as_tensor(rows, device=buf.scores.device)
    s = buf.scores[idx].cpu().double().numpy()
    ref = oracle.topk_pools(s, select_k)
    got = buf.pool_ids[idx].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, ref), "pool ids differ from the oracle's top-k on GPU scores"
    return ref


def check_expand(o, buf, rows=None):
    Q = buf.pool_ids.shape[0]
    rows = list(range(Q)) if rows is None else list(rows)
    idx = torch.as_tensor(rows, device=buf.pool_ids.device)
    qs = None if o["q_seq"] is None else o["q_seq"][np.array(rows)]
    ref, st = oracle.expand_selection(buf.pool_ids[idx].cpu().numpy(), npi(buf.pool_start),
                                      o["cu_pool_cap"], qs, o["kpool"], o["out_width"])
    got = buf.token_ids[idx].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, ref), "token ids differ"
    return st


def mla_tol(ref_out, dtype):
    """1e-2 absolute on the attention output, plus one bf16 spacing at the
    reference value when the output is stored as bf16: both sides round their
    result to bf16, and two values on either side of a rounding boundary land one
    spacing apart (outputs of magnitude 2..4 appear when a query has only a few
    selected rows)."""
    return 1e-2 + (ulp_bf16(ref_out) if dtype == "bf16" else 0.0)


def check_mla(o, buf, rows=None, kv_rows=None):
    """Attention on the GPU's token ids.  kv_rows: optional callable(rows) ->
    float64 latent rows, for workloads too big to copy whole."""
    Q = buf.token_ids.shape[0]
    rows = list(range(Q)) if rows is None else list(rows)
    qsel = np.array(rows)
    tok = buf.token_ids[torch.as_tensor(rows, device=buf.token_ids.device)].cpu().numpy()
    qs = None if o["q_seq"] is None else o["q_seq"][qsel]
    ref_out, ref_lse, st = oracle.mla_selected_decode(o["q_lat"][qsel], o["kv"], o["cu_seqlens"],
                                                      qs, tok, o["sm_scale"], o["dtype"])
    idx = torch.as_tensor(rows, device=buf.out.device)
    out = buf.out[idx].cpu().double().numpy()
    lse = buf.lse[idx].cpu().double().numpy()
    err = np.abs(out - ref_out)
    assert np.all(err <= mla_tol(ref_out, o["dtype"])), f"attention out error {err.max():.3g}"
    if o["dtype"] == "bf16":
        ref32, _, _ = oracle.mla_selected_decode(o["q_lat"][qsel], o["kv"], o["cu_seqlens"], qs,
                                                 tok, o["sm_scale"], "f32")
        tol = 1e-2 + 0.5 * np.maximum(ulp_bf16(ref32), ulp_bf16(out))
        err32 = np.abs(out - ref32)
        assert np.all(err32 <= tol), f"attention out vs unrounded: worst {err32.max():.3g}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.abs(lse[fin] - ref_lse[fin]) <= 1e-3 * np.maximum(1.0, np.abs(ref_lse[fin])))
    return st
