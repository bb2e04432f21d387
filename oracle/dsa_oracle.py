"""CPU oracle for DSA kpool token selection + selected-row NoPE MLA decode.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA path never imports, calls or links anything here, and nothing here
imports the CUDA path: the two share no code, constants or helpers.

Plain, slow, obviously correct numpy in float64.  Every input arrives as float64
arrays holding the exact values the GPU sees (bf16 and fp32 widen exactly to
float64).  The only roundings are the storage points the pages fix:

* the indexer key LayerNorm output is stored in the activation dtype before it
  is pooled (module glm5next_dsa, Constants, LAYERNORM_MODULE: a BF16 LayerNorm);
* pooled keys are stored in the activation dtype;
* scores are fp32 (module glm5next_dsa::tp, "Why the indexer is REPLICATED":
  65 536 pools x 4 B per decode token);
* the attention output is stored in the activation dtype.

Rounding to bf16 is written out below (round-to-nearest-even on the bf16 grid);
rounding to fp32 is numpy's float64->float32 cast, which is round-to-nearest-even.

Sources, by page and section (the pages print no code and no worked values):

* module glm5next_dsa, "Shape of the pipeline": the five stages and their I/O.
* module glm5next_dsa, "Traps carried from Slice 8": k_norm is a LayerNorm with
  bias (not RMSNorm); the pool softmax runs over the slot axis per channel;
  pooling starts at the first valid token; only full, all-valid pools count;
  NoPE (no rotary part); the -1 sentinel destination is written in full.
* module glm5next_dsa::tp, "Why the indexer is REPLICATED": the score is a plain
  sum over heads of weights[h] * relu(scale * dot); the tie order is higher
  score first, then the smaller pool index.
* module glm5next_dsa, Constants, KERNEL_MAX_KPOOL: at most 8 slots per pool.
* module glm5next_dsa, Constants, MASKED_ATTN_MAX_KEYS: dense masked attention
  is the attention oracle (here: dense softmax over exactly the selected rows).

Readings where the pages are silent: LayerNorm uses the population variance and an explicit epsilon; ``ape`` is a
[kpool, D] fp32 bias added to the gate logits per slot and channel; the causal
rule counts a pool when its last token is at or before the query position; the
attention output stays in latent space with an explicit softmax scale; an empty
selection gives out = 0, lse = -inf.  The projections before a1 (hidden state
and query latent to k, gate, weights, q and the latent-space query) are
bias-free linear maps: the pages name the tensors but give no formula.

The paged-cache attention (the pages' paged decode and its fp8 variant) reads
its rows through a block table and decodes E4M3 codes with one fp32 scale per
row: readings of a layout the pages do not give.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(hand-worked values, closed forms, invariants, brute force on tiny inputs,
textbook routines).  No function is left unpinned.
"""
from __future__ import annotations

import numpy as np

KPOOL_MAX = 8  # module glm5next_dsa, Constants, KERNEL_MAX_KPOOL

# Device status bits the oracle reports in the same encoding as the library.
ST_POOL_OVERFLOW = 1 << 1     # more complete pools than the cache slice holds
ST_POOL_UNCOVERED = 1 << 2    # complete pools beyond pool_begin + max_pools
ST_BAD_TOKEN = 1 << 0         # a selected token id outside its sequence
ST_BAD_POOL_ID = 1 << 3       # a pool id outside its cache slice
ST_BAD_QSEQ = 1 << 4          # a query's sequence index outside [0, B)
ST_POOL_RANGE = 1 << 5        # n_pools beyond the cache slice or the score row
ST_BAD_PAGE = 1 << 8          # paged cache: a token's block outside the table or its page


# --------------------------------------------------------------------------
# storage roundings
# --------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the fp32
    exponent range.  For |x| in [2^(e-1), 2^e) the grid spacing is 2^(e-8);
    below the smallest normal (2^-126) the spacing is fixed at 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                 # subnormal range: fixed spacing
    spacing = np.ldexp(1.0, e - 8)
    r = np.rint(x / spacing) * spacing      # np.rint rounds half to even
    big = np.abs(r) > 3.3895313892515355e38  # largest finite bfloat16
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, x), r)
    return np.where(x == 0, x, r)


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_store(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return round_f32(x)
    raise ValueError(f"unknown storage dtype {dtype!r}")


# --------------------------------------------------------------------------
# a1: indexer key LayerNorm
# --------------------------------------------------------------------------
def layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """Mean-subtracting LayerNorm with bias over the last axis.

    module glm5next_dsa, "Traps carried from Slice 8": indexer.k_norm is an
    nn.LayerNorm (mean removed, bias added), not an RMSNorm.  Population
    variance, epsilon inside the square root, as nn.LayerNorm defines it.
    """
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


# --------------------------------------------------------------------------
# a2: kpool_compress
# --------------------------------------------------------------------------
def first_valid(valid_b) -> int:
    """Index of the first valid token of one sequence (its length if none)."""
    nz = np.flatnonzero(np.asarray(valid_b) != 0)
    return int(nz[0]) if nz.size else int(len(valid_b))


def kpool_compress(k, gate, valid, ape, gamma, beta, eps, cu_seqlens, cu_pool_cap,
                   kpool: int, dtype: str, pool_begin=None, max_pools=None,
                   pool_keys=None, pool_start=None, pool_valid=None):
    """Pool LayerNorm'd indexer keys kpool tokens at a time.

    module glm5next_dsa, "Shape of the pipeline" (k, gate, valid, ape ->
    kpool_compress -> pool keys / indices / valid) and "Traps carried from
    Slice 8" (slot-axis softmax per channel; start at the first valid token;
    only full, all-valid pools count).

    For sequence b with tokens [0, T_b) on its own token axis:
      t0 = first valid token, P_b = floor((T_b - t0) / kpool);
      pool p covers tokens t0 + p*kpool + s, s = 0..kpool-1;
      logit[s, d] = gate[token, d] + ape[s, d];
      w[s, d] = softmax over s of logit[., d];
      key[p, d] = sum_s w[s, d] * round(LN(k[token]))[d], stored rounded;
      valid[p] = every slot's token is valid.
    Pools p in [begin_b, min(begin_b + max_pools, cap_b)) are written: computed
    when p < P_b, otherwise set to the sentinel (start -1, valid 0, key 0).
    Pools outside that range keep whatever the passed-in arrays hold.
    Returns (pool_keys, pool_start, pool_valid, n_pools, status).
    """
    if not (1 <= kpool <= KPOOL_MAX):
        raise ValueError("kpool must be in [1, 8]")  # Constants, KERNEL_MAX_KPOOL
    valid = np.asarray(valid)
    ape = np.asarray(ape, np.float64).reshape(kpool, -1)
    B = len(cu_seqlens) - 1
    D = k.shape[1]
    total_cap = int(cu_pool_cap[B])
    if pool_keys is None:
        pool_keys = np.zeros((total_cap, D), np.float64)
    if pool_start is None:
        pool_start = np.full(total_cap, -1, np.int64)
    if pool_valid is None:
        pool_valid = np.zeros(total_cap, np.uint8)
    pool_keys = np.array(pool_keys, np.float64)
    pool_start = np.array(pool_start, np.int64)
    pool_valid = np.array(pool_valid, np.uint8)
    n_pools = np.zeros(B, np.int64)
    status = 0
    for b in range(B):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        T = hi - lo
        cap_lo, cap_hi = int(cu_pool_cap[b]), int(cu_pool_cap[b + 1])
        cap = cap_hi - cap_lo
        begin = 0 if pool_begin is None else int(pool_begin[b])
        end = cap if max_pools is None else min(begin + int(max_pools), cap)
        t0 = first_valid(valid[lo:hi])
        P = (T - t0) // kpool
        if P > cap:
            status |= ST_POOL_OVERFLOW
        P_eff = min(P, cap)
        if P_eff > end:
            status |= ST_POOL_UNCOVERED
        n_pools[b] = P_eff
        # sentinel entries: pools of the range that are not complete pools
        first = max(begin, 0)                    # negative pool ids do not exist
        tail = np.arange(max(first, P_eff), end)
        pool_keys[cap_lo + tail] = 0.0
        pool_start[cap_lo + tail] = -1
        pool_valid[cap_lo + tail] = 0
        # complete pools of the range, all at once: axis 0 = pool, 1 = slot, 2 = channel
        pools = np.arange(first, min(end, P_eff))
        if pools.size == 0:
            continue
        tok = lo + t0 + pools[:, None] * kpool + np.arange(kpool)[None, :]   # [n, kpool]
        kk = np.asarray(k[tok.reshape(-1)], np.float64)
        kn = round_store(layernorm(kk, gamma, beta, eps), dtype).reshape(len(pools), kpool, -1)
        logit = np.asarray(gate[tok.reshape(-1)], np.float64).reshape(len(pools), kpool, -1)
        logit = logit + ape[None, :, :]
        m = logit.max(axis=1, keepdims=True)
        e = np.exp(logit - m)
        w = e / e.sum(axis=1, keepdims=True)                                 # softmax over slots
        pool_keys[cap_lo + pools] = round_store((w * kn).sum(axis=1), dtype)
        pool_start[cap_lo + pools] = t0 + pools * kpool
        pool_valid[cap_lo + pools] = np.all(valid[tok] != 0, axis=1).astype(np.uint8)
    return pool_keys, pool_start, pool_valid, n_pools, status


# --------------------------------------------------------------------------
# a3: index_scores
# --------------------------------------------------------------------------
def index_scores(q, weights, scale: float, pool_keys, pool_start, pool_valid, n_pools,
                 cu_pool_cap, q_seq, q_pos, kpool: int, P_ld: int):
    """score[q, p] = sum_h weights[q, h] * max(0, scale * <q[q, h, :], key[p, :]>).

    module glm5next_dsa::tp, "Why the indexer is REPLICATED": a plain sum over
    heads of weights[h] * relu(scale * dot).  module glm5next_dsa, "Shape of the
    pipeline": [Q, P] scores plus candidate validity, encoded here as -inf for
    a non-candidate.  A pool is a candidate for query q when p < P_b, it is a
    valid pool, and (if q_pos is given) its last token is at or before q_pos.
    Scores are rounded to fp32 and -0 becomes +0.
    q_seq None means every query reads sequence 0.
    """
    q = np.asarray(q, np.float64)
    w = np.asarray(weights, np.float64)
    Q = q.shape[0]
    out = np.full((Q, P_ld), -np.inf, np.float64)
    status = 0
    B = len(cu_pool_cap) - 1
    for i in range(Q):
        b = 0 if q_seq is None else int(q_seq[i])
        if not (0 <= b < B):
            status |= ST_BAD_QSEQ
            continue
        base = int(cu_pool_cap[b])
        cap = int(cu_pool_cap[b + 1]) - base
        P = min(int(n_pools[b]), cap, P_ld)
        if int(n_pools[b]) > P:
            status |= ST_POOL_RANGE
        idx = np.arange(P)
        cand = np.asarray(pool_valid[base:base + P]) != 0
        if q_pos is not None:
            last_tok = np.asarray(pool_start[base:base + P], np.int64) + kpool - 1
            cand &= last_tok <= int(q_pos[i])
        keys = np.asarray(pool_keys[base:base + P], np.float64)     # [P, D]
        dots = keys @ q[i].T                                         # [P, H]
        s = (np.maximum(0.0, scale * dots) * w[i][None, :]).sum(axis=1)
        s = round_f32(s) + 0.0                                       # fp32, -0 -> +0
        out[i, idx[cand]] = s[cand]
    return out, status


# --------------------------------------------------------------------------
# a4: topk_pools
# --------------------------------------------------------------------------
def topk_pools(scores, select_k: int):
    """Per row: candidates (score > -inf) ordered by score descending, then pool
    index ascending; the first min(select_k, n) are kept, the rest is -1.

    module glm5next_dsa::tp, "Why the indexer is REPLICATED" (deterministic tie
    order: higher score, then smaller pool index) and module glm5next_dsa,
    "Shape of the pipeline" ([Q, select_k] pool ids).  -0 and +0 are equal.
    """
    scores = np.asarray(scores, np.float64)
    Q, P = scores.shape
    out = np.full((Q, select_k), -1, np.int64)
    for i in range(Q):
        row = scores[i]
        cand = np.flatnonzero(row > -np.inf)             # NaN and -inf are not candidates
        s = row[cand] + 0.0
        order = np.lexsort((cand, -s))                   # primary: -score, secondary: index
        take = cand[order[:select_k]]
        out[i, :take.size] = take
    return out


# --------------------------------------------------------------------------
# a5: expand_selection
# --------------------------------------------------------------------------
def expand_selection(pool_ids, pool_start, cu_pool_cap, q_seq, kpool: int, out_width: int):
    """token[q, j*kpool + s] = pool_start[pool j of q] + s; -1 for an empty slot.

    module glm5next_dsa, "Shape of the pipeline" ([Q, out_width] token ids, -1 =
    invalid) and "Traps carried from Slice 8" (the -1 destination is written in
    full: every column past select_k * kpool is -1).  A pool id outside its
    sequence's cache slice yields -1 and a status bit; an id whose cache entry
    is the sentinel (start -1) is not a pool and yields -1.
    """
    pool_ids = np.asarray(pool_ids, np.int64)
    Q, K = pool_ids.shape
    if out_width < K * kpool:
        raise ValueError("out_width < select_k * kpool")
    out = np.full((Q, out_width), -1, np.int64)
    status = 0
    B = len(cu_pool_cap) - 1
    for i in range(Q):
        b = 0 if q_seq is None else int(q_seq[i])
        if not (0 <= b < B):
            status |= ST_BAD_QSEQ
            continue
        base, cap = int(cu_pool_cap[b]), int(cu_pool_cap[b + 1]) - int(cu_pool_cap[b])
        for j in range(K):
            p = int(pool_ids[i, j])
            if p < 0:
                continue
            if p >= cap:
                status |= ST_BAD_POOL_ID
                continue
            start = int(pool_start[base + p])
            if start < 0:                                # sentinel entry: not a pool
                continue
            for s in range(kpool):
                out[i, j * kpool + s] = start + s
    return out, status


# --------------------------------------------------------------------------
# a6: NoPE MLA decode over the selected latent rows
# --------------------------------------------------------------------------
def mla_selected_decode(q_lat, kv, cu_seqlens, q_seq, token_ids, sm_scale: float, dtype: str):
    """Absorbed NoPE MLA decode restricted to the selected latent-KV rows.

    module glm5next_dsa, "Shape of the pipeline" (NoPE MLA restricted to the
    selected tokens), Modules, attend (selected-index NoPE MLA decode) and
    "Traps carried from Slice 8" (NoPE: no rotary slice).  For query q, head h,
    over the selected rows c_j = kv[cu_seqlens[b] + tok_j] (tok_j >= 0):
      z_j = sm_scale * <q_lat[q, h], c_j>,  out = sum_j softmax(z)_j c_j,
      lse = log sum_j exp(z_j).
    The value of an MLA latent row is the row itself (the up-projection is
    absorbed upstream).  Empty selection: out = 0, lse = -inf.  A token id
    outside [0, T_b) is skipped and flagged.
    """
    q_lat = np.asarray(q_lat, np.float64)
    token_ids = np.asarray(token_ids, np.int64)
    Q, Hm, L = q_lat.shape
    out = np.zeros((Q, Hm, L), np.float64)
    lse = np.full((Q, Hm), -np.inf, np.float64)
    status = 0
    B = len(cu_seqlens) - 1
    for i in range(Q):
        b = 0 if q_seq is None else int(q_seq[i])
        if not (0 <= b < B):
            status |= ST_BAD_QSEQ
            continue
        lo, T = int(cu_seqlens[b]), int(cu_seqlens[b + 1]) - int(cu_seqlens[b])
        toks = token_ids[i]
        sel = toks[toks >= 0]
        if np.any(sel >= T):
            status |= ST_BAD_TOKEN
            sel = sel[sel < T]
        if sel.size == 0:
            continue
        C = np.asarray(kv[lo + sel], np.float64)          # [n, L]
        out[i], lse[i] = attend_rows(q_lat[i], C, sm_scale)
    return round_store(out, dtype), lse, status


def attend_rows(q_i, C, sm_scale: float):
    """Softmax attention of the heads q_i [Hm, L] over the latent rows C [n, L]
    (n >= 1): z = sm_scale * q_i C^T, out = softmax(z) C, lse = log sum exp z."""
    z = sm_scale * (q_i @ C.T)                        # [Hm, n]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    den = e.sum(axis=1, keepdims=True)
    return (e @ C) / den, (m + np.log(den))[:, 0]


# --------------------------------------------------------------------------
# a6 on a paged latent cache (bf16 or fp8 E4M3 rows)
# --------------------------------------------------------------------------
def fp8_e4m3_decode(codes) -> np.ndarray:
    """Values of 8-bit floating-point codes in the E4M3 encoding.

    The attention's fp8 twin (module glm5next_dsa, Constants, KERNEL_KV_LORA_DIM:
    the mla_paged_decode kernel and its _fp8 variant) stores latent rows in 8
    bits; the pages do not spell out the encoding, read here as the E4M3 format
    of the OCP 8-bit floating-point specification: bit 7 is the sign, bits 6..3
    the exponent with bias 7, bits 2..0 the mantissa.  Exponent 0 encodes the
    subnormals (m / 8) * 2^-6; exponents 1..15 encode (1 + m / 8) * 2^(e - 7);
    exponent 15 with mantissa 7 is NaN, and there is no infinity.
    """
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def mla_paged_decode(q_lat, pages, row_scale, kv_dtype: str, block_table, seq_lens,
                     page_size: int, q_seq, token_ids, sm_scale: float, dtype: str):
    """The selected-row attention (a6) reading its latent rows from a paged cache.

    module glm5next_dsa, Modules, attend (the selected-index NoPE MLA paged
    decode) and Constants, KERNEL_KV_LORA_DIM (its mla_paged_decode kernel and
    the _fp8 variant).  The pages give no layout; the reading used here:

    * the cache is ``pages`` [n_pages * page_size, L]: page g holds the rows
      g * page_size .. g * page_size + page_size - 1;
    * ``block_table`` [B, max_pages]: token t of sequence b lives in page
      block_table[b, t // page_size], row t % page_size of it;
    * ``kv_dtype`` "bf16" or "f32": ``pages`` holds the row values; "fp8_e4m3": ``pages``
      holds E4M3 codes and a row's value is decode(code) * row_scale[row]
      (one fp32 scale per physical row).

    A token id at or past seq_lens[b] is skipped and flagged ST_BAD_TOKEN; a
    token whose block is past the table, or whose page is outside
    [0, n_pages), is skipped and flagged ST_BAD_PAGE.  The attention over the
    rows kept is that of ``mla_selected_decode``.
    """
    q_lat = np.asarray(q_lat, np.float64)
    token_ids = np.asarray(token_ids, np.int64)
    block_table = np.asarray(block_table, np.int64)
    Q, Hm, L = q_lat.shape
    B, max_pages = block_table.shape
    n_pages = pages.shape[0] // page_size
    out = np.zeros((Q, Hm, L), np.float64)
    lse = np.full((Q, Hm), -np.inf, np.float64)
    status = 0
    for i in range(Q):
        b = 0 if q_seq is None else int(q_seq[i])
        if not (0 <= b < B):
            status |= ST_BAD_QSEQ
            continue
        toks = token_ids[i]
        sel = toks[toks >= 0]
        if np.any(sel >= int(seq_lens[b])):
            status |= ST_BAD_TOKEN
            sel = sel[sel < int(seq_lens[b])]
        blk = sel // page_size
        inside = blk < max_pages
        page = np.where(inside, block_table[b, np.minimum(blk, max_pages - 1)], -1)
        ok = (page >= 0) & (page < n_pages)
        if not np.all(ok):
            status |= ST_BAD_PAGE
        rows = page[ok] * page_size + sel[ok] % page_size
        if rows.size == 0:
            continue
        if kv_dtype == "fp8_e4m3":
            C = fp8_e4m3_decode(pages[rows]) * np.asarray(row_scale, np.float64)[rows][:, None]
        elif kv_dtype in ("bf16", "f32"):
            C = np.asarray(pages[rows], np.float64)
        else:
            raise ValueError(f"unknown kv dtype {kv_dtype!r}")
        out[i], lse[i] = attend_rows(q_lat[i], C, sm_scale)
    return round_store(out, dtype), lse, status


# --------------------------------------------------------------------------
# the projections before a1: hidden state / query latent -> the path's inputs
# --------------------------------------------------------------------------
def linear(inp, w, alpha: float = 1.0) -> np.ndarray:
    """out[t, f] = alpha * sum_k w[f, k] * inp[t, k], exactly (float64, no bias).

    Module glm5next_dsa, Modules: build and layer name the block's projection
    tensors but print no formula; a bias-free linear map is the plain reading.
    """
    inp = np.asarray(inp, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    return alpha * (inp @ w.T)


def absorb_query(q_nope, w_uk_t) -> np.ndarray:
    """Latent-space MLA query: q_lat[t, h, l] = sum_n q_nope[t, h, n] * W_uk_h[n, l].

    ``w_uk_t[h]`` is W_uk_h transposed ([L, nope]).  With the key up-projection
    k_h = W_uk_h c of a latent row c, <q_nope_h, k_h> = <q_lat_h, c>: the
    attention scores the latent cache directly (module glm5next_dsa, the NoPE MLA
    over the selected tokens, whose output stays in latent space).
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    w_uk_t = np.asarray(w_uk_t, dtype=np.float64)
    T, Hm, nope = q_nope.shape
    out = np.zeros((T, Hm, w_uk_t.shape[1]))
    for h in range(Hm):
        out[:, h, :] = q_nope[:, h, :] @ w_uk_t[h].T
    return out


def indexer_project(x, w_kgw, cq, w_q, w_uk_t, H: int, D: int, Hm: int, nope: int,
                    weights_scale: float, rounded: bool = True) -> dict:
    """The per-token inputs of the path from a layer's activations.

    * x [T, hidden] through w_kgw [2D + H, hidden]: rows 0..D-1 give the indexer
      key k (LayerNorm'ed later by kpool_compress), rows D..2D-1 its slot-logit
      gate, rows 2D.. the per-head weights, times ``weights_scale``;
    * the query latent cq [T, q_rank] through w_q [H*D + Hm*nope, q_rank]: the
      indexer query (head h from rows h*D..h*D+D-1), then the MLA no-rope query;
    * the no-rope query through the transposed key up-projection (absorb_query).

    With ``rounded`` the stored outputs are rounded as the library stores them:
    bf16 for k, gate, q, q_nope and q_lat, fp32 for the weights; q_lat is then
    computed from the stored (bf16) q_nope, the tensor the latent projection reads.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    hid = linear(x, w_kgw)
    k, gate = hid[:, :D], hid[:, D:2 * D]
    weights = weights_scale * hid[:, 2 * D:2 * D + H]
    qq = linear(cq, w_q)
    q = qq[:, :H * D].reshape(T, H, D)
    q_nope = qq[:, H * D:H * D + Hm * nope].reshape(T, Hm, nope)
    if rounded:
        k, gate, q, q_nope = (round_bf16(a) for a in (k, gate, q, q_nope))
        weights = round_f32(weights)
    q_lat = absorb_query(q_nope, w_uk_t)
    if rounded:
        q_lat = round_bf16(q_lat)
    return dict(k=k, gate=gate, weights=weights, q=q, q_nope=q_nope, q_lat=q_lat)


# --------------------------------------------------------------------------
# the whole path, stage after stage
# --------------------------------------------------------------------------
def run_path(inp: dict, pool_begin=None, max_pools=None, cache=None):
    """Run a1..a6 in the pages' order on one batch; returns every stage output.

    ``inp`` holds float64 / integer numpy arrays with the names of the library's
    arguments.  ``cache`` optionally supplies existing pool arrays (decode:
    only pools >= pool_begin are recomputed).
    """
    kp = inp["kpool"]
    cache = cache or {}
    pk, ps, pv, n_pools, st_c = kpool_compress(
        inp["k"], inp["gate"], inp["valid"], inp["ape"], inp["ln_gamma"], inp["ln_beta"],
        inp["ln_eps"], inp["cu_seqlens"], inp["cu_pool_cap"], kp, inp["dtype"],
        pool_begin=pool_begin, max_pools=max_pools,
        pool_keys=cache.get("pool_keys"), pool_start=cache.get("pool_start"),
        pool_valid=cache.get("pool_valid"))
    scores, st_s = index_scores(inp["q"], inp["weights"], inp["scale"], pk, ps, pv, n_pools,
                                inp["cu_pool_cap"], inp.get("q_seq"), inp.get("q_pos"), kp,
                                inp["P_ld"])
    pool_ids = topk_pools(scores, inp["select_k"])
    tok, st_e = expand_selection(pool_ids, ps, inp["cu_pool_cap"], inp.get("q_seq"), kp,
                                 inp["out_width"])
    out, lse, st_m = mla_selected_decode(inp["q_lat"], inp["kv"], inp["cu_seqlens"],
                                         inp.get("q_seq"), tok, inp["sm_scale"], inp["dtype"])
    return dict(pool_keys=pk, pool_start=ps, pool_valid=pv, n_pools=n_pools, scores=scores,
                pool_ids=pool_ids, token_ids=tok, out=out, lse=lse,
                status=st_c | st_s | st_e | st_m)
