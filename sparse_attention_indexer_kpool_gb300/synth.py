"""Seeded synthetic inputs for the DSA kpool selection + selected-row MLA path.

This module only draws random numbers and lays them out in the library's tensor
layout (ragged token axis with ``cu_seqlens``, pool-cache slices with
``cu_pool_cap``).  It holds none of the method's arithmetic, so it may serve
both the CUDA path and the CPU oracle.

The workloads mirror the pages' geometry (32 index heads, head_dim 128, kpool 4,
262 144-token contexts = 65 536 pools, 11 DSA layers) and the value
distributions of the five named workloads:

* ``tiny``      1 x 256 tokens, 3 tokens of left padding, fp32, 4 index heads of
                dim 32, kpool 4 (63 pools), select_k 8, MLA 4 heads x latent 64;
                integer keys/queries/gates in [-2, 2] drawn from a few template
                pools so that exact score ties straddle the top-k cutoff.
* ``single32k`` 1 x 32 768 tokens, bf16, 32 x 128 indexer, kpool 4, select_k 512,
                MLA 64 heads x latent 512.
* ``ragged64``  64 sequences, lengths U{4096..65536}, left padding U{0..7}.
* ``long262k``  4 x 262 144 tokens (one DSA layer; a model step runs 11).
* ``prefill``   4 096 query tokens appended to a 131 072-token context,
                kpool 8, select_k 256, causal.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Geometry:
    """Per-layer DSA geometry; every value is explicit (nothing defaulted)."""
    D: int            # index head_dim
    H: int            # index heads
    kpool: int
    select_k: int
    out_width: int
    Hm: int           # MLA heads
    L: int            # MLA latent dim
    dtype: str        # "bf16" | "f32"
    ln_eps: float = 1e-5


@dataclass
class Batch:
    """One layer's inputs in the library's layout (tensors on one device)."""
    geo: Geometry
    lengths: list          # T_b per sequence (padding included)
    pads: list             # left padding per sequence
    cu_seqlens: torch.Tensor   # [B+1] int32
    cu_pool_cap: torch.Tensor  # [B+1] int32
    P_ld: int
    k: torch.Tensor        # [sum T, D]
    gate: torch.Tensor     # [sum T, D]
    valid: torch.Tensor    # [sum T] uint8
    ape: torch.Tensor      # [kpool, D] fp32
    ln_gamma: torch.Tensor  # [D]
    ln_beta: torch.Tensor   # [D]
    q: torch.Tensor        # [Q, H, D]
    weights: torch.Tensor  # [Q, H] fp32
    q_seq: torch.Tensor | None   # [Q] int32 or None (all queries on sequence 0)
    q_pos: torch.Tensor | None   # [Q] int32 or None (every complete pool visible)
    q_lat: torch.Tensor    # [Q, Hm, L]
    kv: torch.Tensor       # [sum T, L]
    scale: float
    sm_scale: float
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return len(self.lengths)

    @property
    def Q(self):
        return self.q.shape[0]


def torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def _ints(shape, lo, hi, g, device, dtype):
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(dtype)


def make_batch(geo: Geometry, lengths, pads, *, device="cpu", seed=0, queries="decode",
               q_positions=None, q_sequence=0, dist="normal", pool_cap=None,
               weights_std=None) -> Batch:
    """Draw one layer's caches and queries.

    queries="decode": one query per sequence at its last token.
    queries="chunk":  len(q_positions) queries, all on sequence ``q_sequence``
                      (the prefill-chunk form; q_seq is None, so the caller
                      passes that sequence's cache slice).
    dist="normal": k, gate, q, q_lat, kv ~ N(0,1); ape ~ N(0, 0.1);
                   weights ~ N(0, 1/32) (std given by ``weights_std``);
                   LayerNorm gamma = 1, beta ~ N(0, 0.1).
    dist="ints":   k, gate, q, q_lat, kv integers in [-2, 2];
                   weights ~ N(0,1)/2; same ape / gamma / beta.
    """
    dev = torch.device(device)
    g = _gen(dev, seed)
    act = torch_dtype(geo.dtype)
    B = len(lengths)
    lengths = [int(t) for t in lengths]
    pads = [int(p) for p in pads]
    assert len(pads) == B and all(0 <= p <= t for p, t in zip(pads, lengths))
    total = sum(lengths)
    cu = [0]
    for t in lengths:
        cu.append(cu[-1] + t)
    caps = [t // geo.kpool for t in lengths] if pool_cap is None else list(pool_cap)
    cu_cap = [0]
    for c in caps:
        cu_cap.append(cu_cap[-1] + c)
    P_ld = max([1] + caps)
    D, L = geo.D, geo.L
    if dist == "ints":
        k = _ints((total, D), -2, 2, g, dev, act)
        gate = _ints((total, D), -2, 2, g, dev, act)
    else:
        k = _normal((total, D), 1.0, g, dev, act)
        gate = _normal((total, D), 1.0, g, dev, act)
    valid = torch.ones(total, dtype=torch.uint8, device=dev)
    for b in range(B):
        valid[cu[b]:cu[b] + pads[b]] = 0
    ape = _normal((geo.kpool, D), 0.1, g, dev, torch.float32)
    ln_gamma = torch.ones(D, dtype=act, device=dev)
    ln_beta = _normal((D,), 0.1, g, dev, act)

    if queries == "decode":
        Q = B
        q_seq = torch.arange(B, dtype=torch.int32, device=dev)
        q_pos = torch.tensor([t - 1 for t in lengths], dtype=torch.int32, device=dev)
    elif queries == "chunk":
        Q = len(q_positions)
        q_seq = None
        q_pos = torch.tensor(list(q_positions), dtype=torch.int32, device=dev)
    else:
        raise ValueError(queries)
    if dist == "ints":
        q = _ints((Q, geo.H, D), -2, 2, g, dev, act)
        weights = _normal((Q, geo.H), 0.5, g, dev, torch.float32)
        q_lat = _ints((Q, geo.Hm, L), -2, 2, g, dev, act)
        kv = _ints((total, L), -2, 2, g, dev, act)
    else:
        wstd = weights_std if weights_std is not None else math.sqrt(1.0 / 32.0)
        q = _normal((Q, geo.H, D), 1.0, g, dev, act)
        weights = _normal((Q, geo.H), wstd, g, dev, torch.float32)
        q_lat = _normal((Q, geo.Hm, L), 1.0, g, dev, act)
        kv = _normal((total, L), 1.0, g, dev, act)
    return Batch(geo=geo, lengths=lengths, pads=pads,
                 cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=dev),
                 cu_pool_cap=torch.tensor(cu_cap, dtype=torch.int32, device=dev),
                 P_ld=P_ld, k=k, gate=gate, valid=valid, ape=ape, ln_gamma=ln_gamma,
                 ln_beta=ln_beta, q=q, weights=weights, q_seq=q_seq, q_pos=q_pos,
                 q_lat=q_lat, kv=kv, scale=1.0 / math.sqrt(D), sm_scale=1.0 / math.sqrt(L))


def query_set(geo: Geometry, Q: int, *, device="cpu", seed=0, weights_std=None):
    """Another draw of a batch's per-step query inputs (q, weights, q_lat) with
    make_batch's normal distributions: a decode step's queries change from step
    to step while the caches stay."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    act = torch_dtype(geo.dtype)
    wstd = weights_std if weights_std is not None else math.sqrt(1.0 / 32.0)
    q = _normal((Q, geo.H, geo.D), 1.0, g, dev, act)
    weights = _normal((Q, geo.H), wstd, g, dev, torch.float32)
    q_lat = _normal((Q, geo.Hm, geo.L), 1.0, g, dev, act)
    return q, weights, q_lat


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------
GEO_TINY = Geometry(D=32, H=4, kpool=4, select_k=8, out_width=32, Hm=4, L=64, dtype="f32")
GEO_MAIN = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512, dtype="bf16")
GEO_PREFILL = Geometry(D=128, H=32, kpool=8, select_k=256, out_width=2048, Hm=64, L=512,
                       dtype="bf16")


def tiny(device="cpu", seed=0, n_templates=10, select_k=None, out_width=None) -> Batch:
    """1 x 256 tokens, 3 padding tokens, fp32 integers with tie-making templates.

    Each of the 63 full pools (tokens 3..254) copies its k and gate rows from one
    of ``n_templates`` template pools, so equal templates give bit-identical
    pool keys and scores: ties sit throughout the ranking, including the cutoff.
    """
    geo = Geometry(**{**GEO_TINY.__dict__})
    if select_k is not None:
        geo.select_k = select_k
    if out_width is not None:
        geo.out_width = out_width
    elif select_k is not None:
        geo.out_width = select_k * geo.kpool
    bt = make_batch(geo, [256], [3], device=device, seed=seed, dist="ints")
    g = _gen(torch.device(device), seed + 7919)
    kp, t0, P = geo.kpool, 3, (256 - 3) // geo.kpool
    tmpl = torch.randint(0, n_templates, (P,), generator=g, device=device).tolist()
    src_k = bt.k[t0:t0 + n_templates * kp].clone()
    src_g = bt.gate[t0:t0 + n_templates * kp].clone()
    for p in range(P):
        j = tmpl[p]
        bt.k[t0 + p * kp:t0 + (p + 1) * kp] = src_k[j * kp:(j + 1) * kp]
        bt.gate[t0 + p * kp:t0 + (p + 1) * kp] = src_g[j * kp:(j + 1) * kp]
    bt.extra["templates"] = tmpl
    bt.scale = 1.0 / math.sqrt(geo.D)
    bt.sm_scale = 1.0 / 8.0
    return bt


def single32k(device="cpu", seed=1000) -> Batch:
    return make_batch(GEO_MAIN, [32768], [0], device=device, seed=seed)


def ragged_lengths(B=64, lo=4096, hi=65536, max_pad=7, seed=2000):
    g = torch.Generator()
    g.manual_seed(seed)
    lengths = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    pads = torch.randint(0, max_pad + 1, (B,), generator=g).tolist()
    return lengths, pads


def ragged64(device="cpu", seed=2000) -> Batch:
    lengths, pads = ragged_lengths(seed=seed)
    return make_batch(GEO_MAIN, lengths, pads, device=device, seed=seed + 1)


def long262k(device="cpu", layer=0, seed=3000) -> Batch:
    return make_batch(GEO_MAIN, [262144] * 4, [0] * 4, device=device, seed=seed + 100 * layer)


def prefill(device="cpu", seed=4000, n_query=4096, ctx=131072) -> Batch:
    T = ctx + n_query
    return make_batch(GEO_PREFILL, [T], [0], device=device, seed=seed, queries="chunk",
                      q_positions=list(range(ctx, T)))


@dataclass
class PagedCache:
    """A latent cache laid out in pages (the paged attention's input)."""
    pages: torch.Tensor          # [n_pages * page_size, L] bf16 / fp32, or float8_e4m3fn codes
    row_scale: torch.Tensor | None   # [n_pages * page_size] fp32 (E4M3 only)
    block_table: torch.Tensor    # [B, max_pages] int32
    seq_lens: torch.Tensor       # [B] int32
    page_size: int


def paged_cache(kv, cu_seqlens, page_size: int, *, e4m3=False, seed=0, n_spare=3,
                extra_blocks=1) -> PagedCache:
    """Lay the contiguous cache ``kv`` [sum T_b, L] (sequence b at rows
    cu_seqlens[b] ..) out in shuffled pages of ``page_size`` rows.

    Block i of sequence b (tokens i*page_size ..) goes to a page drawn from a
    seeded permutation; ``n_spare`` pages and the rows past each sequence's
    last token hold other values, and the table has ``extra_blocks`` unused
    (-1) columns.  e4m3: each row is stored as E4M3 codes of row / s with
    s = max|row| / 448 (1 for an all-zero row), s kept per row.
    """
    dev = kv.device
    cu = [int(x) for x in cu_seqlens.tolist()]
    B, L = len(cu) - 1, kv.shape[1]
    lengths = [cu[b + 1] - cu[b] for b in range(B)]
    blocks = [-(-T // page_size) for T in lengths]
    n_pages = sum(blocks) + n_spare
    g = _gen(dev, seed)
    perm = torch.randperm(n_pages, generator=g, device=dev)
    table = torch.full((B, max(blocks) + extra_blocks), -1, dtype=torch.int32, device=dev)
    src, dst = [], []
    k = 0
    for b in range(B):
        if blocks[b]:
            table[b, :blocks[b]] = perm[k:k + blocks[b]].to(torch.int32)
        k += blocks[b]
        t = torch.arange(lengths[b], device=dev)
        src.append(cu[b] + t)
        dst.append(table[b, t // page_size].long() * page_size + t % page_size)
    src, dst = torch.cat(src), torch.cat(dst)
    n_rows = n_pages * page_size
    seq_lens = torch.tensor(lengths, dtype=torch.int32, device=dev)
    if not e4m3:
        pages = torch.randn((n_rows, L), generator=g, device=dev, dtype=kv.dtype)
        pages[dst] = kv[src]
        return PagedCache(pages, None, table, seq_lens, page_size)
    codes = (torch.randn((n_rows, L), generator=g, device=dev, dtype=torch.bfloat16) * 100.0
             ).clamp(-448, 448).to(torch.float8_e4m3fn)
    scale = torch.rand(n_rows, generator=g, device=dev) + 0.5
    for c0 in range(0, src.numel(), 1 << 20):           # bounded float32 temporaries
        rows = kv[src[c0:c0 + (1 << 20)]].float()
        s = rows.abs().amax(dim=1) / 448.0
        s = torch.where(s > 0, s, torch.ones_like(s))
        codes[dst[c0:c0 + (1 << 20)]] = (rows / s[:, None]).to(torch.float8_e4m3fn)
        scale[dst[c0:c0 + (1 << 20)]] = s
    return PagedCache(codes, scale.float(), table, seq_lens, page_size)


@dataclass
class ProjectionInputs:
    """One layer's projection inputs (bf16): activations and random-init weights."""
    x: torch.Tensor        # [T, hidden] hidden states
    cq: torch.Tensor       # [T, q_rank] query latent
    w_kgw: torch.Tensor    # [2D + H, hidden] rows of k, gate, weights
    w_q: torch.Tensor      # [H*D + Hm*nope, q_rank] rows of q, then q_nope
    w_uk_t: torch.Tensor   # [Hm, L, nope] key up-projection, transposed per head
    H: int
    D: int
    Hm: int
    nope: int
    L: int


# Shape assumptions for the projections at full size (the pages give the
# indexer's 32 heads of 128 and the latent width 512, but no hidden size,
# query-latent rank or no-rope head size)
PROJ_MAIN = dict(hidden=6144, q_rank=2048, H=32, D=128, Hm=64, nope=192, L=512)


def projection_inputs(T: int, hidden: int, q_rank: int, H: int, D: int, Hm: int, nope: int,
                      L: int, *, device="cpu", seed=0) -> ProjectionInputs:
    """Activations ~ N(0, 1); weights ~ N(0, 1/fan_in), so every output has
    about unit scale."""
    g = _gen(device, seed)
    bf = torch.bfloat16
    return ProjectionInputs(
        x=_normal((T, hidden), 1.0, g, device, bf),
        cq=_normal((T, q_rank), 1.0, g, device, bf),
        w_kgw=_normal((2 * D + H, hidden), hidden ** -0.5, g, device, bf),
        w_q=_normal((H * D + Hm * nope, q_rank), q_rank ** -0.5, g, device, bf),
        w_uk_t=_normal((Hm, L, nope), nope ** -0.5, g, device, bf),
        H=H, D=D, Hm=Hm, nope=nope, L=L)
