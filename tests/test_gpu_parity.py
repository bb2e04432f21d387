"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
from sparse_attention_indexer_kpool_gb300.synth import Geometry
from tests import _parity as par
from tests._util import npf, npi, oracle_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_and_check(bt, expect_status=0, end_to_end=False):
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    st = par.check_compress(o, buf)
    _, st2 = par.check_scores(o, buf)
    par.check_topk(buf, bt.geo.select_k)
    st3 = par.check_expand(o, buf)
    st4 = par.check_mla(o, buf)
    assert int(buf.status.item()) == (st | st2 | st3 | st4 | expect_status)
    if end_to_end:
        r = oracle.run_path(o)
        assert np.array_equal(buf.pool_ids.cpu().numpy(), r["pool_ids"])
        assert np.array_equal(buf.token_ids.cpu().numpy(), r["token_ids"])
    return buf, o


def test_tiny_fp32_all_stages():
    bt = synth.tiny(device=DEV)
    buf, o = run_and_check(bt, end_to_end=True)
    s = buf.scores[0].cpu().double().numpy()
    ids = buf.pool_ids[0].cpu().numpy()
    kth = s[ids[-1]]
    assert any(s[p] == kth for p in range(63) if p not in set(ids)), "tie must straddle cutoff"


def test_tiny_sentinel_tail_and_wide_output():
    bt = synth.tiny(device=DEV, select_k=64)          # 63 pools < 64: -1 tail
    buf, _ = run_and_check(bt, end_to_end=True)
    assert buf.pool_ids[0, 63].item() == -1 and (buf.token_ids[0, 252:] == -1).all()
    bt = synth.tiny(device=DEV, select_k=8, out_width=40)   # columns 32..39 are -1
    buf, _ = run_and_check(bt, end_to_end=True)
    assert (buf.token_ids[0, 32:] == -1).all()


def ragged_small(dtype="bf16", select_k=64, out_width=320, seed=11):
    geo = Geometry(D=128, H=32, kpool=4, select_k=select_k, out_width=out_width, Hm=64, L=512,
                   dtype=dtype)
    # 0 tokens; kpool-1 valid tokens; 5*kpool+3 valid tokens; all padding; two long ones
    lengths = [1203, 0, 3, 23, 50, 2500]
    pads = [5, 0, 0, 0, 50, 1]
    return synth.make_batch(geo, lengths, pads, device=DEV, seed=seed)


def test_ragged_small_bf16_tensor_core_paths():
    bt = ragged_small()
    buf, _ = run_and_check(bt)
    ids = buf.pool_ids.cpu().numpy()
    assert (ids[1] == -1).all() and (ids[2] == -1).all() and (ids[4] == -1).all()
    assert (ids[3, :5] >= 0).all() and (ids[3, 5:] == -1).all()    # 23 tokens -> 5 pools
    tok = buf.token_ids.cpu().numpy()
    assert (tok[:, 256:] == -1).all()
    assert torch.all(buf.out[1] == 0) and torch.isinf(buf.lse[1]).all()


def test_single32k_bf16():
    bt = synth.single32k(device=DEV)
    run_and_check(bt)


def test_generic_kernels_bf16():
    geo = Geometry(D=64, H=8, kpool=3, select_k=16, out_width=48, Hm=8, L=64, dtype="bf16")
    bt = synth.make_batch(geo, [500, 97], [2, 0], device=DEV, seed=5)
    run_and_check(bt)


def test_generic_kernels_fp32_kpool8_and_1():
    for kp in (8, 1):
        geo = Geometry(D=32, H=4, kpool=kp, select_k=8, out_width=8 * kp + 3, Hm=4, L=64,
                       dtype="f32")
        bt = synth.make_batch(geo, [301, 64], [9, 1], device=DEV, seed=6 + kp)
        run_and_check(bt)


def test_incremental_compress_matches_full_build():
    bt = ragged_small(seed=21)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, buf)
    torch.cuda.synchronize()
    # new data arrives for every sequence's last complete pool: rewrite those tokens
    o = oracle_inputs(bt)
    n = buf.n_pools.cpu().numpy()
    begin = np.maximum(n - 1, 0).astype(np.int32)
    for b in range(bt.B):
        if n[b] == 0:
            continue
        lo = int(o["cu_seqlens"][b]) + int(buf.pool_start[int(o["cu_pool_cap"][b]) + n[b] - 1])
        bt.k[lo:lo + 4] = torch.randn(4, 128, device=DEV).to(bt.k.dtype)
        bt.gate[lo:lo + 4] = torch.randn(4, 128, device=DEV).to(bt.k.dtype)
    cache = dict(pool_keys=npf(buf.pool_keys), pool_start=npi(buf.pool_start),
                 pool_valid=buf.pool_valid.cpu().numpy())
    pool_begin = torch.as_tensor(begin, device=DEV)
    pipeline.compress(bt, buf, pool_begin=pool_begin, max_pools=1)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    par.check_compress(o, buf, pool_begin=begin, max_pools=1, cache=cache)
    full = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, full)
    torch.cuda.synchronize()
    assert torch.equal(full.pool_keys, buf.pool_keys)
    assert torch.equal(full.pool_start, buf.pool_start)


@pytest.mark.parametrize("kpool", [1, 3, 4, 8])
def test_bulk_compress_equals_pool_by_pool(kpool):
    """A bulk build (bf16, D = 128: the wide kernel, a half-warp per pool) writes
    the keys that sixteen-pool incremental calls (the warp-per-pool kernel)
    write, bit for bit, on ragged sequences with padding; and both match the
    oracle."""
    geo = Geometry(D=128, H=32, kpool=kpool, select_k=16, out_width=16 * kpool, Hm=64, L=512,
                   dtype="bf16")
    bt = synth.make_batch(geo, [1203, 40, 2500, 7], [5, 0, 1, 2], device=DEV, seed=90 + kpool)
    bulk = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, bulk)                     # max_pools = P_ld: the wide kernel
    inc = pipeline.LayerBuffers.alloc(bt)
    for p0 in range(0, bt.P_ld, 16):                # sixteen pools per call: the warp kernel
        begin = torch.full((bt.B,), p0, dtype=torch.int32, device=DEV)
        pipeline.compress(bt, inc, pool_begin=begin, max_pools=16)
    torch.cuda.synchronize()
    for name in ("pool_keys", "pool_start", "pool_valid", "n_pools"):
        assert torch.equal(getattr(bulk, name), getattr(inc, name)), name
    par.check_compress(oracle_inputs(bt), bulk)


def _topk_gpu(scores, k):
    Q, P = scores.shape
    ws = torch.empty(ops.topk_workspace_bytes(Q, P, k), dtype=torch.uint8, device=DEV)
    ids = torch.full((Q, k), 0x7F7F7F7F, dtype=torch.int32, device=DEV)
    ops.dsa_topk_pools(scores, k, ids, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("P,k", [(1, 1), (17, 8), (1000, 8), (1000, 999), (1000, 1000),
                                 (5000, 4096), (65536, 512), (70000, 2048)])
def test_topk_tie_stress(P, k):
    g = torch.Generator(device=DEV).manual_seed(P * 7 + k)
    Q = 6
    s = torch.randint(-4, 5, (Q, P), generator=g, device=DEV).float() * 0.25     # heavy ties
    s[1] = torch.randn(P, generator=g, device=DEV)                                # distinct
    s[2] = 0.0                                                                    # all equal
    s[2, ::3] = -0.0
    s[3, : P // 2] = -math.inf                                                    # half absent
    s[4] = -math.inf                                                              # no candidate
    s[5, ::5] = float("nan")
    s[5, 1::7] = math.inf
    got = _topk_gpu(s, k)
    ref = oracle.topk_pools(s.cpu().double().numpy(), k)
    assert np.array_equal(got, ref)


def test_topk_tie_list_overflow_path():
    # 20000 equal candidates in one histogram bin exceed the tie list: exact slow path
    s = torch.full((3, 30000), 1.0, device=DEV)
    s[0, 20000:] = 2.0 ** -30                       # lower bin
    s[1, :100] = 5.0                                # 100 sure keys, the rest tied
    s[2, 7::11] = 1.0 + 2.0 ** -20                  # same 12-bit bin, distinct low bits
    for k in (1, 511, 4096):
        assert np.array_equal(_topk_gpu(s, k), oracle.topk_pools(s.cpu().double().numpy(), k))


def test_expand_overwrites_every_entry_and_flags_bad_ids():
    cap = torch.tensor([0, 5, 9], dtype=torch.int32, device=DEV)
    start = torch.tensor([0, 4, 8, 12, 16, 1, 9, 17, -1], dtype=torch.int32, device=DEV)
    ids = torch.tensor([[4, 0, -1], [2, 3, 7], [0, -1, -1]], dtype=torch.int32, device=DEV)
    q_seq = torch.tensor([0, 1, 1], dtype=torch.int32, device=DEV)
    tok = torch.full((3, 14), 0x7F7F7F7F, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.dsa_expand_selection(ids, start, cap, q_seq, 4, tok, st)
    torch.cuda.synchronize()
    ref, rst = oracle.expand_selection(ids.cpu().numpy(), start.cpu().numpy(), [0, 5, 9],
                                       [0, 1, 1], 4, 14)
    assert np.array_equal(tok.cpu().numpy(), ref)
    assert int(st.item()) == rst == ops.DEV_BAD_POOL_ID


def test_mla_bad_tokens_and_empty_rows():
    geo = synth.GEO_MAIN
    bt = synth.make_batch(geo, [300, 700], [0, 0], device=DEV, seed=9)
    W = 2048
    g = torch.Generator(device=DEV).manual_seed(3)
    tok = torch.randint(-1, 300, (2, W), generator=g, device=DEV, dtype=torch.int32)
    tok[1, :] = -1                                 # empty selection
    tok[0, 5] = 300                                # out of range for sequence 0 -> flagged
    Q = 2
    out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(Q, 64, dtype=torch.float32, device=DEV)
    nb = ops.mla_workspace_bytes(Q, 64, 512, W, ops.DSA_BF16)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.dsa_mla_selected_decode(bt.q_lat, bt.kv, bt.cu_seqlens, bt.q_seq, tok, bt.sm_scale, out,
                                lse, ws, st)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    ref, ref_lse, rst = oracle.mla_selected_decode(o["q_lat"], o["kv"], o["cu_seqlens"],
                                                   o["q_seq"], tok.cpu().numpy(), bt.sm_scale,
                                                   "bf16")
    assert np.all(np.abs(out.cpu().double().numpy() - ref) <= par.mla_tol(ref, "bf16"))
    assert int(st.item()) == rst == ops.DEV_BAD_TOKEN
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))


def test_bad_query_sequence_is_flagged_not_faulted():
    bt = ragged_small(seed=31)
    bt.q_seq[2] = 99
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) & ops.DEV_BAD_QSEQ
    assert torch.all(torch.isneginf(buf.scores[2]))
    assert torch.all(buf.token_ids[2] == -1) and torch.all(buf.out[2] == 0)


def test_repeat_runs_are_bitwise_identical():
    bt = synth.single32k(device=DEV, seed=77)
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, a)
    pipeline.run_layer(bt, b)
    torch.cuda.synchronize()
    for name in ("pool_keys", "scores", "pool_ids", "token_ids", "out", "lse"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_fused_select_matches_stage_calls_and_leaves_workspace_zeroed():
    for bt in (ragged_small(seed=41), synth.tiny(device=DEV), synth.single32k(device=DEV, seed=5)):
        a = pipeline.LayerBuffers.alloc(bt)
        b = pipeline.LayerBuffers.alloc(bt)
        pipeline.run_layer(bt, a, fused=True)
        pipeline.run_layer(bt, b, fused=False)
        pipeline.select(bt, a)                      # second call reuses the workspace
        torch.cuda.synchronize()
        for name in ("scores", "pool_ids", "token_ids", "out", "lse"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        hdr = a.ws_select[: 4096 * 4 * bt.Q]
        assert int(hdr.count_nonzero().item()) == 0, "histogram not left zeroed"


def test_select_with_dirty_workspace_falls_back_exactly():
    """A dsa_select workspace that was not zero-filled gives a histogram that does
    not describe the scores; the selection must still be exact (fallback path),
    flagged, and the workspace left zeroed for the next call."""
    for fill in (0xFF, 0x01):
        bt = synth.single32k(device=DEV, seed=91)
        a = pipeline.LayerBuffers.alloc(bt)
        b = pipeline.LayerBuffers.alloc(bt)
        pipeline.compress(bt, a)
        pipeline.compress(bt, b)
        a.ws_select.fill_(fill)
        pipeline.select(bt, a)
        pipeline.select_stages(bt, b)
        torch.cuda.synchronize()
        assert int(a.status.item()) & ops.DEV_HIST_MISMATCH
        for name in ("scores", "pool_ids", "token_ids"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        hdr = a.ws_select[: 4096 * 4 * bt.Q]
        assert int(hdr.count_nonzero().item()) == 0
        a.status.zero_()
        pipeline.select(bt, a)                       # clean again: fast path, no flag
        torch.cuda.synchronize()
        assert int(a.status.item()) == 0
        assert torch.equal(a.pool_ids, b.pool_ids)


def prefill_chunk_small(n_queries, seed, causal=True, T=40000, pad=3, select_k=256):
    """A chunk of queries on one sequence (q_seq absent): the eight-query-group
    form of the tensor-core scoring kernel when there are 64 queries or more.
    Positions cover no complete pool yet, the first pool completing, a new pool
    becoming visible (p*kpool + pad + kpool - 1 and one token earlier) and the
    last token, plus random ones; the groups of eight are ragged inside."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=select_k, out_width=4 * select_k, Hm=64,
                   L=512, dtype="bf16")
    rng = np.random.default_rng(seed)
    edge = [0, pad + 2, pad + 3, pad + 4 * 100 + 2, pad + 4 * 100 + 3, T - 1]
    pos = np.concatenate([edge, rng.integers(0, T, n_queries - len(edge))])
    bt = synth.make_batch(geo, [T], [pad], device=DEV, seed=seed, queries="chunk",
                          q_positions=pos.tolist())
    if not causal:
        bt.q_pos = None
    return bt


@pytest.mark.parametrize("n_queries,causal", [(203, True), (64, True), (63, True), (72, False)])
def test_prefill_chunk_groups_of_eight(n_queries, causal):
    bt = prefill_chunk_small(n_queries, seed=300 + n_queries, causal=causal)
    buf, o = run_and_check(bt)
    if causal:
        fin = torch.isfinite(buf.scores).sum(dim=1).cpu().numpy()
        pos = bt.q_pos.cpu().numpy()
        want = np.clip((pos - 3 + 1) // 4, 0, None)        # complete pools at each position
        assert np.array_equal(fin, np.minimum(want, (40000 - 3) // 4))


def test_prefill_chunk_fused_matches_stage_calls():
    bt = prefill_chunk_small(130, seed=7)
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, a, fused=True)
    pipeline.run_layer(bt, b, fused=False)
    torch.cuda.synchronize()
    for name in ("scores", "pool_ids", "token_ids", "out", "lse"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert int(a.ws_select.count_nonzero().item()) == 0


@pytest.mark.parametrize("Hm,K,W,lengths", [
    (64, 16, 64, [700, 2100]),         # one split of <= 128 rows: output written directly
    (64, 48, 200, [3000, 41, 900]),    # ragged last split (200 = 128 + 72 rows)
    (32, 64, 256, [2500, 1300]),       # 16-head groups on mma.sync (not 64 heads)
    (128, 32, 128, [1800]),            # 16-head groups, 8 groups
])
def test_mla_tensor_core_variants(Hm, K, W, lengths):
    geo = Geometry(D=128, H=32, kpool=4, select_k=K, out_width=W, Hm=Hm, L=512, dtype="bf16")
    bt = synth.make_batch(geo, lengths, [1] * len(lengths), device=DEV, seed=500 + Hm + W)
    run_and_check(bt)


def test_mla_tensor_core_many_queries_merge_kernel():
    """12 queries x 16 splits x 2 head halves: the split partials of many queries
    go through the merge kernel."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512,
                   dtype="bf16")
    rng = np.random.default_rng(12)
    lengths = [int(x) for x in rng.integers(2100, 4200, 12)]
    bt = synth.make_batch(geo, lengths, [0] * 12, device=DEV, seed=612)
    run_and_check(bt)


def _assert_same_outputs(a, b):
    for name in ("pool_keys", "pool_start", "pool_valid", "n_pools", "scores", "pool_ids",
                 "token_ids", "out", "lse", "status"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("decode_form", [False, True])
def test_decode_layer_matches_the_three_calls(decode_form):
    """The fused call writes what compress -> select -> attend write, for a full
    build and for an incremental step.  In the decode form (no query positions:
    every complete pool is visible, as at the last token) the incremental step's
    scoring kernel streams the key tiles below pool_begin before the compress
    kernel has ended."""
    for bt in (ragged_small(seed=51), synth.single32k(device=DEV, seed=52), synth.tiny(device=DEV)):
        if decode_form:
            bt.q_pos = None
        a = pipeline.LayerBuffers.alloc(bt)
        b = pipeline.LayerBuffers.alloc(bt)
        pipeline.decode_layer(bt, a)
        pipeline.run_layer(bt, b)
        torch.cuda.synchronize()
        _assert_same_outputs(a, b)
        begin = (a.n_pools - 1).clamp(min=0).to(torch.int32)
        # new content for each sequence's last complete pool, then one decode step
        for s in range(bt.B):
            lo = int(bt.cu_seqlens[s]) + bt.pads[s] + max(int(a.n_pools[s]) - 1, 0) * bt.geo.kpool
            bt.k[lo:lo + bt.geo.kpool] *= -1
        for buf in (a, b):
            buf.out.zero_()
            buf.scores.fill_(7.0)
        pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=1)
        pipeline.run_layer(bt, b, pool_begin=begin, max_pools=1)
        torch.cuda.synchronize()
        _assert_same_outputs(a, b)
        assert int(a.status.item()) == 0


@pytest.mark.parametrize("decode_form", [False, True])
@pytest.mark.parametrize("step", ["last_pool", "past_last_pool", "half"])
def test_decode_layer_incremental_pool_count_from_the_valid_mask(step, decode_form):
    """Incremental steps on sequences that start with 0, 37, 255, 256 or 1000
    padding tokens, a short fully valid one and an all-padding one.  In the
    decode form (no query positions) the fused call scores the key tiles below
    pool_begin before its compress kernel has ended, with each pool count found
    from the valid mask when the first valid token is among the sequence's
    first 256 tokens (else it reads the count the compress wrote); it must write
    exactly what the three separate calls write."""
    big = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512, dtype="bf16")
    lengths = [3000, 3000, 2900, 3100, 4000, 250, 200]
    pads = [0, 37, 255, 256, 1000, 0, 200]
    bt = synth.make_batch(big, lengths, pads, device=DEV, seed=71)
    if decode_form:
        bt.q_pos = None
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.decode_layer(bt, a)
    pipeline.run_layer(bt, b)
    torch.cuda.synchronize()
    _assert_same_outputs(a, b)
    n = a.n_pools.clone()
    begin = {"last_pool": (n - 1).clamp(min=0), "past_last_pool": n,
             "half": n // 2}[step].to(torch.int32)
    for s in range(bt.B):
        lo = int(bt.cu_seqlens[s]) + bt.pads[s] + max(int(n[s]) - 1, 0) * bt.geo.kpool
        bt.k[lo:lo + bt.geo.kpool] *= -1
    for buf in (a, b):
        buf.out.zero_()
        buf.scores.fill_(7.0)
        buf.status.zero_()
    max_pools = bt.P_ld if step == "half" else 1
    pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=max_pools)
    pipeline.run_layer(bt, b, pool_begin=begin, max_pools=max_pools)
    torch.cuda.synchronize()
    _assert_same_outputs(a, b)
    assert torch.equal(a.n_pools, n)


def test_decode_layer_launches_what_the_three_calls_launch():
    """The library's launch count: the fused call launches as many kernels as
    compress -> select -> attend for a full build, and one fewer for a decode
    step (no query positions, one new pool per sequence), whose compress runs
    inside the scoring kernel; the outputs are the same."""
    bt = ragged_small(seed=54)
    bt.q_pos = None
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    n0 = ops.dsa_kernel_launches()
    pipeline.decode_layer(bt, a)
    n1 = ops.dsa_kernel_launches()
    pipeline.run_layer(bt, b)
    n2 = ops.dsa_kernel_launches()
    torch.cuda.synchronize()
    assert n1 - n0 == n2 - n1 >= 4
    begin = (a.n_pools - 1).clamp(min=0).to(torch.int32)
    pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=1)
    n3 = ops.dsa_kernel_launches()
    pipeline.run_layer(bt, b, pool_begin=begin, max_pools=1)
    torch.cuda.synchronize()
    assert n3 - n2 == n1 - n0 - 1
    assert ops.dsa_kernel_launches() - n3 == n2 - n1
    _assert_same_outputs(a, b)


def test_decode_step_shared_sequence_and_straddling_pools():
    """A decode-form incremental step (the scoring kernel starts before the
    compress ends) with two queries on one sequence, a sequence with no query,
    and recompressed pools that straddle a 128-pool key tile (three pools from
    pool 127): the same outputs as compress -> select -> attend, and the
    oracle's pool keys."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=64, out_width=256, Hm=64, L=512, dtype="bf16")
    bt = synth.make_batch(geo, [3000, 1500, 600, 800], [2, 0, 5, 0], device=DEV, seed=81)
    bt.q_pos = None
    bt.q_seq = torch.tensor([0, 0, 1, 2], dtype=torch.int32, device=DEV)  # sequence 3: no query
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.decode_layer(bt, a)
    pipeline.run_layer(bt, b)
    torch.cuda.synchronize()
    _assert_same_outputs(a, b)
    begin = torch.tensor([127, 300, 126, 10], dtype=torch.int32, device=DEV)
    for s, p0 in enumerate(begin.tolist()):       # new content for the recompressed pools
        lo = int(bt.cu_seqlens[s]) + bt.pads[s] + p0 * geo.kpool
        bt.k[lo:lo + 3 * geo.kpool] *= -1
        bt.gate[lo:lo + 3 * geo.kpool] += 1
    for buf in (a, b):
        buf.scores.fill_(7.0)
    pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=3)
    pipeline.run_layer(bt, b, pool_begin=begin, max_pools=3)
    torch.cuda.synchronize()
    _assert_same_outputs(a, b)
    # complete pools follow the recompressed ones: flagged by both forms alike
    assert int(a.status.item()) == ops.DEV_POOL_UNCOVERED
    o = oracle_inputs(bt)
    par.check_compress(o, a)
    par.check_scores(o, a)
    par.check_topk(a, geo.select_k)


def test_decode_layer_parity_against_the_oracle():
    bt = ragged_small(seed=53)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.decode_layer(bt, buf)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    st = par.check_compress(o, buf)
    _, st2 = par.check_scores(o, buf)
    par.check_topk(buf, bt.geo.select_k)
    st3 = par.check_expand(o, buf)
    st4 = par.check_mla(o, buf)
    assert int(buf.status.item()) == (st | st2 | st3 | st4)


def test_decode_layer_dirty_workspace_falls_back_exactly():
    """In the fused call the attention CTAs select from the scoring kernel's
    histograms; a selection workspace that was not zero-filled must still give
    the exact selection (flagged), and the call leaves the histograms zeroed."""
    for fill in (0xFF, 0x01):
        bt = ragged_small(seed=61)
        a = pipeline.LayerBuffers.alloc(bt)
        b = pipeline.LayerBuffers.alloc(bt)
        a.ws_select.fill_(fill)
        pipeline.decode_layer(bt, a)
        pipeline.run_layer(bt, b, fused=False)
        torch.cuda.synchronize()
        assert int(a.status.item()) & ops.DEV_HIST_MISMATCH
        for name in ("scores", "pool_ids", "token_ids", "out", "lse"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        assert int(a.ws_select[: 4096 * 4 * bt.Q].count_nonzero().item()) == 0
        a.status.zero_()
        pipeline.decode_layer(bt, a)                 # clean again: no flag
        torch.cuda.synchronize()
        assert int(a.status.item()) == 0
        _assert_same_outputs(a, b)


def test_decode_layer_equal_scores():
    """Queries whose index weights are zero score every visible pool 0.0: the
    order among equal scores is pool ascending, in the bin-and-count path (ties
    on chip) and in the exact paths (more ties than fit on chip; more float4
    groups with a tie than the attention kernel stages)."""
    big = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512, dtype="bf16")
    for bt in (ragged_small(seed=62), synth.single32k(device=DEV, seed=63),
               synth.make_batch(big, [70000, 3000], [0, 1], device=DEV, seed=64)):
        bt.weights[0] = 0.0
        a = pipeline.LayerBuffers.alloc(bt)
        b = pipeline.LayerBuffers.alloc(bt)
        pipeline.decode_layer(bt, a)
        pipeline.run_layer(bt, b, fused=False)
        torch.cuda.synchronize()
        _assert_same_outputs(a, b)
        s0 = a.scores[0]
        n0 = int(torch.isfinite(s0).sum().item())
        assert n0 == 0 or bool((s0[torch.isfinite(s0)] == 0).all())
        k = min(bt.geo.select_k, n0)
        ids = a.pool_ids[0].cpu().numpy()
        fin = torch.nonzero(torch.isfinite(s0)).flatten().cpu().numpy()
        assert np.array_equal(ids[:k], fin[:k]) and (ids[k:] == -1).all()
        o = oracle_inputs(bt)
        par.check_topk(a, bt.geo.select_k)
        par.check_mla(o, a)


@pytest.mark.parametrize("tile", [0, 11])
def test_streaming_attention_large_logit_in_a_late_or_first_tile(tile):
    """40 decode queries x 2048 rows run the streaming attention (more than four
    waves of one-tile CTAs).  A selected row aligned with head 0's query, placed
    in tile `tile` of some queries, raises that head's max by far more than the
    lazy-rescale margin (2^8): in a late tile the accumulator is rescaled, in the
    first tile later tiles stay below the reference."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512,
                   dtype="bf16")
    rng = np.random.default_rng(77)
    lengths = [int(x) for x in rng.integers(2100, 3500, 40)]
    bt = synth.make_batch(geo, lengths, [0] * 40, device=DEV, seed=78)
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    for q in (0, 7, 39):
        tok = int(buf.token_ids[q, tile * 128 + 5])
        b = int(bt.q_seq[q])
        row = int(bt.cu_seqlens[b]) + tok
        bt.kv[row] = bt.q_lat[q, 0].to(bt.kv.dtype)
    buf.out.zero_()
    pipeline.attend(bt, buf)
    torch.cuda.synchronize()
    o = oracle_inputs(bt)
    st = par.check_mla(o, buf)
    assert st == 0 and int(buf.status.item()) == 0
    assert float(buf.lse[0, 0]) > float(buf.lse[0, 1]) + 8.0


@pytest.mark.parametrize("seed", [91, 92])
def test_decode_step_fused_compress_shared_and_uncovered_sequences(seed):
    """The decode form whose compress runs inside the scoring kernel (one new
    pool per sequence): two queries on one sequence (both CTAs holding its new
    pool write it), a sequence no query reads (its pool is still written), a
    new pool that is not complete (a sentinel), one at a tile's first pool and
    one mid-tile; the same outputs as compress -> select -> attend, and the
    oracle's pool keys and counts."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=64, out_width=256, Hm=64, L=512, dtype="bf16")
    bt = synth.make_batch(geo, [3000, 1501, 600, 800, 2052], [2, 0, 5, 0, 3], device=DEV,
                          seed=seed)
    bt.q_pos = None
    bt.q_seq = torch.tensor([0, 0, 1, 2, 4], dtype=torch.int32, device=DEV)  # 3: no query
    a = pipeline.LayerBuffers.alloc(bt)
    b = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, a)
    pipeline.run_layer(bt, b)
    torch.cuda.synchronize()
    # pool 128 opens a tile; sequence 1's pool 375 is incomplete (1501 tokens)
    begin = torch.tensor([128, 375, 140, 150, 300], dtype=torch.int32, device=DEV)
    for s_, p0 in enumerate(begin.tolist()):      # new content for the recompressed pool
        lo = int(bt.cu_seqlens[s_]) + bt.pads[s_] + p0 * geo.kpool
        hi = min(lo + geo.kpool, int(bt.cu_seqlens[s_ + 1]))
        bt.k[lo:hi] *= -1
        bt.gate[lo:hi] += 1
    n0 = ops.dsa_kernel_launches()
    pipeline.decode_layer(bt, a, pool_begin=begin, max_pools=1)
    n1 = ops.dsa_kernel_launches()
    pipeline.run_layer(bt, b, pool_begin=begin, max_pools=1)
    n2 = ops.dsa_kernel_launches()
    torch.cuda.synchronize()
    assert n1 - n0 == n2 - n1 - 1                       # the compress ran inside the scoring
    _assert_same_outputs(a, b)
    assert torch.equal(a.pool_keys, b.pool_keys) and torch.equal(a.n_pools, b.n_pools)
    assert torch.equal(a.pool_start, b.pool_start) and torch.equal(a.pool_valid, b.pool_valid)
    o = oracle_inputs(bt)
    par.check_compress(o, a)
