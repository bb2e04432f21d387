"""The selected-row attention on a paged latent cache (module glm5next_dsa,
Modules, attend: the paged decode, and Constants, KERNEL_KV_LORA_DIM: its fp8
twin).  bf16 / fp32 pages give exactly the contiguous attention (the same
kernel reads the same rows); E4M3 pages match the oracle; blocks past the table
and pages outside the cache are flagged and skipped."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
from sparse_attention_indexer_kpool_gb300.synth import Geometry
from tests._parity import mla_tol
from tests._util import npf, npi

pytestmark = pytest.mark.gpu
DEV = "cuda"


def ragged_small(seed):
    geo = Geometry(D=128, H=32, kpool=4, select_k=64, out_width=320, Hm=64, L=512, dtype="bf16")
    return synth.make_batch(geo, [1203, 0, 3, 23, 50, 2500], [5, 0, 0, 0, 50, 1], device=DEV,
                            seed=seed)


def run_paged(bt, token_ids, pc):
    Q, Hm, L = bt.q_lat.shape
    out = torch.full((Q, Hm, L), 7.0, dtype=bt.q_lat.dtype, device=DEV)
    lse = torch.full((Q, Hm), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    n = ops.mla_paged_workspace_bytes(bt.q_lat, pc.pages, token_ids.shape[1])
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
    ops.dsa_mla_paged_decode(bt.q_lat, pc.pages, pc.row_scale, pc.block_table, pc.seq_lens,
                             pc.page_size, bt.q_seq, token_ids, bt.sm_scale, out, lse, ws, st)
    torch.cuda.synchronize()
    return out, lse, int(st.item())


def oracle_paged(bt, token_ids, pc, block_table=None, seq_lens=None):
    e4 = pc.row_scale is not None
    pages = pc.pages.view(torch.uint8).cpu().numpy() if e4 else npf(pc.pages)
    kd = "fp8_e4m3" if e4 else ("bf16" if pc.pages.dtype == torch.bfloat16 else "f32")
    return oracle.mla_paged_decode(
        npf(bt.q_lat), pages, npf(pc.row_scale) if e4 else None, kd,
        npi(pc.block_table if block_table is None else block_table),
        npi(pc.seq_lens if seq_lens is None else seq_lens), pc.page_size, npi(bt.q_seq),
        npi(token_ids), bt.sm_scale, bt.geo.dtype)


def assert_close(out, lse, ref, dtype):
    ref_out, ref_lse, _ = ref
    got = out.cpu().double().numpy()
    err = np.abs(got - ref_out)
    assert np.all(err <= mla_tol(ref_out, dtype)), f"attention out error {err.max():.3g}"
    lse = lse.cpu().double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.abs(lse[fin] - ref_lse[fin]) <= 1e-3 * np.maximum(1.0, np.abs(ref_lse[fin])))


def contiguous(bt):
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    return buf


@pytest.mark.parametrize("which", ["ragged_small", "single32k", "tiny"])
def test_paged_rows_give_exactly_the_contiguous_attention(which):
    bt = {"ragged_small": lambda: ragged_small(71), "single32k": lambda: synth.single32k(DEV, 72),
          "tiny": lambda: synth.tiny(DEV)}[which]()
    buf = contiguous(bt)
    for i, page_size in enumerate((64, 16, 1)):
        pc = synth.paged_cache(bt.kv, bt.cu_seqlens, page_size, seed=80 + i)
        out, lse, st = run_paged(bt, buf.token_ids, pc)
        assert st == 0
        assert torch.equal(out, buf.out), page_size
        assert torch.equal(lse, buf.lse), page_size


@pytest.mark.parametrize("which", ["ragged_small", "single32k", "tiny"])
def test_paged_e4m3_rows_match_the_oracle(which):
    bt = {"ragged_small": lambda: ragged_small(73), "single32k": lambda: synth.single32k(DEV, 74),
          "tiny": lambda: synth.tiny(DEV)}[which]()
    buf = contiguous(bt)
    for page_size in (64, 5):
        pc = synth.paged_cache(bt.kv, bt.cu_seqlens, page_size, e4m3=True, seed=90)
        out, lse, st = run_paged(bt, buf.token_ids, pc)
        ref = oracle_paged(bt, buf.token_ids, pc)
        assert st == ref[2]
        assert_close(out, lse, ref, bt.geo.dtype)


@pytest.mark.parametrize("e4m3", [False, True])
def test_paged_bad_pages_and_tokens_are_flagged_and_skipped(e4m3):
    bt = ragged_small(75)
    buf = contiguous(bt)
    pc = synth.paged_cache(bt.kv, bt.cu_seqlens, 16, e4m3=e4m3, seed=91)
    n_pages = pc.pages.shape[0] // pc.page_size
    tok = buf.token_ids.clone()
    # query 0 (sequence 0): a block with no page, a page past the cache
    b0 = int(bt.q_seq[0]) if bt.q_seq is not None else 0
    t0, t1 = int(tok[0, 0]), int(tok[0, 4])
    table = pc.block_table.clone()
    table[b0, t0 // 16] = -1
    table[b0, t1 // 16] = n_pages + 5
    bad = synth.PagedCache(pc.pages, pc.row_scale, table, pc.seq_lens, pc.page_size)
    out, lse, st = run_paged(bt, tok, bad)
    ref = oracle_paged(bt, tok, bad)
    assert st == ref[2] and st & ops.DEV_BAD_PAGE
    assert_close(out, lse, ref, bt.geo.dtype)
    # a table too narrow for the longest sequence, and a sequence shorter than its ids
    narrow = pc.block_table[:, :40].contiguous()
    lens = pc.seq_lens.clone()
    lens[int(bt.q_seq[-1])] = 100
    short = synth.PagedCache(pc.pages, pc.row_scale, narrow, lens, pc.page_size)
    out, lse, st = run_paged(bt, tok, short)
    ref = oracle_paged(bt, tok, short)
    assert st == ref[2] and st & ops.DEV_BAD_PAGE and st & ops.DEV_BAD_TOKEN
    assert_close(out, lse, ref, bt.geo.dtype)


@pytest.mark.parametrize("e4m3", [False, True])
def test_paged_many_queries_on_the_tensor_cores(e4m3):
    """64 decode queries x 2048 rows: more than four waves of attention CTAs
    (the contiguous call takes its other tensor-core kernel there; the paged one
    keeps the tcgen05 kernel), sampled queries against the oracle."""
    geo = Geometry(D=128, H=32, kpool=4, select_k=512, out_width=2048, Hm=64, L=512,
                   dtype="bf16")
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(2100, 4000, 64)]
    bt = synth.make_batch(geo, lengths, [0] * 64, device=DEV, seed=93)
    buf = contiguous(bt)
    pc = synth.paged_cache(bt.kv, bt.cu_seqlens, 64, e4m3=e4m3, seed=94)
    out, lse, st = run_paged(bt, buf.token_ids, pc)
    assert st == 0
    rows = [0, 17, 40, 63]
    idx = torch.as_tensor(rows, device=DEV)
    sub = synth.Batch(**{**bt.__dict__, "q_lat": bt.q_lat[idx], "q_seq": bt.q_seq[idx]})
    ref = oracle_paged(sub, buf.token_ids[idx], pc)
    assert_close(out[idx], lse[idx], ref, "bf16")


def test_paged_e4m3_long262k_layer():
    """The 262k decode layer (4 x 262144 tokens, 2048 selected rows per query) on
    an E4M3 cache in pages of 64 rows, every query against the oracle."""
    bt = synth.long262k(DEV, layer=0)
    buf = contiguous(bt)
    pc = synth.paged_cache(bt.kv, bt.cu_seqlens, 64, e4m3=True, seed=92)
    del bt.k, bt.gate
    out, lse, st = run_paged(bt, buf.token_ids, pc)
    assert st == 0
    ref = oracle_paged(bt, buf.token_ids, pc)
    assert_close(out, lse, ref, bt.geo.dtype)


@pytest.mark.parametrize("Q", [4, 320])  # the one-tile kernel; the streaming kernel
def test_paged_e4m3_every_code_decodes_exactly(Q):
    """Every E4M3 code but the two NaNs (both zeros, the subnormals, the largest
    normals, both signs) through a one-row selection: the softmax weight of the
    one row is exactly 1, so each output is the code's value times the row's
    scale.  With a power-of-two scale bf16 holds that product exactly (an E4M3
    value has at most four significant bits), so the kernels' outputs must equal
    the oracle's decode bit for bit."""
    L, Hm, page_size, W = 512, 64, 16, 128
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)  # 254 codes
    n_blocks = -(-Q // page_size)
    n_rows = (n_blocks + 1) * page_size
    pages = np.zeros((n_rows, L), np.uint8)
    for r in range(n_rows):  # row r: every code, rotated by r
        pages[r] = np.resize(np.roll(codes, r), L)
    scale = 0.125
    g = torch.Generator(device="cpu").manual_seed(95)
    q_lat = torch.randn((Q, Hm, L), generator=g).to(torch.bfloat16).to(DEV)
    perm = torch.randperm(n_blocks + 1, generator=g)[:n_blocks].to(torch.int32)
    block_table = torch.full((1, n_blocks + 1), -1, dtype=torch.int32)
    block_table[0, :n_blocks] = perm
    token_ids = torch.full((Q, W), -1, dtype=torch.int32)
    token_ids[:, 0] = torch.arange(Q, dtype=torch.int32)   # query q selects token q only
    pc = synth.PagedCache(torch.from_numpy(pages).to(DEV).view(torch.float8_e4m3fn),
                          torch.full((n_rows,), scale, dtype=torch.float32, device=DEV),
                          block_table.to(DEV), torch.tensor([Q], dtype=torch.int32, device=DEV),
                          page_size)
    out = torch.full((Q, Hm, L), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((Q, Hm), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    n = ops.mla_paged_workspace_bytes(q_lat, pc.pages, W)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
    ops.dsa_mla_paged_decode(q_lat, pc.pages, pc.row_scale, pc.block_table, pc.seq_lens, page_size,
                             torch.zeros(Q, dtype=torch.int32, device=DEV), token_ids.to(DEV),
                             0.05, out, lse, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the cache row of token q: page block_table[q // page_size], slot q % page_size
    rows = perm.numpy()[np.arange(Q) // page_size].astype(np.int64) * page_size + np.arange(Q) % page_size
    want = oracle.fp8_e4m3_decode(pages[rows]) * scale               # [Q, L], exact
    got = out.float().cpu().double().numpy()
    assert np.array_equal(got, np.broadcast_to(want[:, None, :], got.shape))
    assert torch.isfinite(lse).all()
