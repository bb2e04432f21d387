"""The C ABI on a machine without a GPU: the library loads, exports every symbol
include/dsa.h declares, and rejects bad arguments on the host before any CUDA
call (so these calls are safe without a device)."""
import ctypes
import os
import re

import pytest

from sparse_attention_indexer_kpool_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|uint64_t|const char\*)\s+(dsa_\w+)\s*\(",
                                 text, re.M)))


def header_define(name):
    m = re.search(rf"#define\s+{name}\s+(\d+)", open(HEADER).read())
    return int(m.group(1))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code in range(6):
        s = lib.dsa_status_string(code).decode()
        assert s.startswith("DSA_")
    assert lib.dsa_status_string(999).decode() == "DSA_ERR_UNKNOWN"
    assert lib.dsa_version() >= 10000


ERR = {n: header_define(n) for n in ("DSA_OK", "DSA_ERR_INVALID_ARG", "DSA_ERR_MISALIGNED",
                                     "DSA_ERR_UNSUPPORTED", "DSA_ERR_WORKSPACE")}
A = 0x10000          # a 16-byte-aligned fake address; never dereferenced by these calls


def compress(lib, **kw):
    a = dict(k=A, gate=A, valid=A, ape=A, g=A, b=A, eps=1e-5, cu=A, cap=A, begin=None, B=1, D=128,
             kpool=4, max_pools=8, dtype=0, pk=A, ps=A, pv=A, np_=A, st=None, stream=None)
    a.update(kw)
    return lib.dsa_kpool_compress(a["k"], a["gate"], a["valid"], a["ape"], a["g"], a["b"],
                                  a["eps"], a["cu"], a["cap"], a["begin"], a["B"], a["D"],
                                  a["kpool"], a["max_pools"], a["dtype"], a["pk"], a["ps"], a["pv"],
                                  a["np_"], a["st"], a["stream"])


def test_compress_validation(lib):
    assert compress(lib, kpool=9) == ERR["DSA_ERR_INVALID_ARG"]     # refuse, never truncate
    assert compress(lib, kpool=0) == ERR["DSA_ERR_INVALID_ARG"]
    assert compress(lib, dtype=7) == ERR["DSA_ERR_INVALID_ARG"]
    assert compress(lib, eps=float("nan")) == ERR["DSA_ERR_INVALID_ARG"]
    assert compress(lib, D=96) == ERR["DSA_ERR_UNSUPPORTED"]
    assert compress(lib, k=None) == ERR["DSA_ERR_INVALID_ARG"]
    assert compress(lib, k=A + 8) == ERR["DSA_ERR_MISALIGNED"]
    assert compress(lib, B=0) == ERR["DSA_OK"]                        # empty batch: no-op
    assert compress(lib, max_pools=-1) == ERR["DSA_ERR_INVALID_ARG"]


def scores_call(lib, **kw):
    a = dict(q=A, w=A, scale=0.088, pk=A, rows=256, ps=A, pv=A, np_=A, cap=A, qs=A, qp=None, Q=4,
             B=4, H=32, D=128, kpool=4, P_ld=64, dtype=0, out=A, st=None, stream=None)
    a.update(kw)
    return lib.dsa_index_scores(a["q"], a["w"], a["scale"], a["pk"], a["rows"], a["ps"], a["pv"],
                                a["np_"],
                                a["cap"], a["qs"], a["qp"], a["Q"], a["B"], a["H"], a["D"],
                                a["kpool"], a["P_ld"], a["dtype"], a["out"], a["st"], a["stream"])


def test_index_scores_validation(lib):
    assert scores_call(lib, kpool=9) == ERR["DSA_ERR_INVALID_ARG"]
    assert scores_call(lib, scale=0.0) == ERR["DSA_ERR_INVALID_ARG"]
    assert scores_call(lib, scale=float("inf")) == ERR["DSA_ERR_INVALID_ARG"]
    assert scores_call(lib, H=65) == ERR["DSA_ERR_UNSUPPORTED"]
    assert scores_call(lib, D=100) == ERR["DSA_ERR_UNSUPPORTED"]
    assert scores_call(lib, qp=A, ps=None) == ERR["DSA_ERR_INVALID_ARG"]   # causal needs starts
    assert scores_call(lib, q=A + 4) == ERR["DSA_ERR_MISALIGNED"]
    assert scores_call(lib, P_ld=0) == ERR["DSA_ERR_INVALID_ARG"]
    assert scores_call(lib, rows=0) == ERR["DSA_ERR_INVALID_ARG"]      # empty pool cache
    assert scores_call(lib, Q=0) == ERR["DSA_OK"]


def test_topk_validation(lib):
    # the histogram and candidate lists live on chip: no workspace is needed
    assert lib.dsa_topk_pools_workspace_size(4, 1000, 16) == 0
    assert lib.dsa_topk_pools(A, 4, 1000, 0, A, None, 0, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert lib.dsa_topk_pools(A, 4, 0, 16, A, None, 0, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert lib.dsa_topk_pools(A, 4, 1000, 4097, A, None, 0, None) == ERR["DSA_ERR_UNSUPPORTED"]
    assert lib.dsa_topk_pools(A + 2, 4, 1000, 16, A, None, 0, None) == ERR["DSA_ERR_MISALIGNED"]
    assert lib.dsa_topk_pools(None, 4, 1000, 16, A, None, 0, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert lib.dsa_topk_pools(A, 0, 1000, 16, A, None, 0, None) == ERR["DSA_OK"]


def test_rejected_and_empty_calls_launch_nothing(lib):
    n = lib.dsa_kernel_launches()
    assert lib.dsa_topk_pools(A, 4, 1000, 0, A, None, 0, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert lib.dsa_topk_pools(A, 0, 1000, 16, A, None, 0, None) == ERR["DSA_OK"]  # no queries
    assert lib.dsa_kernel_launches() == n


def test_failure_drill_setting(lib):
    """The drill switch takes 0 and the defined drills, and refuses others."""
    for name in ("DSA_DRILL_SKIP_ARM", "DSA_DRILL_SKIP_PV_COMMIT"):
        assert lib.dsa_set_failure_drill(header_define(name)) == ERR["DSA_OK"]
    assert lib.dsa_set_failure_drill(0) == ERR["DSA_OK"]
    assert lib.dsa_set_failure_drill(7) == ERR["DSA_ERR_INVALID_ARG"]
    assert lib.dsa_set_failure_drill(-1) == ERR["DSA_ERR_INVALID_ARG"]


def test_expand_validation(lib):
    f = lib.dsa_expand_selection
    assert f(A, A, A, A, 2, 2, 8, 4, 31, A, None, None) == ERR["DSA_ERR_INVALID_ARG"]  # W < K*kp
    assert f(A, A, A, A, 2, 2, 8, 9, 80, A, None, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(A, A, A, A, 2, 2, 8, 4, 32, None, None, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(A, A, A, A, 2, 2, 8, 4, 32, A + 2, None, None) == ERR["DSA_ERR_MISALIGNED"]
    assert f(A, A, A, A, 0, 2, 8, 4, 32, A, None, None) == ERR["DSA_OK"]


def test_mla_validation(lib):
    f = lib.dsa_mla_selected_decode
    ws = lib.dsa_mla_selected_decode_workspace_size(4, 64, 512, 2048, 0)   # split partials
    assert ws > 0
    assert lib.dsa_mla_selected_decode_workspace_size(4, 64, 512, 2048, 1) == 0
    assert lib.dsa_mla_selected_decode_workspace_size(4096, 64, 512, 2048, 0) == 0   # no split
    assert f(A, A, A, A, A, 4, 4, 64, 500, 2048, 0.04, 0, A, A, A, ws, None, None) \
        == ERR["DSA_ERR_UNSUPPORTED"]
    assert f(A, A, A, A, A, 4, 4, 64, 512, 2048, 0.04, 0, A, A, A, ws - 1, None, None) \
        == ERR["DSA_ERR_WORKSPACE"]
    assert f(A, A, A, A, A, 4, 4, 64, 512, 2048, 0.04, 0, A + 8, A, A, ws, None, None) \
        == ERR["DSA_ERR_MISALIGNED"]
    assert f(A, A, A, A, A, 4, 4, 64, 512, 2048, float("nan"), 0, A, A, A, ws, None, None) \
        == ERR["DSA_ERR_INVALID_ARG"]
    assert f(A, A, A, A, A, 0, 4, 64, 512, 2048, 0.04, 0, A, A, A, ws, None, None) == ERR["DSA_OK"]


def test_mla_paged_validation(lib):
    f = lib.dsa_mla_paged_decode
    fp8 = header_define("DSA_FP8_E4M3")
    assert header_define("DSA_DEV_BAD_PAGE") == 256
    ws = lib.dsa_mla_paged_decode_workspace_size(4, 64, 512, 2048, 0, fp8)   # tensor cores, split
    assert ws > 0 and ws == lib.dsa_mla_paged_decode_workspace_size(4, 64, 512, 2048, 0, 0)
    assert lib.dsa_mla_paged_decode_workspace_size(4, 64, 512, 2048, 0, 1) == 0   # generic kernel
    assert lib.dsa_mla_paged_decode_workspace_size(4, 32, 512, 2048, 0, fp8) == 0

    def kv(**kw):
        a = dict(pages=A, row_scale=A, block_table=A, seq_lens=A, n_pages=100, page_size=64,
                 max_pages=8, kv_dtype=fp8)
        a.update(kw)
        return ctypes.byref(_lib.PagedKv(a["pages"], a["row_scale"], a["block_table"],
                                         a["seq_lens"], a["n_pages"], a["page_size"],
                                         a["max_pages"], a["kv_dtype"]))

    def call(k, Q=4, L=512, sm=0.04, out=A, ws_bytes=ws, q_seq=A):
        return f(A, k, q_seq, A, Q, 4, 64, L, 2048, sm, 0, out, A, A, ws_bytes, None, None)

    assert call(kv(), ws_bytes=ws - 1) == ERR["DSA_ERR_WORKSPACE"]
    assert call(kv(row_scale=None)) == ERR["DSA_ERR_INVALID_ARG"]          # E4M3 needs scales
    assert call(kv(kv_dtype=0)) == ERR["DSA_ERR_INVALID_ARG"]              # bf16 takes none
    assert call(kv(kv_dtype=7)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(page_size=0)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(n_pages=0)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(max_pages=0)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(block_table=None)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(seq_lens=None)) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(n_pages=1 << 20, page_size=1 << 12)) == ERR["DSA_ERR_UNSUPPORTED"]
    assert call(kv(pages=A + 8)) == ERR["DSA_ERR_MISALIGNED"]
    assert call(kv(block_table=A + 2)) == ERR["DSA_ERR_MISALIGNED"]
    assert call(kv(), out=A + 8) == ERR["DSA_ERR_MISALIGNED"]
    assert call(kv(), L=500) == ERR["DSA_ERR_UNSUPPORTED"]
    assert call(kv(), sm=float("inf")) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(A, None, A, A, 4, 4, 64, 512, 2048, 0.04, 0, A, A, A, ws, None, None) \
        == ERR["DSA_ERR_INVALID_ARG"]
    assert call(kv(), Q=0) == ERR["DSA_OK"]                                   # nothing to do


def test_select_validation(lib):
    f = lib.dsa_select
    ws = lib.dsa_select_workspace_size(4, 1000, 16)
    assert ws > 0
    args = lambda **kw: [kw.get("q", A), A, kw.get("scale", 0.1), A, kw.get("rows", 256),
                         A, A, A, A, A, None,
                         kw.get("Q", 4), 4, 32, 128, kw.get("kpool", 4), 1000,
                         kw.get("k", 16), kw.get("W", 64), 0, A, A, A, kw.get("ws", A),
                         kw.get("wsb", ws), None, None]
    assert f(*args(kpool=9)) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(*args(W=63)) == ERR["DSA_ERR_INVALID_ARG"]                 # out_width < K*kpool
    assert f(*args(k=5000, W=20000)) == ERR["DSA_ERR_UNSUPPORTED"]
    assert f(*args(wsb=ws - 1)) == ERR["DSA_ERR_WORKSPACE"]
    assert f(*args(ws=None)) == ERR["DSA_ERR_WORKSPACE"]
    assert f(*args(q=A + 2)) == ERR["DSA_ERR_MISALIGNED"]
    assert f(*args(rows=0)) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(*args(Q=0)) == ERR["DSA_OK"]


def test_python_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    from sparse_attention_indexer_kpool_gb300 import ops
    x = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        ops._ptr(x, torch.float32, "x")                          # CPU tensor refused


def test_decode_layer_validation(lib):
    """All three stages are checked on the host before anything is launched."""
    def args(**kw):
        a = _lib.DecodeLayerArgs(k=A, gate=A, valid=A, ape=A, ln_gamma=A, ln_beta=A, ln_eps=1e-5,
                                 cu_seqlens=A, pool_begin=A, max_pools=1, pool_keys=A,
                                 pool_rows=256, pool_start=A, pool_valid=A, n_pools=A,
                                 cu_pool_cap=A, q=A, weights=A, scale=0.088, q_seq=A, q_pos=None,
                                 q_lat=A, kv_latent=A, sm_scale=0.044, Q=4, B=4, H=32, D=128,
                                 kpool=4, P_ld=64, select_k=16, out_width=64, Hm=64, L=512,
                                 dtype=0, scores=A, pool_ids=A, token_ids=A, out=A, lse=A,
                                 ws_select=A, ws_select_bytes=1 << 20, ws_mla=A,
                                 ws_mla_bytes=1 << 24, status_dev=None)
        for n, v in kw.items():
            setattr(a, n, v)
        return ctypes.byref(a)
    f = lib.dsa_decode_layer
    assert f(None, None) == ERR["DSA_ERR_INVALID_ARG"]
    assert f(args(kpool=9), None) == ERR["DSA_ERR_INVALID_ARG"]            # compress and select
    assert f(args(k=None), None) == ERR["DSA_ERR_INVALID_ARG"]             # compress input
    assert f(args(q=A + 8), None) == ERR["DSA_ERR_MISALIGNED"]             # select input
    assert f(args(ws_select_bytes=1), None) == ERR["DSA_ERR_WORKSPACE"]
    assert f(args(out_width=63), None) == ERR["DSA_ERR_INVALID_ARG"]       # W < K * kpool
    assert f(args(kv_latent=None), None) == ERR["DSA_ERR_INVALID_ARG"]     # attention input
    assert f(args(L=500), None) == ERR["DSA_ERR_UNSUPPORTED"]              # attention geometry
    s_sel, s_mla = ctypes.c_size_t(), ctypes.c_size_t()
    tot = lib.dsa_decode_layer_workspace_size(args(Q=4, P_ld=1000, out_width=2048, select_k=512),
                                              ctypes.byref(s_sel), ctypes.byref(s_mla))
    assert s_sel.value == lib.dsa_select_workspace_size(4, 1000, 512)
    assert s_mla.value == lib.dsa_mla_selected_decode_workspace_size(4, 64, 512, 2048, 0)
    assert tot == s_sel.value + s_mla.value


def test_indexer_project_validation(lib):
    f = lib.dsa_indexer_project
    def call(**kw):
        a = dict(x=A, w=A, cq=A, wq=A, wuk=A, T=4, hidden=6144, q_rank=2048, H=32, D=128, Hm=64,
                 nope=192, L=512, ws_scale=0.17, rows=None, k=A, g=A, w_out=A, q=A, qn=A, ql=A,
                 ws=A, ws_bytes=1 << 30, st=None)
        a.update(kw)
        return f(a["x"], a["w"], a["cq"], a["wq"], a["wuk"], a["T"], a["hidden"], a["q_rank"],
                 a["H"], a["D"], a["Hm"], a["nope"], a["L"], a["ws_scale"], a["rows"], a["k"],
                 a["g"], a["w_out"], a["q"], a["qn"], a["ql"], a["ws"], a["ws_bytes"], a["st"],
                 None)
    size = lib.dsa_indexer_project_workspace_size
    assert size(4, 6144, 2048, 32, 128, 64, 192, 512) > 0        # 4 tokens: split contractions
    assert size(0, 6144, 2048, 32, 128, 64, 192, 512) == 0
    assert call(nope=100) == ERR["DSA_ERR_UNSUPPORTED"]           # not whole 64-wide stages
    assert call(hidden=6148) == ERR["DSA_ERR_UNSUPPORTED"]        # row stride not 16 bytes
    assert call(H=0) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(ws_scale=float("nan")) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(x=None) == ERR["DSA_ERR_INVALID_ARG"]
    assert call(x=A + 8) == ERR["DSA_ERR_MISALIGNED"]
    assert call(w_out=A + 2) == ERR["DSA_ERR_MISALIGNED"]
    assert call(ws=None, ws_bytes=0) == ERR["DSA_ERR_WORKSPACE"]
    assert call(ws_bytes=16) == ERR["DSA_ERR_WORKSPACE"]
    n = lib.dsa_kernel_launches()
    assert call(T=0) == ERR["DSA_OK"]                             # no tokens: no-op
    assert lib.dsa_kernel_launches() == n
