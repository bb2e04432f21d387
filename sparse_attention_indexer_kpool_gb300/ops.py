"""Python binding of the libdsa C ABI: same names, torch tensors in.

Argument marshalling only: each function checks device / dtype / contiguity,
passes data pointers and the current CUDA stream to the C entry point of the
same name, and raises ``DsaError`` on a non-zero return code.  Every step of
the path runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

DSA_BF16, DSA_F32, DSA_FP8_E4M3 = 0, 1, 2
DEV_BAD_TOKEN, DEV_POOL_OVERFLOW, DEV_POOL_UNCOVERED = 1, 2, 4
DEV_BAD_POOL_ID, DEV_BAD_QSEQ, DEV_POOL_RANGE, DEV_TIMEOUT = 8, 16, 32, 64
DEV_HIST_MISMATCH, DEV_BAD_PAGE = 128, 256


class DsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.load().dsa_status_string(code).decode()
        super().__init__(f"{fn}: {msg} (code {code})")
        self.code = code


def _dtype_tag(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    if t.dtype == torch.float32:
        return DSA_F32
    raise TypeError(f"activation dtype must be bfloat16 or float32, got {t.dtype}")


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _pool_rows(pool_keys) -> int:
    if pool_keys.dim() != 2:
        raise ValueError("pool_keys must be [pool_rows, D]")
    return pool_keys.shape[0]


def _check(fn, code):
    if code != 0:
        raise DsaError(fn, code)


def dsa_kpool_compress(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens, cu_pool_cap,
                       pool_begin, kpool, max_pools, pool_keys, pool_start, pool_valid, n_pools,
                       status=None, stream=None):
    act = k.dtype
    B = cu_seqlens.numel() - 1
    code = _lib.load().dsa_kpool_compress(
        _ptr(k, act, "k"), _ptr(gate, act, "gate"), _ptr(valid, torch.uint8, "valid"),
        _ptr(ape, torch.float32, "ape"), _ptr(ln_gamma, act, "ln_gamma"),
        _ptr(ln_beta, act, "ln_beta"), float(ln_eps), _ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        _ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), _ptr(pool_begin, torch.int32, "pool_begin"),
        B, k.shape[-1], int(kpool), int(max_pools), _dtype_tag(k),
        _ptr(pool_keys, act, "pool_keys"), _ptr(pool_start, torch.int32, "pool_start"),
        _ptr(pool_valid, torch.uint8, "pool_valid"), _ptr(n_pools, torch.int32, "n_pools"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check("dsa_kpool_compress", code)


def dsa_index_scores(q, weights, scale, pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap,
                     q_seq, q_pos, kpool, scores, status=None, stream=None):
    Q, H, D = q.shape
    act = q.dtype
    code = _lib.load().dsa_index_scores(
        _ptr(q, act, "q"), _ptr(weights, torch.float32, "weights"), float(scale),
        _ptr(pool_keys, act, "pool_keys"), _pool_rows(pool_keys),
        _ptr(pool_start, torch.int32, "pool_start"),
        _ptr(pool_valid, torch.uint8, "pool_valid"), _ptr(n_pools, torch.int32, "n_pools"),
        _ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), _ptr(q_seq, torch.int32, "q_seq"),
        _ptr(q_pos, torch.int32, "q_pos"), Q, cu_pool_cap.numel() - 1, H, D, int(kpool),
        scores.shape[-1], _dtype_tag(q), _ptr(scores, torch.float32, "scores"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check("dsa_index_scores", code)


def topk_workspace_bytes(Q, P_ld, select_k) -> int:
    return int(_lib.load().dsa_topk_pools_workspace_size(Q, P_ld, select_k))


def dsa_topk_pools(scores, select_k, pool_ids, workspace, stream=None):
    Q, P_ld = scores.shape
    code = _lib.load().dsa_topk_pools(
        _ptr(scores, torch.float32, "scores"), Q, P_ld, int(select_k),
        _ptr(pool_ids, torch.int32, "pool_ids"), _ptr(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream))
    _check("dsa_topk_pools", code)


def dsa_expand_selection(pool_ids, pool_start, cu_pool_cap, q_seq, kpool, token_ids, status=None,
                         stream=None):
    Q, K = pool_ids.shape
    code = _lib.load().dsa_expand_selection(
        _ptr(pool_ids, torch.int32, "pool_ids"), _ptr(pool_start, torch.int32, "pool_start"),
        _ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), _ptr(q_seq, torch.int32, "q_seq"), Q,
        cu_pool_cap.numel() - 1, K, int(kpool), token_ids.shape[-1],
        _ptr(token_ids, torch.int32, "token_ids"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_expand_selection", code)


def mla_workspace_bytes(Q, Hm, L, out_width, dtype_tag) -> int:
    return int(_lib.load().dsa_mla_selected_decode_workspace_size(Q, Hm, L, out_width, dtype_tag))


def dsa_mla_selected_decode(q_lat, kv_latent, cu_seqlens, q_seq, token_ids, sm_scale, out, lse,
                            workspace=None, status=None, stream=None):
    Q, Hm, L = q_lat.shape
    act = q_lat.dtype
    code = _lib.load().dsa_mla_selected_decode(
        _ptr(q_lat, act, "q_lat"), _ptr(kv_latent, act, "kv_latent"),
        _ptr(cu_seqlens, torch.int32, "cu_seqlens"), _ptr(q_seq, torch.int32, "q_seq"),
        _ptr(token_ids, torch.int32, "token_ids"), Q, cu_seqlens.numel() - 1, Hm, L,
        token_ids.shape[-1], float(sm_scale), _dtype_tag(q_lat), _ptr(out, act, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_mla_selected_decode", code)


def _kv_tag(pages: torch.Tensor) -> int:
    if pages.dtype == torch.bfloat16:
        return DSA_BF16
    if pages.dtype == torch.float32:
        return DSA_F32
    if pages.dtype in (torch.float8_e4m3fn, torch.uint8):
        return DSA_FP8_E4M3
    raise TypeError(f"pages must be bfloat16, float32 or float8_e4m3fn, got {pages.dtype}")


def mla_paged_workspace_bytes(q_lat, pages, out_width) -> int:
    Q, Hm, L = q_lat.shape
    return int(_lib.load().dsa_mla_paged_decode_workspace_size(
        Q, Hm, L, int(out_width), _dtype_tag(q_lat), _kv_tag(pages)))


def dsa_mla_paged_decode(q_lat, pages, row_scale, block_table, seq_lens, page_size, q_seq,
                         token_ids, sm_scale, out, lse, workspace=None, status=None, stream=None):
    """``pages`` [n_pages * page_size, L] (bf16, fp32, or float8_e4m3fn / uint8 codes with
    ``row_scale`` [n_pages * page_size] fp32); ``block_table`` [B, max_pages] int32."""
    Q, Hm, L = q_lat.shape
    if pages.dim() != 2 or pages.shape[1] != L or pages.shape[0] % int(page_size) != 0:
        raise ValueError("pages must be [n_pages * page_size, L]")
    if block_table.dim() != 2 or seq_lens.numel() != block_table.shape[0]:
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B]")
    act = q_lat.dtype
    kv = _lib.PagedKv(_ptr(pages, pages.dtype, "pages"), _ptr(row_scale, torch.float32, "row_scale"),
                      _ptr(block_table, torch.int32, "block_table"),
                      _ptr(seq_lens, torch.int32, "seq_lens"), pages.shape[0] // int(page_size),
                      int(page_size), block_table.shape[1], _kv_tag(pages))
    code = _lib.load().dsa_mla_paged_decode(
        _ptr(q_lat, act, "q_lat"), ctypes.byref(kv), _ptr(q_seq, torch.int32, "q_seq"),
        _ptr(token_ids, torch.int32, "token_ids"), Q, block_table.shape[0], Hm, L,
        token_ids.shape[-1], float(sm_scale), _dtype_tag(q_lat), _ptr(out, act, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_mla_paged_decode", code)


def select_workspace_bytes(Q, P_ld, select_k) -> int:
    return int(_lib.load().dsa_select_workspace_size(Q, P_ld, select_k))


def dsa_select(q, weights, scale, pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap, q_seq,
               q_pos, kpool, scores, pool_ids, token_ids, workspace, status=None, stream=None):
    """index_scores -> topk_pools -> expand_selection; ``workspace`` must be a
    zero-filled uint8 tensor before its first use (every call leaves it zeroed)."""
    Q, H, D = q.shape
    act = q.dtype
    code = _lib.load().dsa_select(
        _ptr(q, act, "q"), _ptr(weights, torch.float32, "weights"), float(scale),
        _ptr(pool_keys, act, "pool_keys"), _pool_rows(pool_keys),
        _ptr(pool_start, torch.int32, "pool_start"),
        _ptr(pool_valid, torch.uint8, "pool_valid"), _ptr(n_pools, torch.int32, "n_pools"),
        _ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), _ptr(q_seq, torch.int32, "q_seq"),
        _ptr(q_pos, torch.int32, "q_pos"), Q, cu_pool_cap.numel() - 1, H, D, int(kpool),
        scores.shape[-1], pool_ids.shape[-1], token_ids.shape[-1], _dtype_tag(q),
        _ptr(scores, torch.float32, "scores"), _ptr(pool_ids, torch.int32, "pool_ids"),
        _ptr(token_ids, torch.int32, "token_ids"), _ptr(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_select", code)


def dsa_select_noalloc(q, weights, scale, pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap,
                       q_seq, q_pos, kpool, scores, pool_ids, token_ids, status=None, stream=None):
    """dsa_select without a workspace, for callers that cannot allocate device
    memory (stream capture, host frameworks owning all allocations, hot loops
    that forbid allocation): its scratch is a static device array shared by all
    calls on the device, so calls must not overlap on the GPU; Q <= 64."""
    Q, H, D = q.shape
    act = q.dtype
    code = _lib.load().dsa_select_noalloc(
        _ptr(q, act, "q"), _ptr(weights, torch.float32, "weights"), float(scale),
        _ptr(pool_keys, act, "pool_keys"), _pool_rows(pool_keys),
        _ptr(pool_start, torch.int32, "pool_start"),
        _ptr(pool_valid, torch.uint8, "pool_valid"), _ptr(n_pools, torch.int32, "n_pools"),
        _ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), _ptr(q_seq, torch.int32, "q_seq"),
        _ptr(q_pos, torch.int32, "q_pos"), Q, cu_pool_cap.numel() - 1, H, D, int(kpool),
        scores.shape[-1], pool_ids.shape[-1], token_ids.shape[-1], _dtype_tag(q),
        _ptr(scores, torch.float32, "scores"), _ptr(pool_ids, torch.int32, "pool_ids"),
        _ptr(token_ids, torch.int32, "token_ids"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_select_noalloc", code)


def dsa_decode_layer(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens, pool_begin,
                     max_pools, pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap, q,
                     weights, scale, q_seq, q_pos, q_lat, kv_latent, sm_scale, kpool, scores,
                     pool_ids, token_ids, out, lse, ws_select, ws_mla=None, status=None,
                     stream=None):
    """dsa_kpool_compress -> dsa_select -> dsa_mla_selected_decode in one call
    (same outputs); ``ws_select`` must be zero-filled before its first use."""
    act = k.dtype
    Q, H, D = q.shape
    _, Hm, L = q_lat.shape
    a = _lib.DecodeLayerArgs(
        k=_ptr(k, act, "k"), gate=_ptr(gate, act, "gate"), valid=_ptr(valid, torch.uint8, "valid"),
        ape=_ptr(ape, torch.float32, "ape"), ln_gamma=_ptr(ln_gamma, act, "ln_gamma"),
        ln_beta=_ptr(ln_beta, act, "ln_beta"), ln_eps=float(ln_eps),
        cu_seqlens=_ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        pool_begin=_ptr(pool_begin, torch.int32, "pool_begin"), max_pools=int(max_pools),
        pool_keys=_ptr(pool_keys, act, "pool_keys"), pool_rows=_pool_rows(pool_keys),
        pool_start=_ptr(pool_start, torch.int32, "pool_start"),
        pool_valid=_ptr(pool_valid, torch.uint8, "pool_valid"),
        n_pools=_ptr(n_pools, torch.int32, "n_pools"),
        cu_pool_cap=_ptr(cu_pool_cap, torch.int32, "cu_pool_cap"), q=_ptr(q, act, "q"),
        weights=_ptr(weights, torch.float32, "weights"), scale=float(scale),
        q_seq=_ptr(q_seq, torch.int32, "q_seq"), q_pos=_ptr(q_pos, torch.int32, "q_pos"),
        q_lat=_ptr(q_lat, act, "q_lat"), kv_latent=_ptr(kv_latent, act, "kv_latent"),
        sm_scale=float(sm_scale), Q=Q, B=cu_pool_cap.numel() - 1, H=H, D=D, kpool=int(kpool),
        P_ld=scores.shape[-1], select_k=pool_ids.shape[-1], out_width=token_ids.shape[-1], Hm=Hm,
        L=L, dtype=_dtype_tag(q), scores=_ptr(scores, torch.float32, "scores"),
        pool_ids=_ptr(pool_ids, torch.int32, "pool_ids"),
        token_ids=_ptr(token_ids, torch.int32, "token_ids"), out=_ptr(out, act, "out"),
        lse=_ptr(lse, torch.float32, "lse"), ws_select=_ptr(ws_select, torch.uint8, "ws_select"),
        ws_select_bytes=0 if ws_select is None else ws_select.numel(),
        ws_mla=_ptr(ws_mla, torch.uint8, "ws_mla"),
        ws_mla_bytes=0 if ws_mla is None else ws_mla.numel(),
        status_dev=_ptr(status, torch.int32, "status"))
    _check("dsa_decode_layer", _lib.load().dsa_decode_layer(ctypes.byref(a), _stream(stream)))


def indexer_project_workspace_bytes(T, hidden, q_rank, H, D, Hm, nope, L) -> int:
    return int(_lib.load().dsa_indexer_project_workspace_size(T, hidden, q_rank, H, D, Hm, nope,
                                                              L))


def dsa_indexer_project(x, w_kgw, cq, w_q, w_uk_t, weights_scale, k_out, gate_out, weights_out,
                        q_out, q_nope_out, q_lat_out, workspace=None, kv_rows=None, status=None,
                        stream=None):
    """x [T, hidden], w_kgw [2D+H, hidden], cq [T, q_rank], w_q [H*D+Hm*nope, q_rank],
    w_uk_t [Hm, L, nope] (bf16); outputs k_out/gate_out [rows, D], weights_out [T, H] fp32,
    q_out [T, H, D], q_nope_out [T, Hm, nope], q_lat_out [T, Hm, L]."""
    bf = torch.bfloat16
    T, hidden = x.shape
    q_rank = cq.shape[1]
    Hm, L, nope = w_uk_t.shape
    H, D = q_out.shape[1], q_out.shape[2]
    code = _lib.load().dsa_indexer_project(
        _ptr(x, bf, "x"), _ptr(w_kgw, bf, "w_kgw"), _ptr(cq, bf, "cq"), _ptr(w_q, bf, "w_q"),
        _ptr(w_uk_t, bf, "w_uk_t"), T, hidden, q_rank, H, D, Hm, nope, L, float(weights_scale),
        _ptr(kv_rows, torch.int32, "kv_rows"), _ptr(k_out, bf, "k_out"),
        _ptr(gate_out, bf, "gate_out"), _ptr(weights_out, torch.float32, "weights_out"),
        _ptr(q_out, bf, "q_out"), _ptr(q_nope_out, bf, "q_nope_out"),
        _ptr(q_lat_out, bf, "q_lat_out"), _ptr(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check("dsa_indexer_project", code)


def dsa_kernel_launches() -> int:
    """Kernels the library has launched (or recorded into a stream capture) so far."""
    return int(_lib.load().dsa_kernel_launches())


DSA_DRILL_SKIP_ARM = 1
DSA_DRILL_SKIP_PV_COMMIT = 2


def dsa_set_failure_drill(drill: int) -> None:
    """Arm (DSA_DRILL_SKIP_ARM, DSA_DRILL_SKIP_PV_COMMIT) or disarm (0) a give-up
    drill of the tensor-core kernels, process wide (tests of failure detection
    only)."""
    _check("dsa_set_failure_drill", _lib.load().dsa_set_failure_drill(int(drill)))
