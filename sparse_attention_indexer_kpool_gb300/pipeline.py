"""One DSA layer's hot path, stage after stage, on caller-owned buffers.

``LayerBuffers`` allocates every output and workspace once (PyTorch owns the
memory); ``run_layer`` issues the five library calls in the order of the DSA
module page's pipeline (compress -> index_scores -> topk_pools ->
expand_selection -> MLA over the selected rows) on one stream.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import ops
from .synth import Batch


@dataclass
class LayerBuffers:
    pool_keys: torch.Tensor
    pool_start: torch.Tensor
    pool_valid: torch.Tensor
    n_pools: torch.Tensor
    scores: torch.Tensor
    pool_ids: torch.Tensor
    token_ids: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    ws_topk: torch.Tensor
    ws_select: torch.Tensor
    ws_mla: torch.Tensor | None
    status: torch.Tensor

    @staticmethod
    def alloc(bt: Batch, device=None) -> "LayerBuffers":
        dev = device or bt.k.device
        g = bt.geo
        total_cap = int(bt.cu_pool_cap[-1].item())
        Q = bt.Q
        ws_t = ops.topk_workspace_bytes(Q, bt.P_ld, g.select_k)
        ws_s = ops.select_workspace_bytes(Q, bt.P_ld, g.select_k)
        tag = ops.DSA_BF16 if g.dtype == "bf16" else ops.DSA_F32
        ws_m = ops.mla_workspace_bytes(Q, g.Hm, g.L, g.out_width, tag)
        return LayerBuffers(
            pool_keys=torch.zeros(max(total_cap, 1), g.D, dtype=bt.k.dtype, device=dev),
            pool_start=torch.full((max(total_cap, 1),), -1, dtype=torch.int32, device=dev),
            pool_valid=torch.zeros(max(total_cap, 1), dtype=torch.uint8, device=dev),
            n_pools=torch.zeros(bt.B, dtype=torch.int32, device=dev),
            scores=torch.empty(Q, bt.P_ld, dtype=torch.float32, device=dev),
            pool_ids=torch.empty(Q, g.select_k, dtype=torch.int32, device=dev),
            token_ids=torch.empty(Q, g.out_width, dtype=torch.int32, device=dev),
            out=torch.empty(Q, g.Hm, g.L, dtype=bt.q_lat.dtype, device=dev),
            lse=torch.empty(Q, g.Hm, dtype=torch.float32, device=dev),
            ws_topk=torch.empty(max(ws_t, 16), dtype=torch.uint8, device=dev),
            ws_select=torch.zeros(max(ws_s, 16), dtype=torch.uint8, device=dev),
            ws_mla=torch.empty(ws_m, dtype=torch.uint8, device=dev) if ws_m else None,
            status=torch.zeros(1, dtype=torch.int32, device=dev))


def compress(bt: Batch, buf: LayerBuffers, pool_begin=None, max_pools=None, stream=None):
    if max_pools is None:
        max_pools = bt.P_ld
    ops.dsa_kpool_compress(bt.k, bt.gate, bt.valid, bt.ape, bt.ln_gamma, bt.ln_beta, bt.geo.ln_eps,
                           bt.cu_seqlens, bt.cu_pool_cap, pool_begin, bt.geo.kpool, max_pools,
                           buf.pool_keys, buf.pool_start, buf.pool_valid, buf.n_pools, buf.status,
                           stream)


def select_stages(bt: Batch, buf: LayerBuffers, stream=None):
    """index_scores -> topk_pools -> expand_selection as three separate calls."""
    g = bt.geo
    ops.dsa_index_scores(bt.q, bt.weights, bt.scale, buf.pool_keys, buf.pool_start,
                         buf.pool_valid, buf.n_pools, bt.cu_pool_cap, bt.q_seq, bt.q_pos,
                         g.kpool, buf.scores, buf.status, stream)
    ops.dsa_topk_pools(buf.scores, g.select_k, buf.pool_ids, buf.ws_topk, stream)
    ops.dsa_expand_selection(buf.pool_ids, buf.pool_start, bt.cu_pool_cap, bt.q_seq, g.kpool,
                             buf.token_ids, buf.status, stream)


def select(bt: Batch, buf: LayerBuffers, stream=None):
    """The fused select call (same outputs as select_stages)."""
    ops.dsa_select(bt.q, bt.weights, bt.scale, buf.pool_keys, buf.pool_start, buf.pool_valid,
                   buf.n_pools, bt.cu_pool_cap, bt.q_seq, bt.q_pos, bt.geo.kpool, buf.scores,
                   buf.pool_ids, buf.token_ids, buf.ws_select, buf.status, stream)


def attend(bt: Batch, buf: LayerBuffers, stream=None):
    ops.dsa_mla_selected_decode(bt.q_lat, bt.kv, bt.cu_seqlens, bt.q_seq, buf.token_ids,
                                bt.sm_scale, buf.out, buf.lse, buf.ws_mla, buf.status, stream)


def decode_layer(bt: Batch, buf: LayerBuffers, pool_begin=None, max_pools=None, stream=None):
    """compress -> select -> attend as the single fused call (same outputs as
    run_layer)."""
    if max_pools is None:
        max_pools = bt.P_ld
    ops.dsa_decode_layer(bt.k, bt.gate, bt.valid, bt.ape, bt.ln_gamma, bt.ln_beta, bt.geo.ln_eps,
                         bt.cu_seqlens, pool_begin, max_pools, buf.pool_keys, buf.pool_start,
                         buf.pool_valid, buf.n_pools, bt.cu_pool_cap, bt.q, bt.weights, bt.scale,
                         bt.q_seq, bt.q_pos, bt.q_lat, bt.kv, bt.sm_scale, bt.geo.kpool,
                         buf.scores, buf.pool_ids, buf.token_ids, buf.out, buf.lse,
                         buf.ws_select, buf.ws_mla, buf.status, stream)


def run_layer(bt: Batch, buf: LayerBuffers, pool_begin=None, max_pools=None, stream=None,
              fused=True):
    compress(bt, buf, pool_begin, max_pools, stream)
    (select if fused else select_stages)(bt, buf, stream)
    attend(bt, buf, stream)


@dataclass
class ProjectionBuffers:
    """Outputs and workspace of dsa_indexer_project for one layer."""
    k: torch.Tensor          # [rows, D] bf16 (rows = T, or the cache rows kv_rows points into)
    gate: torch.Tensor       # [rows, D] bf16
    weights: torch.Tensor    # [T, H] fp32
    q: torch.Tensor          # [T, H, D] bf16
    q_nope: torch.Tensor     # [T, Hm, nope] bf16
    q_lat: torch.Tensor      # [T, Hm, L] bf16
    ws: torch.Tensor | None  # counters zeroed here, left zero by every call
    status: torch.Tensor

    @staticmethod
    def alloc(pi, rows=None, device=None) -> "ProjectionBuffers":
        dev = device or pi.x.device
        T, hidden = pi.x.shape
        bf = torch.bfloat16
        rows = T if rows is None else rows
        ws = ops.indexer_project_workspace_bytes(T, hidden, pi.cq.shape[1], pi.H, pi.D, pi.Hm,
                                                 pi.nope, pi.L)
        return ProjectionBuffers(
            k=torch.zeros(rows, pi.D, dtype=bf, device=dev),
            gate=torch.zeros(rows, pi.D, dtype=bf, device=dev),
            weights=torch.empty(T, pi.H, dtype=torch.float32, device=dev),
            q=torch.empty(T, pi.H, pi.D, dtype=bf, device=dev),
            q_nope=torch.empty(T, pi.Hm, pi.nope, dtype=bf, device=dev),
            q_lat=torch.empty(T, pi.Hm, pi.L, dtype=bf, device=dev),
            ws=torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None,
            status=torch.zeros(1, dtype=torch.int32, device=dev))


def project(pi, buf: ProjectionBuffers, weights_scale: float, kv_rows=None, stream=None):
    """The indexer projections of one layer: k, gate, weights, q, q_nope, q_lat."""
    ops.dsa_indexer_project(pi.x, pi.w_kgw, pi.cq, pi.w_q, pi.w_uk_t, weights_scale, buf.k,
                            buf.gate, buf.weights, buf.q, buf.q_nope, buf.q_lat, buf.ws,
                            kv_rows, buf.status, stream)
