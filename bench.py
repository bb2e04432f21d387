#!/usr/bin/env python
"""Decode-step benchmark: DSA kpool selection + selected-row NoPE MLA at 262k context.

Workload (default): 4 sequences x 262 144 tokens (65 536 pools each at kpool 4),
32 index heads x head_dim 128, select_k 512 -> 2 048 token ids, MLA 64 heads x
latent 512, bf16, 11 independent DSA layers per step (each with its own seeded
caches and weights).  One step = every layer's decode pass for the 4 query
tokens, one dsa_decode_layer call per layer: incremental kpool_compress of the
just-completed pool -> index_scores -> topk_pools -> expand_selection -> MLA
over the selected rows.  The step is captured in a CUDA graph; caches live in
HBM before the timed region starts and the 11 layers' 704 MB of pool keys
cycle through the 129 MB L2, so every step reads its pool keys from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")   # the CPU oracle legs run on one core

METRIC = "DSA decode queries/sec at 262k ctx; index+attend HBM GB/s vs peak (1 GB300)"
UNIT = "queries/s"
N_LAYERS = 11
N_QUERY_SETS = 4      # seeded query sets per layer that consecutive steps rotate over


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    # profiling helpers (non-default shapes are never reported as the metric)
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--seqlen", type=int, default=262144)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fixed-queries", action="store_true",
                    help="every step reuses one query set (default: steps rotate over "
                         "N_QUERY_SETS seeded sets, so consecutive steps select different rows)")
    ap.add_argument("--breakdown", action="store_true",
                    help="diagnostic: per-stage in-graph times (extra events between stages)")
    ap.add_argument("--leg", choices=["prefill_index", "prefill_attention", "paged_attention",
                                      "projections"],
                    help="run only this side measurement and print its JSON object (for "
                         "profiling one kernel without the decode step)")
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the paged / E4M3 attention leg")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill-chunk scoring measurement")
    ap.add_argument("--per-layer-metadata", action="store_true",
                    help="give every layer its own copy of the batch layout (cu_seqlens, "
                         "cu_pool_cap, q_seq, pool_begin) and padding mask instead of one "
                         "set shared by the layers")
    ap.add_argument("--no-projections", action="store_true",
                    help="skip the projection leg (hidden state -> the path's inputs)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self, n_gpus):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.uuid}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                   "reasons": sorted(reasons), "samples": len(sm)}
        return out


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def algorithmic_bytes(B, P, D, H, Hm, L, K, kp, W):
    """Bytes one decode query-layer must move at minimum (per stage)."""
    idx = P * D * 2 + P * 1 + H * D * 2 + H * 4 + P * 4          # keys, valid, q, w, scores out
    topk = P * 4 + K * 4                                           # scores in, pool ids out
    expand = K * 4 + K * 4 + W * 4                                 # ids, pool starts, token ids
    mla = W * 4 + W * L * 2 + Hm * L * 2 + Hm * L * 2 + Hm * 4    # ids, rows, q_lat, out, lse
    comp = 2 * kp * D * 2 + kp + D * 2 + 4 + 1                     # last pool: k, gate, valid, out
    return dict(index=idx, topk=topk, expand=expand, mla=mla, compress=comp,
                total=idx + topk + expand + mla + comp)


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from its committed ncu summary, or None
    when the kernel's source changed after the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", kernel + "_long262k.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    src = os.path.join(ROOT, "sparse_attention_indexer_kpool_gb300", "csrc",
                       fields.get("source", ""))
    if not os.path.isfile(src) or "traffic_bytes_per_launch" not in fields:
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != fields.get("source_sha256"):
        return None
    return int(fields["traffic_bytes_per_launch"])


def prefill_index(peaks_path, reps=10):
    """The prefill-chunk scoring pass: 4096 queries appended to a 131 072-token
    context (kpool 8, 16 896 pools, causal), one dsa_index_scores launch, L2
    flushed before every timed launch.  Reported against the bf16 tensor peak
    over the causal flops 2*H*D*sum_q(visible pools of q)."""
    import torch

    from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
    bt = synth.prefill(device="cuda")
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    g = bt.geo
    P = int(buf.n_pools[0].item())
    pos = bt.q_pos.to(torch.int64)
    visible = torch.clamp((pos + 1) // g.kpool, max=P)        # no padding: t0 = 0
    flops = 2.0 * g.H * g.D * float(visible.sum().item())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def launch():
        ops.dsa_index_scores(bt.q, bt.weights, bt.scale, buf.pool_keys, buf.pool_start,
                             buf.pool_valid, buf.n_pools, bt.cu_pool_cap, bt.q_seq, bt.q_pos,
                             g.kpool, buf.scores, buf.status)
    for _ in range(3):
        launch()
    times = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    assert int(buf.status.item()) == 0
    us = statistics.median(times) * 1e3
    # the chunk's own pools: compress of the 4096 new tokens (512 pools of 8)
    # into the cache after the context's 16 384, L2 flushed before each call
    n_ctx = int(bt.q_pos[0].item())
    begin = torch.tensor([n_ctx // g.kpool], dtype=torch.int32, device="cuda")
    n_new = bt.Q // g.kpool
    ctimes = []
    for i in range(reps + 3):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pipeline.compress(bt, buf, pool_begin=begin, max_pools=n_new)
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            ctimes.append(a.elapsed_time(b))
    assert int(buf.status.item()) == 0
    c_us = statistics.median(ctimes) * 1e3
    c_bytes = bt.Q * (2 * g.D * 2 + 1) + n_new * (g.D * 2 + 5)
    peak = json.load(open(peaks_path))["bf16_tflops"] if os.path.exists(peaks_path) else 1900.0
    tf = flops / (us * 1e-6) / 1e12
    return {"workload": "prefill: 4096 chunk queries after 131072 ctx, kpool 8, %d pools, "
                        "causal" % P,
            "chunk_compress": {"pools": n_new, "us": round(c_us, 2), "bytes": c_bytes,
                               "gbs": round(c_bytes / (c_us * 1e-6) / 1e9, 1),
                               "kernel": "kpool_compress_wide_kernel<8>",
                               "timing": "median of %d calls, L2 flushed before each" % reps},
            "kernel": "index_scores_umma_kernel (8 queries per key tile)",
            "us": round(us, 2), "flops": flops, "tflops": round(tf, 1), "bound": "tensor",
            "peak_tflops": peak, "peak_source": "measured bf16 burst" if
            os.path.exists(peaks_path) else "fallback", "frac": round(tf / peak, 4),
            "score_bytes": int(buf.scores.numel() * 4),
            "timing": "median of %d launches, L2 flushed before each" % reps}


def prefill_attention(peaks_path, reps=5):
    """The selected-row attention of the prefill chunk: 4096 queries after a
    131 072-token context, 2048 selected rows each (kpool 8, 256 pools), 64
    heads, latent 512, on the streaming tensor-core kernel; the token ids are
    the chunk's own selection.  L2 flushed before every timed call; reported
    against the bf16 tensor peak over 2 * 2 * Hm * L flops per selected row."""
    import torch

    from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
    bt = synth.prefill(device="cuda")
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.compress(bt, buf)
    pipeline.select(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    Q, Hm, L = bt.q_lat.shape
    rows = int((buf.token_ids >= 0).sum().item())
    flops = 4.0 * Hm * L * rows
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        pipeline.attend(bt, buf)
    times = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pipeline.attend(bt, buf)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    assert int(buf.status.item()) == 0
    us = statistics.median(times) * 1e3
    peak = json.load(open(peaks_path))["bf16_tflops"] if os.path.exists(peaks_path) else 1900.0
    tf = flops / (us * 1e-6) / 1e12
    return {"workload": "prefill chunk attention: %d queries x %d selected rows (%d valid), %d "
                        "heads, latent %d" % (Q, buf.token_ids.shape[1], rows, Hm, L),
            "kernel": "mla_stream_kernel (tcgen05, 64 heads per CTA, 128-row tiles)",
            "us": round(us, 1), "flops": flops, "tflops": round(tf, 1), "bound": "tensor",
            "peak_tflops": peak, "frac": round(tf / peak, 4),
            "timing": "median of %d calls, L2 flushed before each" % reps}


def projections(peaks_path, reps=20):
    """The projections before the selection (dsa_indexer_project: hidden state
    and query latent to k, gate, weights, q, q_nope and the latent-space
    query) at the full-size shapes (hidden 6144, query latent 2048, 32 index
    heads of 128, 64 MLA heads with a 192-wide no-rope part, latent 512;
    random-init weights):
    * decode: 4 tokens per layer, 11 layers of distinct weights (915 MB, past
      the L2) called back to back from a CUDA graph: a weight stream, against
      HBM;
    * prefill: one 4096-token chunk, L2 flushed before every call: against the
      bf16 tensor peak."""
    import torch

    from sparse_attention_indexer_kpool_gb300 import pipeline, synth
    g = synth.PROJ_MAIN
    scale = g["H"] ** -0.5
    hbm = json.load(open(peaks_path))["hbm_gbs"] if os.path.exists(peaks_path) else 6800.0
    peak = json.load(open(peaks_path))["bf16_tflops"] if os.path.exists(peaks_path) else 1900.0
    M1, M2 = 2 * g["D"] + g["H"], g["H"] * g["D"] + g["Hm"] * g["nope"]

    def act_bytes(T):  # activations in, outputs out, q_nope written and read back
        return 2 * T * (g["hidden"] + g["q_rank"] + 2 * g["D"] + g["H"] * g["D"]
                        + 2 * g["Hm"] * g["nope"] + g["Hm"] * g["L"]) + 4 * T * g["H"]

    w_bytes = 2 * (M1 * g["hidden"] + M2 * g["q_rank"] + g["Hm"] * g["L"] * g["nope"])
    pis = [synth.projection_inputs(4, **g, device="cuda", seed=5000 + 100 * l)
           for l in range(N_LAYERS)]
    bufs = [pipeline.ProjectionBuffers.alloc(pi) for pi in pis]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up off the default stream, as for capture
        for _ in range(3):
            for pi, b in zip(pis, bufs):
                pipeline.project(pi, b, scale)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()         # one decode step's projections, 11 layers
    with torch.cuda.graph(graph):
        for pi, b in zip(pis, bufs):
            pipeline.project(pi, b, scale)
    graph.replay()
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b_.record()
    torch.cuda.synchronize()
    assert all(int(b.status.item()) == 0 for b in bufs)
    dec_us = a.elapsed_time(b_) * 1e3 / (reps * N_LAYERS)
    dec_bytes = w_bytes + act_bytes(4)
    dec_gbs = dec_bytes / (dec_us * 1e-6) / 1e9
    del pis, bufs
    T = 4096
    pi = synth.projection_inputs(T, **g, device="cuda", seed=6000)
    buf = pipeline.ProjectionBuffers.alloc(pi)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        pipeline.project(pi, buf, scale)
    times = []
    for _ in range(max(3, reps // 4)):
        flush.fill_(1)
        a.record()
        pipeline.project(pi, buf, scale)
        b_.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b_))
    assert int(buf.status.item()) == 0
    pre_us = statistics.median(times) * 1e3
    flops = 2.0 * T * (M1 * g["hidden"] + M2 * g["q_rank"] + g["Hm"] * g["L"] * g["nope"])
    tf = flops / (pre_us * 1e-6) / 1e12
    return {"kernel": "proj_gemm_kernel (tcgen05, 128 output features x 16/64/128/256 tokens "
                      "per tile, split contraction below two CTAs per SM)",
            "shapes": dict(g),
            "decode": {"tokens": 4, "layers": N_LAYERS, "us_per_layer": round(dec_us, 2),
                       "bytes_per_layer": dec_bytes, "gbs": round(dec_gbs, 1), "bound": "hbm",
                       "peak_gbs": hbm, "frac": round(dec_gbs / hbm, 4),
                       "timing": "%d replays of a CUDA graph of %d calls, one per layer"
                                 % (reps, N_LAYERS)},
            "prefill": {"tokens": T, "us": round(pre_us, 1), "flops": flops,
                        "tflops": round(tf, 1), "bound": "tensor", "peak_tflops": peak,
                        "frac": round(tf / peak, 4),
                        "timing": "median of %d calls, L2 flushed before each" % len(times)}}


def paged_attention(reps=20, page_size=64):
    """The selected-row attention of the 64-sequence ragged decode batch (64
    queries, T_b ~ U{4096..65536}, 2048 selected rows each: 128 MiB of bf16
    rows, well past the L2) on the contiguous bf16 cache and on paged caches
    (pages of 64 rows) in bf16 and E4M3: one call each (attention and merge
    kernels), L2 flushed before every timed call.  The token ids are the
    batch's own selection."""
    import torch

    from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth
    bt = synth.ragged64(device="cuda")
    buf = pipeline.LayerBuffers.alloc(bt)
    pipeline.run_layer(bt, buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    del bt.k, bt.gate
    Q, Hm, L = bt.q_lat.shape
    W = buf.token_ids.shape[1]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(buf.out)
    lse = torch.empty_like(buf.lse)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pcs = {"paged_bf16": synth.paged_cache(bt.kv, bt.cu_seqlens, page_size, seed=5),
           "paged_e4m3": synth.paged_cache(bt.kv, bt.cu_seqlens, page_size, e4m3=True, seed=6)}
    ws = torch.empty(max(ops.mla_paged_workspace_bytes(bt.q_lat, bt.kv, W), 16),
                     dtype=torch.uint8, device="cuda")
    calls = {"contiguous_bf16": lambda: ops.dsa_mla_selected_decode(
        bt.q_lat, bt.kv, bt.cu_seqlens, bt.q_seq, buf.token_ids, bt.sm_scale, out, lse,
        buf.ws_mla, st)}
    for name, pc in pcs.items():
        calls[name] = (lambda pc=pc: ops.dsa_mla_paged_decode(
            bt.q_lat, pc.pages, pc.row_scale, pc.block_table, pc.seq_lens, pc.page_size,
            bt.q_seq, buf.token_ids, bt.sm_scale, out, lse, ws, st))
    fixed = W * 4 + 2 * Hm * L * 2 + Hm * 4          # ids, q, out, lse per query
    per_query = {"contiguous_bf16": W * L * 2 + fixed,
                 "paged_bf16": W * L * 2 + W * 4 + fixed,
                 "paged_e4m3": W * L + W * 4 + W * 4 + fixed}
    res = {}
    for name, f in calls.items():
        for _ in range(3):
            f()
        times = []
        for _ in range(reps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        us = statistics.median(times) * 1e3
        nbytes = per_query[name] * Q
        res[name] = {"us": round(us, 2), "bytes": nbytes,
                     "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
    assert int(st.item()) == 0, "device status set by the attention"
    return {"workload": "64-sequence ragged decode batch: %d queries x %d selected rows, %d heads, "
                        "latent %d, pages of %d rows" % (Q, W, Hm, L, page_size),
            "kernels": {"contiguous_bf16": "mla_stream_kernel (tcgen05, bf16 rows) + merge",
                        "paged_bf16": "mla_stream_kernel (tcgen05, paged rows) + merge",
                        "paged_e4m3": "mla_stream_kernel (tcgen05, E4M3 rows) + merge"},
            "calls": res,
            "bytes": "per call: rows (bf16 2 B, E4M3 1 B per value; E4M3 adds a 4 B row "
                     "scale), 4 B token id and (paged) 4 B table entry per row, q, out, lse",
            "timing": "median of %d calls, L2 flushed before each" % reps}


def run_ours(args, dist):
    import torch

    from sparse_attention_indexer_kpool_gb300 import build as libbuild
    from sparse_attention_indexer_kpool_gb300 import ops, pipeline, synth

    libbuild.build()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    uuid = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(dist.local)
    n_layers, T = args.layers, args.seqlen
    full = (n_layers == N_LAYERS and T == 262144)
    geo = synth.GEO_MAIN
    B = 4
    Q = B

    # ---- per-step host I/O lives in contiguous staging buffers: one step's
    # queries of every layer (a query set) per N_QUERY_SETS, and the outputs
    q_bytes = Q * geo.H * geo.D * 2
    w_bytes = Q * geo.H * 4
    ql_bytes = Q * geo.Hm * geo.L * 2
    in_per_layer = q_bytes + w_bytes + ql_bytes
    set_bytes = n_layers * in_per_layer
    out_per_layer = Q * geo.Hm * geo.L * 2 + Q * geo.Hm * 4
    n_sets = 1 if args.fixed_queries else N_QUERY_SETS
    stage_in = torch.empty(n_sets * set_bytes, dtype=torch.uint8, device=dev)
    stage_out = torch.empty(n_layers * out_per_layer, dtype=torch.uint8, device=dev)

    layers = []
    qsets = []   # qsets[l][k]: (q, weights, q_lat) of layer l in query set k
    for l in range(n_layers):
        bt = synth.make_batch(geo, [T] * B, [0] * B, device=dev, seed=3000 + 100 * l)
        bt.q_pos = None                      # decode query at T-1: every complete pool is visible
        if l > 0 and not args.per_layer_metadata:
            # one batch of sequences: its layout (cu_seqlens, cu_pool_cap,
            # q_seq) and padding mask are the same tensors in every layer;
            # caches and queries stay per layer
            b0 = layers[0][0]
            bt.cu_seqlens, bt.cu_pool_cap, bt.q_seq, bt.valid = (
                b0.cu_seqlens, b0.cu_pool_cap, b0.q_seq, b0.valid)
        sets = []
        for k in range(n_sets):
            src = (bt.q, bt.weights, bt.q_lat) if k == 0 else synth.query_set(
                geo, Q, device=dev, seed=900000 + 100 * l + k)
            o = k * set_bytes + l * in_per_layer
            views = []
            for t, nb, dt, shape in ((src[0], q_bytes, torch.bfloat16, (Q, geo.H, geo.D)),
                                     (src[1], w_bytes, torch.float32, (Q, geo.H)),
                                     (src[2], ql_bytes, torch.bfloat16, (Q, geo.Hm, geo.L))):
                view = stage_in[o:o + nb].view(dt).view(shape)
                view.copy_(t)
                views.append(view)
                o += nb
            sets.append(tuple(views))
        bt.q, bt.weights, bt.q_lat = sets[0]
        qsets.append(sets)
        buf = pipeline.LayerBuffers.alloc(bt)
        buf.scores_idx = torch.empty_like(buf.scores)
        o = l * out_per_layer
        ob = Q * geo.Hm * geo.L * 2
        buf.out = stage_out[o:o + ob].view(torch.bfloat16).view(Q, geo.Hm, geo.L)
        buf.lse = stage_out[o + ob:o + out_per_layer].view(torch.float32).view(Q, geo.Hm)
        layers.append((bt, buf))
    torch.cuda.synchronize()

    # ---- full cache build (kpool_compress over every token): built once, then
    # rebuilt three times (the same result) and timed; the median is reported
    for bt, buf in layers:
        pipeline.compress(bt, buf)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    build_times = []
    for _ in range(3):
        torch.cuda.synchronize()
        e0.record()
        for bt, buf in layers:
            pipeline.compress(bt, buf)
        e1.record()
        torch.cuda.synchronize()
        build_times.append(e0.elapsed_time(e1))
    build_ms = statistics.median(build_times)
    build_bytes = n_layers * (B * T * (2 * geo.D * 2 + 1) + B * (T // geo.kpool) * (geo.D * 2 + 5))
    for bt, buf in layers:
        assert int(buf.status.item()) == 0
        buf.pool_begin = (buf.n_pools - 1).clamp(min=0).to(torch.int32)
    if not args.per_layer_metadata:
        for bt, buf in layers[1:]:
            assert torch.equal(buf.pool_begin, layers[0][1].pool_begin)
            buf.pool_begin = layers[0][1].pool_begin

    def step(events=None, qset=0):
        """One decode step over every layer: one dsa_decode_layer call per layer
        (compress of the just-completed pool -> select -> attend), on query set
        ``qset``.  With events, the three stage calls run separately and
        events[layer] = (before, after) the select call (index_scores + top-k +
        expand)."""
        for li, (bt, buf) in enumerate(layers):
            bt.q, bt.weights, bt.q_lat = qsets[li][qset % n_sets]
            if events is None:
                pipeline.decode_layer(bt, buf, pool_begin=buf.pool_begin, max_pools=1)
                continue
            pipeline.compress(bt, buf, pool_begin=buf.pool_begin, max_pools=1)
            events[li][0].record()
            pipeline.select(bt, buf)
            events[li][1].record()
            pipeline.attend(bt, buf)

    # ---- warm-up (eager), then capture
    for w in range(max(3, args.warmup)):
        step(qset=w)
    torch.cuda.synchronize()

    K = args.steps
    S = max(d for d in range(1, min(K, 20) + 1) if K % d == 0)
    R = K // S
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    # g_plain: the production step, kernels chained by programmatic dependent launch
    g_plain = torch.cuda.CUDAGraph()
    n0 = ops.dsa_kernel_launches()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_plain, stream=side):
            for s in range(S):
                step(qset=s)
    # the library's own count of the kernels recorded for S steps
    launches_per_step = (ops.dsa_kernel_launches() - n0) // S
    # g_ev: the same steps with timing events around every select call (the
    # event nodes break the launch chain there, so this graph runs a little slower)
    try:
        ev = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
               for _ in range(n_layers)] for _ in range(S)]
        ev_ok = True
    except TypeError:
        ev, ev_ok = None, False
    g_ev = torch.cuda.CUDAGraph()
    if ev_ok:
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_ev, stream=side):
                for s in range(S):
                    step(ev[s], qset=s)
    g1 = torch.cuda.CUDAGraph()   # one step on query set 0 (the end-to-end leg's staging area)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g1, stream=side):
            step(qset=0)
    # g_idx: the dominant kernel alone (the scoring kernel of every layer, back to
    # back), for its roofline; dsa_index_scores runs the same tcgen05 kernel as
    # the select call, without counting the top-k histogram
    g_idx = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_idx, stream=side):
            for s in range(S):
                for li, (bt, buf) in enumerate(layers):
                    bt.q, bt.weights, bt.q_lat = qsets[li][s % n_sets]
                    ops.dsa_index_scores(bt.q, bt.weights, bt.scale, buf.pool_keys,
                                         buf.pool_start, buf.pool_valid, buf.n_pools,
                                         bt.cu_pool_cap, bt.q_seq, bt.q_pos, geo.kpool,
                                         buf.scores_idx, buf.status)
    torch.cuda.synchronize()
    g_plain.replay()
    torch.cuda.synchronize()
    for bt, buf in layers:
        assert int(buf.status.item()) == 0, "device status set during warm-up"

    # ---- timed region: K steps of the production graph
    sampler = ClockSampler(uuid)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(R):
        g_plain.replay()
    t1.record()
    torch.cuda.synchronize()
    dist.barrier()
    # ---- second timed region: K steps with events around the select calls
    idx_ms, ev_step_ms = None, None
    if ev_ok:
        t2, t3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t2.record()
        for _ in range(R):
            g_ev.replay()
        t3.record()
        torch.cuda.synchronize()
        ev_step_ms = t2.elapsed_time(t3) / K
        durs = [ev[s][l][0].elapsed_time(ev[s][l][1]) for s in range(S) for l in range(n_layers)]
        idx_ms = sum(durs) / len(durs)
    # ---- third timed region: the scoring kernel alone, K steps' worth of launches
    t4, t5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_idx.replay()
    t4.record()
    for _ in range(R):
        g_idx.replay()
    t5.record()
    torch.cuda.synchronize()
    kern_us = dist.max(t4.elapsed_time(t5)) * 1e3 / (K * n_layers)
    clocks = sampler.stop()
    ms = dist.max(t0.elapsed_time(t1))

    # ---- end to end: pinned host inputs -> device, the step, results -> host.
    # Step i copies query set i (rotating over the sets) from pinned host memory
    # into staging slot i % 2, replays the one-step graph that reads that slot
    # and writes that slot's output area, and copies the output area back to a
    # pinned host buffer.  The copies run on a second stream (the copy engines),
    # so the read-back of step i and the upload for step i + 2 overlap step
    # i + 1; events order each slot's upload -> step -> read-back -> next
    # upload.  The serial loop (upload, step, read-back, one after another) is
    # reported beside it.
    e2e = None
    if not args.no_e2e:
        h_in = torch.empty(stage_in.numel(), dtype=torch.uint8, pin_memory=True)
        h_in.copy_(stage_in)
        h_sets = [h_in[k * set_bytes:(k + 1) * set_bytes] for k in range(n_sets)]
        n_slots = min(2, n_sets)
        d_slot = [stage_in[k * set_bytes:(k + 1) * set_bytes] for k in range(n_slots)]
        d_out = [stage_out] + [torch.empty_like(stage_out) for _ in range(n_slots - 1)]
        h_res = [torch.empty(stage_out.numel(), dtype=torch.uint8, pin_memory=True)
                 for _ in range(n_slots)]
        slot_graphs = [g1]
        ob = Q * geo.Hm * geo.L * 2
        saved = [(buf.out, buf.lse) for _, buf in layers]
        for k in range(1, n_slots):
            for l, (bt, buf) in enumerate(layers):
                o = l * out_per_layer
                buf.out = d_out[k][o:o + ob].view(torch.bfloat16).view(Q, geo.Hm, geo.L)
                buf.lse = d_out[k][o + ob:o + out_per_layer].view(torch.float32).view(Q, geo.Hm)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    step(qset=k)
            slot_graphs.append(g)
        for (bt, buf), (o_, l_) in zip(layers, saved):
            buf.out, buf.lse = o_, l_
        copy_stream = torch.cuda.Stream()
        main = torch.cuda.current_stream()

        def serial(first, n):
            for i in range(first, first + n):
                d_slot[0].copy_(h_sets[i % n_sets], non_blocking=True)
                g1.replay()
                h_res[0].copy_(stage_out, non_blocking=True)

        def pipelined(n):
            ready = [torch.cuda.Event() for _ in range(n_slots)]
            done = [torch.cuda.Event() for _ in range(n_slots)]
            copy_stream.wait_stream(main)
            with torch.cuda.stream(copy_stream):
                for k in range(min(n_slots, n)):
                    d_slot[k].copy_(h_sets[k % n_sets], non_blocking=True)
                    ready[k].record()
            for i in range(n):
                k = i % n_slots
                main.wait_event(ready[k])
                slot_graphs[k].replay()
                done[k].record(main)
                with torch.cuda.stream(copy_stream):
                    copy_stream.wait_event(done[k])
                    h_res[k].copy_(d_out[k], non_blocking=True)
                    if i + n_slots < n:
                        d_slot[k].copy_(h_sets[(i + n_slots) % n_sets], non_blocking=True)
                    ready[k].record()
            main.wait_stream(copy_stream)

        # the pipeline's results are the serial loop's, step by step
        expect = []
        for i in range(3):
            serial(i, 1)
            torch.cuda.synchronize()
            expect.append(h_res[0].clone())
        for n in (1, 2, 3):
            pipelined(n)
            torch.cuda.synchronize()
            assert torch.equal(h_res[(n - 1) % n_slots], expect[n - 1]), \
                "pipelined end-to-end step differs from the serial one"

        def timed(fn):
            torch.cuda.synchronize()
            dist.barrier()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            wall0 = time.perf_counter()
            a.record()
            fn()
            b_.record()
            torch.cuda.synchronize()
            wall = time.perf_counter() - wall0
            return dist.max(max(a.elapsed_time(b_), wall * 1e3))

        timed(lambda: serial(0, 3))
        serial_ms = timed(lambda: serial(1, K))
        timed(lambda: pipelined(4))
        e_ms = timed(lambda: pipelined(K))
        e2e = {"value": round(dist.world * Q * K / (e_ms / 1e3), 1), "unit": UNIT,
               "h2d_bytes_per_step": int(set_bytes),
               "d2h_bytes_per_step": int(stage_out.numel()),
               "ms_per_step": round(e_ms / K, 5),
               "overlap": "uploads and read-backs on a second stream, two staging slots",
               "serial_value": round(dist.world * Q * K / (serial_ms / 1e3), 1),
               "serial_ms_per_step": round(serial_ms / K, 5)}

    breakdown = None
    if args.breakdown:
        names = ("compress", "select", "attend")
        evb = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
               for _ in range(n_layers)]
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(gb, stream=side):
                for li, (bt, buf) in enumerate(layers):
                    evb[li][0].record()
                    pipeline.compress(bt, buf, pool_begin=buf.pool_begin, max_pools=1)
                    evb[li][1].record()
                    pipeline.select(bt, buf)
                    evb[li][2].record()
                    pipeline.attend(bt, buf)
                    evb[li][3].record()
        tot = {n: 0.0 for n in names}
        reps = 20
        for _ in range(reps):
            gb.replay()
            torch.cuda.synchronize()
            for li in range(n_layers):
                for i, n in enumerate(names):
                    tot[n] += evb[li][i].elapsed_time(evb[li][i + 1])
        breakdown = {n: round(v / (reps * n_layers) * 1e3, 2) for n, v in tot.items()}
        breakdown["unit"] = "us per layer (in-graph, events between stages)"

    # ---- numbers
    ab = algorithmic_bytes(B, T // geo.kpool, geo.D, geo.H, geo.Hm, geo.L, geo.select_k,
                           geo.kpool, geo.out_width)
    per_step_bytes = ab["total"] * Q * n_layers
    value = dist.world * Q * K / (ms / 1e3)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peaks = json.load(open(peaks_path))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        hbm_peak, peak_src = 6800.0, "fallback"
    idx_bytes = ab["index"] * Q
    achieved = idx_bytes / (kern_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": "index_scores_umma_kernel",
                "achieved": round(achieved, 1), "peak": hbm_peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": profiled_traffic("index_scores_umma_kernel"),
                "bytes_per_launch": idx_bytes, "launch_us": round(kern_us, 2),
                "timing": "CUDA events around %d back-to-back launches (one per layer, %d "
                          "layers cycling, graph replays)" % (K * n_layers, n_layers)}
    sel_bytes = (ab["index"] + ab["topk"] + ab["expand"]) * Q
    select_call = None
    if idx_ms:
        select_call = {"kernels": "index_scores_umma_kernel + topk_select_kernel "
                                  "(three-call form of the step, events around dsa_select)",
                       "us": round(idx_ms * 1e3, 2), "bytes": sel_bytes,
                       "gbs": round(sel_bytes / (idx_ms * 1e-3) / 1e9, 1)}
    step_gbs = per_step_bytes / (ms / K * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) caches/queries, shapes of the pages' 262k workload)",
        "config": {"workload": "long262k" if full else f"profile-{n_layers}x{T}",
                   "sequences": B, "context": T, "pools_per_seq": T // geo.kpool,
                   "layers": n_layers, "index_heads": geo.H, "head_dim": geo.D,
                   "kpool": geo.kpool, "select_k": geo.select_k, "out_width": geo.out_width,
                   "mla_heads": geo.Hm, "latent": geo.L,
                   "l2": "inputs larger than L2: %d layers x %d MiB pool keys cycle through "
                         "the 129 MB L2" % (n_layers, B * (T // geo.kpool) * geo.D * 2 >> 20),
                   "graph": "CUDA graph of %d steps replayed %d times" % (S, R),
                   "queries": ("one seeded query set reused by every step" if n_sets == 1 else
                               "consecutive steps rotate over %d seeded query sets per layer "
                               "(q, weights, q_lat), so they select different rows" % n_sets),
                   "batch_metadata": ("per layer: every layer has its own copy of the batch "
                                      "layout and padding mask" if args.per_layer_metadata else
                                      "shared: the layers read one batch layout (cu_seqlens, "
                                      "cu_pool_cap, q_seq, pool_begin) and padding mask; "
                                      "caches and queries are per layer")},
        "gpu_launches": launches_per_step * K,
        "roofline": roofline, "select_call_in_step": select_call,
        "step_hbm_gbs": round(step_gbs, 1), "step_frac_of_peak": round(step_gbs / hbm_peak, 4),
        "ms_per_step_with_event_nodes": None if ev_step_ms is None else round(ev_step_ms, 5),
        "algorithmic_bytes_per_query_layer": ab,
        "compress_build": {"ms": round(build_ms, 3),
                           "gbs": round(build_bytes / (build_ms * 1e-3) / 1e9, 1),
                           "frac": round(build_bytes / (build_ms * 1e-3) / 1e9 / hbm_peak, 4),
                           "timing": "median of 3 warm rebuilds of the 11 layers' caches "
                                     "(11 launches each; %d MiB moved "
                                     "per rebuild, past the L2)" % (build_bytes >> 20)},
        "clocks": clocks, "e2e": e2e,
    }
    if breakdown:
        out["breakdown"] = breakdown
    if not args.no_prefill:
        out["prefill_index"] = prefill_index(peaks_path)
        out["prefill_attention"] = prefill_attention(peaks_path)
    if not args.no_paged:
        out["paged_attention"] = paged_attention()
    if not args.no_projections:
        out["projections"] = projections(peaks_path)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(layers[0], args.cpu_seconds)
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------
def oracle_query_layer(host, b, n_pools=None):
    """One decode query-layer through the oracle, stage after stage.  With
    ``n_pools`` the scoring, top-k and expansion see only the sequence's first
    n_pools pools (a bounded sample of the query-layer)."""
    import numpy as np

    import oracle
    kp = host["kpool"]
    # incremental compress of the last complete pool of sequence b
    pk, ps, pv, n, _ = oracle.kpool_compress(
        host["k"][b], host["gate"][b], host["valid"][b], host["ape"], host["ln_gamma"],
        host["ln_beta"], host["ln_eps"], [0, host["T"]], [0, host["cap"]], kp, "bf16",
        pool_begin=[host["cap"] - 1], max_pools=1, pool_keys=host["pool_keys"][b],
        pool_start=host["pool_start"][b], pool_valid=host["pool_valid"][b])
    P = host["cap"] if n_pools is None else int(n_pools)
    pk, ps, pv, n = pk[:P], ps[:P], pv[:P], np.minimum(n, P)
    scores, _ = oracle.index_scores(host["q"][b:b + 1], host["w"][b:b + 1], host["scale"], pk, ps,
                                    pv, n, [0, P], None, None, kp, P)
    ids = oracle.topk_pools(scores, host["select_k"])
    tok, _ = oracle.expand_selection(ids, ps, [0, P], None, kp, host["out_width"])
    out, lse, _ = oracle.mla_selected_decode(host["q_lat"][b:b + 1], host["kv"][b], [0, host["T"]],
                                             None, tok, host["sm_scale"], "bf16")
    return out


class _Rows:
    """Row access to a host bf16 tensor that yields exact float64 rows."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        import numpy as np
        import torch
        if isinstance(idx, slice):
            return self.t[idx].to(torch.float64).numpy()
        return self.t[torch.as_tensor(np.asarray(idx))].to(torch.float64).numpy()


def host_layer(layer):
    """Host copies of one layer for the oracle (bf16 kept; rows widen on access)."""
    import torch
    bt, buf = layer
    T, B = bt.lengths[0], bt.B
    cap = T // bt.geo.kpool
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()
    cpu = lambda t: t.detach().to("cpu")
    return {
        "T": T, "cap": cap, "kpool": bt.geo.kpool, "select_k": bt.geo.select_k,
        "out_width": bt.geo.out_width, "scale": bt.scale, "sm_scale": bt.sm_scale,
        "ln_eps": bt.geo.ln_eps, "ape": f(bt.ape), "ln_gamma": f(bt.ln_gamma),
        "ln_beta": f(bt.ln_beta),
        "k": [_Rows(cpu(bt.k[b * T:(b + 1) * T])) for b in range(B)],
        "gate": [_Rows(cpu(bt.gate[b * T:(b + 1) * T])) for b in range(B)],
        "valid": [bt.valid[b * T:(b + 1) * T].cpu().numpy() for b in range(B)],
        "kv": [_Rows(cpu(bt.kv[b * T:(b + 1) * T])) for b in range(B)],
        "pool_keys": [f(buf.pool_keys[b * cap:(b + 1) * cap]) for b in range(B)],
        "pool_start": [buf.pool_start[b * cap:(b + 1) * cap].cpu().numpy() for b in range(B)],
        "pool_valid": [buf.pool_valid[b * cap:(b + 1) * cap].cpu().numpy() for b in range(B)],
        "q": f(bt.q), "w": f(bt.weights), "q_lat": f(bt.q_lat),
    }


def _oracle_loop(host, first, seconds):
    """Decode query-layers through the oracle for about ``seconds`` (sequences
    round-robin from ``first``); returns (query-layers done, seconds taken)."""
    B = len(host["k"])
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_query_layer(host, (first + n) % B)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return n, time.perf_counter() - t0


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def _share(host):
    """The host arrays as shared-memory tensors, so that worker processes receive
    them by handle instead of by copy."""
    import numpy as np
    import torch

    def conv(v):
        if isinstance(v, np.ndarray):
            return _Shared(torch.from_numpy(v).share_memory_())
        if isinstance(v, _Rows):
            return _Rows(v.t.share_memory_())
        if isinstance(v, list):
            return [conv(x) for x in v]
        return v
    return {k: conv(v) for k, v in host.items()}


class _Shared:
    """A shared-memory tensor that the oracle reads as a numpy array."""

    def __init__(self, t):
        self.t = t

    def __reduce__(self):
        return (_Shared, (self.t,))


def _unshare(host):
    def conv(v):
        if isinstance(v, _Shared):
            return v.t.numpy()
        if isinstance(v, list):
            return [conv(x) for x in v]
        return v
    return {k: conv(v) for k, v in host.items()}


def _oracle_worker_shared(job):
    host, first, seconds = job
    return _oracle_loop(_unshare(host), first, seconds)


def cpu_baseline(layer, seconds, cores=None):
    """The oracle on this host's cores: one core, then every core (one process
    per core, each running whole query-layers of the same workload)."""
    host = host_layer(layer)
    n1, dt1 = _oracle_loop(host, 0, seconds)
    v1 = n1 / dt1 / N_LAYERS
    if cores is None:
        cores = (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                 else os.cpu_count())
    v_all, n_all, dt_all = v1, n1, dt1
    if cores > 1:
        import torch.multiprocessing as tmp
        shared = _share(host)
        ctx = tmp.get_context("spawn")     # workers never touch the GPU
        with ctx.Pool(cores) as pool:
            pool.map(_oracle_worker_shared, [(shared, i, 0.5) for i in range(cores)])  # start-up
            res = pool.map(_oracle_worker_shared, [(shared, i, seconds) for i in range(cores)])
        n_all = sum(r[0] for r in res)
        dt_all = max(r[1] for r in res)
        v_all = n_all / dt_all / N_LAYERS
    return {"value": round(v_all, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_all": round(v_all, 4), "cores_all": cores,
            "value_1core": round(v1, 4), "cpu_model": _cpu_model(),
            "sample": f"decode query-layers of the 262k workload (layer 0, sequences "
                      f"round-robin) through the numpy float64 oracle, one query-layer at a "
                      f"time per process (BLAS on one thread): {n_all} query-layers on "
                      f"{cores} cores in {dt_all:.1f} s and {n1} on one core in {dt1:.1f} s; "
                      f"queries/s = query-layers/s / {N_LAYERS} layers"}


def oracle_layer_cache(bt):
    """The pool cache of an equal-length batch, built by the oracle (for the CPU
    legs when no GPU built it)."""
    import numpy as np
    import torch

    import oracle
    T, geo = bt.lengths[0], bt.geo
    cap = T // geo.kpool

    class _Buf:
        pass
    buf = _Buf()
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()
    pk, ps, pv = [], [], []
    for b in range(bt.B):
        o = oracle.kpool_compress(f(bt.k[b * T:(b + 1) * T]), f(bt.gate[b * T:(b + 1) * T]),
                                  bt.valid[b * T:(b + 1) * T].cpu().numpy(), f(bt.ape),
                                  f(bt.ln_gamma), f(bt.ln_beta), geo.ln_eps, [0, T], [0, cap],
                                  geo.kpool, "bf16")
        pk.append(o[0]); ps.append(o[1]); pv.append(o[2])
    buf.pool_keys = torch.tensor(np.concatenate(pk), dtype=torch.float64)
    buf.pool_start = torch.tensor(np.concatenate(ps), dtype=torch.int32)
    buf.pool_valid = torch.tensor(np.concatenate(pv), dtype=torch.uint8)
    return buf


def run_reference(args, dist):
    """The CPU oracle as the reference arm: bounded samples of the same workload."""
    if dist.rank != 0:
        return
    import torch

    from sparse_attention_indexer_kpool_gb300 import synth
    # caches are synthesised on the GPU when one is present (fast), else on the CPU
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    geo = synth.GEO_MAIN
    bt = synth.make_batch(geo, [args.seqlen] * 4, [0] * 4, device=dev, seed=3000)
    import numpy as np

    import oracle
    # the oracle builds its own pool cache for the sample (setup, not timed)
    T = args.seqlen
    cap = T // geo.kpool
    host = host_layer((bt, oracle_layer_cache(bt)))
    # Size each step so that the whole run stays within a few minutes: one
    # query-layer per step, restricted to the first P_s pools of its sequence
    # (the oracle's time is dominated by the scoring pass, linear in the pools).
    c0 = time.perf_counter()
    oracle_query_layer(host, 0)
    t_full = time.perf_counter() - c0
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    P_s = int(min(cap, max(1024, cap * budget / t_full)))
    frac = P_s / cap
    for w in range(args.warmup):
        oracle_query_layer(host, w % 4, P_s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle_query_layer(host, s % 4, P_s)
    dt = time.perf_counter() - t0
    value = args.steps * frac / dt / N_LAYERS
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", "1"))
    sample = (f"each step = one decode query-layer (sequences round-robin) through the numpy "
              f"float64 oracle, scoring/top-k/expansion restricted to the first {P_s} of "
              f"{cap} pools; a step counts as {frac:.4f} query-layer; queries/s = "
              f"query-layers/s / {N_LAYERS} layers (one full query-layer took {t_full:.2f} s)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / max(1, args.steps) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long262k", "sequences": 4, "context": args.seqlen,
                   "layers": N_LAYERS},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    args = parse()
    dist = Dist(args.gpus)
    try:
        if args.leg:
            from sparse_attention_indexer_kpool_gb300 import build as libbuild
            libbuild.build()
            peaks = os.path.join(ROOT, "MEASURED_PEAKS.json")
            legs = {"prefill_index": lambda: prefill_index(peaks),
                    "prefill_attention": lambda: prefill_attention(peaks),
                    "paged_attention": paged_attention,
                    "projections": lambda: projections(peaks)}
            print(json.dumps({args.leg: legs[args.leg]()}), flush=True)
        elif args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
