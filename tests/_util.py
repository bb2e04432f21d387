"""Test helpers: move a synthetic batch to the oracle's float64 numpy form."""
import numpy as np
import torch


def npf(t):
    """Exact float64 copy of a float tensor (bf16/fp32 widen exactly)."""
    return t.detach().to("cpu", torch.float64).numpy()


def npi(t):
    return None if t is None else t.detach().to("cpu", torch.int64).numpy()


def oracle_inputs(bt):
    g = bt.geo
    return dict(
        k=npf(bt.k), gate=npf(bt.gate), valid=bt.valid.cpu().numpy(), ape=npf(bt.ape),
        ln_gamma=npf(bt.ln_gamma), ln_beta=npf(bt.ln_beta), ln_eps=g.ln_eps,
        cu_seqlens=npi(bt.cu_seqlens), cu_pool_cap=npi(bt.cu_pool_cap), kpool=g.kpool,
        dtype=g.dtype, q=npf(bt.q), weights=npf(bt.weights), scale=bt.scale,
        q_seq=npi(bt.q_seq), q_pos=npi(bt.q_pos), P_ld=bt.P_ld, select_k=g.select_k,
        out_width=g.out_width, q_lat=npf(bt.q_lat), kv=npf(bt.kv), sm_scale=bt.sm_scale)


def ulp_bf16(x):
    """Spacing of the bf16 grid at |x| (2^(e-8) for |x| in [2^(e-1), 2^e))."""
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(1.0, e - 8)
