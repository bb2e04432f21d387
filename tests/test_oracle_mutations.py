"""The oracle pins must reject plausible slips.

Each case plants one mistake in a private copy of the oracle (on the CPU, never
in the library) and checks that at least one pin in test_oracle_pins fails.
"""
import importlib.util
import os
import sys
import tempfile

import pytest

import tests.test_oracle_pins as pins

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = open(os.path.join(HERE, "..", "oracle", "dsa_oracle.py")).read()

MUTATIONS = {
    "rmsnorm": ("mu = x.mean(axis=-1, keepdims=True)", "mu = 0.0 * x.mean(axis=-1, keepdims=True)"),
    "unbiased_variance": ("var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)",
                          "var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    "softmax_over_channels": ("m = logit.max(axis=1, keepdims=True)\n        e = np.exp(logit - m)\n"
                              "        w = e / e.sum(axis=1, keepdims=True)",
                              "m = logit.max(axis=2, keepdims=True)\n        e = np.exp(logit - m)\n"
                              "        w = e / e.sum(axis=2, keepdims=True)"),
    "softmax_over_pools": ("m = logit.max(axis=1, keepdims=True)\n        e = np.exp(logit - m)\n"
                           "        w = e / e.sum(axis=1, keepdims=True)",
                           "m = logit.max(axis=0, keepdims=True)\n        e = np.exp(logit - m)\n"
                           "        w = e / e.sum(axis=0, keepdims=True)"),
    "ape_dropped": ("logit = logit + ape[None, :, :]", "logit = logit + 0 * ape[None, :, :]"),
    "pools_from_token_0": ("t0 = first_valid(valid[lo:hi])", "t0 = 0"),
    "partial_pool_kept": ("P = (T - t0) // kpool", "P = -(-(T - t0) // kpool)"),
    "any_valid_slot": ("np.all(valid[tok] != 0, axis=1)", "np.any(valid[tok] != 0, axis=1)"),
    "relu_after_weight": ("s = (np.maximum(0.0, scale * dots) * w[i][None, :]).sum(axis=1)",
                          "s = np.maximum(0.0, scale * dots * w[i][None, :]).sum(axis=1)"),
    "scale_dropped": ("np.maximum(0.0, scale * dots)", "np.maximum(0.0, dots)"),
    "causal_strict": ("cand &= last_tok <= int(q_pos[i])", "cand &= last_tok < int(q_pos[i])"),
    "tie_order_reversed": ("order = np.lexsort((cand, -s))", "order = np.lexsort((-cand, -s))"),
    "expand_without_base": ("start = int(pool_start[base + p])", "start = int(pool_start[p])"),
    "mla_without_row_base": ("C = np.asarray(kv[lo + sel], np.float64)",
                             "C = np.asarray(kv[sel], np.float64)"),
    "mla_scale_dropped": ("z = sm_scale * (q_i @ C.T)", "z = (q_i @ C.T)"),
    "bf16_truncates": ("r = np.rint(x / spacing) * spacing", "r = np.trunc(x / spacing) * spacing"),
    "paged_row_without_page_size": ("rows = page[ok] * page_size + sel[ok] % page_size",
                                    "rows = page[ok] + sel[ok] % page_size"),
    "paged_block_by_modulo": ("blk = sel // page_size", "blk = sel % page_size"),
    "fp8_bias_8": ("np.ldexp(1.0, e - 7)", "np.ldexp(1.0, e - 8)"),
    "fp8_subnormals_as_normals": ("np.where(e == 0, (m / 8.0) * 2.0 ** -6,",
                                  "np.where(e == 0, (1.0 + m / 8.0) * 2.0 ** -7,"),
    "fp8_row_scale_dropped": ("* np.asarray(row_scale, np.float64)[rows][:, None]", "* 1.0"),
    "projection_transposed_weight": ("return alpha * (inp @ w.T)", "return alpha * (inp @ w)"),
    "absorb_untransposed": ("out[:, h, :] = q_nope[:, h, :] @ w_uk_t[h].T",
                            "out[:, h, :] = q_nope[:, h, :] @ w_uk_t[h]"),
    "gate_rows_swapped_with_k": ("k, gate = hid[:, :D], hid[:, D:2 * D]",
                                 "gate, k = hid[:, :D], hid[:, D:2 * D]"),
    "weights_scale_dropped": ("weights = weights_scale * hid[:, 2 * D:2 * D + H]",
                              "weights = hid[:, 2 * D:2 * D + H]"),
    "q_lat_from_unrounded_query": ("k, gate, q, q_nope = (round_bf16(a) for a in (k, gate, q, q_nope))",
                                   "k, gate, q = (round_bf16(a) for a in (k, gate, q))"),
}


def _load_mutant(src):
    d = tempfile.mkdtemp()
    path = os.path.join(d, "mutant_oracle.py")
    open(path, "w").write(src)
    spec = importlib.util.spec_from_file_location("mutant_oracle", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, monkeypatch):
    a, b = MUTATIONS[name]
    assert SRC.count(a) == 1, name
    mutant = _load_mutant(SRC.replace(a, b))
    monkeypatch.setattr(pins, "oracle", mutant)
    failed = []
    for fn_name in sorted(dir(pins)):
        if fn_name.startswith("test_"):
            try:
                getattr(pins, fn_name)()
            except Exception:
                failed.append(fn_name)
    assert failed, f"no pin caught the planted mistake {name!r}"
