"""Shared helpers of the GPU parity tests: run a drafting round through the C ABI and through
the oracle on the same seeded inputs, and compare them under the stated rules."""
from __future__ import annotations

from collections.abc import Mapping

import numpy as np
import torch

import oracle as O
import workloads as WL
from eagle_speculative_decoding_eagle3_gb300 import harness as HN

GAP = 1e-2          # argmax decisions are compared exactly where the oracle's top-2 gap exceeds this
TOL_BF16 = 2e-2     # max row-relative error of hidden states and logits (bf16 storage, fp32 accumulate)
TOL_F32 = 1e-4      # the same for the fp32 workload (fp32 storage and arithmetic throughout)


def row_rel_err(g, o):
    """max over rows of ||g - o||_inf / ||o||_inf."""
    g = np.asarray(g, dtype=np.float64).reshape(-1, np.shape(g)[-1])
    o = np.asarray(o, dtype=np.float64).reshape(-1, np.shape(o)[-1])
    return float(np.max(np.abs(g - o).max(axis=1) / np.abs(o).max(axis=1)))


FP8_NAMES = ("fc", "q_a", "kv_a", "q_b", "o", "gate", "up", "down", "lm_head")


class QuantOracleWeights(Mapping):
    """The oracle's view of a quantized head: the nine projection matrices replaced by the oracle's own
    quantization of the stored weights (dequantized, fp64), every other tensor widened as stored.  FP8
    matrices are quantized in blocks of rows (the rule is per row); NVFP4 matrices whole (one scale per
    matrix); each once."""

    def __init__(self, stored, fmt):
        self._s = stored
        self._fmt = fmt
        self._f = WL.F64Cache(stored)
        self._q = {}

    def __getitem__(self, k):
        if k not in FP8_NAMES:
            return self._f[k]
        if k not in self._q:
            W = WL.as_f32(self._s[k])
            if self._fmt == "fp8":
                self._q[k] = np.concatenate([O.quantize_rows_e4m3(W[r:r + 2048])[2] for r in range(0, len(W), 2048)])
            else:
                self._q[k] = O.quantize_nvfp4(W)[3]
        return self._q[k]

    def __iter__(self):
        return iter(self._s)

    def __len__(self):
        return len(self._s)


def run_round(w, seqs=None, absorbed=False, with_logits=True, stored=None, d2t_override="default", fp8=False,
              nvfp4=False, gpu_inputs=None, oracle_inputs=None):
    """GPU round (extend + gamma-1 decode steps + accept) and the oracle's forced-continuation round.

    ``seqs``: sequences the oracle checks (all by default); the GPU always runs the whole batch.
    ``fp8`` / ``nvfp4``: the head stores its projection matrices as FP8 E4M3 with row scales (NVFP4 with
    block and matrix scales), quantized on the GPU by eagle3_quantize_e4m3 (eagle3_quantize_nvfp4); the
    oracle runs on its own quantization of the same weights.
    ``gpu_inputs(ex, paged, d2t) -> d2t`` may edit the GPU's extend inputs and cache in place (and return
    the GPU's vocab map); ``oracle_inputs(exs, d2t) -> d2t`` does the same for the oracle's (rows of the
    checked sequences only).  Both default to the seeded inputs unchanged.
    """
    stored = WL.make_weights(w) if stored is None else stored
    lengths = WL.context_lengths(w)
    paged = WL.make_cache(w, lengths)
    ex = WL.make_extend(w, lengths)
    d2t = WL.make_d2t(w) if d2t_override == "default" else d2t_override
    d2t_orc = d2t
    if gpu_inputs is not None:
        d2t = gpu_inputs(ex, paged, d2t)
    head = HN.DeviceHead(w, stored, fp8=fp8, nvfp4=nvfp4)
    try:
        dc = head.cache(paged)
        din = head.extend_inputs(ex)
        B, G, H = w.batch, w.gamma, w.hidden
        hid = torch.zeros((G, B, H), dtype=torch.float32, device="cuda")
        lg = torch.zeros((G, B, w.draft_vocab), dtype=torch.float32, device="cuda") if with_logits else None
        toks = torch.zeros((B, G), dtype=torch.int32, device="cuda")
        d2t_dev = HN.to_device(d2t) if d2t is not None else None
        head.extend(din, dc, hidden_out=hid[0], logits_out=lg[0] if with_logits else None)
        head.decode(G, d2t_dev, dc, toks, hidden_out=hid[1:] if G > 1 else None,
                    logits_out=lg[1:] if (with_logits and G > 1) else None)
        torch.cuda.synchronize()
        gpu = dict(tokens=toks.cpu().numpy(), hidden=hid.cpu().numpy(),
                   logits=lg.cpu().numpy() if with_logits else None,
                   lengths=dc.lengths.cpu().numpy(), cache=dc.data.cpu(), err=head.error_word())
        # acceptance against synthetic targets built from the GPU's drafts
        tgt = WL.synthetic_targets(w, gpu["tokens"])
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        hist = torch.full((G + 1,), -1, dtype=torch.int32, device="cuda")
        from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
        E.eagle3_accept(toks, HN.to_device(tgt), B, G, acc, hist)
        torch.cuda.synchronize()
        gpu.update(target=tgt, acc=acc.cpu().numpy(), hist=hist.cpu().numpy())
    finally:
        head.close()

    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    W = QuantOracleWeights(stored, "fp8" if fp8 else "nvfp4") if (fp8 or nvfp4) else WL.F64Cache(stored)
    caches = [O.SeqCache(WL.as_f32(WL.cache_rows(w, b, int(lengths[b]))), w.max_ctx) for b in seqs]
    exs = WL.make_extend(w, lengths, seqs=seqs)
    if oracle_inputs is not None:
        d2t_orc = oracle_inputs(exs, d2t_orc)
    aux = [WL.as_f32(a) for a in exs.aux]
    orc = O.draft_round(w.hyper(), W, d2t_orc, w.gamma, aux, exs.tokens, exs.positions, exs.row_offsets, caches,
                        absorbed=absorbed, forced=gpu["tokens"][seqs])
    orc["caches"] = caches
    orc["lengths"] = lengths
    orc["d2t"] = d2t_orc
    return gpu, orc, seqs, paged


def check_round(w, gpu, orc, seqs, paged, tol, err=0):
    """Assert every parity rule; returns a dict of the measured errors.  ``err``: the device error word
    the round must leave (0 for valid inputs)."""
    G = w.gamma
    assert gpu["err"] == err, f"device error word {gpu['err']}, expected {err}"
    rep = {}
    # hidden states of every step
    rep["hidden"] = row_rel_err(gpu["hidden"][:, seqs], orc["hidden"])
    assert rep["hidden"] <= tol, rep
    # logits and argmax decisions
    if gpu["logits"] is not None:
        rep["logits"] = row_rel_err(gpu["logits"][:, seqs], orc["logits"])
        assert rep["logits"] <= tol, rep
    ties = 0
    d2t = orc["d2t"]        # the vocab map the oracle's round used
    for s in range(G):
        for i, b in enumerate(seqs):
            lg = orc["logits"][s, i]
            gap = O.top2_gap(lg)
            g_tok = int(gpu["tokens"][b, s])
            o_tok = int(orc["tokens"][i, s])
            if gap > GAP:
                assert g_tok == o_tok, (s, b, g_tok, o_tok, gap)
            else:
                ties += 1
                # the GPU's choice must be a near-maximal draft id whose remap is its token
                cand = np.flatnonzero(lg >= lg.max() - GAP)
                assert g_tok in set(O.d2t_remap(cand, d2t).tolist()), (s, b, g_tok)
    rep["near_ties"] = ties
    # cache: lengths and the appended latent rows
    exp_len = orc["lengths"][seqs] + w.t_new + G - 1
    np.testing.assert_array_equal(gpu["lengths"][seqs], exp_len)
    data = gpu["cache"]
    if data.dtype == torch.bfloat16:
        data = data.float()
    data = data.numpy()
    worst = 0.0
    for i, b in enumerate(seqs):
        L0 = int(orc["lengths"][b])
        n_new = w.t_new + G - 1
        rows = WL.read_rows(data, paged.block_table[b], L0, n_new, w.page_size).astype(np.float64)
        ref = orc["caches"][i].data[L0:L0 + n_new]
        worst = max(worst, row_rel_err(rows, ref))
        # rows below the old length are untouched
        old = WL.read_rows(data, paged.block_table[b], 0, L0, w.page_size)
        np.testing.assert_array_equal(old, WL.as_f32(WL.read_rows(paged.data, paged.block_table[b], 0, L0,
                                                                 w.page_size)))
    rep["cache"] = worst
    assert worst <= tol, rep
    # acceptance: bit-exact against the oracle rule on the same drafts and targets
    acc, hist = O.accept(gpu["tokens"], gpu["target"])
    np.testing.assert_array_equal(gpu["acc"], acc)
    np.testing.assert_array_equal(gpu["hist"], hist)
    return rep
