"""A sampled drafting round through the C ABI: extend (its logits give token 0), eagle3_draft_decode_sampled
for the other gamma - 1 tokens, then residual acceptance against synthetic target distributions.

The oracle follows the GPU's drawn tokens (forced continuation) and must agree on every hidden state and
logit within the usual tolerance.  Each drawn token must be the oracle's filtered sample of the GPU's own
logits for that step with the same uniform (near-boundary draws may take either neighbour, see
test_gpu_sampling), and the acceptance must match the oracle's residual rule."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import TOL_BF16, TOL_F32, row_rel_err

pytestmark = pytest.mark.gpu
EPS = 1e-4


def _sampled_round(w, T, k, p, seed, tol, philox_seed=None):
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    build.build()
    stored = WL.make_weights(w)
    lengths = WL.context_lengths(w)
    paged = WL.make_cache(w, lengths)
    ex = WL.make_extend(w, lengths)
    d2t = WL.make_d2t(w)
    d2t_np = np.zeros(w.draft_vocab, np.int64) if d2t is None else np.asarray(d2t, np.int64)
    B, G, H, Vd, Vt = w.batch, w.gamma, w.hidden, w.draft_vocab, w.target_vocab
    rng = np.random.default_rng(seed)
    u = rng.random((G, B)).astype(np.float32)
    u_dev = torch.from_numpy(u).cuda()
    if philox_seed is not None:
        # the draws come from the device generator (no host copy); the oracle takes the same stream from
        # its own statement of the generator
        u_dev = torch.empty(G * B, dtype=torch.float32, device="cuda")
        E.eagle3_philox_uniforms(philox_seed, 0, G * B, u_dev)
        u = O.philox_uniforms(philox_seed, 0, G * B).astype(np.float32).reshape(G, B)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u_dev.cpu().numpy().reshape(G, B), u)
        u_dev = u_dev.view(G, B)
    head = HN.DeviceHead(w, stored)
    try:
        dc = head.cache(paged)
        din = head.extend_inputs(ex)
        hid = torch.zeros((G, B, H), dtype=torch.float32, device="cuda")
        lg = torch.zeros((G, B, Vd), dtype=torch.float32, device="cuda")
        toks = torch.zeros((B, G), dtype=torch.int32, device="cuda")
        probs = torch.zeros((B, G, Vt), dtype=torch.float32, device="cuda")
        d2t_dev = HN.to_device(d2t) if d2t is not None else None
        head.extend(din, dc, hidden_out=hid[0], logits_out=lg[0])
        head.decode_sampled(G, d2t_dev, dc, T, k, p, lg[0], u_dev, toks, probs, Vt, True,
                            hidden_out=hid[1:] if G > 1 else None, logits_out=lg[1:] if G > 1 else None)
        torch.cuda.synchronize()
        assert head.error_word() == 0
        g_tok, g_hid, g_lg, g_probs = toks.cpu().numpy(), hid.cpu().numpy(), lg.cpu().numpy(), probs.cpu().numpy()
        # residual acceptance against synthetic target distributions over the target vocabulary
        tp = rng.dirichlet(np.ones(Vt) * 0.5, size=(B, G + 1)).astype(np.float32)
        q = g_probs
        for b in range(B):                              # some positions where the target agrees with the draft
            tp[b, 0] = q[b, 0]
        ua = rng.random((B, G)).astype(np.float32)
        ur = rng.random((B, G)).astype(np.float32)
        if philox_seed is not None:
            off = (G * B + 3) // 4
            ua = O.philox_uniforms(philox_seed, off, B * G).astype(np.float32).reshape(B, G)
            ur = O.philox_uniforms(philox_seed, off + (B * G + 3) // 4, B * G).astype(np.float32).reshape(B, G)
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        hist = torch.zeros(G + 1, dtype=torch.int32, device="cuda")
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        E.eagle3_accept_residual(dev(g_tok), dev(q), dev(tp), dev(ua), dev(ur), B, G, Vt, acc, nxt, hist)
        torch.cuda.synchronize()
        g_acc, g_nxt, g_hist = acc.cpu().numpy(), nxt.cpu().numpy(), hist.cpu().numpy()
    finally:
        head.close()

    # the oracle on the GPU's drawn tokens
    W = WL.F64Cache(stored)
    caches = [O.SeqCache(WL.as_f32(WL.cache_rows(w, b, int(lengths[b]))), w.max_ctx) for b in range(B)]
    aux = [WL.as_f32(a) for a in ex.aux]
    orc = O.draft_round(w.hyper(), W, d2t, G, aux, ex.tokens, ex.positions, ex.row_offsets, caches,
                        absorbed=True, forced=g_tok)
    assert row_rel_err(g_hid, orc["hidden"]) <= tol
    assert row_rel_err(g_lg, orc["logits"]) <= tol
    # every drawn token is the filtered sample of the GPU's own logits with the same uniform
    for s in range(G):
        for b in range(B):
            t_o, pr_o = O.sample_filtered(g_lg[s, b], T, k, p, float(u[s, b]))
            want = int(t_o + d2t_np[t_o])
            if int(g_tok[b, s]) != want:
                near = {int(a + d2t_np[a]) for du in (-EPS, 0.0, EPS) for dp in ((-EPS, 0.0, EPS) if p < 1 else (0.0,))
                        for a in [O.sample_filtered(g_lg[s, b], T, k, min(1.0, p + dp),
                                                    min(max(float(u[s, b]) + du, 0.0), 1 - 1e-9))[0]]}
                assert int(g_tok[b, s]) in near, (s, b, int(g_tok[b, s]), want)
    o_acc, o_nxt, o_hist = O.accept_residual(g_tok, q, tp, ua, ur)
    np.testing.assert_array_equal(g_acc, o_acc)
    np.testing.assert_array_equal(g_hist, o_hist)
    return g_tok, g_acc


def test_tiny_f32_sampled_round():
    w = WL.workload("tiny_f32", gamma=4, accept_p=(0.7,) * 4)
    _sampled_round(w, 0.8, 50, 0.9, 31, TOL_F32)


def test_tiny_f32_sampled_round_whole_vocab():
    w = WL.workload("tiny_f32", batch=3, gamma=3, seed=1001)
    _sampled_round(w, 1.2, 0, 1.0, 32, TOL_F32)


def test_mla_shaped_bf16_sampled_round():
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048, target_vocab=8192,
                    draft_vocab=4096, batch=3, ctx=(100, 700), t_new=2, gamma=4, accept_p=(0.7,) * 4, seed=83)
    _sampled_round(w, 0.7, 20, 0.8, 33, TOL_BF16)


def test_tiny_f32_sampled_round_device_uniforms():
    # every uniform of the round from the device Philox stream (seed counter): no host draw
    w = WL.workload("tiny_f32", gamma=4, accept_p=(0.7,) * 4, seed=1002)
    _sampled_round(w, 0.9, 40, 0.95, 35, TOL_F32, philox_seed=0x5EED)


def test_mha_tiny_f32_sampled_round():
    # the MHA head through the same sampled decode and residual acceptance
    w = WL.workload("mha_tiny_f32", gamma=4, accept_p=(0.7,) * 4)
    _sampled_round(w, 0.8, 50, 0.9, 34, TOL_F32)
