"""Pins of the oracle's elementary operations against facts fixed independently of its code:
hand examples, closed forms, invariants, library routines and brute force."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _hyper(d=64, theta=1e4, factor=40.0, L0=4096, bf=32.0, bs=1.0, ms=1.0, msa=1.0, dn=128, nh=2, dv=8, dc=16):
    return dict(qk_rope_dim=d, rope_theta=theta, yarn_factor=factor, yarn_original_max_pos=L0,
                yarn_beta_fast=bf, yarn_beta_slow=bs, yarn_mscale=ms, yarn_mscale_all_dim=msa,
                qk_nope_dim=dn, n_heads=nh, v_head_dim=dv, kv_lora_rank=dc)


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_hand_example():
    # x = (3, 4): mean square 12.5, so y = x / sqrt(12.5) * w when eps = 0
    y = O.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    assert y[0] == pytest.approx(3.0 / math.sqrt(12.5), rel=1e-15)
    assert y[1] == pytest.approx(8.0 / math.sqrt(12.5), rel=1e-15)
    # with eps the denominator is sqrt(12.5 + eps)
    y = O.rms_norm(np.array([3.0, 4.0]), np.ones(2), 0.5)
    assert y[1] == pytest.approx(4.0 / math.sqrt(13.0), rel=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 300))
    y = O.rms_norm(x, np.ones(300), 1e-6)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, np.ones(300), 0.0), O.rms_norm(x, np.ones(300), 0.0), rtol=1e-13)
    # the weight multiplies elementwise after normalisation
    w = rng.standard_normal(300)
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), y * w, rtol=1e-13)


# ---------------------------------------------------------------- YaRN
def test_yarn_factor_one_is_plain_rope():
    inv = O.yarn_inv_freq(64, 1e4, 1.0, 4096, 32.0, 1.0)
    plain = np.array([1.0 / (10000.0 ** (2 * i / 64)) for i in range(32)])
    np.testing.assert_allclose(inv, plain, rtol=1e-14)


def test_yarn_golden_band_edges_dsv3():
    g = json.load(open(os.path.join(GOLD, "yarn_dsv3.json")))
    d, theta, L0, f = g["d"], g["theta"], g["original_max_pos"], g["factor"]
    inv = O.yarn_inv_freq(d, theta, f, L0, g["beta_fast"], g["beta_slow"])
    plain = np.array([theta ** (-2 * i / d) for i in range(d // 2)])
    lo, hi = g["lo"], g["hi"]
    # below the band the plain frequency is kept; above it the frequency is divided by the factor
    np.testing.assert_allclose(inv[:lo + 1], plain[:lo + 1], rtol=1e-14)
    np.testing.assert_allclose(inv[hi:], plain[hi:] / f, rtol=1e-14)
    # inside the band it is strictly between the two
    mid = slice(lo + 1, hi)
    assert np.all(inv[mid] < plain[mid]) and np.all(inv[mid] > plain[mid] / f)
    # YaRN's defining property: kept pairs turn at least beta_fast times over the original window,
    # fully interpolated pairs at most beta_slow times
    turns = L0 * plain / (2 * math.pi)
    assert np.all(turns[:lo + 1] >= g["beta_fast"])
    assert np.all(turns[hi:] <= g["beta_slow"])
    assert turns[lo] == pytest.approx(g["rotations_pair10"], abs=0.01)
    assert turns[hi] == pytest.approx(g["rotations_pair23"], abs=0.001)
    # the blended frequency falls monotonically with the pair index
    assert np.all(np.diff(inv) < 0)


def test_yarn_mscale_golden_and_special_cases():
    g = json.load(open(os.path.join(GOLD, "yarn_dsv3.json")))
    assert O.yarn_mscale(40.0, 1.0) == pytest.approx(g["mscale_factor40_mu1"], rel=1e-15)
    assert O.yarn_mscale(1.0, 1.0) == 1.0          # no scaling without extension
    assert O.yarn_mscale(math.e ** 10, 1.0) == pytest.approx(2.0, rel=1e-15)
    # equal mscale and mscale_all_dim leave cos/sin unscaled
    h = _hyper()
    c, s = O.rope_cos_sin(np.array([0, 5]), h)
    assert np.allclose(c[0], 1.0) and np.allclose(s[0], 0.0)
    np.testing.assert_allclose(c ** 2 + s ** 2, 1.0, rtol=1e-14)
    # factor 1: sigma is the textbook 1/sqrt(d_qk)
    assert O.softmax_scale(_hyper(factor=1.0)) == pytest.approx(1 / math.sqrt(192), rel=1e-15)
    assert O.softmax_scale(_hyper()) == pytest.approx(g["mscale_factor40_mu1"] ** 2 / math.sqrt(192), rel=1e-14)


# ---------------------------------------------------------------- RoPE
def test_rope_hand_quarter_turn():
    # one pair, frequency chosen so that position 1 is a quarter turn: (1, 0) -> (0, 1)
    h = _hyper(d=2, theta=1e4, factor=1.0)
    # with d = 2 the only pair has omega = theta^0 = 1 rad per position
    x = np.array([[1.0, 0.0]])
    y = O.rope_interleaved(x, np.array([math.pi / 2]), h)
    np.testing.assert_allclose(y, [[0.0, 1.0]], atol=1e-15)
    y = O.rope_interleaved(np.array([[0.0, 1.0]]), np.array([math.pi / 2]), h)
    np.testing.assert_allclose(y, [[-1.0, 0.0]], atol=1e-15)


def test_rope_matches_complex_multiplication():
    h = _hyper()
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 64))
    pos = rng.integers(0, 100000, size=7)
    y = O.rope_interleaved(x, pos, h)
    inv = O.yarn_inv_freq(64, 1e4, 40.0, 4096, 32.0, 1.0)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos[:, None] * inv[None, :])
    np.testing.assert_allclose(y[:, 0::2], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[:, 1::2], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_invariants():
    h = _hyper()
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    # position 0 is the identity, pair norms are preserved
    np.testing.assert_allclose(O.rope_interleaved(q, np.array([0]), h), q, rtol=0, atol=0)
    y = O.rope_interleaved(q, np.array([12345]), h)
    np.testing.assert_allclose(y[0, 0::2] ** 2 + y[0, 1::2] ** 2, q[0, 0::2] ** 2 + q[0, 1::2] ** 2, rtol=1e-12)
    # relative-position invariance of the dot product
    def dot(pq, pk):
        return float((O.rope_interleaved(q, np.array([pq]), h) @ O.rope_interleaved(k, np.array([pk]), h).T)[0, 0])
    assert dot(100, 37) == pytest.approx(dot(1063, 1000), rel=1e-9)
    # composition R(a) R(b) = R(a + b)
    ab = O.rope_interleaved(O.rope_interleaved(q, np.array([300]), h), np.array([45]), h)
    np.testing.assert_allclose(ab, O.rope_interleaved(q, np.array([345]), h), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- linear / SiLU
def test_linear_brute_force():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 5))
    W = rng.standard_normal((4, 5))
    y = O.linear(x, W)
    for i in range(3):
        for j in range(4):
            s = 0.0
            for k in range(5):
                s += x[i, k] * W[j, k]
            assert y[i, j] == pytest.approx(s, rel=1e-14, abs=1e-15)


def test_silu_library_and_closed_form():
    x = np.linspace(-20, 20, 81)
    ref = torch.nn.functional.silu(torch.tensor(x, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(O.silu(x), ref, rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


# ---------------------------------------------------------------- attention
def _attn_case(seed, T=3, L=9, nh=3, dn=4, dr=2, dv=5, dc=6):
    rng = np.random.default_rng(seed)
    h = _hyper(d=dr, dn=dn, nh=nh, dv=dv, dc=dc, factor=4.0, L0=16)
    q = rng.standard_normal((T, nh, dn + dr))
    cache = rng.standard_normal((L, dc + dr))
    kv_b = rng.standard_normal((nh * (dn + dv), dc))
    pos = np.arange(L - T, L)
    return h, q, cache, kv_b, pos


def test_attention_matches_torch_sdpa():
    h, q, cache, kv_b, pos = _attn_case(4)
    nh, dn, dv, dc = h["n_heads"], h["qk_nope_dim"], h["v_head_dim"], h["kv_lora_rank"]
    o = O.mla_attention(q, pos, cache, kv_b, h)
    # explicit per-head keys / values from the raw kv_b rows
    W = kv_b.reshape(nh, dn + dv, dc)
    c, kr = cache[:, :dc], cache[:, dc:]
    sigma = O.softmax_scale(h)
    for i, p in enumerate(pos):
        for hh in range(nh):
            K = np.concatenate([c[:p + 1] @ W[hh, :dn].T, kr[:p + 1]], axis=1)
            V = c[:p + 1] @ W[hh, dn:].T
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[i, hh][None, None, None]), torch.tensor(K[None, None]),
                torch.tensor(V[None, None]), scale=sigma)[0, 0, 0].numpy()
            np.testing.assert_allclose(o[i, hh], ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    h, q, cache, kv_b, _ = _attn_case(5, T=1, L=6)
    nh, dn, dv, dc = h["n_heads"], h["qk_nope_dim"], h["v_head_dim"], h["kv_lora_rank"]
    W = kv_b.reshape(nh, dn + dv, dc)
    # a row at position 0 sees only slot 0: output is exactly slot 0's value projection
    o = O.mla_attention(q, np.array([0]), cache, kv_b, h)
    for hh in range(nh):
        np.testing.assert_allclose(o[0, hh], W[hh, dn:] @ cache[0, :dc], rtol=1e-13)
    # all-equal keys: the output is the mean of the values (equal scores)
    c2 = cache.copy()
    c2[:, dc:] = c2[0, dc:]              # same rope key everywhere
    kv2 = kv_b.reshape(nh, dn + dv, dc).copy()
    kv2[:, :dn] = 0.0                    # no-position keys contribute nothing
    o = O.mla_attention(q, np.array([5]), c2, kv2.reshape(-1, dc), h)
    for hh in range(nh):
        np.testing.assert_allclose(o[0, hh], kv2[hh, dn:] @ c2[:6, :dc].mean(axis=0), rtol=1e-12)


def test_absorbed_equals_unabsorbed():
    for seed in range(3):
        h, q, cache, kv_b, pos = _attn_case(10 + seed, T=4, L=12)
        a = O.mla_attention(q, pos, cache, kv_b, h, absorbed=False)
        b = O.mla_attention(q, pos, cache, kv_b, h, absorbed=True)
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_attention_is_convex_combination():
    # softmax rows sum to one: with W_UV = identity-like, outputs stay in the hull of the latents
    h, q, cache, kv_b, pos = _attn_case(6, T=2, L=7, dv=6, dc=6)
    nh, dn, dv, dc = h["n_heads"], h["qk_nope_dim"], h["v_head_dim"], h["kv_lora_rank"]
    W = kv_b.reshape(nh, dn + dv, dc).copy()
    W[:, dn:] = np.eye(dc)
    o = O.mla_attention(q, pos, cache, W.reshape(-1, dc), h)
    ones = np.ones(dc)
    cache1 = cache.copy()
    cache1[:, :dc] = 1.0  # every latent equal to one: any convex combination returns one
    o1 = O.mla_attention(q, pos, cache1, W.reshape(-1, dc), h)
    np.testing.assert_allclose(o1, np.broadcast_to(ones, o1.shape), rtol=1e-13)
    for i, p in enumerate(pos):
        lo = cache[:p + 1, :dc].min(axis=0)
        hi = cache[:p + 1, :dc].max(axis=0)
        assert np.all(o[i] >= lo - 1e-12) and np.all(o[i] <= hi + 1e-12)


# ---------------------------------------------------------------- argmax / d2t / accept
def test_argmax_brute_force_and_ties():
    rng = np.random.default_rng(7)
    for _ in range(50):
        v = rng.integers(-5, 5, size=37).astype(np.float64)   # many ties
        best = None
        for i, x in enumerate(v):
            if best is None or x > v[best]:
                best = i
        assert O.argmax_lowest(v) == best
    v = np.zeros(10)
    v[3] = v[7] = 2.0
    assert O.argmax_lowest(v) == 3
    assert O.top2_gap(np.array([1.0, 5.0, 4.5])) == pytest.approx(0.5)


def test_d2t_remap():
    d = np.array([0, 5, 9])
    assert list(O.d2t_remap(d, np.zeros(10, dtype=np.int32))) == [0, 5, 9]
    assert list(O.d2t_remap(d, None)) == [0, 5, 9]
    table = np.arange(10, dtype=np.int32) * 3
    assert list(O.d2t_remap(d, table)) == [0, 5 + 15, 9 + 27]


def test_accept_cases_and_brute_force():
    rng = np.random.default_rng(8)
    d = rng.integers(0, 5, size=(40, 6))
    acc, hist = O.accept(d, d)
    assert np.all(acc == 6) and hist[6] == 40 and hist.sum() == 40
    t = d.copy()
    t[:, 0] += 1
    acc, hist = O.accept(d, t)
    assert np.all(acc == 0) and hist[0] == 40
    t = rng.integers(0, 2, size=(40, 6))
    d = rng.integers(0, 2, size=(40, 6))
    acc, hist = O.accept(d, t)
    for b in range(40):
        k = next((i for i in range(6) if d[b, i] != t[b, i]), 6)
        assert acc[b] == k
    assert list(hist) == [int((acc == k).sum()) for k in range(7)]


def _sorted_topk(rng, B, G, K, vocab):
    """Distinct candidate ids per position with strictly descending log-probabilities."""
    ids = np.stack([np.stack([rng.choice(vocab, size=K, replace=False) for _ in range(G)]) for _ in range(B)])
    gaps = rng.uniform(0.05, 0.5, size=(B, G, K))
    lp = -np.cumsum(gaps, axis=2)
    return ids.astype(np.int32), lp


def test_accept_relaxed_hand_example():
    # one position, candidates 5, 9, 2 with log-probabilities -0.1, -0.5, -0.8; default delta 0.6
    ids = np.array([[[5, 9, 2]]])
    lp = np.array([[[-0.1, -0.5, -0.8]]])
    for tok, think, want in [(5, False, 1), (9, False, 0), (9, True, 1), (2, True, 0), (7, True, 0), (5, True, 1)]:
        acc, _ = O.accept_relaxed(np.array([[tok]]), ids, lp, [think], 0.6)
        assert acc[0] == want, (tok, think)


def test_accept_relaxed_reduces_to_greedy():
    rng = np.random.default_rng(11)
    B, G, K = 30, 5, 4
    ids, lp = _sorted_topk(rng, B, G, K, 12)
    # drafts: mostly the best candidate, sometimes another candidate or an outside token
    draft = ids[:, :, 0].copy()
    pick = rng.integers(0, 3, size=(B, G))
    draft[pick == 1] = ids[:, :, 1][pick == 1]
    draft[pick == 2] = 99
    greedy, ghist = O.accept(draft, ids[:, :, 0])
    # rows outside thinking follow the greedy rule whatever delta is
    acc, hist = O.accept_relaxed(draft, ids, lp, np.zeros(B, bool), 5.0)
    np.testing.assert_array_equal(acc, greedy)
    np.testing.assert_array_equal(hist, ghist)
    # a delta below every log-probability gap, or a single candidate, is greedy too
    acc, _ = O.accept_relaxed(draft, ids, lp, np.ones(B, bool), 0.01)
    np.testing.assert_array_equal(acc, greedy)
    acc, _ = O.accept_relaxed(draft, ids[:, :, :1], lp[:, :, :1], np.ones(B, bool), 5.0)
    np.testing.assert_array_equal(acc, greedy)
    # a delta above every gap accepts any listed candidate
    acc, _ = O.accept_relaxed(draft, ids, lp, np.ones(B, bool), 100.0)
    for b in range(B):
        k = 0
        while k < G and draft[b, k] != 99:
            k += 1
        assert acc[b] == k


def test_accept_relaxed_monotone_in_delta():
    rng = np.random.default_rng(12)
    B, G, K = 40, 6, 5
    ids, lp = _sorted_topk(rng, B, G, K, 10)
    draft = np.where(rng.random((B, G)) < 0.8, ids[np.arange(B)[:, None], np.arange(G)[None, :],
                                                     rng.integers(0, K, size=(B, G))], 77)
    think = rng.random(B) < 0.5
    prev = None
    for delta in [0.0, 0.1, 0.3, 0.6, 1.0, 3.0]:
        acc, hist = O.accept_relaxed(draft, ids, lp, think, delta)
        assert hist.sum() == B
        if prev is not None:
            assert np.all(acc >= prev)
        prev = acc


def test_sample_filtered_greedy_and_top1():
    l = np.array([0.5, 2.0, 2.0, -1.0], dtype=np.float32)
    for T in (0.0, 0.7):
        k = 1 if T > 0 else 0
        for u in (0.0, 0.5, 0.999):
            t, probs = O.sample_filtered(l, T, k, 1.0, u)
            assert t == 1 and probs[1] == 1.0 and probs.sum() == 1.0


def test_sample_filtered_frequencies_match_softmax():
    # inverse-CDF sampling over a fine grid of u reproduces the renormalised softmax of the kept set
    l = np.array([1.0, 0.2, -0.5, 1.5, 0.0, 0.7], dtype=np.float32)
    T = 0.8
    x = l.astype(np.float64) / T
    for top_k, top_p, keep in [(0, 1.0, [0, 1, 2, 3, 4, 5]), (3, 1.0, [3, 0, 5]), (6, 0.5, [3, 0])]:
        w = np.zeros(6)
        w[keep] = np.exp(x[keep] - x[keep].max())
        want = w / w.sum()
        n = 20000
        counts = np.zeros(6)
        for i in range(n):
            t, probs = O.sample_filtered(l, T, top_k, top_p, (i + 0.5) / n)
            counts[t] += 1
        np.testing.assert_allclose(probs, want, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(counts / n, want, atol=2e-4)


def test_sample_filtered_top_p_and_tie_order_hand_cases():
    l = np.array([2.0, 1.0, 0.0, -1.0], dtype=np.float32)    # softmax 0.644, 0.237, 0.087, 0.032
    for u in (0.0, 0.3, 0.99):
        assert O.sample_filtered(l, 1.0, 4, 0.6, u)[0] == 0
    _, probs = O.sample_filtered(l, 1.0, 4, 0.7, 0.5)
    np.testing.assert_array_equal(probs > 0, [True, True, False, False])
    # equal logits at the top-k boundary: lower indices are kept first
    _, probs = O.sample_filtered(np.array([1.0, 3.0, 3.0, 3.0, 0.0], np.float32), 1.0, 2, 1.0, 0.5)
    np.testing.assert_array_equal(probs > 0, [False, True, True, False, False])


def test_accept_residual_emits_the_target_distribution():
    # the speculative-sampling theorem: the token emitted at a position (the accepted draft, or the
    # residual draw after a rejection) is distributed as the target's p, whatever the draft's q
    rng = np.random.default_rng(13)
    V = 5
    q = rng.dirichlet(np.ones(V))
    p = rng.dirichlet(np.ones(V))
    n = 400
    out = np.zeros(V)
    for x in range(V):                       # the draft token, drawn from q
        for ia in range(n):                  # u_accept grid
            for ir in range(0, n, 8):        # u_resample grid (coarser)
                ua, ur = (ia + 0.5) / n, (ir + 4) / n
                acc, nxt, _ = O.accept_residual([[x]], q[None, None, :], np.stack([p, p])[None], [[ua]], [[ur]])
                tok = x if acc[0] == 1 else nxt[0]
                out[tok] += q[x] / (n * (n // 8))
    np.testing.assert_allclose(out, p, atol=4e-3)


def test_accept_residual_special_cases():
    p = np.array([[[0.1, 0.6, 0.3], [0.2, 0.2, 0.6], [0.5, 0.25, 0.25]]])
    # a draft distribution equal to the target's is always accepted; the bonus comes from p[gamma]
    acc, nxt, hist = O.accept_residual([[1, 2]], p[:, :2], p, [[0.999, 0.999]], [[0.1, 0.7]])
    assert acc[0] == 2 and nxt[0] == 1 and hist[2] == 1
    # a drafted token the target gives no mass is rejected; the residual excludes it
    q = np.array([[[0.0, 0.0, 1.0], [1.0, 0.0, 0.0]]])
    p0 = np.array([[[0.5, 0.5, 0.0], [1.0, 0.0, 0.0], [1.0, 0.0, 0.0]]])
    acc, nxt, _ = O.accept_residual([[2, 0]], q, p0, [[0.0, 0.0]], [[0.75, 0.0]])
    assert acc[0] == 0 and nxt[0] == 1


def test_e4m3_table_and_round_trip():
    # published E4M3 facts: largest finite 448, smallest subnormal 2^-9, smallest normal 2^-6, one NaN code
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0xFE) == -448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9 and O.e4m3_decode(0x08) == 2.0 ** -6
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    assert O.e4m3_decode(0x38) == 1.0 and O.e4m3_decode(0x40) == 2.0 and O.e4m3_decode(0x3C) == 1.5
    for c in list(range(0x7F)) + list(range(0x81, 0xFF)):
        assert O.e4m3_encode(O.e4m3_decode(c)) == c, hex(c)


def test_e4m3_rounding_ties_and_saturation():
    assert O.e4m3_encode(1.0625) == 0x38          # midpoint of 1.0 (even code 0x38) and 1.125 -> even
    assert O.e4m3_encode(1.1875) == 0x3A          # midpoint of 1.125 (0x39) and 1.25 (0x3A) -> even
    assert O.e4m3_encode(1.07) == 0x39
    assert O.e4m3_encode(1e6) == 0x7E and O.e4m3_encode(-1e6) == 0xFE
    assert O.e4m3_encode(2.0 ** -11) == 0x00     # below half the smallest subnormal


def test_e4m3_array_encoder_matches_the_scalar_rule():
    # every code value, every midpoint between neighbours (and a hair to each side), zeros, tiny and
    # saturating magnitudes, a random sweep over 2^-12 .. 2^10; both signs
    pos = np.array([O.e4m3_decode(c) for c in range(0x7F)])
    mids = (pos[1:] + pos[:-1]) / 2
    xs = np.concatenate([pos, mids, mids * (1 + 1e-9), mids * (1 - 1e-9), [0.0, 2.0 ** -11, 2.0 ** -10, 449.0,
                         464.0, 480.0, 1e6], np.exp2(np.random.default_rng(15).uniform(-12, 10, 3000))])
    xs = np.concatenate([xs, -xs])
    got = O.e4m3_encode_array(xs)
    ref = np.array([O.e4m3_encode(v) for v in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)
    assert O.e4m3_encode_array(np.array([-0.0]))[0] == O.e4m3_encode(-0.0) == 0x80


def test_quantize_rows_e4m3_error_bound():
    rng = np.random.default_rng(14)
    W = (rng.normal(0, 0.02, size=(9, 40))).astype(np.float32)
    W[3] = 0.0
    codes, scales, deq = O.quantize_rows_e4m3(W)
    assert codes.dtype == np.uint8 and scales.shape == (9,)
    # the per-element rule, written out with the scalar encoder and fp32 quotients
    for n in range(9):
        assert [O.e4m3_encode(np.float32(v) / scales[n]) for v in W[n]] == codes[n].tolist()
        assert np.all(deq[n] == np.array([O.e4m3_decode(c) for c in codes[n]]) * np.float64(scales[n]))
    amax = np.abs(W).max(axis=1)
    # each row's largest magnitude maps to 448 exactly; relative error of E4M3 <= 2^-4 per element
    for n in range(9):
        if amax[n] == 0:
            assert scales[n] == 1.0 and np.all(deq[n] == 0)
            continue
        assert np.max(np.abs(deq[n])) == pytest.approx(amax[n], rel=1e-6)
        err = np.abs(deq[n] - W[n])
        assert np.all(err <= np.maximum(np.abs(W[n]) * 2.0 ** -4, scales[n] * 2.0 ** -10) * (1 + 1e-6))


# ---------------------------------------------------------------- MHA head: rotate-half RoPE, GQA attention
def _mha_hyper(nh=4, nkv=2, d=8, factor=1.0, L0=16):
    h = _hyper(d=d, factor=factor, L0=L0)
    h.update(attention="mha", n_heads=nh, n_kv_heads=nkv, head_dim=d)
    return h


def test_rope_half_hand_quarter_turn_and_pairing():
    # d = 2: the only pair is (x_0, x_1) with omega = 1 rad per position, as in the interleaved layout
    h = _mha_hyper(d=2)
    np.testing.assert_allclose(O.rope_half(np.array([[1.0, 0.0]]), np.array([math.pi / 2]), h), [[0.0, 1.0]],
                               atol=1e-15)
    # d = 4: dimension 0 pairs with 2 (omega 1) and dimension 1 with 3 (omega theta^-1/2); the interleaved
    # layout would pair 0 with 1 instead
    h = _mha_hyper(d=4)
    y = O.rope_half(np.array([[1.0, 0.0, 0.0, 0.0]]), np.array([math.pi / 2]), h)
    np.testing.assert_allclose(y, [[0.0, 0.0, 1.0, 0.0]], atol=1e-15)


def test_rope_half_matches_complex_multiplication_and_invariants():
    h = _mha_hyper(d=64, factor=40.0, L0=4096)
    rng = np.random.default_rng(21)
    x = rng.standard_normal((7, 3, 64))
    pos = rng.integers(0, 100000, size=7)
    y = O.rope_half(x, pos, h)
    inv = O.yarn_inv_freq(64, 1e4, 40.0, 4096, 32.0, 1.0)
    z = (x[..., :32] + 1j * x[..., 32:]) * np.exp(1j * pos[:, None, None] * inv[None, None, :])
    np.testing.assert_allclose(y[..., :32], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[..., 32:], z.imag, rtol=1e-12, atol=1e-12)
    q, k = rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    np.testing.assert_allclose(O.rope_half(q, np.array([0]), h), q, rtol=0, atol=0)

    def dot(pq, pk):
        return float((O.rope_half(q, np.array([pq]), h) @ O.rope_half(k, np.array([pk]), h).T)[0, 0])
    assert dot(100, 37) == pytest.approx(dot(1063, 1000), rel=1e-9)


def test_mha_attention_matches_torch_sdpa_with_grouped_heads():
    h = _mha_hyper(nh=6, nkv=2, d=8, factor=4.0)
    rng = np.random.default_rng(22)
    T, L = 3, 11
    q = rng.standard_normal((T, 6, 8))
    cache = rng.standard_normal((L, 2 * 2 * 8))
    pos = np.arange(L - T, L)
    o = O.mha_attention(q, pos, cache, h)
    k = torch.tensor(cache[:, :16].reshape(L, 2, 8)).permute(1, 0, 2)        # [n_kv, L, d]
    v = torch.tensor(cache[:, 16:].reshape(L, 2, 8)).permute(1, 0, 2)
    kk, vv = k.repeat_interleave(3, dim=0), v.repeat_interleave(3, dim=0)     # query heads 3g..3g+2 -> g
    mask = torch.tensor(np.arange(L)[None, :] <= pos[:, None])                  # [T, L]: slot <= position
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).permute(1, 0, 2), kk, vv, attn_mask=mask, scale=O.softmax_scale(h)).permute(1, 0, 2)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)
    # the softmax scale of the MHA head: d^-1/2 times the squared YaRN attention factor
    m = 0.1 * math.log(4.0) + 1.0
    assert O.softmax_scale(h) == pytest.approx(8 ** -0.5 * m * m, rel=1e-15)


def test_mha_attention_single_slot_and_equal_keys():
    h = _mha_hyper(nh=4, nkv=1, d=8)
    rng = np.random.default_rng(23)
    q = rng.standard_normal((1, 4, 8))
    cache = rng.standard_normal((5, 16))
    # position 0 sees one slot: every head returns that slot's value row
    o = O.mha_attention(q, np.array([0]), cache, h)
    np.testing.assert_allclose(o[0], np.repeat(cache[0:1, 8:], 4, axis=0), rtol=1e-14)
    # equal keys give the mean of the visible values
    cache[:, :8] = cache[0, :8]
    o = O.mha_attention(q, np.array([4]), cache, h)
    np.testing.assert_allclose(o[0], np.repeat(cache[:, 8:].mean(axis=0, keepdims=True), 4, axis=0), rtol=1e-12)


# ---------------------------------------------------------------- NVFP4 (E2M1 codes, E4M3 block scales)
def test_e2m1_table_ties_and_saturation():
    # OCP FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    assert [O.e2m1_decode(c) for c in range(8)] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [O.e2m1_decode(c) for c in range(8, 16)] == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    # every code round-trips; midpoints go to the even code: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2,
    # 2.5 -> 2, 3.5 -> 4, 5 -> 4; above 6 saturates
    vals = np.array([O.e2m1_decode(c) for c in range(16)])
    np.testing.assert_array_equal(O.e2m1_encode_array(vals)[[c for c in range(16) if c != 8]],
                                  [c for c in range(16) if c != 8])
    got = O.e2m1_encode_array(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 1e9, -5.0, 0.26, -0.1]))
    np.testing.assert_array_equal(got, [0, 2, 2, 4, 4, 6, 6, 7, 7, 14, 1, 8])


def test_quantize_nvfp4_rule_and_error_bound():
    rng = np.random.default_rng(31)
    W = rng.normal(0, 0.02, size=(5, 64)).astype(np.float32)
    W[2, 16:32] = 0.0                                       # an all-zero block: scale code 0, codes 0
    W[4, :16] = np.float32(1e-9)                            # a block whose scale underflows E4M3
    codes, sb, g, deq = O.quantize_nvfp4(W)
    assert codes.shape == (5, 64) and sb.shape == (5, 4) and codes.max() <= 15
    amax = np.float32(np.abs(W).max())
    assert g == np.float32(amax / np.float32(2688.0))
    # the rule written out for every block, with the scalar E4M3 encoder
    six_g = np.float32(np.float32(6.0) * g)
    for n in range(5):
        for b in range(4):
            blk = W[n, 16 * b:16 * b + 16]
            s = O.e4m3_encode(np.float32(np.abs(blk).max()) / six_g)
            assert s == sb[n, b]
            eff = np.float32(np.float32(O.e4m3_decode(s)) * g)
            for k in range(16):
                q = np.float32(blk[k]) / eff if eff > 0 else 0.0
                assert O.e2m1_encode_array(np.array([q]))[0] == codes[n, 16 * b + k]
    assert np.all(sb[2, 1] == 0) and np.all(codes[2, 16:32] == 0)
    # error bound: within half a step of the E2M1 grid (<= 1 at the top of the range) times the block's
    # effective scale, plus the scale's own E4M3 rounding (the largest element maps to 6 * (1 +- 2^-4))
    for n in range(5):
        for b in range(4):
            blk = W[n, 16 * b:16 * b + 16].astype(np.float64)
            eff = O.e4m3_decode(sb[n, b]) * float(g)
            if eff == 0:
                continue
            err = np.abs(deq[n, 16 * b:16 * b + 16] - blk)
            assert np.all(err <= np.maximum(np.abs(blk) * 0.25, 0.25 * eff) * (1 + 1e-6) + 1e-12)


# ---- typical acceptance (Medusa's rule, a reading of the strategy named in the MAX walkthrough §10)
def test_accept_typical_one_hot_targets_reduce_to_greedy():
    # a one-hot target distribution has zero entropy: the threshold is min(eps, delta) < 1, so a drafted
    # token is accepted exactly when it is the target's argmax
    rng = np.random.default_rng(31)
    B, G, V = 30, 5, 17
    tgt = rng.integers(0, V, size=(B, G))
    p = np.zeros((B, G, V))
    p[np.arange(B)[:, None], np.arange(G)[None, :], tgt] = 1.0
    draft = np.where(rng.random((B, G)) < 0.75, tgt, (tgt + 1 + rng.integers(0, V - 1, size=(B, G))) % V)
    for eps, dlt in ((0.09, 0.3), (0.5, 0.9), (0.99, 0.01)):
        acc, hist = O.accept_typical(draft, p, eps, dlt)
        g_acc, g_hist = O.accept(draft, tgt)
        np.testing.assert_array_equal(acc, g_acc)
        np.testing.assert_array_equal(hist, g_hist)


def test_accept_typical_uniform_target_closed_form():
    # uniform over V: H = ln V, so the threshold is min(eps, delta / V) and p(x) = 1 / V; acceptance
    # happens exactly when delta < 1 or eps < 1 / V
    V = 10
    p = np.full((1, 1, V), 1.0 / V)
    for eps, dlt, want in ((0.09, 0.3, 1), (0.5, 1.5, 0), (0.05, 1.5, 1), (0.5, 0.99, 1), (0.2, 2.0, 0)):
        acc, _ = O.accept_typical([[3]], p, eps, dlt)
        assert acc[0] == want, (eps, dlt)


def test_accept_typical_entropy_against_library_and_product_identity():
    import scipy.stats
    # two-point distribution (0.9, 0.1): exp(-H) = 0.9^0.9 * 0.1^0.1 = 0.72247... (product identity)
    q = np.array([0.9, 0.1, 0.0])
    e_minus_h = 0.9 ** 0.9 * 0.1 ** 0.1
    assert abs(math.exp(-scipy.stats.entropy(q)) - e_minus_h) < 1e-15
    p = q[None, None, :]
    # delta exp(-H) just above / below p(x) = 0.1 decides the minority token
    dlt_hi = 0.1 / e_minus_h * (1 + 1e-9)
    dlt_lo = 0.1 / e_minus_h * (1 - 1e-9)
    assert O.accept_typical([[1]], p, 1.0, dlt_hi)[0][0] == 0
    assert O.accept_typical([[1]], p, 1.0, dlt_lo)[0][0] == 1
    # random distributions: the rule evaluated with scipy's entropy gives the same lengths
    rng = np.random.default_rng(32)
    B, G, V = 25, 4, 40
    p = rng.dirichlet(np.ones(V) * 0.2, size=(B, G))
    draft = np.argsort(-p, axis=2)[:, :, 0]
    draft = np.where(rng.random((B, G)) < 0.5, draft, rng.integers(0, V, size=(B, G)))
    eps, dlt = 0.09, 0.3
    want = np.zeros(B, dtype=np.int32)
    for b in range(B):
        k = 0
        while k < G and p[b, k, draft[b, k]] > min(eps, dlt * math.exp(-scipy.stats.entropy(p[b, k]))):
            k += 1
        want[b] = k
    np.testing.assert_array_equal(O.accept_typical(draft, p, eps, dlt)[0], want)


def test_accept_typical_monotone_in_thresholds():
    rng = np.random.default_rng(33)
    B, G, V = 40, 6, 30
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, G))
    draft = rng.integers(0, V, size=(B, G))
    prev = None
    for eps in (0.5, 0.2, 0.09, 0.03, 0.0):
        acc, hist = O.accept_typical(draft, p, eps, 0.3)
        assert hist.sum() == B
        if prev is not None:
            assert np.all(acc >= prev)
        prev = acc
    # a token outside the vocabulary is never accepted
    assert O.accept_typical([[V + 2]], p[:1, :1], 0.0, 0.0)[0][0] == 0


# ---- Philox4x64-10 (the device generator of the sampled rounds' uniforms)
def test_philox_matches_numpy_philox():
    # numpy.random.Philox is an independent implementation of the same generator; it increments its
    # counter before producing each block
    U64 = (1 << 64) - 1
    for key in ([0, 0], [123, 456], [U64, 7], [0xdeadbeefcafebabe, 0x0123456789abcdef]):
        for ctr in ([0, 0, 0, 0], [5, 0, 0, 0], [U64 - 2, 0, 0, 0], [U64, U64, 3, 9]):
            g = np.random.Philox(counter=np.array(ctr, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
            raw = [int(x) for x in g.random_raw(8)]
            c = ctr[0] + (ctr[1] << 64) + (ctr[2] << 128) + (ctr[3] << 192)
            blocks = []
            for j in (1, 2):
                cj = (c + j) & ((1 << 256) - 1)
                blocks += O.philox4x64_10([(cj >> (64 * w)) & U64 for w in range(4)], key)
            assert blocks == raw, (key, ctr)


def test_philox_uniform_stream_properties():
    u = O.philox_uniforms(2024, 0, 4000)
    assert np.all(u >= 0.0) and np.all(u < 1.0)
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)      # exact in fp32
    assert abs(u.mean() - 0.5) < 0.02 and abs(u.var() - 1.0 / 12) < 0.01
    # element i of (seed, offset) is element i + 4 * offset of (seed, 0)
    np.testing.assert_array_equal(O.philox_uniforms(2024, 3, 20), u[12:32])
    # a different seed gives a different stream
    assert not np.array_equal(O.philox_uniforms(2025, 0, 64), u[:64])
