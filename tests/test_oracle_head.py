"""Composition and structural invariants of the oracle's whole-head calls (tiny fp32 workload)."""
import numpy as np
import pytest

import oracle as O
import workloads as WL


@pytest.fixture(scope="module", params=["tiny_f32", "mha_tiny_f32"])
def tiny(request):
    w = WL.workload(request.param)
    W = WL.F32View(WL.make_weights(w))
    return w, W


def _caches(w, lengths, seqs=None):
    seqs = range(w.batch) if seqs is None else seqs
    return [O.SeqCache(WL.as_f32(WL.cache_rows(w, b, int(lengths[b]))), w.max_ctx) for b in seqs]


def test_extend_equals_sequence_of_single_row_extends(tiny):
    """One T-row extend gives the same cache rows and last hidden as T one-row extends."""
    w, W = tiny
    hy = w.hyper()
    L = WL.context_lengths(w)
    ex = WL.make_extend(w, L)
    c_all = _caches(w, L)
    out = O.draft_extend(hy, W, ex.aux, ex.tokens, ex.positions, ex.row_offsets, c_all)
    c_one = _caches(w, L)
    for b in range(w.batch):
        r0, r1 = ex.row_offsets[b], ex.row_offsets[b + 1]
        for r in range(r0, r1):
            one = O.draft_extend(hy, W, [a[r:r + 1] for a in ex.aux], ex.tokens[r:r + 1],
                                 ex.positions[r:r + 1], np.array([0, 1]), [c_one[b]])
        np.testing.assert_allclose(one["h2"][0], out["h2"][b], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(c_one[b].data, c_all[b].data, rtol=1e-11, atol=1e-11)
        assert c_one[b].length == c_all[b].length == L[b] + w.t_new


def test_batch_independence(tiny):
    """A sequence's result does not depend on its batch-mates."""
    w, W = tiny
    hy = w.hyper()
    L = WL.context_lengths(w)
    ex = WL.make_extend(w, L)
    both = O.draft_extend(hy, W, ex.aux, ex.tokens, ex.positions, ex.row_offsets, _caches(w, L))
    ex1 = WL.make_extend(w, L, seqs=[1])
    solo = O.draft_extend(hy, W, ex1.aux, ex1.tokens, ex1.positions, ex1.row_offsets, _caches(w, L, [1]))
    np.testing.assert_allclose(solo["h2"][0], both["h2"][1], rtol=1e-12)
    assert solo["d"][0] == both["d"][1]


def test_residual_pass_through(tiny):
    """Zeroed o_proj and down projections leave h2 equal to the fused hidden (the residual)."""
    w, W = tiny
    hy = w.hyper()
    W0 = dict(W)
    W0["o"] = np.zeros_like(W["o"])
    W0["down"] = np.zeros_like(W["down"])
    L = WL.context_lengths(w)
    ex = WL.make_extend(w, L)
    out = O.draft_extend(hy, W0, ex.aux, ex.tokens, ex.positions, ex.row_offsets, _caches(w, L))
    fused = O.linear(np.concatenate(list(ex.aux), axis=1), W["fc"])
    last = ex.row_offsets[1:] - 1
    np.testing.assert_allclose(out["h2"], fused[last], rtol=1e-13, atol=1e-15)
    # a zero value projection makes the attention output vanish: h1 == fused (the MHA head's new
    # value rows are zero, but its cached prefix is not, so only the MLA head's kv_b zeroes them all)
    if w.attention == "mla":
        W1 = dict(W)
        kvb = np.array(W["kv_b"]).reshape(w.n_heads, w.qk_nope_dim + w.v_head_dim, w.kv_lora_rank).copy()
        kvb[:, w.qk_nope_dim:] = 0
        W1["kv_b"] = kvb.reshape(-1, w.kv_lora_rank)
        W1["down"] = np.zeros_like(W["down"])
        out = O.draft_extend(hy, W1, ex.aux, ex.tokens, ex.positions, ex.row_offsets, _caches(w, L))
        np.testing.assert_allclose(out["h2"], fused[last], rtol=1e-13, atol=1e-15)


def test_decode_carries_previous_hidden(tiny):
    """A decode step's residual stream is the previous step's h2 (fc is skipped)."""
    w, W = tiny
    hy = w.hyper()
    W0 = dict(W)
    W0["o"] = np.zeros_like(W["o"])
    W0["down"] = np.zeros_like(W["down"])
    L = WL.context_lengths(w)
    rng = np.random.default_rng(0)
    h_prev = rng.standard_normal((w.batch, w.hidden))
    st = O.draft_decode_step(hy, W0, h_prev, np.array([5, 6]), _caches(w, L))
    np.testing.assert_allclose(st["h2"], h_prev, rtol=1e-14)


def test_fc_only_on_its_input_width(tiny):
    # fc takes exactly fc_inputs aux states (3 for the MLA head; 2 for the tiny MHA head)
    w, W = tiny
    L = WL.context_lengths(w)
    ex = WL.make_extend(w, L)
    assert len(ex.aux) == w.fc_inputs
    with pytest.raises(AssertionError):
        O.draft_extend(w.hyper(), W, ex.aux[:-1], ex.tokens, ex.positions, ex.row_offsets, _caches(w, L))


def test_decode_step_equals_one_row_extend_with_given_hidden(tiny):
    """Decode (hidden carried) and extend (hidden from fc) run the same decoder chain: feeding the
    decode step's hidden through an fc equal to [I 0 0] reproduces it."""
    w, W = tiny
    hy = w.hyper()
    L = WL.context_lengths(w)
    rng = np.random.default_rng(1)
    h_prev = rng.standard_normal((w.batch, w.hidden))
    toks = np.array([17, 1999])
    st = O.draft_decode_step(hy, W, h_prev, toks, _caches(w, L))
    Wi = dict(W)
    Wi["fc"] = np.concatenate([np.eye(w.hidden), np.zeros((w.hidden, (w.fc_inputs - 1) * w.hidden))], axis=1)
    aux = [h_prev] + [np.zeros_like(h_prev)] * (w.fc_inputs - 1)
    ex = O.draft_extend(hy, Wi, aux, toks, L.astype(np.int64), np.arange(w.batch + 1), _caches(w, L))
    np.testing.assert_allclose(ex["h2"], st["h2"], rtol=1e-12)
    np.testing.assert_allclose(ex["logits"], st["logits"], rtol=1e-11, atol=1e-12)


def test_round_structure_and_forced_continuation(tiny):
    w, W = tiny
    hy = w.hyper()
    L = WL.context_lengths(w)
    ex = WL.make_extend(w, L)
    d2t = WL.make_d2t(w)
    r = O.draft_round(hy, W, d2t, w.gamma, ex.aux, ex.tokens, ex.positions, ex.row_offsets, _caches(w, L))
    assert r["tokens"].shape == (w.batch, w.gamma)
    np.testing.assert_array_equal(r["tokens"], O.d2t_remap(r["draft"].T, d2t))
    assert np.all(r["tokens"] < w.target_vocab) and np.all(r["tokens"] >= 0)
    for s in range(w.gamma):
        for b in range(w.batch):
            assert r["draft"][s, b] == O.argmax_lowest(r["logits"][s, b])
    # forcing the oracle's own tokens changes nothing
    f = O.draft_round(hy, W, d2t, w.gamma, ex.aux, ex.tokens, ex.positions, ex.row_offsets, _caches(w, L),
                      forced=r["tokens"])
    np.testing.assert_array_equal(f["tokens"], r["tokens"])
    np.testing.assert_allclose(f["hidden"], r["hidden"], rtol=1e-13)


def test_workload_generators_are_valid():
    for name in ("tiny_f32", "dsv3_b1", "mha_tiny_f32", "mha_b1"):
        w = WL.workload(name)
        d2t = WL.make_d2t(w)
        t = np.arange(w.draft_vocab) + d2t
        assert t.min() >= 0 and t.max() < w.target_vocab
        if w.d2t == "sorted":
            assert np.all(np.diff(t) > 0)        # injective and monotone
    w = WL.workload("dsv3_b256")
    L = WL.context_lengths(w)
    assert L.min() >= 4096 and L.max() <= 16384
    draft = np.random.default_rng(0).integers(0, w.target_vocab, size=(w.batch, w.gamma))
    tgt = WL.synthetic_targets(w, draft)
    eq = (tgt == draft)
    assert np.all(tgt[~eq] != draft[~eq]) and np.all((tgt >= 0) & (tgt < w.target_vocab))
    # subset regeneration reproduces the same rows
    sub = WL.synthetic_targets(w, draft[[3, 7]], seqs=[3, 7])
    np.testing.assert_array_equal(sub, tgt[[3, 7]])
    # bf16 rounding: nearest-even on hand cases
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], dtype=np.float32)
    r = WL.bf16_to_f32(WL.f32_to_bf16_bits(x))
    np.testing.assert_array_equal(r, np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], dtype=np.float32))
