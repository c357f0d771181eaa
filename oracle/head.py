"""fp64 oracle of the EAGLE-3 draft heads (MLA, and the Llama-style MHA variant) — test
infrastructure only (see package docstring).

Notation: H hidden, n_h heads, d_q q_lora_rank, d_c kv_lora_rank, d_n qk_nope, d_r qk_rope,
d_v v_head, I intermediate, V_t target vocab, V_d draft vocab; MHA: n_kv key/value heads, d head_dim.  Weights follow nn.Linear:
W[out, in], y = x W^T.  ``hyper`` is a plain dict with those sizes and the YaRN / norm
constants; ``W`` maps weight names to arrays (any float dtype, widened to fp64 on use).
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


# ----------------------------------------------------------------------------
# Elementary operations
# ----------------------------------------------------------------------------
def rms_norm(x, w, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w.

    The draft head normalises both input streams and every sub-layer input this way,
    with rms_norm_eps = 1e-6 ([MAX-API] Eagle3DeepseekV3DraftConfig; [MAX-walkthrough] §4).
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(w)


def linear(x, W):
    """Bias-free linear layer y = x W^T with W stored [out, in] ([MAX-walkthrough] §4: fc,
    o_proj and the dense MLP carry no bias; attention_bias=False in [MAX-API])."""
    return _f64(x) @ _f64(W).T


def silu(x):
    """SiLU(x) = x * sigmoid(x) (hidden_act='silu', [MAX-API])."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


# ----------------------------------------------------------------------------
# DeepSeek YaRN rotary embedding (interleaved pairs)
# ----------------------------------------------------------------------------
def yarn_inv_freq(d, theta, factor, original_max_pos, beta_fast, beta_slow):
    """Per-pair angular frequencies of YaRN ("DeepseekYarnRotaryEmbedding", [MAX-walkthrough] §4,
    with rope_scaling beta_fast / beta_slow, §5).

    The pages name the method but do not print it; this is YaRN's published construction:
    pair i < d/2 has the plain RoPE frequency theta^(-2i/d) ("extrapolated") or that
    frequency divided by ``factor`` ("interpolated").  A pair whose wavelength fits at least
    beta_fast times into the original context keeps the plain frequency, one that fits
    fewer than beta_slow times is fully interpolated, and a linear ramp over the pair index
    blends the band in between.  The band edges are the (real) pair indices at which the
    rotation count over the original context equals beta:
        corr(beta) = d * ln(L0 / (2 pi beta)) / (2 ln theta),
    lo = max(floor(corr(beta_fast)), 0), hi = min(ceil(corr(beta_slow)), d - 1).
    """
    i = np.arange(d // 2, dtype=F64)
    extra = theta ** (-2.0 * i / d)
    inter = extra / factor

    def corr(beta):
        return d * math.log(original_max_pos / (2.0 * math.pi * beta)) / (2.0 * math.log(theta))

    lo = max(math.floor(corr(beta_fast)), 0)
    hi = min(math.ceil(corr(beta_slow)), d - 1)
    if lo == hi:
        hi += 0.001
    ramp = np.clip((i - lo) / (hi - lo), 0.0, 1.0)
    return inter * ramp + extra * (1.0 - ramp)


def yarn_mscale(factor, mscale):
    """YaRN magnitude factor m(f, mu) = 0.1 mu ln f + 1 for f > 1, else 1 (reading: not printed)."""
    if factor <= 1.0:
        return 1.0
    return 0.1 * mscale * math.log(factor) + 1.0


def rope_dim(hyper):
    """Rotated width: d_r of the MLA head; the whole head_dim d of the MHA head."""
    return hyper["head_dim"] if hyper.get("attention", "mla") == "mha" else hyper["qk_rope_dim"]


def rope_cos_sin(positions, hyper):
    """cos/sin [len(positions), d/2] (d = rope_dim) of angle p * omega_i, scaled by
    m(f, mscale) / m(f, mscale_all_dim) (reading)."""
    d = rope_dim(hyper)
    inv = yarn_inv_freq(d, hyper["rope_theta"], hyper["yarn_factor"], hyper["yarn_original_max_pos"],
                        hyper["yarn_beta_fast"], hyper["yarn_beta_slow"])
    ang = _f64(positions)[:, None] * inv[None, :]
    scale = yarn_mscale(hyper["yarn_factor"], hyper["yarn_mscale"]) / \
        yarn_mscale(hyper["yarn_factor"], hyper["yarn_mscale_all_dim"])
    return np.cos(ang) * scale, np.sin(ang) * scale


def rope_interleaved(x, positions, hyper):
    """Rotate interleaved pairs (x_2i, x_2i+1) by angle p * omega_i (rope_interleave=True,
    [MAX-API]); reading: the pairs are rotated in place, counter-clockwise:
        x'_2i   = x_2i cos - x_2i+1 sin
        x'_2i+1 = x_2i sin + x_2i+1 cos.
    ``x`` is [T, ..., d_r] with one position per leading row."""
    x = _f64(x)
    cos, sin = rope_cos_sin(positions, hyper)
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (cos.shape[1],)
    cos = cos.reshape(shape)
    sin = sin.reshape(shape)
    a = x[..., 0::2]
    b = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


def rope_half(x, positions, hyper):
    """Llama-style rotary embedding of the MHA head (LlamaForCausalLMEagle3, "Eagle3 DeepseekV3 in
    MAX" §11): dimension i pairs with i + d/2 (reading: the Llama "rotate half" layout), both rotated
    by angle p * omega_i counter-clockwise:
        x'_i       = x_i cos - x_{i+d/2} sin
        x'_{i+d/2} = x_i sin + x_{i+d/2} cos.
    ``x`` is [T, ..., d] with one position per leading row."""
    x = _f64(x)
    cos, sin = rope_cos_sin(positions, hyper)
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (cos.shape[1],)
    cos = cos.reshape(shape)
    sin = sin.reshape(shape)
    h = x.shape[-1] // 2
    a = x[..., :h]
    b = x[..., h:]
    return np.concatenate([a * cos - b * sin, a * sin + b * cos], axis=-1)


def softmax_scale(hyper):
    """sigma = d_qk^(-1/2) * m(f, mscale_all_dim)^2 with d_qk = d_n + d_r (MLA) or head_dim (MHA)
    (reading: YaRN attention scaling folded into the softmax scale, as DeepSeek's MLA does)."""
    m = yarn_mscale(hyper["yarn_factor"], hyper["yarn_mscale_all_dim"])
    if hyper.get("attention", "mla") == "mha":
        return hyper["head_dim"] ** -0.5 * m * m
    return (hyper["qk_nope_dim"] + hyper["qk_rope_dim"]) ** -0.5 * m * m


# ----------------------------------------------------------------------------
# MLA attention over a one-layer latent cache
# ----------------------------------------------------------------------------
def split_kv_b(kv_b, hyper):
    """kv_b [n_h (d_n + d_v), d_c] -> (W_UK [n_h, d_n, d_c], W_UV [n_h, d_v, d_c]).

    Reading: kv_b's output is viewed per head as [d_n | d_v] (key part first)."""
    nh, dn, dv, dc = hyper["n_heads"], hyper["qk_nope_dim"], hyper["v_head_dim"], hyper["kv_lora_rank"]
    w = _f64(kv_b).reshape(nh, dn + dv, dc)
    return w[:, :dn, :], w[:, dn:, :]


def mla_attention(q, positions, cache, kv_b, hyper, absorbed=False):
    """Attention of query rows over one sequence's latent cache ([MAX-walkthrough] §4: a single
    MLA decoder layer; its cache is a one-layer view of the target's, [MAX-API]).

    q        [T, n_h, d_n + d_r]   (q_pe part already rotated)
    cache    [L, d_c + d_r]        rows [c_kv_hat | k_r_rot] indexed by position
    returns  o [T, n_h, d_v]

    Row i at position p attends to cache slots 0..p (causal; a decode row sees itself).
    Unabsorbed (the definition): k_h,t = [W_UK,h c_t ; k_r,t], v_h,t = W_UV,h c_t,
    s_t = sigma q_h . k_h,t, o_h = sum_t softmax(s)_t v_h,t.
    ``absorbed=True`` evaluates the same quantity as q_lat,h = W_UK,h^T q_nope,h,
    s_t = sigma (q_lat,h . c_t + q_pe,h . k_r,t), o_h = W_UV,h (sum_t p_t c_t); the tests pin
    it to the unabsorbed form, and large parity cases use it to keep the fp64 cost low.
    """
    q = _f64(q)
    cache = _f64(cache)
    dn, dc = hyper["qk_nope_dim"], hyper["kv_lora_rank"]
    sigma = softmax_scale(hyper)
    W_UK, W_UV = split_kv_b(kv_b, hyper)
    T, nh = q.shape[0], q.shape[1]
    out = np.empty((T, nh, hyper["v_head_dim"]), dtype=F64)
    maxp = int(np.max(positions)) + 1
    c = cache[:maxp, :dc]
    kr = cache[:maxp, dc:]
    if not absorbed:
        k_nope = np.einsum("tc,hnc->htn", c, W_UK)   # [n_h, L, d_n]
        v = np.einsum("tc,hvc->htv", c, W_UV)        # [n_h, L, d_v]
    for i in range(T):
        n = int(positions[i]) + 1
        q_nope = q[i, :, :dn]
        q_pe = q[i, :, dn:]
        rope_part = q_pe @ kr[:n].T                                   # [n_h, n]
        if absorbed:
            q_lat = np.einsum("hn,hnc->hc", q_nope, W_UK)             # [n_h, d_c]
            s = sigma * (q_lat @ c[:n].T + rope_part)
        else:
            s = sigma * (np.einsum("hn,htn->ht", q_nope, k_nope[:, :n]) + rope_part)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        if absorbed:
            o_lat = p @ c[:n]                                         # [n_h, d_c]
            out[i] = np.einsum("hc,hvc->hv", o_lat, W_UV)
        else:
            out[i] = np.einsum("ht,htv->hv", p, v[:, :n])
    return out


def mha_attention(q, positions, cache, hyper):
    """Grouped-query attention of the MHA head over its own one-layer cache ("Eagle3 DeepseekV3 in
    MAX" §11: the Llama-style Eagle3 head; [MAX-API] Eagle3MHADeepseekV3DraftArchConfig: its own KV,
    one layer, bf16).

    q        [T, n_h, d]          (rotated)
    cache    [L, 2 n_kv d]        rows [k_rot (n_kv x d) | v (n_kv x d)] indexed by position
    returns  o [T, n_h, d]

    Query head h reads key/value head h // (n_h / n_kv) (reading: consecutive query heads share a
    key/value head, as Llama's grouped-query attention repeats them).  Row i at position p attends
    to slots 0..p: s_t = sigma q_h . k_g,t, o_h = sum_t softmax(s)_t v_g,t.
    """
    q = _f64(q)
    cache = _f64(cache)
    nh, nkv, d = hyper["n_heads"], hyper["n_kv_heads"], hyper["head_dim"]
    G = nh // nkv
    sigma = softmax_scale(hyper)
    T = q.shape[0]
    k = cache[:, :nkv * d].reshape(-1, nkv, d)
    v = cache[:, nkv * d:].reshape(-1, nkv, d)
    out = np.empty((T, nh, d), dtype=F64)
    for i in range(T):
        n = int(positions[i]) + 1
        for h in range(nh):
            g = h // G
            s = sigma * (k[:n, g] @ q[i, h])
            s = s - s.max()
            p = np.exp(s)
            p /= p.sum()
            out[i, h] = p @ v[:n, g]
    return out


# ----------------------------------------------------------------------------
# The decoder chain
# ----------------------------------------------------------------------------
class SeqCache:
    """One sequence's logical latent cache: fp64 rows [capacity, d_c + d_r] and its length."""

    def __init__(self, rows, capacity):
        rows = _f64(rows)
        self.data = np.zeros((capacity, rows.shape[1]), dtype=F64)
        self.data[:rows.shape[0]] = rows
        self.length = rows.shape[0]

    def copy(self):
        c = SeqCache(self.data[:0], self.data.shape[0])
        c.data = self.data.copy()
        c.length = self.length
        return c


def decoder_rows(hyper, W, f, tokens, positions, cache: SeqCache, absorbed=False, trace=None):
    """One decoder pass over T rows of one sequence ([MAX-walkthrough] §4, Eagle3MLADraft.__call__).

    f       [T, H]  fused hidden: fc output (extend) or the previous step's h2 (decode);
                    it is also the residual stream (reading)
    tokens  [T]     target-vocab ids; the embedding is the target's table ([MAX-walkthrough] §5)
    Appends the rows' latent entries at their positions, returns h2 [T, H] (before the final norm).
    """
    eps = hyper["rms_eps"]
    nh, dn, dr, dc = hyper["n_heads"], hyper["qk_nope_dim"], hyper["qk_rope_dim"], hyper["kv_lora_rank"]
    f = _f64(f)
    T = f.shape[0]
    positions = np.asarray(positions, dtype=np.int64)
    e = _f64(W["embed"][np.asarray(tokens, dtype=np.int64)])
    # two streams normalised separately, then concatenated to 2H: [norm(embed) | norm(fused)]
    # ([ModelOpt-EAGLE] part 3; [MAX-walkthrough] §4; the order is a reading)
    x = np.concatenate([rms_norm(e, W["input_norm"], eps), rms_norm(f, W["hidden_norm"], eps)], axis=1)
    need = int(positions.max()) + 1
    if need > cache.data.shape[0]:
        grow = np.zeros((need - cache.data.shape[0], cache.data.shape[1]), dtype=F64)
        cache.data = np.concatenate([cache.data, grow], axis=0)
    if hyper.get("attention", "mla") == "mha":
        # Llama-style attention at 2H input ("Eagle3 DeepseekV3 in MAX" §11; [ModelOpt-EAGLE] part 3):
        # q, k, v projections, rotary on q and k, own cache append, grouped-query attention
        nkv, d = hyper["n_kv_heads"], hyper["head_dim"]
        q = rope_half(linear(x, W["q_proj"]).reshape(T, nh, d), positions, hyper)
        k = rope_half(linear(x, W["k_proj"]).reshape(T, nkv, d), positions, hyper)
        v = linear(x, W["v_proj"])
        cache.data[positions] = np.concatenate([k.reshape(T, nkv * d), v], axis=1)
        cache.length = max(cache.length, need)
        o = mha_attention(q, positions, cache.data, hyper)
        h1 = linear(o.reshape(T, -1), W["o"]) + f
        y = rms_norm(h1, W["post_attn_norm"], eps)
        m = silu(linear(y, W["gate"])) * linear(y, W["up"])
        h2 = linear(m, W["down"]) + h1
        if trace is not None:
            trace.update(x=x, q=q, k=k, v=v, o=o, h1=h1, y=y, m=m, h2=h2)
        return h2
    # MLA projections at 2H input ([ModelOpt-EAGLE] part 3: first-layer q/k/v input doubled)
    c_q = rms_norm(linear(x, W["q_a"]), W["q_a_norm"], eps)
    kv = linear(x, W["kv_a"])
    c_kv = rms_norm(kv[:, :dc], W["kv_a_norm"], eps)
    k_r = rope_interleaved(kv[:, dc:], positions, hyper)
    q = linear(c_q, W["q_b"]).reshape(T, nh, dn + dr)
    q[:, :, dn:] = rope_interleaved(q[:, :, dn:], positions, hyper)
    # latent KV append: slot = position
    cache.data[positions] = np.concatenate([c_kv, k_r], axis=1)
    cache.length = max(cache.length, need)
    o = mla_attention(q, positions, cache.data, W["kv_b"], hyper, absorbed=absorbed)
    # o_proj (heads * v_head_dim -> H) and residual; post-attention norm; dense SiLU MLP; residual
    h1 = linear(o.reshape(T, -1), W["o"]) + f
    y = rms_norm(h1, W["post_attn_norm"], eps)
    m = silu(linear(y, W["gate"])) * linear(y, W["up"])
    h2 = linear(m, W["down"]) + h1
    if trace is not None:
        trace.update(x=x, c_q=c_q, c_kv=c_kv, k_r=k_r, q=q, o=o, h1=h1, y=y, m=m, h2=h2)
    return h2


def final_logits(hyper, W, h2):
    """Final RMSNorm and the head's own lm_head over the draft vocabulary
    ([MAX-walkthrough] §4; [ModelOpt-EAGLE] part 4: bias-free Linear(H, draft_vocab))."""
    z = rms_norm(h2, W["final_norm"], hyper["rms_eps"])
    return linear(z, W["lm_head"])


def argmax_lowest(v):
    """Index of the maximum of a 1-D vector; among equal maxima the lowest index (reading)."""
    v = _f64(v)
    return int(np.flatnonzero(v == v.max())[0])


def top2_gap(v):
    """Difference between the largest and second-largest entries of a 1-D vector."""
    s = np.sort(_f64(v))
    return float(s[-1] - s[-2])


def d2t_remap(d, d2t):
    """Draft id -> target id by adding the per-id offset: t = d + d2t[d]
    ([ModelOpt-EAGLE] part 4); identity when no table is given."""
    d = np.asarray(d, dtype=np.int64)
    if d2t is None:
        return d.astype(np.int32)
    return (d + np.asarray(d2t, dtype=np.int64)[d]).astype(np.int32)


# ----------------------------------------------------------------------------
# Head calls
# ----------------------------------------------------------------------------
def draft_extend(hyper, W, aux, tokens, positions, row_offsets, caches, absorbed=False):
    """Extend: fc fuses the aux states (three for the MLA head: early, middle, late; two or three for
    the MHA head, as fc's width says, "Eagle3 DeepseekV3 in MAX" §11) to H with no bias
    ([MAX-walkthrough] §4; [ModelOpt-EAGLE] part 2), then the decoder chain over each
    sequence's new rows; the last row of each sequence is scored ([MAX-walkthrough] §4:
    last-token gather by input_row_offsets).

    aux: fc_inputs arrays [N, H] (3 unless hyper says otherwise); caches: list of SeqCache (mutated).
    Returns dict(h2 [B, H], logits [B, V_d], d [B]).
    """
    B = len(row_offsets) - 1
    fused_in = np.concatenate([_f64(a) for a in aux], axis=1)        # [N, fc_inputs H]
    assert fused_in.shape[1] == hyper.get("fc_inputs", 3) * hyper["hidden"], "fc's input width"
    h2_last, logits = [], []
    for b in range(B):
        r0, r1 = int(row_offsets[b]), int(row_offsets[b + 1])
        f = linear(fused_in[r0:r1], W["fc"])
        h2 = decoder_rows(hyper, W, f, tokens[r0:r1], positions[r0:r1], caches[b], absorbed)
        h2_last.append(h2[-1])
        logits.append(final_logits(hyper, W, h2[-1:])[0])
    logits = np.stack(logits)
    return dict(h2=np.stack(h2_last), logits=logits, d=np.array([argmax_lowest(l) for l in logits]))


def draft_decode_step(hyper, W, h_prev, tokens, caches, absorbed=False):
    """One autoregressive draft step ([MAX-walkthrough] §9: decode steps, one token per sequence;
    [ModelOpt-EAGLE] TTT section: each step feeds on the previous step's own hidden state).
    The carried H-wide hidden skips fc ([MAX-walkthrough] §4).  Token of sequence b sits at
    position = current cache length of b."""
    B = len(tokens)
    h2s, logits = [], []
    for b in range(B):
        pos = np.array([caches[b].length])
        h2 = decoder_rows(hyper, W, _f64(h_prev[b])[None, :], np.array([tokens[b]]), pos, caches[b], absorbed)
        h2s.append(h2[0])
        logits.append(final_logits(hyper, W, h2)[0])
    logits = np.stack(logits)
    return dict(h2=np.stack(h2s), logits=logits, d=np.array([argmax_lowest(l) for l in logits]))


def draft_round(hyper, W, d2t, gamma, aux, tokens, positions, row_offsets, caches,
                absorbed=False, forced=None):
    """A drafting round: the extend gives the first draft token, then gamma - 1 decode steps;
    every draft id is mapped to the target vocab before it is output and before it is
    embedded (reading; the embedding table is the target's).

    ``forced`` [B, gamma] (optional) feeds those tokens forward instead of the oracle's own
    choices (used where a near-tie lets a correct implementation pick another token).
    Returns dict(tokens [B, gamma] (oracle's own choices), hidden [gamma, B, H],
    logits [gamma, B, V_d], draft [gamma, B]).
    """
    ext = draft_extend(hyper, W, aux, tokens, positions, row_offsets, caches, absorbed)
    B = len(row_offsets) - 1
    toks = np.zeros((B, gamma), dtype=np.int32)
    hid, lgs, drafts = [ext["h2"]], [ext["logits"]], [ext["d"]]
    toks[:, 0] = d2t_remap(ext["d"], d2t)
    h = ext["h2"]
    for s in range(1, gamma):
        feed = toks[:, s - 1] if forced is None else np.asarray(forced)[:, s - 1]
        st = draft_decode_step(hyper, W, h, feed, caches, absorbed)
        toks[:, s] = d2t_remap(st["d"], d2t)
        hid.append(st["h2"])
        lgs.append(st["logits"])
        drafts.append(st["d"])
        h = st["h2"]
    return dict(tokens=toks, hidden=np.stack(hid), logits=np.stack(lgs), draft=np.stack(drafts))


def accept(draft, target):
    """Greedy acceptance ([MAX-walkthrough] §10: greedy argmax acceptance): the accepted length of a
    sequence is the number of leading positions where the drafted token equals the target's.
    Returns (acc [B], hist [gamma + 1]) with hist[k] = number of sequences with acc == k."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    B, G = draft.shape
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        k = 0
        while k < G and draft[b, k] == target[b, k]:
            k += 1
        acc[b] = k
    hist = np.zeros(G + 1, dtype=np.int32)
    for k in acc:
        hist[k] += 1
    return acc, hist


def accept_relaxed(draft, topk_ids, topk_logprobs, in_thinking, delta):
    """Relaxed acceptance inside thinking blocks ([MAX-walkthrough] §10: use_relaxed_acceptance_for_
    thinking with relaxed_topk and relaxed_delta; §8: the per-row in_thinking_phase flag).

    Reading of the pages: a row in its thinking phase accepts a drafted token when it is one of the
    target's top-k candidates whose log-probability is at least the best candidate's minus delta; a row
    outside it accepts only the target's best candidate (the greedy rule; among equal best
    log-probabilities the first listed wins).  The accepted length counts leading accepted positions.
    draft [B, G]; topk_ids, topk_logprobs [B, G, k]; in_thinking [B] (bool).  Returns (acc, hist) like
    ``accept``.  The comparison lp >= best - delta is the plain real-number one on the given values:
    the log-probabilities and delta are single-precision inputs, widened exactly to fp64, where the
    threshold is formed."""
    draft = np.asarray(draft)
    ids = np.asarray(topk_ids)
    lp = np.asarray(topk_logprobs, dtype=np.float32).astype(np.float64)
    delta = float(np.float32(delta))
    think = np.asarray(in_thinking, dtype=bool)
    B, G = draft.shape
    K = ids.shape[2]

    def matches(b, i):
        best = max(lp[b, i, j] for j in range(K))
        if not think[b]:
            first = min(j for j in range(K) if lp[b, i, j] == best)
            return draft[b, i] == ids[b, i, first]
        return any(ids[b, i, j] == draft[b, i] and lp[b, i, j] >= best - delta for j in range(K))

    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        k = 0
        while k < G and matches(b, k):
            k += 1
        acc[b] = k
    hist = np.zeros(G + 1, dtype=np.int32)
    for k in acc:
        hist[k] += 1
    return acc, hist


def sample_filtered(logits, temperature, top_k, top_p, u):
    """Sampled draft token ([MAX-walkthrough] §3.1 and §10: sampling parameters of the drafts; §8: a seed
    counter feeds the sampler).  The uniform u in [0, 1) is an input, so both sides draw the same number.

    Reading of the pages, which name the parameters but not their composition: temperature 0 is the
    greedy argmax (lowest index among equal maxima).  Otherwise x = logits / temperature (in fp64 from
    the given logits); top_k > 0 keeps the top_k largest x, lower indices first among equal values;
    top_p < 1 then keeps the shortest prefix of those, in the order (x descending, index ascending), whose softmax
    mass reaches top_p of the kept mass.  The kept tokens' softmax weights are renormalised and u picks
    the token by inverse CDF over the kept tokens in ascending index order.
    Returns (token, probs) with probs [V] the final distribution (zero outside the kept set)."""
    l = np.asarray(logits, dtype=np.float32)
    V = l.shape[0]
    probs = np.zeros(V, dtype=np.float64)
    if temperature == 0.0:
        t = int(np.flatnonzero(l == l.max())[0])
        probs[t] = 1.0
        return t, probs
    x = l.astype(np.float64) / float(temperature)
    order = sorted(range(V), key=lambda i: (-float(x[i]), i))
    kept = order[:top_k] if top_k > 0 else order
    m = float(x[kept[0]])
    w = np.array([math.exp(float(x[i]) - m) for i in kept])
    if top_p < 1.0:
        cum, n = 0.0, 0
        total = w.sum()
        while n < len(kept):
            cum += w[n]
            n += 1
            if cum >= top_p * total:
                break
        kept, w = kept[:n], w[:n]
    by_index = sorted(range(len(kept)), key=lambda j: kept[j])
    total = w.sum()
    cum, token = 0.0, kept[by_index[-1]]
    for j in by_index:
        cum += w[j]
        if u * total < cum:
            token = kept[j]
            break
    for j, i in enumerate(kept):
        probs[i] = w[j] / total
    return int(token), probs


def accept_residual(draft, draft_probs, target_probs, u_accept, u_resample):
    """Residual (rejection-sampling) acceptance ([MAX-walkthrough] §10: the residual strategy of
    --rejection-sampling-strategy).  The speculative-sampling rule: position i accepts its drafted
    token x with probability min(1, p_i(x) / q_i(x)), tested as u_accept[b, i] * q_i(x) < p_i(x); the
    first rejected position instead emits a token drawn from the residual max(0, p_i - q_i),
    renormalised, by inverse CDF in ascending token order with u_resample[b, i]; if every position is
    accepted the bonus token is drawn from p_gamma with u_resample[b, gamma - 1].
    draft [B, G] target-vocab ids; draft_probs [B, G, V] (the drafts' final distributions mapped to
    the target vocabulary); target_probs [B, G + 1, V].  Returns (acc [B], next_token [B], hist)."""
    draft = np.asarray(draft)
    q = np.asarray(draft_probs, dtype=np.float64)
    p = np.asarray(target_probs, dtype=np.float64)
    ua = np.asarray(u_accept, dtype=np.float64)
    ur = np.asarray(u_resample, dtype=np.float64)
    B, G = draft.shape
    V = p.shape[2]

    def inverse_cdf(w, u):
        total = w.sum()
        cum = 0.0
        last = max(i for i in range(V) if w[i] > 0) if total > 0 else V - 1
        for i in range(V):
            cum += w[i]
            if w[i] > 0 and u * total < cum:
                return i
        return last

    acc = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        k = 0
        while k < G:
            x = int(draft[b, k])
            if ua[b, k] * q[b, k, x] < p[b, k, x]:
                k += 1
                continue
            break
        acc[b] = k
        if k < G:
            nxt[b] = inverse_cdf(np.maximum(p[b, k] - q[b, k], 0.0), ur[b, k])
        else:
            nxt[b] = inverse_cdf(p[b, G], ur[b, G - 1])
    hist = np.zeros(G + 1, dtype=np.int32)
    for k in acc:
        hist[k] += 1
    return acc, nxt, hist


# --------------------------------------------------------------------------- FP8 draft weights
def e4m3_decode(code):
    """Value of an FP8 E4M3 code (OCP 8-bit floating point, E4M3: sign, 4 exponent bits with bias 7, 3
    mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 is NaN, largest finite 448)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_POS = np.array([e4m3_decode(c) for c in range(0x7F)])      # codes 0 .. 126, ascending values
_E4M3_ALL = np.array([e4m3_decode(c) for c in range(256)])       # value of every code (NaN at 0x7F, 0xFF)


def e4m3_encode(x):
    """Nearest E4M3 code of x, ties to the even code, saturating at +-448 (the satfinite conversion)."""
    x = float(x)
    sign = 0x80 if (x < 0 or (x == 0 and math.copysign(1.0, x) < 0)) else 0
    a = min(abs(x), 448.0)
    i = int(np.searchsorted(_E4M3_POS, a))          # first code with value >= a
    if i == 0:
        return sign
    lo, hi = i - 1, min(i, 0x7E)
    dl, dh = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    if dl < dh or (dl == dh and lo % 2 == 0):
        return sign | lo
    return sign | hi


def e4m3_encode_array(x):
    """e4m3_encode over an array (the same nearest-code rule, ties to the even code, saturation at
    +-448), for matrices too large for the scalar loop.  Returns uint8 codes of x's shape."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    a = np.minimum(np.abs(x), 448.0)
    i = np.searchsorted(_E4M3_POS, a)               # first code with value >= a
    lo = np.maximum(i - 1, 0)
    hi = np.minimum(i, 0x7E)
    dl = a - _E4M3_POS[lo]
    dh = _E4M3_POS[hi] - a
    pick_lo = (dl < dh) | ((dl == dh) & (lo % 2 == 0))
    code = np.where(i == 0, 0, np.where(pick_lo, lo, hi)).astype(np.uint8)
    return code | sign


def quantize_rows_e4m3(W):
    """Per-output-row FP8 weights ("EAGLE head deep dive", deployment: the drafter quantized to FP8 by
    post-training quantization with weight scales).  Reading: scale_n = max_k |W[n, k]| / 448 (1 for an
    all-zero row), q[n, k] = E4M3(W[n, k] / scale_n), both in fp32 as the GPU forms them; the weight the
    head then uses is decode(q) * scale_n.  Returns (codes uint8 [N, K], scales fp32 [N], dequantized
    fp64 [N, K])."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    amax = np.abs(W).max(axis=1)
    scales = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    inv = (W / scales[:, None]).astype(np.float32)   # fp32 division, as the GPU divides
    codes = e4m3_encode_array(inv)
    deq = _E4M3_ALL[codes] * scales[:, None].astype(np.float64)
    return codes, scales, deq


# --------------------------------------------------------------------------- NVFP4 draft weights
_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])     # codes 0..7 (sign in bit 3)


def e2m1_decode(code):
    """Value of a 4-bit E2M1 code (OCP FP4: sign bit 3, 2 exponent bits with bias 1, 1 mantissa bit,
    subnormal 0.5 at exponent 0, largest 6, no infinities or NaN)."""
    code = int(code) & 0xF
    v = _E2M1_POS[code & 7]
    return -v if code & 8 else v


def e2m1_encode_array(x):
    """Nearest E2M1 code of each x, ties to the even code, magnitudes above 6 saturating to 6."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 8, 0).astype(np.uint8)
    a = np.minimum(np.abs(x), 6.0)
    i = np.searchsorted(_E2M1_POS, a)
    lo = np.maximum(i - 1, 0)
    hi = np.minimum(i, 7)
    dl = a - _E2M1_POS[lo]
    dh = _E2M1_POS[hi] - a
    pick_lo = (dl < dh) | ((dl == dh) & (lo % 2 == 0))
    code = np.where(i == 0, 0, np.where(pick_lo, lo, hi)).astype(np.uint8)
    return code | sign


def quantize_nvfp4(W):
    """NVFP4 weights ("EAGLE head deep dive", deployment: the drafter quantized to NVFP4 by post-training
    quantization; the format is not printed).  Reading, the published NVFP4 layout: E2M1 values, one
    E4M3 scale per 16 consecutive weights of a row, one fp32 scale per matrix, all formed in fp32 as the
    GPU forms them:
        g   = max |W| / (448 * 6)                           (1 for an all-zero matrix)
        s_b = E4M3(max_{k in b} |W[n, k]| / (6 g))          (6 g rounded first)
        e_b = decode(s_b) * g                               (the block's effective scale, fp32)
        q   = E2M1(W / e_b), or 0 where e_b == 0
    and the head uses decode(q) * decode(s_b) * g.  Returns (codes uint8 [N, K] (one code per element,
    0..15), block scale codes uint8 [N, K/16], g fp32, dequantized fp64 [N, K])."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 16 == 0
    amax = np.float32(np.abs(W).max())
    g = np.float32(amax / np.float32(2688.0)) if amax > 0 else np.float32(1.0)
    six_g = np.float32(np.float32(6.0) * g)
    blocks = W.reshape(N, K // 16, 16)
    bmax = np.abs(blocks).max(axis=2)
    sb = e4m3_encode_array((bmax / six_g).astype(np.float32))                 # fp32 quotient
    eff = (_E4M3_ALL[sb].astype(np.float32) * g).astype(np.float32)          # fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = np.where(eff[:, :, None] > 0, blocks / eff[:, :, None], np.float32(0.0)).astype(np.float32)
    codes = e2m1_encode_array(quot).reshape(N, K)
    vals = np.where(codes & 8, -1.0, 1.0) * _E2M1_POS[codes & 7]
    deq = vals.reshape(N, K // 16, 16) * _E4M3_ALL[sb][:, :, None] * np.float64(g)
    return codes, sb, g, deq.reshape(N, K)


def accept_typical(draft, target_probs, epsilon, delta):
    """Typical acceptance ([MAX-walkthrough] §10 names "typical-acceptance" among the values of
    --rejection-sampling-strategy without stating the rule).

    Reading: the published typical-acceptance rule of Medusa (Cai et al. 2024): the drafted token x at
    position i is accepted when the target's probability of it exceeds min(epsilon, delta exp(-H(p_i))),
    with H(p_i) = -sum_v p_i(v) ln p_i(v) the entropy (nats) of the target's distribution there.  The
    accepted length counts leading accepted positions; a token outside the vocabulary is never
    accepted.  draft [B, G] ids; target_probs [B, G, V].  Returns (acc [B], hist [G + 1])."""
    draft = np.asarray(draft)
    p = np.asarray(target_probs, dtype=np.float64)
    B, G = draft.shape
    V = p.shape[2]
    eps, dlt = float(epsilon), float(delta)

    def entropy(q):
        h = 0.0
        for v in np.flatnonzero(q > 0):
            h -= q[v] * math.log(q[v])
        return h

    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        k = 0
        while k < G:
            x = int(draft[b, k])
            if not 0 <= x < V:
                break
            thr = min(eps, dlt * math.exp(-entropy(p[b, k])))
            if not p[b, k, x] > thr:
                break
            k += 1
        acc[b] = k
    hist = np.zeros(G + 1, dtype=np.int32)
    for k in acc:
        hist[k] += 1
    return acc, hist


# Philox4x64-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
# ten rounds of two 64 x 64 -> 128-bit multiplications on a 4-word counter, with a 2-word key bumped by
# the Weyl constants after each round.
_PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
_PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)
_U64 = (1 << 64) - 1


def philox4x64_10(counter, key):
    """One Philox4x64-10 block: four 64-bit words from a 4-word counter and a 2-word key."""
    x = [int(w) & _U64 for w in counter]
    k0, k1 = int(key[0]) & _U64, int(key[1]) & _U64
    for _ in range(10):
        p0 = _PHILOX_M[0] * x[0]
        p1 = _PHILOX_M[1] * x[2]
        x = [((p1 >> 64) ^ x[1] ^ k0) & _U64, p1 & _U64, ((p0 >> 64) ^ x[3] ^ k1) & _U64, p0 & _U64]
        k0 = (k0 + _PHILOX_W[0]) & _U64
        k1 = (k1 + _PHILOX_W[1]) & _U64
    return x


def philox_uniforms(seed, offset, n):
    """The stream of uniforms in [0, 1) of the device generator (eagle3_philox_uniforms): element i is
    word i mod 4 of the Philox4x64-10 block whose counter is the 256-bit integer offset + floor(i / 4)
    (little-endian words) under key (seed, 0), its top 24 bits scaled by 2^-24 (exact in fp32).
    Returns float64 values (all exactly representable in float32)."""
    out = np.zeros(int(n), dtype=np.float64)
    for i in range(int(n)):
        c = int(offset) + i // 4
        words = philox4x64_10([(c >> (64 * j)) & _U64 for j in range(4)], (int(seed), 0))
        out[i] = (words[i % 4] >> 40) * 2.0 ** -24
    return out
