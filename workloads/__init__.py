"""Seeded synthetic workloads for the EAGLE-3 draft heads (MLA, and the Llama-style MHA variant).

This module is the ONLY code shared by the fp64 oracle side (``oracle/``) and the
CUDA side (the ``eagle_speculative_decoding_eagle3_gb300`` package).  It holds no
arithmetic of the method: it only names the five workloads (shapes, value
distributions, batch/context mix) and draws their inputs from seeded generators.

Every tensor is drawn on the host from a counter-addressed stream:
chunk ``c`` of tensor ``name`` comes from ``PCG64(SeedSequence([seed, crc32(name), c]))``,
so any tensor (or any one sequence's cache rows) can be regenerated alone and the
result does not depend on the order of generation or on the number of threads.
bf16 values are produced by round-to-nearest-even of an fp32 draw and are kept
as raw ``uint16`` bit patterns; :func:`bf16_to_f32` widens them exactly.

The workloads follow the head configuration of the DeepseekV3 draft
(MAX API reference "max.pipelines.architectures.eagle3_deepseekV3",
class Eagle3DeepseekV3DraftConfig defaults: hidden 7168, 128 heads, q_lora 1536,
kv_lora 512, rope 64, nope 128, v 128, intermediate 18432, vocab 129280,
rms_norm_eps 1e-6, rope_theta 1e4, rope_interleave True).  The pages measure on
no dataset this code could use; synthetic acceptance (a calibrated per-position
acceptance probability, the benchmarking knob named in "Eagle3 DeepseekV3 in MAX",
§10) stands in for real target tokens.
"""
from __future__ import annotations

import math
import os
import zlib
from collections.abc import Mapping
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

CHUNK = 1 << 22  # elements per independently seeded chunk


# ----------------------------------------------------------------------------
# Workload specifications
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_heads: int
    q_lora_rank: int
    kv_lora_rank: int
    qk_nope_dim: int
    qk_rope_dim: int
    v_head_dim: int
    intermediate: int
    target_vocab: int
    draft_vocab: int
    dtype: str                      # "f32" or "bf16": storage type of weights, aux states, cache
    batch: int
    ctx: tuple                      # (lo, hi) inclusive range of cached tokens per sequence
    t_new: int                      # new tokens per sequence in the extend call
    gamma: int                      # draft tokens per round (extend gives the first)
    d2t: str | None                 # None, "uniform" (offsets U[0, V_t-V_d)), "sorted" (distinct ids)
    accept_p: tuple = ()            # per-position acceptance probability of synthetic targets
    rope_theta: float = 10000.0
    yarn_factor: float = 1.0
    yarn_original_max_pos: int = 4096
    yarn_beta_fast: float = 32.0
    yarn_beta_slow: float = 1.0
    yarn_mscale: float = 1.0
    yarn_mscale_all_dim: float = 1.0
    rms_eps: float = 1e-6
    page_size: int = 64
    seed: int = 1000
    weight_std: float = 0.02
    norm_std: float = 0.01
    # the Llama-style MHA head ("Eagle3 DeepseekV3 in MAX" §11); the MLA sizes above are unused by it
    attention: str = "mla"          # "mla" or "mha"
    n_kv_heads: int = 0
    head_dim: int = 0
    fc_inputs: int = 3              # aux states fused by fc (the MLA head always takes 3)

    # derived sizes ----------------------------------------------------------
    @property
    def qk_head_dim(self) -> int:
        return self.qk_nope_dim + self.qk_rope_dim

    @property
    def latent_dim(self) -> int:
        return self.kv_lora_rank + self.qk_rope_dim

    @property
    def cache_dim(self) -> int:
        """Width of one cache row: [c_kv | k_rope] (MLA) or [k (n_kv x d) | v (n_kv x d)] (MHA)."""
        return 2 * self.n_kv_heads * self.head_dim if self.attention == "mha" else self.latent_dim

    @property
    def max_ctx(self) -> int:
        return self.ctx[1] + self.t_new + self.gamma

    @property
    def max_pages_per_seq(self) -> int:
        return -(-self.max_ctx // self.page_size)

    def hyper(self) -> dict:
        """Plain hyper-parameter dict (what both sides are configured with)."""
        keys = ("hidden", "n_heads", "q_lora_rank", "kv_lora_rank", "qk_nope_dim", "qk_rope_dim",
                "v_head_dim", "intermediate", "target_vocab", "draft_vocab", "rope_theta",
                "yarn_factor", "yarn_original_max_pos", "yarn_beta_fast", "yarn_beta_slow",
                "yarn_mscale", "yarn_mscale_all_dim", "rms_eps", "attention", "n_kv_heads", "head_dim",
                "fc_inputs")
        return {k: getattr(self, k) for k in keys}

    def weight_shapes(self) -> dict:
        H, nh = self.hidden, self.n_heads
        if self.attention == "mha":
            d, nkv = self.head_dim, self.n_kv_heads
            return {
                "embed": (self.target_vocab, H),
                "fc": (H, self.fc_inputs * H),
                "input_norm": (H,),
                "hidden_norm": (H,),
                "q_proj": (nh * d, 2 * H),
                "k_proj": (nkv * d, 2 * H),
                "v_proj": (nkv * d, 2 * H),
                "o": (H, nh * d),
                "post_attn_norm": (H,),
                "gate": (self.intermediate, H),
                "up": (self.intermediate, H),
                "down": (H, self.intermediate),
                "final_norm": (H,),
                "lm_head": (self.draft_vocab, H),
            }
        return {
            "embed": (self.target_vocab, H),
            "fc": (H, 3 * H),
            "input_norm": (H,),
            "hidden_norm": (H,),
            "q_a": (self.q_lora_rank, 2 * H),
            "q_a_norm": (self.q_lora_rank,),
            "q_b": (nh * self.qk_head_dim, self.q_lora_rank),
            "kv_a": (self.latent_dim, 2 * H),
            "kv_a_norm": (self.kv_lora_rank,),
            "kv_b": (nh * (self.qk_nope_dim + self.v_head_dim), self.kv_lora_rank),
            "o": (H, nh * self.v_head_dim),
            "post_attn_norm": (H,),
            "gate": (self.intermediate, H),
            "up": (self.intermediate, H),
            "down": (H, self.intermediate),
            "final_norm": (H,),
            "lm_head": (self.draft_vocab, H),
        }


_DSV3 = dict(hidden=7168, n_heads=128, q_lora_rank=1536, kv_lora_rank=512, qk_nope_dim=128,
             qk_rope_dim=64, v_head_dim=128, intermediate=18432, target_vocab=129280, dtype="bf16",
             yarn_factor=40.0, yarn_original_max_pos=4096, yarn_beta_fast=32.0, yarn_beta_slow=1.0,
             yarn_mscale=1.0, yarn_mscale_all_dim=1.0)

WORKLOADS: dict[str, Workload] = {
    # tiny fp32 head: correctness workload the oracle finishes in well under a second
    "tiny_f32": Workload(
        name="tiny_f32", hidden=256, n_heads=4, q_lora_rank=64, kv_lora_rank=32, qk_nope_dim=32,
        qk_rope_dim=16, v_head_dim=32, intermediate=512, target_vocab=2048, draft_vocab=1024,
        dtype="f32", batch=2, ctx=(64, 64), t_new=4, gamma=3, d2t="uniform", accept_p=(0.7, 0.7, 0.7),
        yarn_factor=4.0, yarn_original_max_pos=32, page_size=16, seed=1000),
    # DSV3-shaped head, batch-1 decode (the headline workload)
    "dsv3_b1": Workload(
        name="dsv3_b1", draft_vocab=32000, batch=1, ctx=(4096, 4096), t_new=1, gamma=3, d2t="sorted",
        accept_p=(0.7, 0.7, 0.7), seed=1001, **_DSV3),
    # the batch-1 layer shapes and context with a small vocabulary: keeps profiler captures (which save
    # and restore device memory around every replay pass) to about 1.5 GB on the device
    "dsv3_b1_small": Workload(
        name="dsv3_b1_small", draft_vocab=4096, batch=1, ctx=(4096, 4096), t_new=1, gamma=3, d2t="sorted",
        accept_p=(0.7, 0.7, 0.7), seed=1005, **dict(_DSV3, target_vocab=8192)),
    # batch-64 decode, ragged contexts, full-vocab head without d2t
    "dsv3_b64": Workload(
        name="dsv3_b64", draft_vocab=129280, batch=64, ctx=(1024, 8192), t_new=1, gamma=5, d2t=None,
        accept_p=(0.7,) * 5, seed=1002, **_DSV3),
    # extend / prefill: 8 sequences x 2048 new tokens on an empty cache
    "dsv3_extend": Workload(
        name="dsv3_extend", draft_vocab=32000, batch=8, ctx=(0, 0), t_new=2048, gamma=1, d2t="sorted",
        accept_p=(0.7,), seed=1003, **_DSV3),
    # one sequence of the extend above (2048 new rows): the same kernels at a size a profiler capture of
    # every section can hold
    "dsv3_extend_small": Workload(
        name="dsv3_extend_small", draft_vocab=32000, batch=1, ctx=(0, 0), t_new=2048, gamma=1, d2t="sorted",
        accept_p=(0.7,), seed=1006, **_DSV3),
    # batch-256 decode, long ragged contexts, gamma 7, acceptance decaying 0.9 -> 0.5
    "dsv3_b256": Workload(
        name="dsv3_b256", draft_vocab=32000, batch=256, ctx=(4096, 16384), t_new=1, gamma=7, d2t="sorted",
        accept_p=tuple(0.9 * (0.5 / 0.9) ** (i / 6) for i in range(7)), seed=1004, **_DSV3),
    # the batch-256 attention shape (contexts U[4096, 16384]) on 32 sequences with a small vocabulary: a
    # profiler capture of the latent attention holds about 2 GB on the device
    "dsv3_b256_small": Workload(
        name="dsv3_b256_small", draft_vocab=4096, batch=32, ctx=(4096, 16384), t_new=1, gamma=3, d2t="sorted",
        accept_p=(0.9, 0.8, 0.7), seed=1007, **dict(_DSV3, target_vocab=8192)),
    # the batch-64 decode shape with a 32000-entry vocabulary (no d2t): its lm_head still has more output
    # tiles than SMs (the persistent GEMM), while a profiler capture holds about 3 GB on the device
    "dsv3_b64_small": Workload(
        name="dsv3_b64_small", draft_vocab=32000, batch=64, ctx=(1024, 8192), t_new=1, gamma=3, d2t=None,
        accept_p=(0.7, 0.7, 0.7), seed=1008, **dict(_DSV3, target_vocab=32000)),
    # the Llama-style MHA head on the same target: tiny fp32 head (2-way fc, 4 query heads per key/value
    # head) and a DeepseekV3-width head (hidden 7168 = 56 heads x 128, 8 key/value heads, 3-way fc) at
    # batch 1; no MHA head configuration is printed on the pages, these sizes are a reading
    "mha_tiny_f32": Workload(
        name="mha_tiny_f32", hidden=256, n_heads=8, q_lora_rank=0, kv_lora_rank=0, qk_nope_dim=0, qk_rope_dim=0,
        v_head_dim=0, intermediate=512, target_vocab=2048, draft_vocab=1024, dtype="f32", batch=2, ctx=(64, 64),
        t_new=4, gamma=3, d2t="uniform", accept_p=(0.7, 0.7, 0.7), yarn_factor=4.0, yarn_original_max_pos=32,
        page_size=16, seed=1010, attention="mha", n_kv_heads=2, head_dim=32, fc_inputs=2),
    "mha_b1": Workload(
        name="mha_b1", hidden=7168, n_heads=56, q_lora_rank=0, kv_lora_rank=0, qk_nope_dim=0, qk_rope_dim=0,
        v_head_dim=0, intermediate=18432, target_vocab=129280, draft_vocab=32000, dtype="bf16", batch=1,
        ctx=(4096, 4096), t_new=1, gamma=3, d2t="sorted", accept_p=(0.7, 0.7, 0.7), yarn_factor=40.0,
        yarn_original_max_pos=4096, seed=1011, attention="mha", n_kv_heads=8, head_dim=128, fc_inputs=3),
}


def workload(name: str, **overrides) -> Workload:
    """Return a named workload, optionally with fields replaced (for reduced parity cases)."""
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


# ----------------------------------------------------------------------------
# Seeded streams
# ----------------------------------------------------------------------------
def _tid(name: str) -> int:
    return zlib.crc32(name.encode())


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _chunk_gen(seed: int, name: str, c: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _tid(name), c])))


def _fill(n: int, seed: int, name: str, draw) -> np.ndarray:
    """Fill n float32 values chunk by chunk; ``draw(gen, count) -> float32 array``."""
    out = np.empty(n, dtype=np.float32)
    nchunks = -(-n // CHUNK)

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        out[lo:hi] = draw(_chunk_gen(seed, name, c), hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal(shape, std: float, seed: int, name: str, mean: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1

    def draw(g, k):
        v = g.standard_normal(k, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        return v
    return _fill(n, seed, name, draw).reshape(shape)


def uniform01(shape, seed: int, name: str) -> np.ndarray:
    """float64 uniforms in [0, 1) (single stream; used for small index draws)."""
    g = _chunk_gen(seed, name, 0)
    return g.random(shape)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    n = flat_in.size
    step = CHUNK

    def work(lo):
        b = flat_in[lo:lo + step].copy()
        b += np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
        flat_out[lo:lo + step] = (b >> np.uint32(16)).astype(np.uint16)

    starts = range(0, n, step)
    if n > step:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(work, starts))
    else:
        for s in starts:
            work(s)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return x32 if dtype == "f32" else f32_to_bf16_bits(x32)


def as_f32(a: np.ndarray) -> np.ndarray:
    """View any stored tensor (fp32 or bf16 bits) as exact fp32 values."""
    return bf16_to_f32(a) if a.dtype == np.uint16 else a


class StoredTensors(Mapping):
    """name -> stored array (fp32, or uint16 bf16 bits); ``.f32(name)`` widens exactly."""

    def __init__(self, arrays: dict):
        self._a = arrays

    def __getitem__(self, k):
        return self._a[k]

    def __iter__(self):
        return iter(self._a)

    def __len__(self):
        return len(self._a)

    def f32(self, k) -> np.ndarray:
        return as_f32(self._a[k])


class F32View(Mapping):
    """Read-only mapping that widens stored tensors to fp32 on access (for the oracle)."""

    def __init__(self, stored: Mapping):
        self._s = stored

    def __getitem__(self, k):
        return as_f32(self._s[k])

    def __iter__(self):
        return iter(self._s)

    def __len__(self):
        return len(self._s)


class F64Cache(Mapping):
    """Read-only mapping that widens stored tensors to fp64 once and keeps them (for repeated oracle
    calls on large heads; exact, since bf16 and fp32 values are representable in fp64)."""

    def __init__(self, stored: Mapping):
        self._s = stored
        self._c = {}

    def __getitem__(self, k):
        if k not in self._c:
            self._c[k] = as_f32(self._s[k]).astype(np.float64)
        return self._c[k]

    def __iter__(self):
        return iter(self._s)

    def __len__(self):
        return len(self._s)


# ----------------------------------------------------------------------------
# Weights
# ----------------------------------------------------------------------------
_NORMS = ("input_norm", "hidden_norm", "q_a_norm", "kv_a_norm", "post_attn_norm", "final_norm")


def make_weights(w: Workload, names=None) -> StoredTensors:
    """Random-init weights: linear layers and the embedding N(0, 0.02); norm weights 1 + N(0, 0.01)."""
    out = {}
    for name, shape in w.weight_shapes().items():
        if names is not None and name not in names:
            continue
        if name in _NORMS:
            v = normal(shape, w.norm_std, w.seed, "w." + name, mean=1.0)
        else:
            v = normal(shape, w.weight_std, w.seed, "w." + name)
        out[name] = _store(v, w.dtype)
    return StoredTensors(out)


def make_d2t(w: Workload) -> np.ndarray | None:
    """Draft-to-target offsets (int32 [V_d]); t = d + d2t[d] lands in [0, V_t)."""
    if w.d2t is None:
        return None
    if w.d2t == "uniform":
        span = w.target_vocab - w.draft_vocab
        u = uniform01(w.draft_vocab, w.seed, "d2t")
        return np.minimum((u * span).astype(np.int64), span - 1).astype(np.int32)
    if w.d2t == "sorted":
        g = _chunk_gen(w.seed, "d2t", 0)
        ids = np.sort(g.choice(w.target_vocab, size=w.draft_vocab, replace=False))
        return (ids - np.arange(w.draft_vocab)).astype(np.int32)
    raise ValueError(w.d2t)


# ----------------------------------------------------------------------------
# Cache and extend inputs
# ----------------------------------------------------------------------------
def context_lengths(w: Workload) -> np.ndarray:
    lo, hi = w.ctx
    if lo == hi:
        return np.full(w.batch, lo, dtype=np.int32)
    u = uniform01(w.batch, w.seed, "ctx_len")
    return (lo + np.minimum((u * (hi - lo + 1)).astype(np.int64), hi - lo)).astype(np.int32)


def cache_rows(w: Workload, b: int, length: int) -> np.ndarray:
    """Stored cache rows [length, d_c + d_r] of sequence b (taken as already normalised/rotated)."""
    v = normal((length, w.cache_dim), 1.0, w.seed, f"cache.{b}")
    return _store(v, w.dtype)


@dataclass
class PagedCache:
    data: np.ndarray          # [num_pages, page_size, latent] stored dtype
    block_table: np.ndarray   # int32 [B, max_pages_per_seq]
    lengths: np.ndarray       # int32 [B]
    page_size: int


def page_assignment(w: Workload) -> np.ndarray:
    """Block table: every sequence owns max_pages_per_seq pages, placed by a seeded permutation."""
    P = w.max_pages_per_seq
    g = _chunk_gen(w.seed, "pages", 0)
    perm = g.permutation(w.batch * P).astype(np.int32)
    return perm.reshape(w.batch, P)


def make_cache(w: Workload, lengths=None, fill=True) -> PagedCache:
    lengths = context_lengths(w) if lengths is None else np.asarray(lengths, dtype=np.int32)
    bt = page_assignment(w)
    num_pages = w.batch * w.max_pages_per_seq
    dt = np.float32 if w.dtype == "f32" else np.uint16
    data = np.zeros((num_pages, w.page_size, w.cache_dim), dtype=dt)
    if fill:
        def one(b):
            write_rows(data, bt[b], 0, cache_rows(w, b, int(lengths[b])), w.page_size)
        if w.batch > 1:
            with ThreadPoolExecutor(max_workers=min(_threads(), w.batch)) as ex:
                list(ex.map(one, range(w.batch)))
        else:
            one(0)
    return PagedCache(data=data, block_table=bt, lengths=lengths.copy(), page_size=w.page_size)


def write_rows(data, bt_row, start, rows, page_size):
    """Scatter logical rows [start, start+len) of one sequence into its pages."""
    n = rows.shape[0]
    t = 0
    while t < n:
        slot = start + t
        page, off = divmod(slot, page_size)
        k = min(page_size - off, n - t)
        data[bt_row[page], off:off + k] = rows[t:t + k]
        t += k


def read_rows(data, bt_row, start, n, page_size):
    """Gather logical rows [start, start+n) of one sequence from its pages."""
    out = np.empty((n, data.shape[2]), dtype=data.dtype)
    t = 0
    while t < n:
        slot = start + t
        page, off = divmod(slot, page_size)
        k = min(page_size - off, n - t)
        out[t:t + k] = data[bt_row[page], off:off + k]
        t += k
    return out


@dataclass
class ExtendInputs:
    aux: list                 # fc_inputs stored arrays [N, H] (early, (middle,) late)
    tokens: np.ndarray        # int32 [N]
    positions: np.ndarray     # int32 [N]
    row_offsets: np.ndarray   # int32 [B+1]


def make_extend(w: Workload, lengths: np.ndarray, seqs=None) -> ExtendInputs:
    """New rows: t_new per sequence at positions L_b .. L_b + t_new - 1; aux ~ N(0,1); tokens uniform.

    ``seqs`` restricts generation to a subset of sequences (rows of other sequences are
    not generated); the values of a sequence's rows never depend on the subset.
    """
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    T, H = w.t_new, w.hidden
    aux = [[] for _ in range(w.fc_inputs)]
    toks, pos = [], []
    for b in seqs:
        for j in range(w.fc_inputs):
            aux[j].append(_store(normal((T, H), 1.0, w.seed, f"aux{j}.{b}"), w.dtype))
        g = _chunk_gen(w.seed, f"tok.{b}", 0)
        toks.append(g.integers(0, w.target_vocab, size=T, dtype=np.int64).astype(np.int32))
        pos.append(np.arange(lengths[b], lengths[b] + T, dtype=np.int32))
    row_offsets = np.arange(0, (len(seqs) + 1) * T, T, dtype=np.int32)
    return ExtendInputs(aux=[np.concatenate(a, 0) for a in aux], tokens=np.concatenate(toks),
                        positions=np.concatenate(pos), row_offsets=row_offsets)


def synthetic_targets(w: Workload, draft: np.ndarray, seqs=None) -> np.ndarray:
    """Target tokens from draft tokens: equal with probability p_i, else a guaranteed-different id.

    Draws for sequence b come from its own stream, so a subset reproduces the same rows.
    """
    draft = np.asarray(draft, dtype=np.int64)
    B, G = draft.shape
    seqs = list(range(B)) if seqs is None else list(seqs)
    out = np.empty_like(draft)
    p = np.asarray(w.accept_p[:G] if len(w.accept_p) >= G else (w.accept_p + (w.accept_p[-1],) * G)[:G])
    for r, b in enumerate(seqs):
        g = _chunk_gen(w.seed, f"target.{b}", 0)
        u = g.random(G)
        u2 = g.random(G)
        alt = (draft[r] + 1 + np.minimum((u2 * (w.target_vocab - 1)).astype(np.int64), w.target_vocab - 2)) \
            % w.target_vocab
        out[r] = np.where(u < p, draft[r], alt)
    return out.astype(np.int32)
