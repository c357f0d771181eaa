"""fp64 CPU oracle of the EAGLE-3 MLA draft-head step — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` may import or call this package.  The product path (the
C-ABI library and its Python binding) never does; it shares no code with it.

Sources (cited by title and section):
  [MAX-walkthrough]  "Eagle3 DeepseekV3 speculative decoding architecture: a full
                     walkthrough of MAX's eagle3_deepseekV3 module" (xxmr.cn/news/219581)
  [MAX-API]          "max.pipelines.architectures.eagle3_deepseekV3" API reference
                     (max.modular.com), class Eagle3DeepseekV3DraftConfig
  [ModelOpt-EAGLE]   "EAGLE head deep dive: inside Model Optimizer's speculative-decoding
                     draft model" (discosf.com/news/5068204)

Every function is a plain fp64 numpy statement of its definition (no blocking,
fusion or reordering).  Pins (``tests/test_oracle_*.py``):
  rms_norm          closed form on a hand example, scale invariance, unit-RMS output
  yarn_inv_freq     factor 1 == plain RoPE; YaRN's defining rotation-count property on
                    the DeepseekV3 parameters; hand-computed band edges (golden file)
  yarn_mscale       hand value 1 + 0.1 ln 40 (golden file)
  rope_interleaved  complex-multiplication formulation, norm preservation, position 0
                    identity, relative-position invariance, composition R(a)R(b)=R(a+b)
  linear / silu     brute-force triple loop; torch.nn.functional.silu in fp64
  mla_attention     torch scaled_dot_product_attention (fp64) on explicit K/V; single key
                    returns its value; equal keys return the mean; causal first row;
                    absorbed == unabsorbed to fp64 round-off
  rope_half         (MHA head) hand quarter turn and the (i, i + d/2) pairing; complex multiplication;
                    identity at 0, relative-position invariance
  mha_attention     torch SDPA in fp64 with key/value heads repeated per group and the causal mask;
                    single visible slot; equal keys give the mean value
  argmax_lowest     brute force with planted ties
  d2t_remap         zero offsets give identity; brute force
  accept            full match gives gamma; first mismatch gives 0; brute force
  e4m3_*            every code decodes per the OCP E4M3 table (max 448, one NaN pattern); encode(decode(c)) ==
                    c; midpoints round to the even code; values saturate at 448; the array
                    encoder equals the scalar one on every code, midpoint and a random sweep
  e2m1_* / nvfp4    the eight E2M1 magnitudes and their signs; every midpoint rounds to the even code;
                    saturation at 6; the NVFP4 rule restated element by element; the block error bound
  accept_relaxed    rows outside thinking == greedy accept; k = 1 or delta below every gap ==
                    greedy; hand example with the default delta 0.6; monotone in delta
  accept_typical    one-hot targets reduce it to greedy acceptance; uniform targets give the closed
                    form 1/V > min(eps, delta / V); the entropy against scipy.stats.entropy and the
                    identity exp(-H) = prod p^p on a hand distribution; monotone in eps and delta
  philox4x64_10 /   bit-exact against numpy.random.Philox (an independent implementation of the same
  philox_uniforms   published generator); uniforms exact in fp32, in [0, 1), mean and variance
  draft_extend /    composition invariants: one T-row extend == T one-row extends
  draft_decode_step (same cache rows and hidden); batch and page-placement independence;
                    residual pass-through with zeroed projections; fc only on 3H input
The whole head has no worked numeric example on the pages: beyond the invariants
above its parity is unpinned (the 2H concat order is a reading that only permutes
weight columns and cannot be pinned).
"""
from .head import (  # noqa: F401
    F64, rms_norm, linear, silu, yarn_inv_freq, yarn_mscale, rope_cos_sin, rope_interleaved, rope_half, rope_dim,
    softmax_scale, split_kv_b, mla_attention, mha_attention, decoder_rows, final_logits, argmax_lowest,
    top2_gap, d2t_remap, SeqCache, draft_extend, draft_decode_step, draft_round, accept, accept_relaxed,
    sample_filtered, accept_residual, e4m3_decode, e4m3_encode, e4m3_encode_array, quantize_rows_e4m3,
    e2m1_decode, e2m1_encode_array, quantize_nvfp4, accept_typical, philox4x64_10, philox_uniforms,
)
