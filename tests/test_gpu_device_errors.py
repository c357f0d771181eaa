"""The device-side error convention of the C ABI, on the GPU.

A token outside the target vocabulary, a position at or past max_ctx, a d2t entry that maps outside the
target vocabulary and a block-table page outside the cache are not host-checkable (they live in device
memory).  The kernels clamp them, set a bit of the handle's sticky error word and carry on, so a call
never faults and every output stays finite and in range ("Eagle3 DeepseekV3 in MAX" §10: the decode loop
is one captured graph that reports rather than raises).  Where the clamp has a plain meaning (a token
clamped to the nearest valid id, a remap clamped to the last target id) the round must equal the
oracle's round on the clamped inputs; elsewhere the other sequences of the batch must be untouched
(sequences are independent).  eagle3_draft_clear_error resets the word."""
import numpy as np
import pytest
import torch

import workloads as WL
from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E

from parity import TOL_BF16, TOL_F32, check_round, run_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from eagle_speculative_decoding_eagle3_gb300 import build
    build.build()


def _sane(w, gpu, seq):
    """Outputs of a sequence that met a device range error: finite, tokens in the target vocabulary."""
    assert np.all(np.isfinite(gpu["hidden"][:, seq]))
    if gpu["logits"] is not None:
        assert np.all(np.isfinite(gpu["logits"][:, seq]))
    t = gpu["tokens"][seq]
    assert np.all((t >= 0) & (t < w.target_vocab)), t


def test_token_out_of_vocab_is_clamped():
    w = WL.workload("tiny_f32")
    Vt, T = w.target_vocab, w.t_new

    def gpu_in(ex, paged, d2t):
        ex.tokens[1] = Vt + 7            # sequence 0: past the vocabulary
        ex.tokens[T + 2] = -3            # sequence 1: negative
        return d2t

    def orc_in(exs, d2t):
        exs.tokens[1] = Vt - 1
        exs.tokens[T + 2] = 0
        return d2t

    gpu, orc, seqs, paged = run_round(w, gpu_inputs=gpu_in, oracle_inputs=orc_in)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32, err=E.DEVERR_TOKEN))


def test_d2t_out_of_range_is_clamped():
    w = WL.workload("tiny_f32", seed=1003)
    Vt, Vd = w.target_vocab, w.draft_vocab
    bad = np.full(Vd, Vt, dtype=np.int32)                          # d + d2t[d] >= V_t for every d
    last = (Vt - 1 - np.arange(Vd)).astype(np.int32)               # every d remaps to V_t - 1

    gpu, orc, seqs, paged = run_round(w, gpu_inputs=lambda ex, paged, d2t: bad,
                                      oracle_inputs=lambda exs, d2t: last)
    assert np.all(gpu["tokens"] == Vt - 1)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32, err=E.DEVERR_D2T))


def test_position_past_max_ctx_is_clamped():
    w = WL.workload("tiny_f32", seed=1004)
    T = w.t_new

    def gpu_in(ex, paged, d2t):
        ex.positions[:T] = w.max_ctx + 3      # every new row of sequence 0
        return d2t

    gpu, orc, seqs, paged = run_round(w, seqs=[1], gpu_inputs=gpu_in)
    _sane(w, gpu, 0)
    assert gpu["lengths"][0] == w.max_ctx
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32, err=E.DEVERR_POSITION))


def _bad_append_page(w):
    lengths = WL.context_lengths(w)
    page = int(lengths[0]) // w.page_size

    def gpu_in(ex, paged, d2t):
        paged.block_table[0, page] = paged.data.shape[0] + 100   # the page that takes sequence 0's new rows
        return d2t
    return gpu_in


@pytest.mark.parametrize("name,tol,over", [
    ("tiny_f32", TOL_F32, {}),
    ("mha_tiny_f32", TOL_F32, {}),
    # the bf16 tensor-core path (24 rows per decode step): the mma.sync attention kernel's page check
    ("dsv3_b1", TOL_BF16, dict(hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048, target_vocab=8192,
                               draft_vocab=4096, batch=24, ctx=(30, 300), t_new=2, gamma=3, accept_p=(0.7,) * 3,
                               seed=84)),
    # 128 heads, 16 rows per step: the tcgen05 latent attention's producer fills the page's tiles with zeros
    ("dsv3_b1", TOL_BF16, dict(hidden=1024, n_heads=128, q_lora_rank=256, intermediate=2048, target_vocab=8192,
                               draft_vocab=4096, batch=16, ctx=(100, 300), t_new=2, gamma=3, accept_p=(0.7,) * 3,
                               seed=89)),
])
def test_block_table_page_outside_cache(name, tol, over):
    w = WL.workload(name, **over)
    gpu, orc, seqs, paged = run_round(w, seqs=[1], gpu_inputs=_bad_append_page(w))
    _sane(w, gpu, 0)
    print(check_round(w, gpu, orc, seqs, paged, tol, err=E.DEVERR_PAGE))


def test_clear_error_resets_the_word():
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    w = WL.workload("tiny_f32", seed=1005)
    stored = WL.make_weights(w)
    lengths = WL.context_lengths(w)
    head = HN.DeviceHead(w, stored)
    try:
        B, G = w.batch, w.gamma
        toks = torch.zeros((B, G), dtype=torch.int32, device="cuda")
        d2t = HN.to_device(WL.make_d2t(w))
        ex = WL.make_extend(w, lengths)
        ex.tokens[0] = w.target_vocab + 1
        dc = head.cache(WL.make_cache(w, lengths))
        head.extend(head.extend_inputs(ex), dc)
        head.decode(G, d2t, dc, toks)
        torch.cuda.synchronize()
        assert head.error_word() == E.DEVERR_TOKEN
        E.eagle3_draft_clear_error(head.handle)
        torch.cuda.synchronize()
        assert head.error_word() == 0
        # the handle stays usable: a valid round on a fresh cache leaves the word clear
        dc = head.cache(WL.make_cache(w, lengths))
        head.extend(head.extend_inputs(WL.make_extend(w, lengths)), dc)
        head.decode(G, d2t, dc, toks)
        torch.cuda.synchronize()
        assert head.error_word() == 0
        t = toks.cpu().numpy()
        assert np.all((t >= 0) & (t < w.target_vocab))
    finally:
        head.close()
