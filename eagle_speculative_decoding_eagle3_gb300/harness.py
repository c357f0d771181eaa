"""Device-side harness: puts a seeded workload's tensors in HBM and drives the C ABI.

Used by the tests, ``bench.py`` and ``__graft_entry__.smoke``.  It only moves data (host arrays
from ``workloads`` to torch device tensors) and calls the binding; every step of the head runs
in libeagle3's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import eagle3 as E


def to_device(arr: np.ndarray, device="cuda") -> torch.Tensor:
    """Stored array (fp32, int32, or uint16 bf16 bits) -> device tensor of the same bits."""
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(arr).to(device)


def config_for(w, max_batch=None, max_tokens=None, fp8=False, nvfp4=False) -> E.eagle3_config_t:
    return E.make_config(
        hidden=w.hidden, n_heads=w.n_heads, q_lora_rank=w.q_lora_rank, kv_lora_rank=w.kv_lora_rank,
        qk_nope_dim=w.qk_nope_dim, qk_rope_dim=w.qk_rope_dim, v_head_dim=w.v_head_dim,
        intermediate=w.intermediate, target_vocab=w.target_vocab, draft_vocab=w.draft_vocab,
        max_batch=max_batch or w.batch, max_tokens_per_extend=max_tokens or max(w.batch * w.t_new, w.batch),
        max_ctx=w.max_ctx, page_size=w.page_size, max_pages_per_seq=w.max_pages_per_seq,
        rms_eps=w.rms_eps, rope_theta=w.rope_theta, yarn_factor=w.yarn_factor, yarn_beta_fast=w.yarn_beta_fast,
        yarn_beta_slow=w.yarn_beta_slow, yarn_mscale=w.yarn_mscale, yarn_mscale_all_dim=w.yarn_mscale_all_dim,
        yarn_original_max_pos=w.yarn_original_max_pos, rope_interleave=1,
        dtype=E.BF16 if w.dtype == "bf16" else E.F32, weight_format=E.WEIGHTS_NVFP4 if nvfp4 else (E.WEIGHTS_FP8 if fp8 else E.WEIGHTS_DTYPE),
        attention=E.ATTN_MHA if w.attention == "mha" else E.ATTN_MLA, n_kv_heads=w.n_kv_heads,
        head_dim=w.head_dim, fc_inputs=w.fc_inputs)


@dataclass
class DeviceCache:
    data: torch.Tensor
    block_table: torch.Tensor
    lengths: torch.Tensor
    num_pages: int

    def kv(self) -> E.eagle3_kv_t:
        return E.make_kv(self.data, self.block_table, self.lengths, self.num_pages)


def quantize_fp8(t: torch.Tensor):
    """Device FP8 E4M3 codes and row scales of a bf16 / fp32 device matrix, by eagle3_quantize_e4m3."""
    N, K = t.shape
    codes = torch.empty((N, K), dtype=torch.uint8, device=t.device)
    scales = torch.empty((N,), dtype=torch.float32, device=t.device)
    E.eagle3_quantize_e4m3(t, E.BF16 if t.dtype == torch.bfloat16 else E.F32, N, K, codes, scales)
    return codes, scales


def quantize_nvfp4(t: torch.Tensor):
    """Device NVFP4 codes, E4M3 block scales and fp32 matrix scale of a bf16 / fp32 device matrix, by
    eagle3_quantize_nvfp4."""
    N, K = t.shape
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=t.device)
    block = torch.empty((N, K // 16), dtype=torch.uint8, device=t.device)
    g = torch.empty((1,), dtype=torch.float32, device=t.device)
    E.eagle3_quantize_nvfp4(t, E.BF16 if t.dtype == torch.bfloat16 else E.F32, N, K, codes, block, g)
    return codes, block, g


class DeviceHead:
    """A created draft head whose weights live in device tensors owned by this object.

    fp8=True (nvfp4=True) stores the projection matrices as FP8 E4M3 codes with per-row scales (NVFP4
    codes with block and matrix scales), quantized on the device from the given weights (the bf16 copies
    of those matrices are released)."""

    def __init__(self, w, stored_weights, device="cuda", max_batch=None, max_tokens=None, fp8=False, nvfp4=False):
        self.w = w
        self.device = device
        self.tensors = {}
        self.scales = {}
        self.matrix_scales = torch.ones(len(E.FP8_WEIGHT_NAMES), dtype=torch.float32, device=device) if nvfp4 else None
        for n in E.WEIGHT_NAMES + E.MHA_WEIGHT_NAMES:
            if n not in stored_weights:
                continue                       # the other head kind's weights
            t = to_device(stored_weights[n], device)
            if fp8 and n in E.FP8_WEIGHT_NAMES:
                t, self.scales[n] = quantize_fp8(t)
            elif nvfp4 and n in E.FP8_WEIGHT_NAMES:
                t, self.scales[n], g = quantize_nvfp4(t)
                self.matrix_scales[E.FP8_WEIGHT_NAMES.index(n)] = g[0]
            self.tensors[n] = t
        self.config = config_for(w, max_batch, max_tokens, fp8, nvfp4)
        self.handle = E.eagle3_draft_create(self.config, E.make_weights(self.tensors, self.scales or None,
                                                                        self.matrix_scales))

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None   # the library frees the handle even when it reports an error
            E.eagle3_draft_destroy(h)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- inputs ----------------------------------------------------------------------------
    def cache(self, paged) -> DeviceCache:
        return DeviceCache(data=to_device(paged.data, self.device),
                           block_table=to_device(paged.block_table, self.device),
                           lengths=to_device(paged.lengths.astype(np.int32), self.device),
                           num_pages=paged.data.shape[0])

    def extend_inputs(self, ex):
        return dict(aux=[to_device(a, self.device) for a in ex.aux],
                    tokens=to_device(ex.tokens, self.device), positions=to_device(ex.positions, self.device),
                    row_offsets=to_device(ex.row_offsets, self.device))

    # -- calls -----------------------------------------------------------------------------
    def extend(self, dev_in, cache: DeviceCache, hidden_out=None, logits_out=None, stream=None):
        batch = dev_in["row_offsets"].numel() - 1
        E.eagle3_draft_extend(self.handle, dev_in["aux"], dev_in["tokens"], dev_in["positions"],
                              dev_in["row_offsets"], batch, dev_in["tokens"].numel(), cache.kv(),
                              hidden_out, logits_out, stream)

    def decode(self, gamma, d2t, cache: DeviceCache, draft_tokens, hidden_out=None, logits_out=None, stream=None):
        E.eagle3_draft_decode(self.handle, gamma, d2t, cache.kv(), draft_tokens, hidden_out, logits_out, stream)

    def decode_sampled(self, gamma, d2t, cache: DeviceCache, temperature, top_k, top_p, first_logits, uniforms,
                       draft_tokens, draft_probs=None, probs_len=0, probs_in_target=False, hidden_out=None,
                       logits_out=None, stream=None):
        E.eagle3_draft_decode_sampled(self.handle, gamma, d2t, cache.kv(), temperature, top_k, top_p, first_logits,
                                      uniforms, draft_tokens, draft_probs, probs_len, probs_in_target, hidden_out,
                                      logits_out, stream)

    def error_word(self) -> int:
        return E.eagle3_draft_get_error(self.handle)
