"""ctypes binding of libeagle3 (include/eagle3.h): argument marshalling only.

Every function here has the C name and forwards to the library; all compute runs in its CUDA
kernels.  Pointer arguments accept a torch tensor (its data_ptr), an int address, or None.
The library must be built first (``build.build()``); loading fails loudly if it is missing.
"""
from __future__ import annotations

import ctypes as C
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libeagle3.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_STATE, ERR_OOM, ERR_CUDA, ERR_DEVICE_RANGE, ERR_SCRATCH_LIMIT = range(8)
NOALLOC_SCRATCH_BYTES = 16 << 20   # EAGLE3_NOALLOC_SCRATCH_BYTES
F32, BF16 = 0, 1
WEIGHTS_DTYPE, WEIGHTS_FP8, WEIGHTS_NVFP4 = 0, 1, 2   # eagle3_weight_format_t
ATTN_MLA, ATTN_MHA = 0, 1           # eagle3_attention_t
DEVERR_TOKEN, DEVERR_POSITION, DEVERR_D2T, DEVERR_PAGE, DEVERR_ROWS = 1, 2, 4, 8, 16


class eagle3_config_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_heads", "q_lora_rank", "kv_lora_rank", "qk_nope_dim", "qk_rope_dim", "v_head_dim",
        "intermediate", "target_vocab", "draft_vocab", "max_batch", "max_tokens_per_extend", "max_ctx",
        "page_size", "max_pages_per_seq")] + [(n, C.c_float) for n in (
            "rms_eps", "rope_theta", "yarn_factor", "yarn_beta_fast", "yarn_beta_slow", "yarn_mscale",
            "yarn_mscale_all_dim")] + [("yarn_original_max_pos", C.c_int32), ("rope_interleave", C.c_int32),
                                       ("dtype", C.c_int32), ("weight_format", C.c_int32),
                                       ("attention", C.c_int32), ("n_kv_heads", C.c_int32),
                                       ("head_dim", C.c_int32), ("fc_inputs", C.c_int32)]


WEIGHT_NAMES = ("embed", "fc", "input_norm", "hidden_norm", "q_a", "q_a_norm", "q_b", "kv_a", "kv_a_norm", "kv_b",
                "o", "post_attn_norm", "gate", "up", "down", "final_norm", "lm_head")


# the projection matrices that EAGLE3_WEIGHTS_FP8 stores as E4M3 codes with per-row scales
FP8_WEIGHT_NAMES = ("fc", "q_a", "kv_a", "q_b", "o", "gate", "up", "down", "lm_head")
# the MHA head's own projections (its unused MLA fields stay NULL)
MHA_WEIGHT_NAMES = ("q_proj", "k_proj", "v_proj")


class eagle3_weights_t(C.Structure):
    _fields_ = ([(n, C.c_void_p) for n in WEIGHT_NAMES] + [(n + "_scale", C.c_void_p) for n in FP8_WEIGHT_NAMES]
                + [(n, C.c_void_p) for n in MHA_WEIGHT_NAMES] + [("matrix_scales", C.c_void_p)])


class eagle3_kv_t(C.Structure):
    _fields_ = [("data", C.c_void_p), ("block_table", C.c_void_p), ("lengths", C.c_void_p),
                ("num_pages", C.c_int32)]


class eagle3_sampling_t(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_k", C.c_int32), ("top_p", C.c_float)]


class Eagle3Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _lib().eagle3_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cudaError {_lib().eagle3_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{status}]")


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libeagle3.so is not built ({_LIB_PATH}); run build.build() first")
        lib = C.CDLL(_LIB_PATH)
        P = C.c_void_p
        lib.eagle3_status_string.restype = C.c_char_p
        lib.eagle3_status_string.argtypes = [C.c_int]
        lib.eagle3_last_cuda_error.restype = C.c_int32
        lib.eagle3_draft_create.argtypes = [C.POINTER(eagle3_config_t), C.POINTER(eagle3_weights_t), C.POINTER(P)]
        lib.eagle3_draft_workspace_bytes.argtypes = [C.POINTER(eagle3_config_t), C.POINTER(C.c_size_t)]
        lib.eagle3_draft_extend.argtypes = [P, C.POINTER(P), P, P, P, C.c_int32, C.c_int32, C.POINTER(eagle3_kv_t),
                                            P, P, P]
        lib.eagle3_draft_decode.argtypes = [P, C.c_int32, P, C.POINTER(eagle3_kv_t), P, P, P, P]
        lib.eagle3_accept.argtypes = [P, P, C.c_int32, C.c_int32, P, P, P]
        lib.eagle3_accept_relaxed.argtypes = [P, P, P, P, C.c_int32, C.c_int32, C.c_int32, C.c_float, P, P, P]
        lib.eagle3_sample.argtypes = [P, C.c_int32, C.c_int32, C.c_int64, C.POINTER(eagle3_sampling_t), P, P,
                                      C.c_int32, P, P, P, C.c_int32, C.c_int32, P]
        lib.eagle3_accept_residual.argtypes = [P, P, P, P, P, C.c_int32, C.c_int32, C.c_int32, P, P, P, P]
        lib.eagle3_accept_typical.argtypes = [P, P, C.c_int32, C.c_int32, C.c_int32, C.c_float, C.c_float, P, P, P]
        lib.eagle3_philox_uniforms.argtypes = [C.c_uint64, C.c_uint64, C.c_int64, P, P]
        lib.eagle3_draft_decode_sampled.argtypes = [P, C.c_int32, P, C.POINTER(eagle3_kv_t),
                                                    C.POINTER(eagle3_sampling_t), P, P, P, P, C.c_int32, C.c_int32,
                                                    P, P, P]
        lib.eagle3_linear.argtypes = [P, P, P, P, C.c_int32, C.c_int32, C.c_int32, P]
        lib.eagle3_linear_noalloc.argtypes = [P, P, P, C.c_int32, C.c_int32, C.c_int32, P]
        lib.eagle3_quantize_e4m3.argtypes = [P, C.c_int32, C.c_int32, C.c_int32, P, P, P]
        lib.eagle3_quantize_nvfp4.argtypes = [P, C.c_int32, C.c_int32, C.c_int32, P, P, P, P]
        lib.eagle3_draft_get_error.argtypes = [P, C.POINTER(C.c_int32)]
        lib.eagle3_draft_clear_error.argtypes = [P, P]
        lib.eagle3_draft_destroy.argtypes = [P]
        lib.eagle3_draft_profile_enable.argtypes = [P, C.c_int32]
        lib.eagle3_draft_profile_read.argtypes = [P, C.c_int32, C.POINTER(C.c_double), C.POINTER(C.c_int64),
                                                  C.POINTER(C.c_int64), C.POINTER(C.c_char_p)]
        lib.eagle3_draft_profile_reset.argtypes = [P]
        for f in ("eagle3_draft_profile_enable", "eagle3_draft_profile_read", "eagle3_draft_profile_reset",
                  "eagle3_draft_create", "eagle3_draft_workspace_bytes", "eagle3_draft_extend", "eagle3_draft_decode",
                  "eagle3_accept", "eagle3_accept_relaxed", "eagle3_sample", "eagle3_accept_residual", "eagle3_accept_typical", "eagle3_philox_uniforms", "eagle3_draft_decode_sampled", "eagle3_linear", "eagle3_linear_noalloc", "eagle3_draft_get_error", "eagle3_draft_clear_error", "eagle3_draft_destroy"):
            getattr(lib, f).restype = C.c_int
        _L = lib
    return _L


def library_path() -> str:
    return _LIB_PATH


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, status):
    if status != OK:
        raise Eagle3Error(fn, status)


def make_config(**fields) -> eagle3_config_t:
    c = eagle3_config_t()
    defaults = dict(rms_eps=1e-6, rope_theta=1e4, yarn_factor=1.0, yarn_beta_fast=32.0, yarn_beta_slow=1.0,
                    yarn_mscale=1.0, yarn_mscale_all_dim=1.0, yarn_original_max_pos=4096, rope_interleave=1)
    defaults.update(fields)
    for k, v in defaults.items():
        setattr(c, k, v)
    return c


def make_weights(tensors, scales=None, matrix_scales=None) -> eagle3_weights_t:
    """Weight pointers; `scales` (quantized heads) maps each of FP8_WEIGHT_NAMES to its FP8 row scales or
    NVFP4 block scales; `matrix_scales` (NVFP4) is the fp32 [9] tensor of the matrices' scales."""
    w = eagle3_weights_t()
    for n in WEIGHT_NAMES + MHA_WEIGHT_NAMES:
        setattr(w, n, _ptr(tensors.get(n)))
    for n in FP8_WEIGHT_NAMES if scales else ():
        setattr(w, n + "_scale", _ptr(scales[n]))
    w.matrix_scales = _ptr(matrix_scales)
    return w


def make_kv(data, block_table, lengths, num_pages) -> eagle3_kv_t:
    return eagle3_kv_t(_ptr(data), _ptr(block_table), _ptr(lengths), int(num_pages))


def eagle3_status_string(status: int) -> str:
    return _lib().eagle3_status_string(status).decode()


def eagle3_draft_workspace_bytes(config: eagle3_config_t) -> int:
    n = C.c_size_t()
    _check("eagle3_draft_workspace_bytes", _lib().eagle3_draft_workspace_bytes(C.byref(config), C.byref(n)))
    return n.value


def eagle3_draft_create(config: eagle3_config_t, weights: eagle3_weights_t) -> int:
    h = C.c_void_p()
    _check("eagle3_draft_create", _lib().eagle3_draft_create(C.byref(config), C.byref(weights), C.byref(h)))
    return h.value


def eagle3_draft_extend(handle, aux_hidden, tokens, positions, row_offsets, batch, num_tokens, cache: eagle3_kv_t,
                        hidden_out=None, logits_out=None, stream=None):
    aux = (C.c_void_p * 3)(*[_ptr(a) for a in aux_hidden] + [None] * (3 - len(aux_hidden)))
    _check("eagle3_draft_extend", _lib().eagle3_draft_extend(
        handle, aux, _ptr(tokens), _ptr(positions), _ptr(row_offsets), int(batch), int(num_tokens), C.byref(cache),
        _ptr(hidden_out), _ptr(logits_out), _stream(stream)))


def eagle3_draft_decode(handle, gamma, d2t, cache: eagle3_kv_t, draft_tokens, hidden_out=None, logits_out=None,
                        stream=None):
    _check("eagle3_draft_decode", _lib().eagle3_draft_decode(
        handle, int(gamma), _ptr(d2t), C.byref(cache), _ptr(draft_tokens), _ptr(hidden_out), _ptr(logits_out),
        _stream(stream)))


def eagle3_linear(handle, x, w, y, M, N, K, stream=None):
    _check("eagle3_linear", _lib().eagle3_linear(handle, _ptr(x), _ptr(w), _ptr(y), int(M), int(N), int(K),
                                                 _stream(stream)))


def eagle3_linear_noalloc(x, w, y, M, N, K, stream=None):
    """eagle3_linear without a handle and without any device allocation, for callers that cannot allocate
    (its split-K scratch is a fixed array in the library; M * N <= 2^21; overlapping calls race)."""
    _check("eagle3_linear_noalloc", _lib().eagle3_linear_noalloc(_ptr(x), _ptr(w), _ptr(y), int(M), int(N),
                                                                 int(K), _stream(stream)))


def eagle3_quantize_e4m3(w, dtype, N, K, codes, scales, stream=None):
    """Per-row FP8 E4M3 codes [N, K] (uint8) and fp32 scales [N] of the bf16 / fp32 matrix w [N, K]."""
    _check("eagle3_quantize_e4m3", _lib().eagle3_quantize_e4m3(_ptr(w), int(dtype), int(N), int(K), _ptr(codes),
                                                               _ptr(scales), _stream(stream)))


def eagle3_quantize_nvfp4(w, dtype, N, K, codes, block_scales, global_scale, stream=None):
    """NVFP4 codes [N, K/2] (uint8, two per byte), E4M3 block scales [N, K/16] (uint8) and the fp32 matrix
    scale [1] of the bf16 / fp32 matrix w [N, K]."""
    _check("eagle3_quantize_nvfp4", _lib().eagle3_quantize_nvfp4(_ptr(w), int(dtype), int(N), int(K), _ptr(codes),
                                                                 _ptr(block_scales), _ptr(global_scale),
                                                                 _stream(stream)))


def eagle3_accept(draft, target, batch, gamma, accepted_len, hist=None, stream=None):
    _check("eagle3_accept", _lib().eagle3_accept(_ptr(draft), _ptr(target), int(batch), int(gamma),
                                                 _ptr(accepted_len), _ptr(hist), _stream(stream)))


def eagle3_accept_relaxed(draft, topk_ids, topk_logprobs, in_thinking, batch, gamma, k, delta, accepted_len,
                          hist=None, stream=None):
    _check("eagle3_accept_relaxed", _lib().eagle3_accept_relaxed(
        _ptr(draft), _ptr(topk_ids), _ptr(topk_logprobs), _ptr(in_thinking), int(batch), int(gamma), int(k),
        float(delta), _ptr(accepted_len), _ptr(hist), _stream(stream)))


def eagle3_sample(logits, rows, V, ld, temperature, top_k, top_p, uniforms, d2t, target_vocab, tokens,
                  token_prob=None, probs=None, probs_len=0, probs_in_target=False, stream=None):
    prm = eagle3_sampling_t(float(temperature), int(top_k), float(top_p))
    _check("eagle3_sample", _lib().eagle3_sample(
        _ptr(logits), int(rows), int(V), int(ld), C.byref(prm), _ptr(uniforms), _ptr(d2t), int(target_vocab),
        _ptr(tokens), _ptr(token_prob), _ptr(probs), int(probs_len), int(bool(probs_in_target)), _stream(stream)))


def eagle3_draft_decode_sampled(handle, gamma, d2t, kv, temperature, top_k, top_p, first_logits, uniforms,
                                draft_tokens, draft_probs=None, probs_len=0, probs_in_target=False, hidden_out=None,
                                logits_out=None, stream=None):
    prm = eagle3_sampling_t(float(temperature), int(top_k), float(top_p))
    _check("eagle3_draft_decode_sampled", _lib().eagle3_draft_decode_sampled(
        handle, int(gamma), _ptr(d2t), C.byref(kv), C.byref(prm), _ptr(first_logits), _ptr(uniforms),
        _ptr(draft_tokens), _ptr(draft_probs), int(probs_len), int(bool(probs_in_target)), _ptr(hidden_out),
        _ptr(logits_out), _stream(stream)))


def eagle3_accept_residual(draft, draft_probs, target_probs, u_accept, u_resample, batch, gamma, V, accepted_len,
                           next_token, hist=None, stream=None):
    _check("eagle3_accept_residual", _lib().eagle3_accept_residual(
        _ptr(draft), _ptr(draft_probs), _ptr(target_probs), _ptr(u_accept), _ptr(u_resample), int(batch),
        int(gamma), int(V), _ptr(accepted_len), _ptr(next_token), _ptr(hist), _stream(stream)))


def eagle3_accept_typical(draft, target_probs, batch, gamma, V, epsilon, delta, accepted_len, hist=None, stream=None):
    _check("eagle3_accept_typical", _lib().eagle3_accept_typical(
        _ptr(draft), _ptr(target_probs), int(batch), int(gamma), int(V), float(epsilon), float(delta),
        _ptr(accepted_len), _ptr(hist), _stream(stream)))


def eagle3_philox_uniforms(seed, offset, n, out, stream=None):
    _check("eagle3_philox_uniforms", _lib().eagle3_philox_uniforms(
        int(seed), int(offset), int(n), _ptr(out), _stream(stream)))


def eagle3_draft_get_error(handle) -> int:
    v = C.c_int32()
    st = _lib().eagle3_draft_get_error(handle, C.byref(v))
    if st not in (OK, ERR_DEVICE_RANGE):
        raise Eagle3Error("eagle3_draft_get_error", st)
    return v.value


def eagle3_draft_clear_error(handle, stream=None):
    _check("eagle3_draft_clear_error", _lib().eagle3_draft_clear_error(handle, _stream(stream)))


PROF_KINDS = 24


def eagle3_draft_profile_enable(handle, kind_mask=-1):
    """Time the launches of the kinds in `kind_mask` (bit k = kind k; -1 all, 0 off)."""
    _check("eagle3_draft_profile_enable", _lib().eagle3_draft_profile_enable(handle, int(kind_mask)))


def eagle3_draft_profile_read(handle, kind):
    """(name, total_ms, timed_launches, launches) of one kernel kind since the last reset (synchronises)."""
    ms, t, n, name = C.c_double(), C.c_int64(), C.c_int64(), C.c_char_p()
    _check("eagle3_draft_profile_read", _lib().eagle3_draft_profile_read(
        handle, int(kind), C.byref(ms), C.byref(t), C.byref(n), C.byref(name)))
    return name.value.decode(), ms.value, t.value, n.value


def eagle3_draft_profile_reset(handle):
    _check("eagle3_draft_profile_reset", _lib().eagle3_draft_profile_reset(handle))


def eagle3_draft_destroy(handle):
    _check("eagle3_draft_destroy", _lib().eagle3_draft_destroy(handle))
