"""Thin Python binding of libmtp (include/mtp.h): ctypes mirrors of the C structs and the
entry points under the same names. Argument marshalling only -- every step of the drafter
runs in the CUDA library; there is no Python or CPU fallback. Device buffers are passed as
raw pointers (e.g. torch CUDA tensors' data_ptr()).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmtp.so")

MTP_MAX_LAYERS = 8
MTP_OK, MTP_ERR_INVALID_ARG, MTP_ERR_UNSUPPORTED_SHAPE, MTP_ERR_BAD_ORDERING, MTP_ERR_CUDA, MTP_ERR_TIMEOUT = range(6)
MTP_DTYPE_BF16, MTP_DTYPE_F32 = 0, 1
MTP_LAYER_SLIDING, MTP_LAYER_FULL = 0, 1

# Every symbol include/mtp.h declares.
EXPORTS = ("mtp_init_weights", "mtp_draft_block", "mtp_centroid_head", "mtp_verify_greedy", "mtp_get_status",
           "mtp_set_path", "mtp_destroy", "mtp_last_error", "mtp_centroid_head_noalloc", "mtp_set_logit_mask",
           "mtp_verify_sample", "mtp_set_sparse_head", "mtp_set_debug")
MASK_NEG_1E30, MASK_MIN_MINUS_ONE = 0, 1  # enum mtp_logit_mask
HEAD_AUTO, HEAD_PER_SEQUENCE, HEAD_CLUSTER_MAJOR = 0, 1, 2  # enum mtp_sparse_head


class MtpError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} failed with code {code}: {msg}")
        self.code = code


class mtp_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "backbone", "hidden", "n_layers", "n_head", "head_dim_swa", "head_dim_full", "n_kv_head", "ffn", "vocab",
        "n_centroids", "top_k", "window", "use_ordered_embeddings", "dtype", "max_batch", "max_ctx")] + [
        ("layer_type", ctypes.c_uint8 * MTP_MAX_LAYERS),
        ("rms_eps", ctypes.c_float), ("attn_scale", ctypes.c_float),
        ("rope_theta_swa", ctypes.c_float), ("rope_theta_full", ctypes.c_float)]


class mtp_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "q", "o", "gate", "up", "down", "q_norm", "attn_norm", "post_attn_norm", "ffn_norm", "post_ffn_norm")] + [
        ("layer_scalar", ctypes.c_float)]


class mtp_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "pre_proj", "post_proj", "token_embd", "centroids", "out_norm", "token_ordering")] + [
        ("layer", mtp_layer_weights * MTP_MAX_LAYERS)]


class mtp_kv(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("stride_b", ctypes.c_int64), ("stride_t", ctypes.c_int64), ("max_ctx", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmtp.so (built by build.py). Raises when it is missing: no fallback exists."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmtp.so not found at {path}; build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.mtp_init_weights.argtypes = [ctypes.POINTER(mtp_config), ctypes.POINTER(mtp_weights), vp,
                                     ctypes.POINTER(vp)]
    lib.mtp_draft_block.argtypes = [vp, vp, vp, ctypes.POINTER(mtp_kv), ctypes.POINTER(mtp_kv), vp, i32, i32, vp, vp,
                                    vp]
    lib.mtp_centroid_head.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.mtp_verify_greedy.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.mtp_verify_sample.argtypes = [vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp, vp]
    lib.mtp_centroid_head_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.mtp_get_status.argtypes = [vp]
    lib.mtp_set_path.argtypes = [vp, i32]
    lib.mtp_set_logit_mask.argtypes = [vp, i32]
    lib.mtp_set_sparse_head.argtypes = [vp, i32]
    lib.mtp_set_debug.argtypes = [vp, i32, ctypes.c_int64]
    lib.mtp_destroy.argtypes = [vp]
    lib.mtp_destroy.restype = None
    lib.mtp_last_error.argtypes = []
    lib.mtp_last_error.restype = ctypes.c_char_p
    for name in ("mtp_init_weights", "mtp_draft_block", "mtp_centroid_head", "mtp_verify_greedy",
                 "mtp_get_status", "mtp_set_path", "mtp_centroid_head_noalloc", "mtp_set_logit_mask",
                 "mtp_verify_sample", "mtp_set_sparse_head", "mtp_set_debug"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int, where: str) -> None:
    if rc != MTP_OK:
        raise MtpError(rc, where, mtp_last_error())


def mtp_last_error() -> str:
    return load_library().mtp_last_error().decode(errors="replace")


def mtp_init_weights(config: mtp_config, weights: mtp_weights, target_embed: int) -> int:
    h = ctypes.c_void_p()
    _check(load_library().mtp_init_weights(ctypes.byref(config), ctypes.byref(weights), target_embed,
                                           ctypes.byref(h)), "mtp_init_weights")
    return h.value


def mtp_draft_block(handle: int, hidden: int, last_token: int, kv_sliding, kv_full, pos: int, B: int,
                    n_draft: int, out_tokens: int, out_hidden: int = 0, stream: int = 0) -> None:
    _check(load_library().mtp_draft_block(handle, hidden, last_token,
                                          ctypes.byref(kv_sliding) if kv_sliding is not None else None,
                                          ctypes.byref(kv_full) if kv_full is not None else None,
                                          pos, B, n_draft, out_tokens, out_hidden or None, stream or None),
           "mtp_draft_block")


def mtp_centroid_head(handle: int, y: int, B: int, out_logits: int, out_token: int, out_centroids: int,
                      stream: int = 0) -> None:
    _check(load_library().mtp_centroid_head(handle, y, B, out_logits or None, out_token, out_centroids or None,
                                            stream or None), "mtp_centroid_head")


def mtp_verify_greedy(target_logits: int, draft: int, B: int, n: int, V: int, accept_len: int, out_tokens: int,
                      stream: int = 0) -> None:
    _check(load_library().mtp_verify_greedy(target_logits, draft or None, B, n, V, accept_len, out_tokens,
                                            stream or None), "mtp_verify_greedy")


def mtp_verify_sample(target_logits: int, draft: int, B: int, n: int, V: int, temperature: float, u_accept: int,
                      u_sample: int, accept_len: int, out_tokens: int, stream: int = 0) -> None:
    _check(load_library().mtp_verify_sample(target_logits, draft or None, B, n, V, float(temperature),
                                            u_accept or None, u_sample, accept_len, out_tokens, stream or None),
           "mtp_verify_sample")


def mtp_centroid_head_noalloc(y: int, centroids: int, token_ordering: int, token_embd: int, dtype: int, B: int,
                              hidden: int, n_centroids: int, top_k: int, vocab: int, out_logits: int, out_token: int,
                              out_centroids: int, stream: int = 0) -> None:
    """Centroid head without a handle and without any device allocation (static scratch of
    MTP_NOALLOC_SCRATCH_BYTES); for callers that cannot allocate device memory."""
    _check(load_library().mtp_centroid_head_noalloc(y, centroids, token_ordering, token_embd, dtype, B, hidden,
                                                    n_centroids, top_k, vocab, out_logits or None, out_token,
                                                    out_centroids or None, stream or None),
           "mtp_centroid_head_noalloc")


def mtp_get_status(handle: int) -> int:
    return load_library().mtp_get_status(handle)


def mtp_set_path(handle: int, path: int) -> None:
    _check(load_library().mtp_set_path(handle, path), "mtp_set_path")


def mtp_set_logit_mask(handle: int, mode: int) -> None:
    _check(load_library().mtp_set_logit_mask(handle, mode), "mtp_set_logit_mask")


def mtp_set_sparse_head(handle: int, mode: int) -> None:
    _check(load_library().mtp_set_sparse_head(handle, mode), "mtp_set_sparse_head")


def mtp_set_debug(handle: int, skip_arrival_cta: int, spin_limit_cycles: int) -> None:
    _check(load_library().mtp_set_debug(handle, skip_arrival_cta, spin_limit_cycles), "mtp_set_debug")


def mtp_destroy(handle: int) -> None:
    load_library().mtp_destroy(handle)
