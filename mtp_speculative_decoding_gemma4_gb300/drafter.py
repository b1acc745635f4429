"""Torch-facing convenience layer over the C ABI: holds the device tensors a handle borrows,
fills the ctypes structs from them and allocates outputs. Marshalling only; the drafter
runs entirely in libmtp.so.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B

_DT = {"bf16": (B.MTP_DTYPE_BF16, torch.bfloat16), "f32": (B.MTP_DTYPE_F32, torch.float32)}


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _need_cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def make_config(shape, max_batch: int, max_ctx: int) -> B.mtp_config:
    """mtp_config from any object with the drafter-shape attributes (dtype, backbone, hidden,
    layer_types ('S'/'F'), n_head, head_dim_swa/full, n_kv_head, ffn, vocab, n_centroids,
    top_k, window, use_ordered_embeddings, rms_eps, attn_scale, rope_theta_swa/full)."""
    c = B.mtp_config()
    for f in ("backbone", "hidden", "n_head", "head_dim_swa", "head_dim_full", "n_kv_head", "ffn", "vocab",
              "n_centroids", "top_k", "window"):
        setattr(c, f, int(getattr(shape, f)))
    c.n_layers = len(shape.layer_types)
    c.use_ordered_embeddings = 1 if shape.use_ordered_embeddings else 0
    c.dtype = _DT[shape.dtype][0]
    c.max_batch, c.max_ctx = int(max_batch), int(max_ctx)
    for i, t in enumerate(shape.layer_types):
        c.layer_type[i] = B.MTP_LAYER_FULL if t == "F" else B.MTP_LAYER_SLIDING
    c.rms_eps, c.attn_scale = float(shape.rms_eps), float(shape.attn_scale)
    c.rope_theta_swa, c.rope_theta_full = float(shape.rope_theta_swa), float(shape.rope_theta_full)
    return c


def make_kv(k: torch.Tensor, ctx_len: torch.Tensor, v: Optional[torch.Tensor] = None) -> B.mtp_kv:
    """mtp_kv for a right-padded K tensor [B][Lmax][n_kv][d] (and optional V of that shape)."""
    _need_cuda(k, "k")
    kv = B.mtp_kv()
    kv.k, kv.v, kv.ctx_len = _ptr(k), _ptr(v), _ptr(ctx_len)
    kv.stride_b, kv.stride_t, kv.max_ctx = k.stride(0), k.stride(1), k.shape[1]
    return kv


class Drafter:
    """One drafter (weights + workspace) on the current CUDA device."""

    def __init__(self, shape, weights, target_embed: torch.Tensor, max_batch: int, max_ctx: int):
        self.shape = shape
        self.torch_dtype = _DT[shape.dtype][1]
        self._keep = [target_embed]
        self.config = make_config(shape, max_batch, max_ctx)
        w = B.mtp_weights()
        for f in ("pre_proj", "post_proj", "token_embd", "centroids", "out_norm", "token_ordering"):
            t = weights.get(f)
            if t is not None:
                _need_cuda(t, f)
                self._keep.append(t)
            setattr(w, f, _ptr(t))
        for i, L in enumerate(weights["layers"]):
            for f in ("q", "o", "gate", "up", "down", "q_norm", "attn_norm", "post_attn_norm", "ffn_norm",
                      "post_ffn_norm"):
                t = _need_cuda(L[f], f)
                self._keep.append(t)
                setattr(w.layer[i], f, _ptr(t))
            w.layer[i].layer_scalar = float(L["layer_scalar"])
        self.weights = w
        self.handle = B.mtp_init_weights(self.config, w, _ptr(_need_cuda(target_embed, "target_embed")))

    # ------------------------------------------------------------------ calls
    def draft_block(self, hidden, last_token, k_swa, k_full, ctx_len, pos, n_draft: int, want_hidden: bool = True,
                    v_swa=None, v_full=None, out_tokens=None, out_hidden=None, stream: int = 0):
        Bn = hidden.shape[0]
        dev = hidden.device
        if out_tokens is None:
            out_tokens = torch.empty((Bn, n_draft), dtype=torch.int32, device=dev)
        if out_hidden is None and want_hidden:
            out_hidden = torch.empty((Bn, n_draft, self.shape.backbone), dtype=torch.float32, device=dev)
        kv_s = make_kv(k_swa, ctx_len, v_swa) if k_swa is not None else None
        kv_f = make_kv(k_full, ctx_len, v_full) if k_full is not None else None
        B.mtp_draft_block(self.handle, _ptr(hidden), _ptr(last_token), kv_s, kv_f, _ptr(pos), Bn, n_draft,
                          _ptr(out_tokens), _ptr(out_hidden), stream)
        return out_tokens, out_hidden

    def centroid_head(self, y: torch.Tensor, want_logits: bool = False, want_centroids: bool = False,
                      stream: int = 0):
        Bn = y.shape[0]
        dev = y.device
        tok = torch.empty(Bn, dtype=torch.int32, device=dev)
        logits = torch.empty((Bn, self.shape.vocab), dtype=torch.float32, device=dev) if want_logits else None
        cents = (torch.empty((Bn, self.shape.top_k), dtype=torch.int32, device=dev)
                 if want_centroids and self.shape.use_ordered_embeddings else None)
        B.mtp_centroid_head(self.handle, _ptr(_need_cuda(y, "y")), Bn, _ptr(logits), _ptr(tok), _ptr(cents), stream)
        return tok, logits, cents

    def set_path(self, path: int) -> None:
        B.mtp_set_path(self.handle, path)

    def set_logit_mask(self, mode: int) -> None:
        """Mask of the rows centroid_head materialises: binding.MASK_NEG_1E30 (default) or
        binding.MASK_MIN_MINUS_ONE (smallest selected logit minus one)."""
        B.mtp_set_logit_mask(self.handle, mode)

    def set_sparse_head(self, mode: int) -> None:
        """Traversal of the centroid head's candidate rows: binding.HEAD_AUTO (default),
        HEAD_PER_SEQUENCE, or HEAD_CLUSTER_MAJOR (each selected cluster read once per step)."""
        B.mtp_set_sparse_head(self.handle, mode)

    def set_debug(self, skip_arrival_cta: int = -1, spin_limit_cycles: int = 0) -> None:
        """Testing only: make one CTA of the persistent kernel miss its first grid-barrier
        arrival (the bounded waits then report MTP_ERR_TIMEOUT) and / or shorten the wait bound."""
        B.mtp_set_debug(self.handle, skip_arrival_cta, spin_limit_cycles)

    def status(self) -> int:
        return B.mtp_get_status(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            B.mtp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def verify_sample(target_logits: torch.Tensor, drafts: torch.Tensor, temperature: float, u_accept: torch.Tensor,
                  u_sample: torch.Tensor, accept_len=None, out_tokens=None, stream: int = 0):
    """Sampled verification at a temperature: target_logits bf16 [B][n+1][V], drafts int32
    [B][n], uniforms fp32 u_accept [B][n] and u_sample [B][n+1] (device tensors)."""
    Bn, n1, V = target_logits.shape
    dev = target_logits.device
    if accept_len is None:
        accept_len = torch.empty(Bn, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((Bn, n1), dtype=torch.int32, device=dev)
    B.mtp_verify_sample(_ptr(_need_cuda(target_logits, "target_logits")), _ptr(drafts), Bn, n1 - 1, V, temperature,
                        _ptr(u_accept), _ptr(_need_cuda(u_sample, "u_sample")), _ptr(accept_len), _ptr(out_tokens),
                        stream)
    return accept_len, out_tokens


def verify_greedy(target_logits: torch.Tensor, drafts: torch.Tensor, accept_len=None, out_tokens=None,
                  stream: int = 0):
    """Greedy accept-prefix check: target_logits bf16 [B][n+1][V], drafts int32 [B][n]."""
    Bn, n1, V = target_logits.shape
    dev = target_logits.device
    if accept_len is None:
        accept_len = torch.empty(Bn, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((Bn, n1), dtype=torch.int32, device=dev)
    B.mtp_verify_greedy(_ptr(_need_cuda(target_logits, "target_logits")), _ptr(drafts), Bn, n1 - 1, V,
                        _ptr(accept_len), _ptr(out_tokens), stream)
    return accept_len, out_tokens
