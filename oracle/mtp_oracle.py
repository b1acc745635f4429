"""CPU oracle of the Gemma-4-assistant MTP drafter step, draft block, greedy verify and
sampled (temperature) verify.

TEST INFRASTRUCTURE ONLY. Only the test-suite, the package smoke check and the benchmark's
CPU-baseline leg may import this module. The CUDA library never calls it, and it shares
no code with the CUDA library.

Plain NumPy in float64: stored bf16 values are upcast exactly, every sum / dot product
accumulates in fp64 (NumPy matrix-vector products are used as the dot-product primitive),
one sequence at a time, in the order the pages describe the step.

Precision contract shared with the CUDA path (the pages fix no precision):
  * stored tensors (weights, K, embeddings, hidden input, target logits) are bf16, except
    in fp32 shapes where everything is fp32;
  * every activation stays in floating point wider than storage: fp64 here, fp32 in the
    kernels; no activation is rounded to bf16 between operations, and the post-projected
    hidden state carried to the next draft step is not rounded either. (Rounding every
    projection input to bf16 makes the step discontinuous: a one-ulp change of a single
    input element was measured to move the post-projected hidden state by 0.6 % and to
    flip a later drafted token, so fp32-vs-fp64 accumulation differences would cascade
    into whole-ulp differences.)
  * top-k and argmax decisions are taken on fp32 values (ties: lower centroid index,
    lower vocabulary id);
  * RoPE angles are formed in fp64.

Readings where the pages are silent or disagree (each is stated again where it is used):
  * concatenation order [target_last_hidden ; embed(last_token)];
  * embed() is a raw row of the target's input embedding table [V][bb];
  * norm form v / sqrt(mean(v^2) + eps) * g with eps 1e-6; sandwich norms around attention
    and FFN; layer_scalar multiplies the whole residual stream after the block;
  * attention scale 1/sqrt(head_dim) unless configured; q-only RoPE at the caller's
    constant position, NeoX half-split, theta 1e4 (sliding) / 1e6 (full);
  * sliding layers attend the most recent `window` keys [max(0, L-W), L); the full layer
    attends [0, L); q_len is 1 so both masks are bidirectional;
  * head i reads KV head i // (n_head / n_kv_head);
  * token_ordering viewed row-major [C][vsc]: centroid c owns ids ordering[c*vsc:(c+1)*vsc];
  * unselected vocabulary entries of the materialised row are -1e30 (fp32), or, in the
    other variant the pages give, the smallest candidate logit minus one;
  * sampled verification (the pages only say that accept rates vary with temperature):
    speculative sampling with the drafter's proposal as a point mass on the drafted token,
    uniforms passed in by the caller.

Pins: every helper and the centroid head, top-k, attention, verify and the shape counts are
pinned by the not-gpu tests against closed forms, invariants, brute force and the values
the pages print. A whole drafter step is pinned through special cases written out by
hand (zero queries, one planted key at several positions, the MLP path alone, zero
blocks); with a general query and every path active at once it is "parity unpinned" beyond
those: the pages publish no logit or token for any input.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

MASK_VALUE = np.float32(-1e30)


# ---------------------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def decode(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Storage form -> float64 values: uint16 bf16 bits, or float32."""
    if dtype == "bf16":
        return decode_bf16(arr)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------
# Elementwise pieces
# ---------------------------------------------------------------------------------------

def rms_norm(v: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm with a plain gain over the last axis.

    The tensor schema of "Gemma 4 Multi-Token Prediction (MTP) drafter" ("Tensor schema":
    attn_norm, post_attention_norm, ffn_norm, post_ffw_norm, output_norm, attn_q_norm)
    names the norms and their [hidden] / [head_dim] gains; the form and eps are a reading.
    """
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def rope(q: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary embedding of one head vector at a single position, NeoX half-split.

    The drafter predicts at one constant position ("Gemma 4 Assistant 使用指南", section
    二.2 "position_ids 恒定"); which rotary convention applies is a reading. theta == 0
    disables the rotation. Angles are formed in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    if theta == 0.0:
        return q.copy()
    d = q.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = float(pos) * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = q[..., :half], q[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ---------------------------------------------------------------------------------------
# Attention over the target's shared K (V = K)
# ---------------------------------------------------------------------------------------

def key_range(layer_type: str, ctx_len: int, window: int):
    """Keys a q_len=1 drafter query attends.

    Full layer: all of [0, L) -- with one query the causal and the bidirectional mask are
    the same ("Gemma 4 Assistant 使用指南", section 二.4, create_attention_masks).
    Sliding layer: the flipped window, i.e. the most recent `window` keys [max(0, L-W), L)
    ("Gemma 4 Multi-Token Prediction (MTP) drafter", "Runtime implementation", piece 2;
    the same blog section, swa_mask flip).
    """
    if layer_type == "F":
        return 0, int(ctx_len)
    return max(0, int(ctx_len) - int(window)), int(ctx_len)


def attention_q_only(q: np.ndarray, k: np.ndarray, v: Optional[np.ndarray], scale: float) -> np.ndarray:
    """Single-query attention of n_head query heads over external keys.

    q: [n_head][d]; k: [L][n_kv][d] already cut to the attended range; v: same shape or
    None, meaning V = K (attention_k_eq_v: "Gemma 4 Assistant tensor inventory", "Notes for
    llama.cpp port" item 2). Query head h reads KV head h // (n_head / n_kv).
    Softmax: subtract the maximum, exponentiate, normalise, all fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    vv = k if v is None else np.asarray(v, dtype=np.float64)
    n_head, d = q.shape
    n_kv = k.shape[1]
    group = n_head // n_kv
    out = np.empty((n_head, d), dtype=np.float64)
    for h in range(n_head):
        g = h // group
        s = scale * (k[:, g, :] @ q[h])
        p = np.exp(s - np.max(s))
        p /= np.sum(p)
        out[h] = p @ vv[:, g, :]
    return out


# ---------------------------------------------------------------------------------------
# Shapes and weights
# ---------------------------------------------------------------------------------------

@dataclass
class Shape:
    """Drafter hyper-parameters (plain numbers; built from the caller's description)."""
    dtype: str
    backbone: int
    hidden: int
    layer_types: Sequence[str]
    n_head: int
    head_dim_swa: int
    head_dim_full: int
    n_kv_head: int
    ffn: int
    vocab: int
    n_centroids: int
    top_k: int
    window: int
    use_ordered_embeddings: bool
    rms_eps: float = 1e-6
    attn_scale: float = 0.0
    rope_theta_swa: float = 1.0e4
    rope_theta_full: float = 1.0e6

    @classmethod
    def of(cls, s) -> "Shape":
        names = cls.__dataclass_fields__.keys()
        return cls(**{n: getattr(s, n) for n in names})

    def head_dim(self, t: str) -> int:
        return self.head_dim_full if t == "F" else self.head_dim_swa

    def scale(self, t: str) -> float:
        return self.attn_scale if self.attn_scale else 1.0 / math.sqrt(self.head_dim(t))

    def theta(self, t: str) -> float:
        return self.rope_theta_full if t == "F" else self.rope_theta_swa

    @property
    def vsc(self) -> int:
        return self.vocab // self.n_centroids


@dataclass
class DecodedWeights:
    """Weights as float64 (decoded once from storage form)."""
    pre_proj: np.ndarray
    post_proj: np.ndarray
    out_norm: np.ndarray
    token_embd: np.ndarray
    centroids: Optional[np.ndarray]
    token_ordering: Optional[np.ndarray]
    target_embed_raw: np.ndarray     # storage form; rows decoded on demand
    dtype: str
    layers: List[Dict[str, object]] = field(default_factory=list)

    def target_row(self, tok: int) -> np.ndarray:
        return decode(self.target_embed_raw[int(tok)], self.dtype)


def decode_weights(w) -> DecodedWeights:
    """Decode a weight set given in storage form (attributes as in the tensor schema)."""
    dt = w.dtype
    layers = []
    for L in w.layers:
        layers.append({k: (float(v) if k == "layer_scalar" else
                           (np.asarray(v, dtype=np.float64) if k.endswith("norm") else decode(v, dt)))
                       for k, v in L.items()})
    return DecodedWeights(
        pre_proj=decode(w.pre_proj, dt), post_proj=decode(w.post_proj, dt),
        out_norm=np.asarray(w.out_norm, dtype=np.float64), token_embd=decode(w.token_embd, dt),
        centroids=None if w.centroids is None else decode(w.centroids, dt),
        token_ordering=None if w.token_ordering is None else np.asarray(w.token_ordering, dtype=np.int64),
        target_embed_raw=w.target_embed, dtype=dt, layers=layers)


def param_count(s: Shape) -> int:
    """Trainable parameters of the drafter per the tensor schema (token_ordering is a
    buffer, not a parameter): token_embd, output_norm, pre/post projection, centroids and
    per block q, q_norm, o, four norms, gate/up/down and layer_scalar ("Gemma 4
    Multi-Token Prediction (MTP) drafter", "Tensor schema")."""
    H, bb = s.hidden, s.backbone
    n = s.vocab * H + H + 2 * bb * H + H * bb
    if s.use_ordered_embeddings:
        n += H * s.n_centroids
    for t in s.layer_types:
        d = s.head_dim(t)
        n += 2 * H * s.n_head * d + d + 4 * H + 3 * H * s.ffn + 1
    return n


def checkpoint_bytes(s: Shape) -> int:
    """bf16 parameters plus the token_ordering buffer stored as F32 ("Tensor schema" note:
    the 1-D ordering is force-stored F32)."""
    b = 2 * param_count(s)
    if s.use_ordered_embeddings:
        b += 4 * s.vocab
    return b


# ---------------------------------------------------------------------------------------
# Heads
# ---------------------------------------------------------------------------------------

def topk_desc(values32: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest fp32 values, largest first; equal values: lower index first."""
    v = np.asarray(values32, dtype=np.float32)
    order = np.lexsort((np.arange(v.size), -v.astype(np.float64)))
    return order[:k].astype(np.int64)


def argmax_lowest(values32: np.ndarray, ids: Optional[np.ndarray] = None) -> int:
    """Id of the largest fp32 value; equal values: the lowest id wins.

    `ids` maps positions to vocabulary ids (sparse candidates); None means position = id.
    """
    v = np.asarray(values32, dtype=np.float32)
    m = v.max()
    pos = np.nonzero(v == m)[0]
    if ids is None:
        return int(pos.min())
    return int(np.asarray(ids)[pos].min())


def top2_gap(values: np.ndarray) -> float:
    v = np.sort(np.asarray(values, dtype=np.float64))
    return float(v[-1] - v[-2]) if v.size > 1 else math.inf


@dataclass
class HeadResult:
    token: int
    centroid_logits: Optional[np.ndarray] = None   # fp64 [C]
    selected: Optional[np.ndarray] = None          # [k] centroid ids, best first
    ids: Optional[np.ndarray] = None               # [k*vsc] candidate vocab ids
    logits: Optional[np.ndarray] = None            # fp64 logits of the candidates (or all V)
    logit_gap: float = math.inf                    # top-2 gap of the token logits (fp64)
    kth_gap: float = math.inf                      # k-th minus (k+1)-th centroid logit


def centroid_head(s: Shape, W: DecodedWeights, yb: np.ndarray) -> HeadResult:
    """Centroid-clustered sparse LM head on one final-normed hidden state.

    Steps as in "Gemma 4 Assistant tensor inventory", section "Centroid / ordered embeddings
    LM head", steps 1-4, and "Gemma 4 Assistant 使用指南" section 五 (use_ordered_embeddings
    steps 1-3): centroid logits; top-k centroids; gather the vsc token ids each selected
    centroid owns from token_ordering viewed [C][vsc]; dot the gathered token_embd rows with
    the hidden state. The token is the argmax over the candidates (greedy drafting).
    """
    assert s.vocab % s.n_centroids == 0
    c = W.centroids @ yb
    sel = topk_desc(c.astype(np.float32), s.top_k)
    srt = np.sort(c.astype(np.float32).astype(np.float64))[::-1]
    kth_gap = float(srt[s.top_k - 1] - srt[s.top_k]) if s.top_k < s.n_centroids else math.inf
    ids = W.token_ordering.reshape(s.n_centroids, s.vsc)[sel].reshape(-1)
    logits = W.token_embd[ids] @ yb
    tok = argmax_lowest(logits.astype(np.float32), ids)
    return HeadResult(token=tok, centroid_logits=c, selected=sel, ids=ids, logits=logits,
                      logit_gap=top2_gap(logits), kth_gap=kth_gap)


def materialise_row(s: Shape, head: HeadResult, mask: str = "neg_1e30") -> np.ndarray:
    """Full-vocabulary fp32 row with the sparse logits scattered at their ids.

    mask "neg_1e30": every other entry is -1e30 ("Gemma 4 Assistant tensor inventory",
    "Centroid / ordered embeddings LM head", step 5: a dense -1e30 fill, then the rows set).
    mask "min_minus_one": every other entry is the smallest candidate logit minus one, both
    in fp32 ("Gemma 4 Assistant 使用指南", section 五, use_ordered_embeddings step 3, where the
    unscored positions take a mask value one below the smallest logit; the tensor-inventory
    page names it as the MLX variant)."""
    vals = head.logits.astype(np.float32)
    if mask == "neg_1e30":
        fill = MASK_VALUE
    elif mask == "min_minus_one":
        fill = np.float32(np.float32(vals.min()) - np.float32(1.0))
    else:
        raise ValueError(f"unknown mask {mask!r}")
    row = np.full(s.vocab, fill, dtype=np.float32)
    row[head.ids] = vals
    return row


def dense_head(s: Shape, W: DecodedWeights, yb: np.ndarray) -> HeadResult:
    """Dense tied LM head: logits over every vocabulary row of token_embd, then argmax
    (use_ordered_embeddings = false: "Gemma 4 Assistant tensor inventory", "HF config
    highlights"; "Gemma 4 Assistant 使用指南" section 五)."""
    logits = W.token_embd @ yb
    return HeadResult(token=argmax_lowest(logits.astype(np.float32)), logits=logits,
                      logit_gap=top2_gap(logits))


# ---------------------------------------------------------------------------------------
# One drafter step for one sequence
# ---------------------------------------------------------------------------------------

@dataclass
class StepResult:
    token: int
    hidden_out: np.ndarray          # post_projection output h' (fp64, [bb])
    head: HeadResult
    x_layers: List[np.ndarray]      # residual stream after each block
    q: List[np.ndarray]             # attention query per block (after q_norm and RoPE)
    o: List[np.ndarray]             # attention output per block [n_head][d]
    y: np.ndarray                   # final normed hidden (before rounding)


def drafter_step(s: Shape, W: DecodedWeights, h: np.ndarray, tok: int,
                 k_by_type: Dict[str, np.ndarray], v_by_type: Dict[str, Optional[np.ndarray]],
                 ctx_len: int, pos: int) -> StepResult:
    """One drafter forward at q_len = 1 for one sequence.

    h: target (or previous step's) hidden state [bb], float64 holding stored values.
    k_by_type: {"S": K [Lmax][n_kv][d_s], "F": K [Lmax][n_kv][d_f]} in storage form.

    Order of operations:
      1. u = [h ; embed(tok)] with embed() a row of the target's input embedding table;
         x = pre_projection(u) ("Gemma 4 Multi-Token Prediction (MTP) drafter", "What it
         is", 2x backbone input; "Gemma 4 drafter explained", "Target Activations").
      2. per block: a = norm(x); q = W_q a; per head q_norm then RoPE at the constant
         position; attention over the target's shared K of the block's type with V = K;
         x += norm(W_o o); f = norm(x); x += norm(W_down(gelu_tanh(W_gate f) * W_up f));
         x *= layer_scalar ("Tensor schema" per-block tensors; "What it is": Q-only
         attention and the per-layer scalar gate).
      3. y = output_norm(x); h' = post_projection(y) ("Tensor schema"; "Gemma 4 Assistant
         使用指南" section 六: last_hidden_state is post-projected).
      4. head on y (centroid or dense) -> greedy token.
    Activations are fp64 throughout (no intermediate rounding).
    """
    dt = s.dtype
    u = np.concatenate([np.asarray(h, dtype=np.float64), W.target_row(tok)])
    x = W.pre_proj @ u
    x_layers, qs, os_ = [], [], []
    for li, t in enumerate(s.layer_types):
        L = W.layers[li]
        d = s.head_dim(t)
        a = rms_norm(x, L["attn_norm"], s.rms_eps)
        q = (L["q"] @ a).reshape(s.n_head, d)
        q = rms_norm(q, L["q_norm"], s.rms_eps)
        q = np.stack([rope(q[hh], pos, s.theta(t)) for hh in range(s.n_head)])
        lo, hi = key_range(t, ctx_len, s.window)
        k = decode(k_by_type[t][lo:hi], dt)
        v = v_by_type.get(t)
        v = None if v is None else decode(v[lo:hi], dt)
        o = attention_q_only(q, k, v, s.scale(t))
        attn = L["o"] @ o.reshape(-1)
        x = x + rms_norm(attn, L["post_attn_norm"], s.rms_eps)
        f = rms_norm(x, L["ffn_norm"], s.rms_eps)
        m = gelu_tanh(L["gate"] @ f) * (L["up"] @ f)
        x = x + rms_norm(L["down"] @ m, L["post_ffn_norm"], s.rms_eps)
        x = x * L["layer_scalar"]
        x_layers.append(x.copy()); qs.append(q); os_.append(o)
    y = rms_norm(x, W.out_norm, s.rms_eps)
    h_out = W.post_proj @ y
    head = centroid_head(s, W, y) if s.use_ordered_embeddings else dense_head(s, W, y)
    return StepResult(token=head.token, hidden_out=h_out, head=head, x_layers=x_layers,
                      q=qs, o=os_, y=y)


def next_hidden(h_out: np.ndarray) -> np.ndarray:
    """Hidden state fed to the next draft step: the post-projected output itself
    ("Gemma 4 drafter explained", "Target Activations": later rounds use the drafter's own
    up-projected activations), carried without rounding."""
    return np.asarray(h_out, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# Draft block
# ---------------------------------------------------------------------------------------

@dataclass
class BlockResult:
    tokens: np.ndarray        # [B][n] int64
    hidden_out: np.ndarray    # [B][n][bb] fp64 (post_projection output of every step)
    logit_gap: np.ndarray     # [B][n] top-2 gap of the token logits
    kth_gap: np.ndarray       # [B][n] k-th vs (k+1)-th centroid logit gap
    selected: Optional[np.ndarray]  # [B][n][k]
    steps: List[List[StepResult]]


def draft_block(s: Shape, W: DecodedWeights, hidden, last_token, k_swa, k_full, ctx_len, pos,
                n_draft: int, v_swa=None, v_full=None, keep_steps: bool = False) -> BlockResult:
    """Iterate the drafter step n_draft times per sequence.

    The first step consumes the target's hidden state and last token; each later step
    consumes the previous step's greedy token and its post-projected hidden state
    ("Gemma 4 Assistant 使用指南" section 二.3, the table of the "last seen token";
    "Gemma 4 drafter explained", "Target Activations", rounds 2 and 3).
    The K (and hence the position) stays the same for the whole block (section 二.2).
    """
    B = len(last_token)
    bb = s.backbone
    toks = np.zeros((B, n_draft), dtype=np.int64)
    hout = np.zeros((B, n_draft, bb), dtype=np.float64)
    lgap = np.zeros((B, n_draft)); kgap = np.full((B, n_draft), math.inf)
    sel = np.zeros((B, n_draft, s.top_k), dtype=np.int64) if s.use_ordered_embeddings else None
    steps: List[List[StepResult]] = []
    for b in range(B):
        h = decode(hidden[b], s.dtype)
        tok = int(last_token[b])
        kb = {}
        vb = {}
        if k_swa is not None:
            kb["S"] = k_swa[b]; vb["S"] = None if v_swa is None else v_swa[b]
        if k_full is not None:
            kb["F"] = k_full[b]; vb["F"] = None if v_full is None else v_full[b]
        row = []
        for i in range(n_draft):
            r = drafter_step(s, W, h, tok, kb, vb, int(ctx_len[b]), int(pos[b]))
            toks[b, i] = r.token
            hout[b, i] = r.hidden_out
            lgap[b, i] = r.head.logit_gap
            kgap[b, i] = r.head.kth_gap
            if sel is not None:
                sel[b, i] = r.head.selected
            if keep_steps:
                row.append(r)
            tok = r.token
            h = next_hidden(r.hidden_out)
        steps.append(row)
    return BlockResult(tokens=toks, hidden_out=hout, logit_gap=lgap, kth_gap=kgap, selected=sel, steps=steps)


# ---------------------------------------------------------------------------------------
# Greedy verification
# ---------------------------------------------------------------------------------------

def verify_greedy(target_logits: np.ndarray, drafts: np.ndarray, logits_dtype: str = "bf16"):
    """Greedy accept-prefix check of a draft against the target's logits.

    target_logits: [B][n+1][V] (bf16 bits or fp32); drafts: [B][n].
    Row i's target token is the argmax of row i (lowest id on ties). Drafts are accepted
    while they equal the target's token; at the first disagreement the target's token
    replaces the rejected draft; when all n are accepted the target's token of row n is
    appended ("Gemma 4 drafter explained", "What is Speculative Decoding?"; greedy
    acceptance as with --temp 0 in "Gemma 4 Multi-Token Prediction (MTP) drafter",
    "Runtime implementation").
    Returns accept_len [B] and out_tokens [B][n+1] padded with -1.
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    B, n = drafts.shape
    acc = np.zeros(B, dtype=np.int64)
    out = np.full((B, n + 1), -1, dtype=np.int64)
    for b in range(B):
        a = 0
        while True:
            row = decode(target_logits[b, a], logits_dtype).astype(np.float32)
            t = argmax_lowest(row)
            if a < n and int(drafts[b, a]) == t:
                out[b, a] = t
                a += 1
                continue
            out[b, a] = t
            break
        acc[b] = a
    return acc, out


def accept_rate(n_accept: int, n_drafted: int) -> float:
    """Acceptance rate as the pages report it: accepted drafts over drafted tokens
    ("Gemma 4 Multi-Token Prediction (MTP) drafter", "Runtime implementation")."""
    return n_accept / n_drafted


def verify_sample(target_logits: np.ndarray, drafts: np.ndarray, temperature: float, u_accept: np.ndarray,
                  u_sample: np.ndarray, logits_dtype: str = "bf16"):
    """Sampled verification of a greedy draft at a temperature.

    The pages give the accept-until-disagreement structure ("Gemma 4 drafter explained",
    "What is Speculative Decoding?") and note that the accept rate varies with temperature
    ("Gemma 4 Multi-Token Prediction (MTP) drafter", "Status"); they give no stochastic
    acceptance rule. This follows speculative sampling (Leviathan, Kalman, Matias 2023;
    Chen et al. 2023) with the drafter's proposal q = a point mass on the drafted token d_i
    (the drafter drafts greedily):
      p_i = softmax(target_logits[i] / T);
      accept d_i when u_accept[i] < min(1, p_i(d_i) / q(d_i)) = p_i(d_i);
      at the first rejection emit a sample of the residual max(0, p_i - q) / Z, i.e. p_i with
      d_i removed and renormalised (inverse CDF over increasing ids: the smallest v whose
      cumulative residual mass exceeds u_sample[i] * Z);
      when every draft is accepted emit a sample of p_n with u_sample[n].
    The emitted tokens are then distributed as sampling from the target at temperature T.
    T = 0 is greedy verification (verify_greedy).

    target_logits: [B][n+1][V] (bf16 bits or fp32); drafts [B][n]; u_accept [B][n] and
    u_sample [B][n+1] uniforms in [0, 1). Returns accept_len [B], out_tokens [B][n+1] (-1
    padded) and, per sequence, the smallest distance (relative to the mass compared against)
    between a uniform and the boundary that decided the outcome, in fp64.
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    B, n = drafts.shape
    if temperature == 0.0:
        acc, out = verify_greedy(target_logits, drafts, logits_dtype)
        return acc, out, np.full(B, np.inf)
    if temperature < 0.0:
        raise ValueError("temperature must be >= 0")
    acc = np.zeros(B, dtype=np.int64)
    out = np.full((B, n + 1), -1, dtype=np.int64)
    margin = np.full(B, np.inf)
    for b in range(B):
        i = 0
        while True:
            z = decode(target_logits[b, i], logits_dtype).astype(np.float64) / temperature
            w = np.exp(z - z.max())
            Z = w.sum()
            if i < n:
                d = int(drafts[b, i])
                pd = w[d] / Z
                ua = float(u_accept[b, i])
                margin[b] = min(margin[b], abs(ua - pd))
                if ua < pd:
                    out[b, i] = d
                    i += 1
                    continue
                w = w.copy()
                w[d] = 0.0
            c = np.cumsum(w)
            target = float(u_sample[b, i]) * c[-1]
            t = int(np.searchsorted(c, target, side="right"))
            t = min(t, len(c) - 1)
            lo = c[t - 1] if t > 0 else 0.0
            margin[b] = min(margin[b], min(target - lo, c[t] - target) / c[-1])
            out[b, i] = t
            break
        acc[b] = i
    return acc, out, margin
