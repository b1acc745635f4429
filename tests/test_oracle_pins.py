"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the pages
print (tests/golden/*.json, with citations), a closed form, an invariant, a library
routine for a special case, or brute force on a tiny input.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from mtp_synth import configs as C
from mtp_synth import gen as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ number formats

def test_decode_bf16_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F7F], dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.decode_bf16(bits), ref)


# ------------------------------------------------------------------ elementwise pieces

def test_rms_norm_constant_vector_and_scale_invariance():
    g = np.linspace(0.5, 1.5, 64)
    for c in (3.0, -0.25):
        out = O.rms_norm(np.full(64, c), g, 1e-6)
        np.testing.assert_allclose(out, np.sign(c) * g * abs(c) / math.sqrt(c * c + 1e-6), rtol=1e-15)
    v = np.random.default_rng(1).standard_normal(256)
    np.testing.assert_allclose(O.rms_norm(7.0 * v, 1.0, 0.0), O.rms_norm(v, 1.0, 0.0), rtol=1e-13)
    assert np.all(O.rms_norm(np.zeros(8), 1.0, 1e-6) == 0.0)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((5, 96))
    g = 1 + 0.02 * rng.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(v), (96,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(v, g, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_gelu_tanh_closed_forms_and_torch():
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    x = np.linspace(-9, 9, 1001)
    np.testing.assert_allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, atol=1e-12)   # odd part is x/2
    np.testing.assert_allclose(O.gelu_tanh(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(O.gelu_tanh(x), ref, rtol=1e-12, atol=1e-14)


def test_rope_identity_norm_composition_relative():
    rng = np.random.default_rng(3)
    d = 64
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    np.testing.assert_array_equal(O.rope(q, 0, 1e4), q)
    np.testing.assert_array_equal(O.rope(q, 123, 0.0), q)
    r = O.rope(q, 4097, 1e6)
    assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
    np.testing.assert_allclose(O.rope(O.rope(q, 5, 1e4), 9, 1e4), O.rope(q, 14, 1e4), atol=1e-12)
    # dot products depend only on the position difference
    a = O.rope(q, 100, 1e4) @ O.rope(k, 37, 1e4)
    b = O.rope(q, 63, 1e4) @ k
    assert abs(a - b) < 1e-10
    # d = 2: a plain rotation by `pos` radians (inverse frequency 1)
    v = np.array([1.0, 0.0])
    np.testing.assert_allclose(O.rope(v, 1, 10.0), [math.cos(1.0), math.sin(1.0)], atol=1e-15)


# ------------------------------------------------------------------ attention

def _sdpa(q, k, scale):
    # torch's scaled_dot_product_attention over an explicit all-true mask (bidirectional)
    nh, d = q.shape
    n_kv = k.shape[1]
    kk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(nh // n_kv, dim=0)  # [nh][L][d]
    qq = torch.from_numpy(q)[:, None, :]
    mask = torch.ones(nh, 1, k.shape[0], dtype=torch.bool)
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, kk, attn_mask=mask, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("nh,n_kv,d,L", [(2, 1, 32, 64), (8, 2, 16, 300), (4, 4, 8, 5)])
def test_attention_full_equals_bidirectional_sdpa(nh, n_kv, d, L):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((nh, d)); k = rng.standard_normal((L, n_kv, d))
    np.testing.assert_allclose(O.attention_q_only(q, k, None, 0.3), _sdpa(q, k, 0.3), rtol=1e-12, atol=1e-13)


def test_attention_invariants():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 16)); k = rng.standard_normal((50, 1, 16))
    o = O.attention_q_only(q, k, None, 0.25)
    # key order does not matter (q_len = 1: no position in the mask)
    np.testing.assert_allclose(O.attention_q_only(q, k[::-1], None, 0.25), o, rtol=1e-13)
    # one key -> that key; identical keys -> that key
    np.testing.assert_allclose(O.attention_q_only(q, k[:1], None, 0.25), np.repeat(k[0], 4, 0), rtol=0, atol=0)
    same = np.repeat(k[:1], 7, axis=0)
    np.testing.assert_allclose(O.attention_q_only(q, same, None, 0.25), np.repeat(k[0], 4, 0), atol=1e-15)
    # V = None is V = K, bit for bit
    np.testing.assert_array_equal(O.attention_q_only(q, k, k, 0.25), o)


def test_attention_gqa_head_mapping():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 8)); k = rng.standard_normal((20, 2, 8))
    o = O.attention_q_only(q, k, None, 0.5)
    # heads 0,1 read kv head 0; heads 2,3 read kv head 1
    np.testing.assert_allclose(o[:2], O.attention_q_only(q[:2], k[:, :1], None, 0.5), rtol=1e-14)
    np.testing.assert_allclose(o[2:], O.attention_q_only(q[2:], k[:, 1:], None, 0.5), rtol=1e-14)


def test_sliding_window_is_the_flipped_mask():
    for L, W in [(4096, 512), (300, 512), (512, 512), (513, 512), (1, 4)]:
        lo, hi = O.key_range("S", L, W)
        # flip construction: in reversed key order the window is the first W positions;
        # flipping back gives the mask over the original order
        rev_mask = np.arange(L) < W
        mask = rev_mask[::-1]
        np.testing.assert_array_equal(np.nonzero(mask)[0], np.arange(lo, hi))
        assert hi - lo == min(L, W)
        if L > W:
            assert lo == L - W          # the key at distance exactly W is excluded
        assert O.key_range("F", L, W) == (0, L)


def test_sliding_equals_full_when_context_fits_window():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 8)); k = rng.standard_normal((30, 1, 8))
    lo, hi = O.key_range("S", 30, 64)
    np.testing.assert_array_equal(O.attention_q_only(q, k[lo:hi], None, 0.3),
                                  O.attention_q_only(q, k, None, 0.3))


# ------------------------------------------------------------------ heads

def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(8)
    for trial in range(300):
        n = int(rng.integers(1, 65)); k = int(rng.integers(1, n + 1))
        v = rng.integers(-4, 5, size=n).astype(np.float32)      # many exact ties
        brute = [i for _, i in sorted((-float(v[i]), i) for i in range(n))][:k]
        assert list(O.topk_desc(v, k)) == brute


def test_argmax_lowest_id_on_ties():
    v = np.array([1.0, 3.0, 3.0, 2.0], dtype=np.float32)
    assert O.argmax_lowest(v) == 1
    assert O.argmax_lowest(v, ids=np.array([40, 30, 20, 10])) == 20


def _tiny_head_shape(V=512, Cn=16, k=3, H=24):
    return O.Shape(dtype="bf16", backbone=8, hidden=H, layer_types=("F",), n_head=1, head_dim_swa=8,
                   head_dim_full=8, n_kv_head=1, ffn=8, vocab=V, n_centroids=Cn, top_k=k, window=0,
                   use_ordered_embeddings=True)


def _tiny_head_weights(s, seed):
    rng = np.random.default_rng(seed)
    W = O.DecodedWeights(pre_proj=None, post_proj=None, out_norm=None,
                         token_embd=O.decode_bf16(G.bf16_bits(0.02 * rng.standard_normal((s.vocab, s.hidden)))),
                         centroids=O.decode_bf16(G.bf16_bits(0.02 * rng.standard_normal((s.n_centroids, s.hidden)))),
                         token_ordering=rng.permutation(s.vocab), target_embed_raw=None, dtype="bf16")
    return W


def test_centroid_head_matches_dense_on_selected_clusters():
    s = _tiny_head_shape()
    hits = 0
    for seed in range(100):
        W = _tiny_head_weights(s, seed)
        y = np.random.default_rng(100 + seed).standard_normal(s.hidden)
        head = O.centroid_head(s, W, y)
        dense = O.dense_head(s, W, y)
        # sparse logits equal the dense logits at the gathered ids
        np.testing.assert_array_equal(head.logits, dense.logits[head.ids])
        # the gathered ids are exactly the members of the selected clusters
        members = W.token_ordering.reshape(s.n_centroids, s.vsc)[head.selected]
        assert set(head.ids.tolist()) == set(members.reshape(-1).tolist())
        assert len(head.ids) == s.top_k * s.vsc
        # materialised row: -1e30 exactly outside the candidates
        row = O.materialise_row(s, head)
        mask = np.ones(s.vocab, bool); mask[head.ids] = False
        assert np.all(row[mask] == np.float32(-1e30)) and np.sum(~mask) == s.top_k * s.vsc
        np.testing.assert_array_equal(row[head.ids], head.logits.astype(np.float32))
        # when the dense argmax lies in a selected cluster the sparse argmax equals it
        if dense.token in set(head.ids.tolist()):
            hits += 1
            assert head.token == dense.token
    assert hits >= 5


def test_min_minus_one_mask_orders_every_unselected_entry_below_the_candidates():
    # "Gemma 4 Assistant 使用指南" section 五, use_ordered_embeddings step 3: the entries no
    # cluster scored take a mask value one below the smallest logit. Invariants: the argmax is
    # the head's token under both masks; every masked entry lies strictly below every
    # candidate (a dropped "- 1", a "+ 1" or a max in place of the min breaks this) and one
    # unit below the smallest; the candidates are the same under both masks.
    s = _tiny_head_shape()
    for seed in range(40):
        W = _tiny_head_weights(s, seed)
        y = np.random.default_rng(300 + seed).standard_normal(s.hidden)
        head = O.centroid_head(s, W, y)
        r0 = O.materialise_row(s, head)
        r1 = O.materialise_row(s, head, mask="min_minus_one")
        unsel = np.ones(s.vocab, bool)
        unsel[head.ids] = False
        cand = r1[~unsel]
        np.testing.assert_array_equal(cand, r0[~unsel])
        assert np.all(r1[unsel] < cand.min())
        assert len(np.unique(r1[unsel])) == 1
        assert abs(float(cand.min()) - float(r1[unsel][0]) - 1.0) < 1e-6 * max(1.0, abs(float(cand.min())))
        assert int(np.argmax(r1)) == int(np.argmax(r0)) == head.token
    with pytest.raises(ValueError):
        O.materialise_row(s, head, mask="zero")


def test_centroid_head_recovers_planted_token():
    # clusters built around centroid directions: y along a member of cluster 5 selects that
    # cluster first, and the dense winner is found inside it
    s = _tiny_head_shape(V=256, Cn=8, k=2, H=32)
    rng = np.random.default_rng(9)
    cent = rng.standard_normal((s.n_centroids, s.hidden))
    order = rng.permutation(s.vocab)
    T = np.empty((s.vocab, s.hidden))
    for c in range(s.n_centroids):
        T[order[c * s.vsc:(c + 1) * s.vsc]] = cent[c] + 0.1 * rng.standard_normal((s.vsc, s.hidden))
    W = O.DecodedWeights(None, None, None, T, cent, order, None, "f32")
    target = order[5 * s.vsc + 7]
    y = T[target] * 3.0
    head = O.centroid_head(s, W, y)
    assert head.selected[0] == 5 and head.token == O.dense_head(s, W, y).token
    assert head.token in set(order[5 * s.vsc:6 * s.vsc].tolist()) and target in set(head.ids.tolist())


def test_near_tie_gaps_are_the_decision_margins():
    # the gaps that decide whether a GPU/oracle token difference is tolerated: top2_gap is the
    # largest minus the second largest value (0 for a tie, inf for one value); the head's
    # kth_gap is the k-th minus the (k+1)-th centroid logit and its logit_gap the top-2 gap of
    # the candidate logits. Planted on a unit y so every logit is a chosen number.
    assert O.top2_gap(np.array([3.0, 1.0, 2.0])) == 1.0
    assert O.top2_gap(np.array([2.0, 2.0, 1.0])) == 0.0
    assert O.top2_gap(np.array([-1.0, -4.0])) == 3.0
    assert O.top2_gap(np.array([7.0])) == math.inf
    s = _tiny_head_shape(V=64, Cn=8, k=3, H=4)
    order = np.random.default_rng(4).permutation(s.vocab)
    cent = np.zeros((s.n_centroids, s.hidden))
    # sorted: 5, 4, 3 | 2.625, 2, ...: the k-th minus (k+1)-th gap is 0.375; the neighbouring
    # index mistakes would give 0.625 or 1.0
    cent[:, 0] = [1.0, 5.0, 2.625, 4.0, 0.5, 3.0, -1.0, 2.0]
    T = np.zeros((s.vocab, s.hidden))
    members = order.reshape(s.n_centroids, s.vsc)
    a, b = members[3, 2], members[5, 6]
    T[a, 0], T[b, 0] = 1.25, 1.0                              # best candidate 1.25, runner-up 1.0
    T[members[2, 0], 0] = 9.0                                 # in an unselected cluster: ignored
    W = O.DecodedWeights(None, None, None, T, cent, order, None, "f32")
    y = np.array([1.0, 0.0, 0.0, 0.0])
    head = O.centroid_head(s, W, y)
    assert sorted(head.selected.tolist()) == [1, 3, 5] and head.selected[0] == 1
    assert head.kth_gap == 0.375
    assert head.token == a and head.logit_gap == 0.25
    T[b, 0] = 1.25                                            # an exact tie: gap 0, lowest id
    head = O.centroid_head(s, W, y)
    assert head.logit_gap == 0.0 and head.token == min(a, b)


def test_vocab_divisible_and_ordering_permutation():
    for cfg in C.CONFIGS:
        s = cfg.shape
        if s.use_ordered_embeddings:
            assert s.vocab % s.n_centroids == 0
    g = _golden("published_shapes.json")["centroid_head"]
    assert g["vocab"] % g["n_centroids"] == 0
    assert g["vocab"] // g["n_centroids"] * g["top_k"] == 4096


# ------------------------------------------------------------------ shapes pinned by printed sizes

def test_param_count_and_checkpoint_size_match_pages():
    g = _golden("published_shapes.json")
    e2b, e4b = O.Shape.of(C.E2B), O.Shape.of(C.E4B)
    assert e2b.hidden == g["e2b"]["hidden"] and e2b.backbone == g["e2b"]["backbone"]
    assert e4b.backbone == g["e4b"]["backbone"]
    # "~78 M" read as within 1 % of 78e6; "~158 MB" as within 0.5 % of 158e6
    near = lambda v, ref, tol: abs(v / ref - 1.0) < tol
    assert near(O.param_count(e2b), 1e6 * g["e2b"]["params_approx_millions"], 0.01)
    assert near(O.param_count(e4b), 1e6 * g["e4b"]["params_approx_millions"], 0.01)
    assert near(O.checkpoint_bytes(e4b), 1e6 * g["e4b"]["checkpoint_mb_bf16_approx"], 0.005)
    assert O.param_count(e2b) == 77_731_332
    # a half-width FFN, or separate K/V projections, would break the printed sizes
    half_ffn = O.Shape.of(C.E2B); half_ffn.ffn = 1024
    assert not near(O.param_count(half_ffn), 78e6, 0.01)
    kv_proj = 2 * sum(O.Shape.of(C.E4B).head_dim(t) * 256 for t in C.E4B.layer_types) * 2
    assert not near(O.checkpoint_bytes(e4b) + kv_proj, 158e6, 0.005)
    assert C.A4B_DENSE.backbone == g["a4b_backbone"]["backbone"]
    assert C.A4B_DENSE.hidden == g["a4b_backbone"]["hidden"]
    assert float(O.MASK_VALUE) == np.float32(g["mask_value"]["value"])


def test_accept_rate_printed_value():
    g = _golden("accept_rate.json")
    assert round(100 * O.accept_rate(g["n_accept"], g["n_drafted"]), 1) == g["accept_rate_percent_1dp"]


# ------------------------------------------------------------------ verify

def _rows_with_argmax(targets, V, rng):
    rows = rng.standard_normal((len(targets), V)).astype(np.float32)
    for i, t in enumerate(targets):
        rows[i, t] = rows[i].max() + 1.0
    return rows


def test_verify_worked_example():
    g = _golden("verify_worked_example.json")
    rng = np.random.default_rng(10)
    for case in g["cases"]:
        logits = _rows_with_argmax(case["target_argmax"], g["vocab_size"], rng)[None]
        acc, out = O.verify_greedy(logits, np.array([case["drafts"]]), logits_dtype="f32")
        assert acc[0] == case["accept_len"], case["name"]
        assert out[0].tolist() == case["out_tokens"], case["name"]


def test_verify_ties_take_lowest_id():
    logits = np.zeros((1, 2, 6), dtype=np.float32)
    logits[0, 0, [2, 4]] = 5.0
    logits[0, 1, [1, 3]] = 2.0
    acc, out = O.verify_greedy(logits, np.array([[2]]), logits_dtype="f32")
    assert acc[0] == 1 and out[0].tolist() == [2, 1]
    acc, out = O.verify_greedy(logits, np.array([[4]]), logits_dtype="f32")
    assert acc[0] == 0 and out[0].tolist() == [2, -1]


def test_verify_bf16_input_decoded():
    bits = G.bf16_bits(np.array([[[0.5, 2.0, 1.0], [3.0, 0.0, 0.0]]], dtype=np.float32))
    acc, out = O.verify_greedy(bits, np.array([[1]]))
    assert acc[0] == 1 and out[0].tolist() == [1, 0]


def test_verify_expected_accept_length_closed_form():
    # agreement ~ Bernoulli(p) per position, independent: P(accept >= i) = p^i, so
    # E[accept] = sum_{i=1..n} p^i and E[accept^2] = sum_i (2i-1) p^i
    p, n, V, B = 0.6, 8, 64, 4000
    rng = np.random.default_rng(11)
    drafts = rng.integers(0, V, size=(B, n))
    agree, alt_raw = G.round_tables(B, n, V, p, seed=77, r=0)
    tgt = G.planted_targets(drafts, agree, alt_raw, V)
    logits = rng.standard_normal((B, n + 1, V)).astype(np.float32)
    logits[np.arange(B)[:, None], np.arange(n + 1)[None, :], tgt] = 16.0
    acc, out = O.verify_greedy(logits, drafts, logits_dtype="f32")
    mean = sum(p ** i for i in range(1, n + 1))
    var = sum((2 * i - 1) * p ** i for i in range(1, n + 1)) - mean ** 2
    assert abs(acc.mean() - mean) < 3 * math.sqrt(var / B)
    assert abs(mean - 1.4748) < 1e-4
    # the token after the accepted prefix is the planted target of that row
    np.testing.assert_array_equal(out[np.arange(B), acc], tgt[np.arange(B), acc])


# ------------------------------------------------------------------ whole step: reduction cases

def _tiny_model(seed=0, dtype="f32", layer_types=("S", "F"), zero_blocks=False):
    cfg = C.TINY_F32 if dtype == "f32" else C.E2B
    from dataclasses import replace
    shape = replace(C.TINY_F32, dtype=dtype, layer_types=layer_types, window=8)
    w = G.make_weights(shape, seed)
    if zero_blocks:
        for L in w.layers:
            L["o"] = np.zeros_like(L["o"]); L["down"] = np.zeros_like(L["down"])
    wl = C.Workload(batch=2, ctx=40, ctx_lo=10, n_draft=3)
    inp = G.make_step_inputs(shape, wl, seed)
    return shape, w, inp


def test_zero_blocks_reduce_to_scaled_preprojection():
    # with W_o = W_down = 0 every block only multiplies the residual by layer_scalar, and
    # the final norm removes the scale (up to eps): y = norm(pre_projection([h; e]))
    shape, w, inp = _tiny_model(zero_blocks=True)
    s = O.Shape.of(shape); W = O.decode_weights(w)
    b = 0
    h = O.decode(inp.hidden[b], s.dtype)
    r = O.drafter_step(s, W, h, int(inp.last_token[b]), {"S": inp.k_swa[b], "F": inp.k_full[b]},
                       {}, int(inp.ctx_len[b]), int(inp.pos[b]))
    u = np.concatenate([h, O.decode(w.target_embed[int(inp.last_token[b])], s.dtype)])
    x0 = W.pre_proj @ u
    lam = np.prod([L["layer_scalar"] for L in W.layers])
    np.testing.assert_allclose(r.x_layers[-1], lam * x0, rtol=1e-12)
    np.testing.assert_allclose(r.y, O.rms_norm(lam * x0, W.out_norm, s.rms_eps), rtol=1e-12)
    np.testing.assert_allclose(r.y, O.rms_norm(x0, W.out_norm, 0.0), rtol=1e-3)


def test_concat_order_reading():
    # pre_projection = [I | 0] selects the hidden state, [0 | I] the embedding row
    shape, w, inp = _tiny_model(zero_blocks=True)
    s = O.Shape.of(shape)
    H, bb = s.hidden, s.backbone
    for sel, which in ((0, "h"), (bb, "e")):
        w.pre_proj = np.zeros((H, 2 * bb), np.float32); w.pre_proj[np.arange(H), sel + np.arange(H)] = 1
        W = O.decode_weights(w)
        h = O.decode(inp.hidden[0], s.dtype)
        tok = int(inp.last_token[0])
        r = O.drafter_step(s, W, h, tok, {"S": inp.k_swa[0], "F": inp.k_full[0]}, {}, int(inp.ctx_len[0]), 5)
        lam = np.prod([L["layer_scalar"] for L in W.layers])
        src = h if which == "h" else O.decode(w.target_embed[tok], s.dtype)
        np.testing.assert_allclose(r.x_layers[-1], lam * src[:H], rtol=1e-12)


def test_last_layer_scalar_cancels_in_final_norm():
    shape, w, inp = _tiny_model()
    s = O.Shape.of(shape)
    def y_of(w_):
        W = O.decode_weights(w_)
        return O.drafter_step(s, W, O.decode(inp.hidden[1], s.dtype), int(inp.last_token[1]),
                              {"S": inp.k_swa[1], "F": inp.k_full[1]}, {}, int(inp.ctx_len[1]), 7).y
    y0 = y_of(w)
    w.layers[-1]["layer_scalar"] *= 2.0
    np.testing.assert_allclose(y_of(w), y0, rtol=1e-5, atol=1e-6)
    w.layers[-1]["layer_scalar"] /= 2.0
    w.layers[0]["layer_scalar"] *= 2.0
    assert np.max(np.abs(y_of(w) - y0)) > 1e-3


def test_draft_block_feeds_token_and_hidden_forward():
    shape, w, inp = _tiny_model(dtype="bf16")
    s = O.Shape.of(shape); W = O.decode_weights(w)
    blk = O.draft_block(s, W, inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos, 3,
                        keep_steps=True)
    for b in range(2):
        h = O.decode(inp.hidden[b], "bf16"); tok = int(inp.last_token[b])
        for i in range(3):
            r = O.drafter_step(s, W, h, tok, {"S": inp.k_swa[b], "F": inp.k_full[b]}, {},
                               int(inp.ctx_len[b]), int(inp.pos[b]))
            assert r.token == blk.tokens[b, i]
            np.testing.assert_array_equal(r.hidden_out, blk.hidden_out[b, i])
            h = r.hidden_out; tok = r.token


def test_step_is_continuous_in_its_inputs():
    # no intermediate rounding: a tiny input change moves every output by a comparably tiny
    # amount (a rounding step inside would turn it into whole-ulp jumps)
    shape, w, inp = _tiny_model(dtype="bf16")
    s = O.Shape.of(shape); W = O.decode_weights(w)
    h = O.decode(inp.hidden[0], "bf16")
    kw = dict(tok=int(inp.last_token[0]), k_by_type={"S": inp.k_swa[0], "F": inp.k_full[0]}, v_by_type={},
              ctx_len=int(inp.ctx_len[0]), pos=int(inp.pos[0]))
    r0 = O.drafter_step(s, W, h, **kw)
    dh = np.zeros_like(h); dh[5] = 1e-9
    r1 = O.drafter_step(s, W, h + dh, **kw)
    assert 0 < np.max(np.abs(r1.hidden_out - r0.hidden_out)) < 1e-7
    assert np.max(np.abs(r1.head.logits - r0.head.logits)) < 1e-7


def test_ragged_padding_is_never_read():
    # K padding is NaN: a NaN anywhere in the outputs would mean the padding was attended
    shape, w, inp = _tiny_model(dtype="bf16")
    s = O.Shape.of(shape); W = O.decode_weights(w)
    assert np.any(np.isnan(O.decode(inp.k_full, "bf16")))
    blk = O.draft_block(s, W, inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos, 2)
    assert np.all(np.isfinite(blk.hidden_out))


def _step_y(shape, w, inp, b=0):
    s = O.Shape.of(shape); W = O.decode_weights(w)
    return O.drafter_step(s, W, O.decode(inp.hidden[b], s.dtype), int(inp.last_token[b]),
                          {"S": inp.k_swa[b], "F": inp.k_full[b]}, {}, int(inp.ctx_len[b]), 11)


def test_norms_make_projection_scale_irrelevant():
    # post-attention, post-FFN and q norms remove any positive scale (4: exact in fp32) of W_o, W_down, W_q and
    # W_up (W_up enters the gated product linearly); W_gate enters through the GELU and is
    # not scale-free. A dropped norm or swapped gate/up would break one of these.
    from dataclasses import replace
    shape, w, inp = _tiny_model(dtype="f32")
    shape = replace(shape, rms_eps=0.0)        # exact scale invariance without eps
    ref = _step_y(shape, w, inp)
    for name, changes in (("o", False), ("down", False), ("q", False), ("up", False), ("gate", True)):
        w2 = G.make_weights(shape, 0)
        w2.layers[0][name] = (w2.layers[0][name] * 4.0).astype(np.float32)
        r = _step_y(shape, w2, inp)
        diff = np.max(np.abs(r.y - ref.y))
        assert (diff > 1e-3) if changes else (diff < 1e-9), (name, diff)


def test_layer_types_read_their_own_k_and_window():
    shape, w, inp = _tiny_model(dtype="f32")
    b = int(np.argmax(inp.ctx_len))
    L = int(inp.ctx_len[b]); W_ = shape.window
    assert L > W_
    ref = _step_y(shape, w, inp, b)
    k_swa = inp.k_swa.copy(); k_swa[b, :L - W_] += 5.0      # outside the sliding window
    r = _step_y(shape, w, G.StepInputs(inp.hidden, inp.last_token, inp.ctx_len, inp.pos, k_swa, inp.k_full), b)
    np.testing.assert_array_equal(r.y, ref.y)
    k_full = inp.k_full.copy(); k_full[b, 0] += 5.0           # the full layer sees key 0
    r = _step_y(shape, w, G.StepInputs(inp.hidden, inp.last_token, inp.ctx_len, inp.pos, inp.k_swa, k_full), b)
    assert np.max(np.abs(r.y - ref.y)) > 1e-4
    k_swa = inp.k_swa.copy(); k_swa[b, L - 1] += 5.0          # the sliding layer sees the newest key
    r = _step_y(shape, w, G.StepInputs(inp.hidden, inp.last_token, inp.ctx_len, inp.pos, k_swa, inp.k_full), b)
    assert np.max(np.abs(r.y - ref.y)) > 1e-4


def _closed_form_uniform_step(shape, w, inp, b):
    """The step written out by hand for W_q = 0, W_o = I, W_down = 0: every query is zero, so
    each block's attention is the plain mean of the keys in its range (V = K), the MLP adds
    nothing, and the residual stream is a chain of sandwich-norm updates."""
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    eps = shape.rms_eps
    L = int(inp.ctx_len[b]); Wn = shape.window
    h = f64(inp.hidden[b]); e = f64(w.target_embed[int(inp.last_token[b])])
    x = f64(w.pre_proj) @ np.concatenate([h, e])
    for li, t in enumerate(shape.layer_types):
        lay = w.layers[li]
        keys = f64(inp.k_full[b] if t == "F" else inp.k_swa[b])[:, 0, :]
        lo = 0 if t == "F" else max(0, L - Wn)
        m = keys[lo:L].mean(axis=0)                      # every head reads the one KV head
        a = np.tile(m, shape.n_head)                     # o, flattened over heads; W_o = I
        x = float(lay["layer_scalar"]) * (x + f64(lay["post_attn_norm"]) * a / math.sqrt(np.mean(a * a) + eps))
    y = f64(w.out_norm) * x / math.sqrt(np.mean(x * x) + eps)
    return y, f64(w.post_proj) @ y


@pytest.mark.parametrize("layer_types", [("S", "F"), ("F", "S", "S"), ("S",)])
def test_zero_query_step_equals_its_closed_form(layer_types):
    # whole-step composition pin: the concatenation [h ; e], the key range of each block type
    # (the flipped sliding window, the full context), V = K, the norm placed after W_o and
    # before the residual add, the layer scalar applied to the updated residual stream, the
    # output norm and post_projection, against the formula written out above (planting any
    # one of: a window one key wider, a dropped post-attention norm, the scalar taken before
    # the add, [e ; h] for [h ; e], or a dropped output-norm gain in the oracle fails it)
    shape, w, inp = _tiny_model(dtype="f32", layer_types=layer_types)
    H = shape.hidden
    assert shape.n_head * shape.head_dim_swa == H and shape.n_head * shape.head_dim_full == H
    for L in w.layers:
        L["q"] = np.zeros_like(L["q"])
        L["o"] = np.eye(H, dtype=np.float32)
        L["down"] = np.zeros_like(L["down"])
        L["layer_scalar"] = 0.75
    s = O.Shape.of(shape); W = O.decode_weights(w)
    for b in range(2):
        assert int(inp.ctx_len[b]) > shape.window      # the window cuts the sliding range
        kf = {"S": inp.k_swa[b] if inp.k_swa is not None else None,
              "F": inp.k_full[b] if inp.k_full is not None else None}
        r = O.drafter_step(s, W, np.asarray(inp.hidden[b], np.float64), int(inp.last_token[b]), kf, {},
                           int(inp.ctx_len[b]), int(inp.pos[b]))
        y, h_out = _closed_form_uniform_step(shape, w, inp, b)
        np.testing.assert_allclose(r.y, y, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r.hidden_out, h_out, rtol=1e-11, atol=1e-11)
    # the inputs make the window matter: one key more in the sliding range moves the result
    if "S" in layer_types:
        from dataclasses import replace
        wider = replace(shape, window=shape.window + 1)
        y1, _ = _closed_form_uniform_step(wider, w, inp, 0)
        assert np.max(np.abs(y1 - _closed_form_uniform_step(shape, w, inp, 0)[0])) > 1e-6


def _rotate_complex(v, pos, theta):
    # the rotary reading as complex multiplication: element i and element i + d/2 form
    # z_i = v_i + j v_{i+d/2}, turned by the angle pos * theta^(-2i/d)
    half = v.shape[-1] // 2
    z = (v[:half] + 1j * v[half:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(half) / v.shape[-1]))
    return np.concatenate([z.real, z.imag])


@pytest.mark.parametrize("t,pos", [("F", 0), ("S", 0), ("F", 4099), ("S", 37)])
def test_one_planted_key_step_equals_its_closed_form(t, pos):
    # whole-step pin of the query path: the query of head h is q_norm of its slice of W_q a
    # (a = attn_norm(x)), turned by the rotary angles of the block type's theta at `pos`
    # (at position 0 the identity); every key in range is zero except one, set along head
    # 0's query, so head h's attention output is p_h k* with p_h = e^s / (e^s + n - 1),
    # s = scale * (q_h . k*) and n the keys in range. Keys outside the range are large
    # noise, so a wrong range, scale, q_norm, theta or softmax shows.
    shape, w, inp = _tiny_model(dtype="f32", layer_types=(t,))
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    H, nh, d, eps = shape.hidden, shape.n_head, shape.head_dim(t), shape.rms_eps
    rng = np.random.default_rng(7)
    lay = w.layers[0]
    lay["o"] = np.eye(H, dtype=np.float32)
    lay["down"] = np.zeros_like(lay["down"])
    s = O.Shape.of(shape); W = O.decode_weights(w)
    b = 0
    L = int(inp.ctx_len[b])
    assert L > shape.window
    lo = 0 if t == "F" else L - shape.window
    n = L - lo
    # closed form up to the query
    h = f64(inp.hidden[b]); e = f64(w.target_embed[int(inp.last_token[b])])
    x0 = f64(w.pre_proj) @ np.concatenate([h, e])
    a = f64(lay["attn_norm"]) * x0 / math.sqrt(np.mean(x0 * x0) + eps)
    qraw = (f64(lay["q"]) @ a).reshape(nh, d)
    gq = f64(lay["q_norm"])
    qh = np.stack([gq * qraw[k] / math.sqrt(np.mean(qraw[k] ** 2) + eps) for k in range(nh)])
    theta = shape.rope_theta_full if t == "F" else shape.rope_theta_swa
    qh = np.stack([_rotate_complex(qh[k], pos, theta) for k in range(nh)])
    scale = 1.0 / math.sqrt(d)
    # keys: zero in range except j*, noise outside the range, NaN padding beyond L
    beta = 3.0 / (scale * np.linalg.norm(qh[0]))
    kstar = (beta * qh[0] / np.linalg.norm(qh[0])).astype(np.float32)
    Lmax = (inp.k_full if t == "F" else inp.k_swa).shape[1]
    K = (50.0 * rng.standard_normal((Lmax, 1, d))).astype(np.float32)
    K[lo:L] = 0.0
    jstar = lo + n // 2
    K[jstar, 0] = kstar
    K[L:] = np.nan
    ks = f64(kstar)
    o = np.concatenate([(lambda sc: math.exp(sc) / (math.exp(sc) + n - 1))(scale * float(qh[k] @ ks)) * ks
                        for k in range(nh)])
    x1 = float(lay["layer_scalar"]) * (x0 + f64(lay["post_attn_norm"]) * o / math.sqrt(np.mean(o * o) + eps))
    y = f64(w.out_norm) * x1 / math.sqrt(np.mean(x1 * x1) + eps)
    r = O.drafter_step(s, W, h, int(inp.last_token[b]), {t: K}, {}, L, pos)
    np.testing.assert_allclose(r.o[0].reshape(-1), o, rtol=1e-6, atol=1e-9)   # kstar is fp32-rounded
    np.testing.assert_allclose(r.y, y, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(r.hidden_out, f64(w.post_proj) @ y, rtol=1e-6, atol=1e-8)


def test_mlp_only_step_equals_its_closed_form():
    # whole-step pin of the MLP path: with W_o = 0 the attention update adds norm(0) = 0, so
    # one block is x1 = lambda (x0 + g_pf * n(W_down m)), m = gelu_tanh(W_gate f) * (W_up f),
    # f = g_ffn * n(x0), n(v) = v / sqrt(ms(v) + eps); GELU from torch, not from the oracle
    shape, w, inp = _tiny_model(dtype="f32", layer_types=("F",))
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    eps = shape.rms_eps
    lay = w.layers[0]
    lay["o"] = np.zeros_like(lay["o"])
    n = lambda v: v / math.sqrt(np.mean(v * v) + eps)
    gelu = lambda v: torch.nn.functional.gelu(torch.from_numpy(v), approximate="tanh").numpy()
    s = O.Shape.of(shape); W = O.decode_weights(w)
    for b in range(2):
        h = f64(inp.hidden[b]); e = f64(w.target_embed[int(inp.last_token[b])])
        x0 = f64(w.pre_proj) @ np.concatenate([h, e])
        f = f64(lay["ffn_norm"]) * n(x0)
        m = gelu(f64(lay["gate"]) @ f) * (f64(lay["up"]) @ f)
        x1 = float(lay["layer_scalar"]) * (x0 + f64(lay["post_ffn_norm"]) * n(f64(lay["down"]) @ m))
        y = f64(w.out_norm) * n(x1)
        r = O.drafter_step(s, W, h, int(inp.last_token[b]), {"F": inp.k_full[b]}, {}, int(inp.ctx_len[b]),
                           int(inp.pos[b]))
        np.testing.assert_allclose(r.x_layers[0], x1, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r.y, y, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------------------
# Sampled verification (speculative sampling with a point-mass proposal on each draft)
# ---------------------------------------------------------------------------------------

def _bf16_rows(rng, shape, scale=1.0):
    return G.bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


def test_verify_sample_at_zero_temperature_is_greedy():
    rng = np.random.default_rng(11)
    B, n, V = 6, 4, 64
    logits = _bf16_rows(rng, (B, n + 1, V))
    drafts = rng.integers(0, V, size=(B, n))
    for b in range(0, B, 2):  # some sequences agree with the target for a while
        drafts[b, :3] = [O.argmax_lowest(O.decode_bf16(logits[b, i]).astype(np.float32)) for i in range(3)]
    u = rng.random((B, n + 1))
    acc, out, _ = O.verify_sample(logits, drafts, 0.0, u[:, :n], u)
    racc, rout = O.verify_greedy(logits, drafts)
    np.testing.assert_array_equal(acc, racc)
    np.testing.assert_array_equal(out, rout)


def test_verify_sample_tends_to_greedy_as_the_temperature_falls():
    rng = np.random.default_rng(12)
    B, n, V = 8, 3, 32
    vals = np.stack([rng.permutation(V) for _ in range(B * (n + 1))]).reshape(B, n + 1, V).astype(np.float32) * 0.25
    logits = G.bf16_bits(vals)  # distinct values 0.25 apart: a unique maximum per row
    drafts = rng.integers(0, V, size=(B, n))
    drafts[::2, 0] = np.argmax(vals[::2, 0], axis=-1)
    u = rng.uniform(0.01, 0.99, size=(B, n + 1))
    acc, out, _ = O.verify_sample(logits, drafts, 1e-3, u[:, :n], u)
    racc, rout = O.verify_greedy(logits, drafts)
    np.testing.assert_array_equal(acc, racc)
    np.testing.assert_array_equal(out, rout)


def test_verify_sample_emits_the_target_distribution():
    # P(first token = v) over (u_accept, u_sample) must equal softmax(logits / T)[v]: the
    # draft is kept with probability p(d), otherwise v != d comes from p without d
    # renormalised. Integrated on a midpoint grid of both uniforms (error <= 1 / grid).
    rng = np.random.default_rng(13)
    V, T, grid = 6, 0.8, 400
    logits = _bf16_rows(rng, (1, 2, V))
    p = torch.softmax(torch.tensor(O.decode_bf16(logits[0, 0]).astype(np.float64)) / T, dim=0).numpy()
    for d in (int(np.argmax(p)), int(np.argmin(p))):
        g = (np.arange(grid) + 0.5) / grid
        ua, us = np.meshgrid(g, g, indexing="ij")
        M = ua.size
        lg = np.broadcast_to(logits, (M, 2, V))
        acc, out, _ = O.verify_sample(lg, np.full((M, 1), d), T, ua.reshape(M, 1), np.repeat(us.reshape(M, 1), 2, 1))
        freq = np.bincount(out[:, 0], minlength=V) / M
        np.testing.assert_allclose(freq, p, atol=2.0 / grid)
        assert abs(np.mean(acc == 1) - p[d]) <= 1.0 / grid  # acceptance probability p(d)


def test_verify_sample_bonus_token_follows_the_last_row():
    rng = np.random.default_rng(14)
    V, T, grid = 8, 1.3, 2000
    logits = _bf16_rows(rng, (1, 3, V))
    vals = O.decode_bf16(logits).astype(np.float32)
    drafts = np.array([[0, 1]])
    for i in range(2):  # the drafts carry (almost) all the mass of their rows
        vals[0, i, :] = -40.0
        vals[0, i, drafts[0, i]] = 40.0
    logits = G.bf16_bits(vals)
    p_last = torch.softmax(torch.tensor(vals[0, 2].astype(np.float64)) / T, dim=0).numpy()
    us = (np.arange(grid) + 0.5) / grid
    M = grid
    lg = np.broadcast_to(logits, (M, 3, V))
    u_s = np.zeros((M, 3))
    u_s[:, 2] = us
    acc, out, _ = O.verify_sample(lg, np.broadcast_to(drafts, (M, 2)), T, np.full((M, 2), 0.5), u_s)
    assert np.all(acc == 2)
    np.testing.assert_allclose(np.bincount(out[:, 2], minlength=V) / M, p_last, atol=1.0 / grid)


def test_verify_sample_margins_locate_the_decision_boundaries():
    # a uniform placed exactly on p(d) sits on the accept boundary: margin 0
    rng = np.random.default_rng(15)
    V, T = 16, 1.0
    logits = _bf16_rows(rng, (1, 2, V))
    p = np.exp(O.decode_bf16(logits[0, 0]).astype(np.float64) / T)
    p /= p.sum()
    d = 5
    _, _, m = O.verify_sample(logits, np.array([[d]]), T, np.array([[p[d]]]), np.array([[0.5, 0.5]]))
    assert m[0] <= 1e-12
