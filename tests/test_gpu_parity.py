"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same seeded
inputs: every benchmark configuration at full size, both implementations of the draft
block (one launch per phase, and the persistent kernel), the head entry point, greedy
verification and the edge cases."""
import numpy as np
import pytest
import torch

import oracle as O
from mtp_synth import configs as C
from mtp_synth import gen as G

from _util import (NEAR_TIE, TOL, compare_block, config_data, decoded, expected_accept, inputs_to_device,
                   oracle_block, to_torch, weights_to_device)

pytestmark = pytest.mark.gpu

PHASES, PERSISTENT, TENSOR, STREAMED, GRID = 1, 2, 5, 6, 7
ONE_SEQ = [STREAMED, GRID]  # the single-sequence paths


def _drafter(index, batch=0, ctx=0, max_batch=0):
    from mtp_speculative_decoding_gemma4_gb300 import Drafter
    shape, wl, w, inp = config_data(index, batch, ctx)
    wd, tgt = weights_to_device(w)
    return (Drafter(shape, wd, tgt, max_batch=max(wl.batch, max_batch), max_ctx=wl.ctx),
            inputs_to_device(inp, shape.dtype))


def _run_block(dr, d, n_draft, path, **kw):
    dr.set_path(path)
    tok, hid = dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"],
                              n_draft, **kw)
    torch.cuda.synchronize()
    assert dr.status() == 0
    return tok.cpu().numpy(), None if hid is None else hid.cpu().numpy()


@pytest.mark.parametrize("index", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("path", [PHASES, PERSISTENT])
def test_draft_block_matches_oracle(index, path):
    shape, wl, w, inp = config_data(index)
    ref = oracle_block(index)
    dr, d = _drafter(index)
    tok, hid = _run_block(dr, d, wl.n_draft, path)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    print(f"config {index} path {path}: {cmp.steps_compared} steps, max hidden err {cmp.max_hidden_err:.3g}, "
          f"near-tie divergences {cmp.tie_divergences}")
    assert len(cmp.tie_divergences) <= max(1, cmp.steps_compared // 50)
    dr.close()


@pytest.mark.parametrize("index", [2, 3, 4])
def test_tensor_core_path_matches_oracle(index):
    # every projection (and the dense head of config 3) as a tcgen05 GEMM; config 2 (B=8)
    # exercises the padding of the staged terms to 32 sequences
    shape, wl, w, inp = config_data(index)
    ref = oracle_block(index)
    dr, d = _drafter(index)
    tok, hid = _run_block(dr, d, wl.n_draft, TENSOR)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    print(f"config {index} tensor-core path: {cmp.steps_compared} steps, max hidden err {cmp.max_hidden_err:.3g}, "
          f"near-tie divergences {cmp.tie_divergences}")
    assert len(cmp.tie_divergences) <= max(1, cmp.steps_compared // 50)
    # same tokens as the CUDA-core phases
    a, _ = _run_block(dr, d, wl.n_draft, PHASES)
    assert np.mean(a == tok) >= 0.98
    dr.close()


@pytest.mark.parametrize("path", ONE_SEQ)
def test_one_sequence_path_matches_oracle_e2b_b1(path):
    shape, wl, w, inp = config_data(1)
    ref = oracle_block(1)
    dr, d = _drafter(1)
    tok, hid = _run_block(dr, d, wl.n_draft, path)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    print(f"path {path} config 1: max hidden err {cmp.max_hidden_err:.3g}, near-ties {cmp.tie_divergences}")
    # more steps than the bench block, and repeated calls (mailbox epochs / barrier phases)
    ref8 = oracle_block(1, n_draft=8)
    for _ in range(3):
        tok, hid = _run_block(dr, d, 8, path)
        compare_block(tok, hid, ref8, shape.dtype)
    # without the hidden output
    tok2, _ = _run_block(dr, d, 8, path, want_hidden=False)
    np.testing.assert_array_equal(tok2, tok)
    dr.close()


@pytest.mark.parametrize("path", ONE_SEQ)
@pytest.mark.parametrize("ctx,n_kv", [(1, 1), (5, 1), (8, 1), (9, 2), (63, 2), (64, 1)])
def test_one_sequence_path_short_and_window_edge_contexts(ctx, n_kv, path):
    from dataclasses import replace
    from mtp_speculative_decoding_gemma4_gb300 import Drafter
    shape = replace(C.TINY_F32, dtype="bf16", layer_types=("S", "F", "S"), window=8, n_head=4, n_kv_head=n_kv)
    wl = C.Workload(batch=1, ctx=64, n_draft=4)
    w = G.make_weights(shape, 31 + ctx)
    inp = G.make_step_inputs(shape, wl, 31 + ctx, ctx_len=np.array([ctx], dtype=np.int32))
    ref = O.draft_block(O.Shape.of(shape), O.decode_weights(w), inp.hidden, inp.last_token, inp.k_swa,
                        inp.k_full, inp.ctx_len, inp.pos, 4)
    wd, tgt = weights_to_device(w)
    dr = Drafter(shape, wd, tgt, max_batch=1, max_ctx=64)
    d = inputs_to_device(inp, "bf16")
    tok, hid = _run_block(dr, d, 4, path)
    compare_block(tok, hid, ref, "bf16")
    dr.close()


def _one_sequence_case(index, ctx_len, storage_ctx, n_draft, seed_offset=0):
    """B = 1 inputs of configuration `index`'s shape (its seeded weights) at an explicit
    context length, with K stored for storage_ctx keys (NaN beyond ctx_len)."""
    shape, wl, w, _ = config_data(index)
    wl1 = C.Workload(batch=1, ctx=storage_ctx, n_draft=n_draft, seed=wl.seed + seed_offset)
    inp = G.make_step_inputs(shape, wl1, wl1.seed, ctx_len=np.array([ctx_len], dtype=np.int32))
    s, W = decoded(index)
    ref = O.draft_block(s, W, inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos, n_draft)
    return shape, w, inp, ref


@pytest.mark.parametrize("path", [0, STREAMED, GRID])
@pytest.mark.parametrize("index,ctx,storage", [
    (2, 32768, 32768),   # E4B backbone at the longest context of its workload
    (2, 20001, 32768),   # E4B, ragged: not a multiple of the 128-key attention chunk
    (1, 511, 1024),      # E2B, one key short of the sliding window
    (1, 512, 1024),      # E2B, exactly the window
    (1, 513, 1024),      # E2B, one key past the window (the sliding layers drop key 0)
])
def test_one_sequence_path_long_ragged_and_window_contexts(index, ctx, storage, path):
    from mtp_speculative_decoding_gemma4_gb300 import Drafter, MtpError, binding
    shape, w, inp, ref = _one_sequence_case(index, ctx, storage, 4)
    wd, tgt = weights_to_device(w)
    dr = Drafter(shape, wd, tgt, max_batch=1, max_ctx=storage)
    d = inputs_to_device(inp, shape.dtype)
    try:
        tok, hid = _run_block(dr, d, 4, path)
    except MtpError as e:
        # a forced single-sequence path may refuse a shape outside its plan (the streamed
        # cluster kernel takes no E4B backbone); the automatic path must always run
        dr.close()
        assert path != 0 and e.code == binding.MTP_ERR_UNSUPPORTED_SHAPE, e
        pytest.skip(f"path {path} does not take this shape: {e}")
    cmp = compare_block(tok, hid, ref, shape.dtype)
    print(f"config {index} ctx {ctx} path {path}: max hidden err {cmp.max_hidden_err:.3g}, "
          f"near-ties {cmp.tie_divergences}")
    dr.close()


@pytest.mark.parametrize("path", [0, STREAMED, GRID])
def test_one_sequence_top_k_with_every_centroid_logit_tied(path):
    """Zero centroid rows make all 2048 centroid logits equal: the top 32 must be centroids
    0..31 (equal values, lower index first: "Centroid / ordered embeddings LM head" step 2
    with the tie rule of the readings). Every candidate key reaches the bound, so the grid
    kernel's tiled top-k overflows its candidate buffer and takes its general form. Tokens
    are compared exactly (the oracle's k-th gap is 0, so the near-tie allowance would excuse
    anything) and the selection is checked on the oracle side."""
    from dataclasses import replace
    from mtp_speculative_decoding_gemma4_gb300 import Drafter
    shape, wl, w, inp = config_data(1)
    w0 = replace(w, centroids=np.zeros_like(w.centroids))
    s = O.Shape.of(shape)
    ref = O.draft_block(s, O.decode_weights(w0), inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len,
                        inp.pos, wl.n_draft)
    assert (ref.selected == np.arange(shape.top_k)).all()
    wd, tgt = weights_to_device(w0)
    dr = Drafter(shape, wd, tgt, max_batch=1, max_ctx=wl.ctx)
    d = inputs_to_device(inp, shape.dtype)
    tok, hid = _run_block(dr, d, wl.n_draft, path)
    # the selection is exact; only a token whose own top-2 logit gap is a near tie may differ
    # (then the later steps are not compared)
    for i in range(wl.n_draft):
        assert np.max(np.abs(hid[0, i].astype(np.float64) - ref.hidden_out[0, i])) <= TOL["bf16"]
        if tok[0, i] != ref.tokens[0, i]:
            assert ref.logit_gap[0, i] < NEAR_TIE["bf16"], (i, tok[0, i], ref.tokens[0, i])
            break
    dr.close()


@pytest.mark.parametrize("path", ONE_SEQ)
def test_one_sequence_paths_reject_batches(path):
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    dr, d = _drafter(2)
    dr.set_path(path)
    with pytest.raises(MtpError) as e:
        dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], 1)
    assert e.value.code == binding.MTP_ERR_UNSUPPORTED_SHAPE
    dr.close()


def test_paths_agree_bitwise_on_tokens():
    # the two implementations run the same phase code; only the grid differs
    dr, d = _drafter(1)
    a, ha = _run_block(dr, d, 4, PHASES)
    b, hb = _run_block(dr, d, 4, PERSISTENT)
    np.testing.assert_array_equal(a, b)
    assert np.max(np.abs(ha - hb)) <= TOL["bf16"]
    dr.close()


def test_one_sequence_paths_agree_on_tokens():
    dr, d = _drafter(1)
    a, ha = _run_block(dr, d, 8, GRID)
    for path in (STREAMED, PERSISTENT):
        b, hb = _run_block(dr, d, 8, path)
        np.testing.assert_array_equal(a, b)
        assert np.max(np.abs(ha - hb)) <= TOL["bf16"]
    dr.close()


def test_removed_paths_are_rejected():
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    dr, _ = _drafter(0)
    for path in (3, 4, 8, -1):
        with pytest.raises(MtpError) as e:
            dr.set_path(path)
        assert e.value.code == binding.MTP_ERR_INVALID_ARG
    dr.close()


def test_repeated_calls_are_deterministic():
    dr, d = _drafter(1)
    a, ha = _run_block(dr, d, 4, PERSISTENT)
    b, hb = _run_block(dr, d, 4, PERSISTENT)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ha, hb)
    dr.close()


@pytest.mark.parametrize("index", [0, 1])
def test_centroid_head_entry_matches_oracle(index):
    shape, wl, w, inp = config_data(index)
    s, W = decoded(index)
    rng = np.random.default_rng(5)
    B = 3
    y = (rng.standard_normal((B, s.hidden)) * 0.8).astype(np.float32)
    dr, _ = _drafter(index, max_batch=B)
    tok, logits, cents = dr.centroid_head(to_torch(y, "f32"), want_logits=True, want_centroids=True)
    torch.cuda.synchronize()
    tok, logits, cents = tok.cpu().numpy(), logits.cpu().numpy(), cents.cpu().numpy()
    tol, delta = TOL[shape.dtype], NEAR_TIE[shape.dtype]
    for b in range(B):
        ref = O.centroid_head(s, W, y[b].astype(np.float64))
        if not np.array_equal(cents[b], ref.selected):
            assert ref.kth_gap < delta, (cents[b], ref.selected, ref.kth_gap)
            continue
        row = O.materialise_row(s, ref)
        unsel = row == np.float32(-1e30)
        # unselected entries are exactly -1e30, selected ones within tolerance
        assert np.array_equal(logits[b] == np.float32(-1e30), unsel)
        assert np.max(np.abs(logits[b][ref.ids].astype(np.float64) - ref.logits)) <= tol
        if tok[b] != ref.token:
            assert ref.logit_gap < delta
    dr.close()


@pytest.mark.parametrize("index", [0, 1])
def test_centroid_head_min_minus_one_mask_matches_oracle(index):
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    shape, wl, w, inp = config_data(index)
    s, W = decoded(index)
    rng = np.random.default_rng(15)
    B = 3
    y = (rng.standard_normal((B, s.hidden)) * 0.8).astype(np.float32)
    dr, _ = _drafter(index, max_batch=B)
    with pytest.raises(MtpError):
        dr.set_logit_mask(2)
    dr.set_logit_mask(binding.MASK_MIN_MINUS_ONE)
    tok, logits, cents = dr.centroid_head(to_torch(y, "f32"), want_logits=True, want_centroids=True)
    torch.cuda.synchronize()
    tok, logits, cents = tok.cpu().numpy(), logits.cpu().numpy(), cents.cpu().numpy()
    tol, delta = TOL[shape.dtype], NEAR_TIE[shape.dtype]
    for b in range(B):
        ref = O.centroid_head(s, W, y[b].astype(np.float64))
        if not np.array_equal(cents[b], ref.selected):
            assert ref.kth_gap < delta, (cents[b], ref.selected, ref.kth_gap)
            continue
        row = O.materialise_row(s, ref, mask="min_minus_one")
        unsel = np.ones(s.vocab, bool)
        unsel[ref.ids] = False
        cand = logits[b][ref.ids]
        assert np.max(np.abs(cand.astype(np.float64) - ref.logits)) <= tol
        # every other entry: the GPU's own smallest candidate minus one (fp32), within
        # tolerance of the oracle's fill
        fill = np.float32(cand.min()) - np.float32(1.0)
        assert np.all(logits[b][unsel] == fill)
        assert abs(float(fill) - float(row[unsel][0])) <= tol
        if tok[b] != ref.token:
            assert ref.logit_gap < delta
        else:
            assert int(np.argmax(logits[b])) == ref.token
    # back to the -1e30 fill
    dr.set_logit_mask(binding.MASK_NEG_1E30)
    _t, logits0, _c = dr.centroid_head(to_torch(y, "f32"), want_logits=True)
    torch.cuda.synchronize()
    l0 = logits0.cpu().numpy()
    assert np.sum(l0 == np.float32(-1e30)) == B * (s.vocab - s.top_k * s.vsc)
    dr.close()


@pytest.mark.parametrize("index,B", [(0, 5), (1, 64)])
def test_cluster_major_head_entry_matches_oracle(index, B):
    # the head with each selected cluster's rows read once for all sequences that chose it:
    # same selected sets and tokens as the per-sequence traversal, logits equal up to fp32
    # summation order, and every row against the oracle. Sequences 0..7 share one hidden
    # state so that some clusters are listed by many sequences at once.
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    shape, wl, w, inp = config_data(index)
    s, W = decoded(index)
    rng = np.random.default_rng(25)
    y = (rng.standard_normal((B, s.hidden)) * 0.8).astype(np.float32)
    y[1:min(B, 8)] = y[0]
    dr, _ = _drafter(index, max_batch=B)
    with pytest.raises(MtpError):
        dr.set_sparse_head(3)
    out = {}
    for mode in (binding.HEAD_PER_SEQUENCE, binding.HEAD_CLUSTER_MAJOR):
        dr.set_sparse_head(mode)
        t, lg, c = dr.centroid_head(to_torch(y, "f32"), want_logits=True, want_centroids=True)
        torch.cuda.synchronize()
        out[mode] = (t.cpu().numpy(), lg.cpu().numpy(), c.cpu().numpy())
    tp, lp, cp = out[binding.HEAD_PER_SEQUENCE]
    tok, logits, cents = out[binding.HEAD_CLUSTER_MAJOR]
    assert np.array_equal(cp, cents)
    fill = lp == np.float32(-1e30)
    assert np.array_equal(fill, logits == np.float32(-1e30))
    assert np.sum(~fill) == B * s.top_k * s.vsc
    sel = ~fill
    assert np.max(np.abs(lp[sel] - logits[sel])) <= 1e-5 * max(1.0, float(np.max(np.abs(lp[sel]))))
    tol, delta = TOL[shape.dtype], NEAR_TIE[shape.dtype]
    for b in range(B):
        ref = O.centroid_head(s, W, y[b].astype(np.float64))
        if not np.array_equal(cents[b], ref.selected):
            assert ref.kth_gap < delta, (cents[b], ref.selected, ref.kth_gap)
            continue
        assert np.max(np.abs(logits[b][ref.ids].astype(np.float64) - ref.logits)) <= tol
        if tok[b] != ref.token or tp[b] != tok[b]:
            assert ref.logit_gap < delta
    dr.close()


@pytest.mark.parametrize("index,batch,path,mode", [(0, 5, PHASES, 2), (1, 3, TENSOR, 2), (2, 0, TENSOR, 2),
                                                   (4, 0, TENSOR, 2), (4, 0, PHASES, 2), (4, 0, PERSISTENT, 2)])
def test_sparse_head_traversals_in_the_draft_block(index, batch, path, mode):
    # the cluster-major traversal (the automatic rule gathers per sequence), two steps at
    # config 4's 64 sequences; the persistent kernel keeps the per-sequence gather whatever
    # the mode
    shape, wl, w, inp = config_data(index, batch)
    n = 2 if index == 4 else wl.n_draft
    ref = oracle_block(index, n_draft=n, batch=batch)
    dr, d = _drafter(index, batch)
    dr.set_sparse_head(mode)
    tok, hid = _run_block(dr, d, n, path)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    print(f"config {index} B={tok.shape[0]} path {path} head mode {mode}: {cmp.steps_compared} steps, "
          f"max hidden err {cmp.max_hidden_err:.3g}, near-tie divergences {cmp.tie_divergences}")
    assert len(cmp.tie_divergences) <= max(1, cmp.steps_compared // 50)
    dr.close()


def test_a_missing_grid_barrier_arrival_times_out_and_the_handle_recovers():
    # failure detection without a fault: CTA 0 of the persistent kernel skips its first
    # grid-barrier arrival, every bounded wait gives up after ~10 ms of cycles, the status
    # word reads MTP_ERR_TIMEOUT, and the next call on the same handle is correct again
    from mtp_speculative_decoding_gemma4_gb300 import binding
    shape, wl, w, inp = config_data(0, 3)
    ref = oracle_block(0, batch=3)
    dr, d = _drafter(0, 3)
    dr.set_path(PERSISTENT)
    dr.set_debug(skip_arrival_cta=0, spin_limit_cycles=20_000_000)
    dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], wl.n_draft)
    torch.cuda.synchronize()
    assert dr.status() == binding.MTP_ERR_TIMEOUT
    assert dr.status() == binding.MTP_OK  # reading the word cleared it
    dr.set_debug()
    tok, hid = _run_block(dr, d, wl.n_draft, PERSISTENT)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    assert len(cmp.tie_divergences) <= 1
    dr.close()


def test_grid_path_timeout_is_reported_and_the_handle_recovers():
    # failure detection without a fault on the default one-sequence path: CTA 0 of the grid
    # kernel does not publish its slice of the first all-reduce, every bounded wait gives up
    # after ~10 ms of cycles, the status word reads MTP_ERR_TIMEOUT, and the next call on the
    # same handle matches the oracle
    from mtp_speculative_decoding_gemma4_gb300 import binding
    shape, wl, w, inp = config_data(1)
    ref = oracle_block(1)
    dr, d = _drafter(1)
    dr.set_path(GRID)
    dr.set_debug(skip_arrival_cta=0, spin_limit_cycles=20_000_000)
    dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], wl.n_draft)
    torch.cuda.synchronize()
    assert dr.status() == binding.MTP_ERR_TIMEOUT
    assert dr.status() == binding.MTP_OK
    dr.set_debug()
    tok, hid = _run_block(dr, d, wl.n_draft, GRID)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    assert len(cmp.tie_divergences) <= 1
    dr.close()


@pytest.mark.parametrize("index,batch,path", [(1, 0, STREAMED), (1, 3, TENSOR)])
def test_cluster_and_tensor_core_timeouts_are_reported_and_the_handle_recovers(index, batch, path):
    # failure detection without a fault, one test per kernel family: on the streamed cluster
    # path (k_block_c2) CTA 0 sends none of its rows in the launch's first exchange; on the
    # tensor-core path the first projection GEMM's CTA 0 (k_tc_gemm) issues no copy for its
    # last k stage. Either way a bounded wait gives up after ~10 ms of cycles, the status word
    # reads MTP_ERR_TIMEOUT, and the next call on the same handle matches the oracle.
    from mtp_speculative_decoding_gemma4_gb300 import binding
    shape, wl, w, inp = config_data(index, batch)
    ref = oracle_block(index, batch=batch)
    dr, d = _drafter(index, batch)
    dr.set_path(path)
    dr.set_debug(skip_arrival_cta=0, spin_limit_cycles=20_000_000)
    dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], wl.n_draft)
    torch.cuda.synchronize()
    assert dr.status() == binding.MTP_ERR_TIMEOUT
    assert dr.status() == binding.MTP_OK
    dr.set_debug()
    tok, hid = _run_block(dr, d, wl.n_draft, path)
    cmp = compare_block(tok, hid, ref, shape.dtype)
    assert len(cmp.tie_divergences) <= max(1, cmp.steps_compared // 50)
    dr.close()


def test_dense_head_entry_matches_oracle():
    shape, wl, w, inp = config_data(3)
    s, W = decoded(3)
    rng = np.random.default_rng(6)
    B = 4
    y = rng.standard_normal((B, s.hidden)).astype(np.float32)
    dr, _ = _drafter(3, max_batch=B)
    tok, logits, _c = dr.centroid_head(to_torch(y, "f32"), want_logits=True)
    torch.cuda.synchronize()
    tok, logits = tok.cpu().numpy(), logits.cpu().numpy()
    for b in range(B):
        ref = O.dense_head(s, W, y[b].astype(np.float64))
        assert np.max(np.abs(logits[b].astype(np.float64) - ref.logits)) <= TOL["bf16"]
        assert tok[b] == ref.token or ref.logit_gap < NEAR_TIE["bf16"]
    dr.close()


# ------------------------------------------------------------------ edge cases of the block

@pytest.mark.parametrize("ctx_lens", [[1, 2, 5, 63], [8, 9, 16, 17], [64, 64, 3, 40]])
def test_short_and_window_edge_contexts(ctx_lens):
    # tiny shape with a sliding layer of window 8: contexts below, at and just above it
    from dataclasses import replace
    from mtp_speculative_decoding_gemma4_gb300 import Drafter
    shape = replace(C.TINY_F32, dtype="bf16", layer_types=("S", "F"), window=8)
    wl = C.Workload(batch=4, ctx=64, n_draft=3)
    w = G.make_weights(shape, 21)
    inp = G.make_step_inputs(shape, wl, 21, ctx_len=np.array(ctx_lens, dtype=np.int32))
    ref = O.draft_block(O.Shape.of(shape), O.decode_weights(w), inp.hidden, inp.last_token, inp.k_swa,
                        inp.k_full, inp.ctx_len, inp.pos, 3)
    wd, tgt = weights_to_device(w)
    dr = Drafter(shape, wd, tgt, max_batch=4, max_ctx=64)
    d = inputs_to_device(inp, "bf16")
    for path in (PHASES, PERSISTENT):
        tok, hid = _run_block(dr, d, 3, path)
        compare_block(tok, hid, ref, "bf16")
    dr.close()


def test_v_equal_k_pointer_is_bit_identical_to_v_null():
    dr, d = _drafter(1)
    dr.set_path(PERSISTENT)
    a, ha = dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], 2)
    b, hb = dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], 2,
                           v_swa=d["k_swa"], v_full=d["k_full"])
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ha, hb)
    dr.close()


def test_missing_kv_and_bad_batch_are_rejected():
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    dr, d = _drafter(0)
    with pytest.raises(MtpError) as e:
        dr.draft_block(d["hidden"], d["last_token"], None, None, d["ctx_len"], d["pos"], 1)
    assert e.value.code == binding.MTP_ERR_INVALID_ARG
    big = torch.zeros((5, d["hidden"].shape[1]), dtype=d["hidden"].dtype, device="cuda")
    with pytest.raises(MtpError) as e:
        dr.draft_block(big, d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], 1)
    assert e.value.code == binding.MTP_ERR_INVALID_ARG
    dr.close()


def test_bad_ordering_is_rejected():
    from mtp_speculative_decoding_gemma4_gb300 import Drafter, MtpError, binding
    shape, wl, w, inp = config_data(0)
    wd, tgt = weights_to_device(w)
    wd["token_ordering"] = wd["token_ordering"].clone()
    wd["token_ordering"][7] = wd["token_ordering"][8]
    with pytest.raises(MtpError) as e:
        Drafter(shape, wd, tgt, max_batch=1, max_ctx=64)
    assert e.value.code == binding.MTP_ERR_BAD_ORDERING


# ------------------------------------------------------------------ greedy verify

def _verify_case(B, n, V, seed, ties=False):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, n + 1, V)).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, n)).astype(np.int32)
    agree = rng.random((B, n)) < 0.7
    for b in range(B):
        for i in range(n):
            t = drafts[b, i] if agree[b, i] else (drafts[b, i] + 1 + rng.integers(0, V - 1)) % V
            logits[b, i, t] = 9.0
        if ties:
            row = logits[b, 0]
            m = int(np.argmax(row))
            row[(m + 3) % V] = row[m]   # an exact tie with another id
    bits = G.bf16_bits(logits)
    return bits, drafts


@pytest.mark.parametrize("B,n,V,ties", [(64, 8, 262144, False), (3, 0, 64, False), (5, 4, 4096, True),
                                        (7, 1, 8, False), (2, 8, 131072, True), (1, 4, 262144, False),
                                        (1, 9, 4096, True), (1, 5, 262144, True)])
def test_verify_matches_oracle(B, n, V, ties):
    from mtp_speculative_decoding_gemma4_gb300 import verify_greedy
    bits, drafts = _verify_case(B, n, V, seed=B * 1000 + n, ties=ties)
    acc, out = verify_greedy(to_torch(bits, "bf16"), to_torch(drafts, "i32"))
    torch.cuda.synchronize()
    racc, rout = O.verify_greedy(bits, drafts)
    np.testing.assert_array_equal(acc.cpu().numpy(), racc)
    np.testing.assert_array_equal(out.cpu().numpy(), rout)


@pytest.mark.parametrize("B,n", [(1, 4), (1, 12), (6, 6)])
def test_verify_ignores_rows_after_the_first_disagreement(B, n):
    """Rows after each sequence's first disagreement are overwritten with NaN (bf16 0x7fc1);
    they share a read batch with the rows before them, yet the result is the oracle's."""
    from mtp_speculative_decoding_gemma4_gb300 import verify_greedy
    V = 8192
    bits, drafts = _verify_case(B, n, V, seed=77 + B * 13 + n, ties=False)
    racc, rout = O.verify_greedy(bits, drafts)
    poisoned = bits.copy()
    for b in range(B):
        poisoned[b, int(racc[b]) + 1:, :] = 0x7FC1
    acc, out = verify_greedy(to_torch(poisoned, "bf16"), to_torch(drafts, "i32"))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), racc)
    np.testing.assert_array_equal(out.cpu().numpy(), rout)


def _sample_case(B, n, V, seed, plant):
    """Target logits N(0, 1) with a planted value at the draft (probability 0.7) or at another
    id, drafts, and seeded uniforms."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, n + 1, V)).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, n)).astype(np.int32)
    agree = rng.random((B, n)) < 0.7
    for b in range(B):
        for i in range(n):
            t = drafts[b, i] if agree[b, i] else (drafts[b, i] + 1 + rng.integers(0, V - 1)) % V
            logits[b, i, t] = plant
    ua = rng.random((B, n)).astype(np.float32)
    us = rng.random((B, n + 1)).astype(np.float32)
    return G.bf16_bits(logits), drafts, ua, us


@pytest.mark.parametrize("B,n,V,T,plant", [(64, 8, 262144, 1.0, 16.0), (64, 8, 262144, 0.7, 12.0),
                                           (5, 4, 4096, 1.0, 4.0), (3, 0, 64, 0.5, 2.0), (7, 1, 8, 2.0, 1.0),
                                           (4, 3, 131072, 1.5, 20.0)])
def test_verify_sample_matches_oracle(B, n, V, T, plant):
    from mtp_speculative_decoding_gemma4_gb300 import verify_sample
    bits, drafts, ua, us = _sample_case(B, n, V, seed=B * 7 + n * 3 + V % 97, plant=plant)
    acc, out = verify_sample(to_torch(bits, "bf16"), to_torch(drafts, "i32"), T,
                             torch.from_numpy(ua).cuda(), torch.from_numpy(us).cuda())
    torch.cuda.synchronize()
    acc, out = acc.cpu().numpy(), out.cpu().numpy()
    racc, rout, margin = O.verify_sample(bits, drafts, T, ua, us)
    # fp32 decisions may differ from the fp64 oracle only for a uniform within 1e-5 of a
    # decision boundary (relative to the mass compared against)
    bad = [b for b in range(B) if acc[b] != racc[b] or not np.array_equal(out[b], rout[b])]
    assert all(margin[b] < 1e-5 for b in bad), (bad, [margin[b] for b in bad])
    assert len(bad) <= max(1, B // 32)


def test_verify_sample_at_zero_temperature_is_greedy_on_the_device():
    from mtp_speculative_decoding_gemma4_gb300 import verify_greedy, verify_sample
    bits, drafts = _verify_case(16, 4, 4096, seed=77, ties=True)
    t = to_torch(bits, "bf16")
    d = to_torch(drafts, "i32")
    u = torch.rand((16, 5), device="cuda")
    a1, o1 = verify_sample(t, d, 0.0, u[:, :4].contiguous(), u)
    a2, o2 = verify_greedy(t, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a1.cpu().numpy(), a2.cpu().numpy())
    np.testing.assert_array_equal(o1.cpu().numpy(), o2.cpu().numpy())


def test_verify_sample_first_token_follows_the_target_distribution():
    # 16384 independent trials of one row: the emitted first token must be distributed as
    # softmax(row / T) (the draft kept with probability p(d), else a residual sample)
    from mtp_speculative_decoding_gemma4_gb300 import verify_sample
    rng = np.random.default_rng(5)
    B, V, T, d = 16384, 16, 0.9, 3
    row = rng.standard_normal(V).astype(np.float32)
    bits = G.bf16_bits(np.broadcast_to(row, (B, 2, V)).copy())
    p = torch.softmax(torch.tensor(O.decode_bf16(bits[0, 0]).astype(np.float64)) / T, dim=0).numpy()
    drafts = np.full((B, 1), d, dtype=np.int32)
    ua = torch.rand((B, 1), device="cuda")
    us = torch.rand((B, 2), device="cuda")
    acc, out = verify_sample(to_torch(bits, "bf16"), to_torch(drafts, "i32"), T, ua, us)
    torch.cuda.synchronize()
    first = out.cpu().numpy()[:, 0]
    freq = np.bincount(first, minlength=V) / B
    sigma = np.sqrt(p * (1 - p) / B)
    assert np.all(np.abs(freq - p) <= 5 * sigma + 1e-4), (freq, p)
    assert abs(np.mean(acc.cpu().numpy() == 1) - p[d]) <= 5 * np.sqrt(p[d] * (1 - p[d]) / B)


def test_verify_rejects_bad_vocab():
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, verify_greedy
    t = torch.zeros((1, 2, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MtpError):
        verify_greedy(t, torch.zeros((1, 1), dtype=torch.int32, device="cuda"))


# ------------------------------------------------------------------ draft + verify loop

def _planted(base, drafts, agree, alt_raw, V):
    """The round's target logits: the base logits with each row's +16 maximum planted."""
    B, n1 = drafts.shape[0], drafts.shape[1] + 1
    tgt = G.planted_targets(drafts, agree, alt_raw, V)
    planted = base.copy()
    planted[np.arange(B)[:, None], np.arange(n1)[None, :], tgt] = G.bf16_bits(np.float32([G.PLANT_VALUE]))[0]
    return tgt, planted


def _loop(dr, d, shape, wl, rounds, seed):
    """Draft+verify rounds of the library against the planted synthetic target; returns per
    round (input tokens, drafts, accept_len, out_tokens). Round r > 0 starts from the
    pregenerated hidden state of round r - 1 and the token emitted after the accepted prefix."""
    B, n, V = wl.batch, wl.n_draft, shape.vocab
    base = G.base_target_logits(B, n + 1, V, seed)
    hist = []
    logits_dev = to_torch(base, "bf16")
    hidden, tok = d["hidden"], d["last_token"]
    for r in range(rounds):
        agree, alt_raw = G.round_tables(B, n, V, wl.agree_p, seed, r)
        tok_in = tok.cpu().numpy().copy()
        drafts, _ = dr.draft_block(hidden, tok, d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], n,
                                   want_hidden=False)
        dnp = drafts.cpu().numpy()
        tgt = G.planted_targets(dnp, agree, alt_raw, V)
        idx = torch.from_numpy(tgt).cuda()
        bi = torch.arange(B, device="cuda")[:, None]
        ri = torch.arange(n + 1, device="cuda")[None, :]
        saved = logits_dev[bi, ri, idx].clone()
        logits_dev[bi, ri, idx] = G.PLANT_VALUE
        acc, out = verify_greedy_(logits_dev, drafts)
        logits_dev[bi, ri, idx] = saved
        a, o = acc.cpu().numpy(), out.cpu().numpy()
        hidden = to_torch(G.next_round_hidden(B, shape.backbone, seed, r), "bf16")
        tok = out[torch.arange(B, device="cuda"), acc.long()].contiguous()
        hist.append((tok_in, dnp.copy(), a.copy(), o.copy()))
    return hist


def verify_greedy_(logits, drafts):
    from mtp_speculative_decoding_gemma4_gb300 import verify_greedy
    return verify_greedy(logits, drafts)


LOOP_ROUNDS_CHECKED = 10


@pytest.mark.parametrize("path", [0, PERSISTENT])
def test_draft_verify_loop_matches_oracle_round_by_round(path):
    # The loop workload (E2B, B=64, draft block 8) for 10 rounds. Each round the oracle drafts
    # from the same inputs the library used (teacher forcing: the library's carried token),
    # so a near-tie divergence in one round does not desynchronise later rounds. Every
    # drafted token must equal the oracle's unless the oracle's own margin at that step is
    # below the near-tie bound (per sequence, through compare_block); verification of the
    # library's drafts against the same planted target is bit-exact.
    shape, wl, w, inp = config_data(4)
    s, W = decoded(4)
    dr, d = _drafter(4)
    dr.set_path(path)
    B, n, V = wl.batch, wl.n_draft, shape.vocab
    g = _loop(dr, d, shape, wl, rounds=LOOP_ROUNDS_CHECKED, seed=wl.seed)
    base = G.base_target_logits(B, n + 1, V, wl.seed)
    ties, compared = [], 0
    for r, (tok_in, gd, ga, go) in enumerate(g):
        hidden = inp.hidden if r == 0 else G.next_round_hidden(B, shape.backbone, wl.seed, r - 1)
        ref = O.draft_block(s, W, hidden, tok_in, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos, n)
        cmp = compare_block(gd, None, ref, shape.dtype)
        compared += cmp.steps_compared
        ties += [(r,) + t for t in cmp.tie_divergences]
        agree, alt_raw = G.round_tables(B, n, V, wl.agree_p, wl.seed, r)
        _, planted = _planted(base, gd, agree, alt_raw, V)
        oa, oo = O.verify_greedy(planted, gd)
        np.testing.assert_array_equal(ga, oa, err_msg=f"accept lengths of round {r}")
        np.testing.assert_array_equal(go, oo, err_msg=f"emitted tokens of round {r}")
    print(f"path {path}: {LOOP_ROUNDS_CHECKED} rounds x {B} sequences, {compared} draft steps compared, "
          f"near-tie divergences (round, sequence, step, oracle margin): {ties}")
    dr.close()


def test_draft_verify_loop_accept_length_statistics():
    # 1000 rounds of B=64, n=8 against a target agreeing with probability 0.6 per position:
    # E[accept] = sum_{i=1..8} 0.6^i = 1.4748
    shape, wl, w, inp = config_data(4)
    dr, d = _drafter(4)
    dr.set_path(PERSISTENT)
    g = _loop(dr, d, shape, wl, rounds=wl.rounds, seed=wl.seed)
    acc = np.concatenate([a for _, _, a, _ in g]).astype(np.float64)
    mean, sd = expected_accept(wl.agree_p, wl.n_draft)
    print(f"mean accept length {acc.mean():.4f} (expected {mean:.4f}) over {acc.size} sequence-rounds")
    assert abs(acc.mean() - mean) < 3 * sd / np.sqrt(acc.size)
    # every output row holds accept_len drafts then the target token, then -1 padding
    for _, dn, a, o in g[:50]:
        for b in range(wl.batch):
            assert np.array_equal(o[b, :a[b]], dn[b, :a[b]])
            assert o[b, a[b]] >= 0 and np.all(o[b, a[b] + 1:] == -1)
    dr.close()


def test_graph_replay_reads_new_contents_and_recaptures_on_new_arguments():
    # the multi-launch paths replay a captured graph when the arguments repeat: new input
    # contents behind the same pointers must be read, and a change of n_draft recaptured
    shape, wl, w, inp = config_data(4)
    dr, d = _drafter(4)
    t1, _ = _run_block(dr, d, 2, TENSOR)
    t2, _ = _run_block(dr, d, 2, TENSOR)          # replay, same inputs
    np.testing.assert_array_equal(t1, t2)
    t4, _ = _run_block(dr, d, 4, TENSOR)          # new n_draft: captured again
    np.testing.assert_array_equal(t4[:, :2], t1)
    d["last_token"].copy_(torch.roll(d["last_token"], 1))  # new contents, same pointers
    t5, _ = _run_block(dr, d, 4, TENSOR)
    dr.close()
    dr2, _ = _drafter(4)
    t6, _ = _run_block(dr2, d, 4, TENSOR)         # a fresh handle with the same inputs
    np.testing.assert_array_equal(t5, t6)
    assert not np.array_equal(t5, t4)
    dr2.close()


@pytest.mark.parametrize("B,path", [(1, 0), (4, TENSOR), (4, PHASES)])
def test_e4b_with_two_kv_heads_matches_oracle(B, path):
    # the E4B drafter with two shared KV heads (two query heads per KV head) on the automatic
    # one-sequence path and on the batched paths
    from mtp_speculative_decoding_gemma4_gb300 import Drafter
    shape = C.E4B_KV2
    wl = C.Workload(batch=B, ctx=4096, ctx_lo=1024 if B > 1 else None, n_draft=3, seed=2024)
    w = G.make_weights(shape, wl.seed)
    inp = G.make_step_inputs(shape, wl, wl.seed)
    ref = O.draft_block(O.Shape.of(shape), O.decode_weights(w), inp.hidden, inp.last_token, inp.k_swa, inp.k_full,
                        inp.ctx_len, inp.pos, wl.n_draft)
    wd, tgt = weights_to_device(w)
    dr = Drafter(shape, wd, tgt, max_batch=B, max_ctx=wl.ctx)
    d = inputs_to_device(inp, "bf16")
    tok, hid = _run_block(dr, d, wl.n_draft, path)
    cmp = compare_block(tok, hid, ref, "bf16")
    assert len(cmp.tie_divergences) <= 1
    dr.close()
