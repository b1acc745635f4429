"""mtp_centroid_head_noalloc, the centroid head for callers that cannot allocate device
memory (code running where cudaMalloc is unavailable, e.g. inside graph capture or under a
runtime that owns all device memory): it must give the same tokens, selected centroids and
logits as mtp_centroid_head on the same tensors, call after call, although its scratch
lives in one static device array shared by all calls.

Collected after the main GPU suite on purpose: those tests have run by the time it runs.
"""
import numpy as np
import pytest
import torch

from _util import TOL, config_data, to_torch, weights_to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("index", [1, 0])
def test_noalloc_head_matches_handle_head_on_two_calls(index):
    from mtp_speculative_decoding_gemma4_gb300 import Drafter, binding
    shape, wl, w, inp = config_data(index)
    wd, tgt = weights_to_device(w)
    B, H, V, k = 4, shape.hidden, shape.vocab, shape.top_k
    dr = Drafter(shape, wd, tgt, max_batch=B, max_ctx=wl.ctx)
    dtype = binding.MTP_DTYPE_BF16 if shape.dtype == "bf16" else binding.MTP_DTYPE_F32
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(17)
    for call in range(2):
        y = to_torch(rng.standard_normal((B, H)).astype(np.float32), "f32")
        tok, logits, cents = dr.centroid_head(y, want_logits=True, want_centroids=True, stream=stream)
        tok2 = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        cents2 = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        logits2 = torch.full((B, V), 123.0, dtype=torch.float32, device="cuda")
        binding.mtp_centroid_head_noalloc(y.data_ptr(), wd["centroids"].data_ptr(), wd["token_ordering"].data_ptr(),
                                          wd["token_embd"].data_ptr(), dtype, B, H, shape.n_centroids, k, V,
                                          logits2.data_ptr(), tok2.data_ptr(), cents2.data_ptr(), stream)
        torch.cuda.synchronize()
        assert torch.equal(tok, tok2), (call, tok, tok2)
        assert torch.equal(cents, cents2), call
        assert float((logits - logits2).abs().max()) <= TOL[shape.dtype], call
        assert torch.equal(logits == -1e30, logits2 == -1e30), call
    dr.close()


def test_noalloc_head_rejects_requests_beyond_its_scratch():
    from mtp_speculative_decoding_gemma4_gb300 import MtpError, binding
    fake = 256   # never dereferenced: the size check fails before any device work
    with pytest.raises(MtpError) as e:
        binding.mtp_centroid_head_noalloc(fake, fake, fake, fake, binding.MTP_DTYPE_BF16, 64, 256, 8192, 32, 262144,
                                          0, fake, 0)
    assert e.value.code == binding.MTP_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
