"""Host-side checks of libmtp.so that need no GPU: the library loads, exports every entry
point include/mtp.h declares, and rejects invalid arguments before touching the device."""
import ctypes
import os
import re

import pytest

from mtp_speculative_decoding_gemma4_gb300 import binding as B
from mtp_speculative_decoding_gemma4_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load_library()


def _declared():
    with open(os.path.join(ROOT, "include", "mtp.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^MTP_API (?:int|void|const char \*)\s*\**(mtp_\w+)\(", text, flags=re.M)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(B.EXPORTS)


def test_header_enum_values_match_binding():
    # every enumerator of include/mtp.h against the binding's constant of the same value
    with open(os.path.join(ROOT, "include", "mtp.h")) as f:
        text = f.read()
    enums = {}
    for body in re.findall(r"enum \w+ \{([^}]*)\}", text):
        for name, val in re.findall(r"(MTP_\w+)\s*=\s*(\d+)", body):
            enums[name] = int(val)
    assert len(enums) >= 15
    for name, val in enums.items():
        py = name if hasattr(B, name) else name[len("MTP_"):]
        assert getattr(B, py) == val, name


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_no_cpu_fallback_symbols(lib):
    # the library is the CUDA implementation only: its exported C symbols are the ABI
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = sorted(set(re.findall(r" T (mtp_\w+)", out)))
    assert exported == sorted(B.EXPORTS)


def test_null_arguments_are_rejected_without_a_device(lib):
    assert lib.mtp_init_weights(None, None, None, None) == B.MTP_ERR_INVALID_ARG
    assert "non-NULL" in B.mtp_last_error()
    assert lib.mtp_draft_block(None, None, None, None, None, None, 1, 1, None, None, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_centroid_head(None, None, 1, None, None, None, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_greedy(None, None, 1, 1, 8, None, None, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_set_path(None, 1) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_set_logit_mask(None, B.MASK_MIN_MINUS_ONE) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_set_sparse_head(None, B.HEAD_CLUSTER_MAJOR) == B.MTP_ERR_INVALID_ARG
    assert "MTP_HEAD_CLUSTER_MAJOR" in B.mtp_last_error()
    assert lib.mtp_set_debug(None, -1, 0) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_get_status(None) == B.MTP_ERR_INVALID_ARG
    lib.mtp_destroy(None)


def _tiny_config(**over):
    c = B.mtp_config()
    vals = dict(backbone=128, hidden=64, n_layers=1, n_head=2, head_dim_swa=32, head_dim_full=32, n_kv_head=1,
                ffn=256, vocab=4096, n_centroids=64, top_k=4, window=16, use_ordered_embeddings=1,
                dtype=B.MTP_DTYPE_F32, max_batch=1, max_ctx=64)
    vals.update(over)
    for k, v in vals.items():
        setattr(c, k, v)
    c.layer_type[0] = B.MTP_LAYER_FULL
    c.rms_eps = 1e-6
    return c


@pytest.mark.parametrize("over,code", [
    (dict(vocab=4000), B.MTP_ERR_BAD_ORDERING),            # vocab % n_centroids != 0
    (dict(n_layers=0), B.MTP_ERR_INVALID_ARG),
    (dict(n_layers=9), B.MTP_ERR_INVALID_ARG),
    (dict(dtype=7), B.MTP_ERR_INVALID_ARG),
    (dict(top_k=65), B.MTP_ERR_UNSUPPORTED_SHAPE),
    (dict(n_head=3), B.MTP_ERR_UNSUPPORTED_SHAPE),         # not a multiple of n_kv_head... 3 % 1 ok; head dim check
    (dict(head_dim_full=48), B.MTP_ERR_UNSUPPORTED_SHAPE),
    (dict(hidden=66), B.MTP_ERR_UNSUPPORTED_SHAPE),
    (dict(max_batch=0), B.MTP_ERR_INVALID_ARG),
])
def test_invalid_configs_are_rejected_before_the_device(lib, over, code):
    if over == dict(n_head=3):
        over = dict(n_head=3, n_kv_head=2)
    c = _tiny_config(**over)
    w = B.mtp_weights()
    h = ctypes.c_void_p()
    rc = lib.mtp_init_weights(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == code, B.mtp_last_error()
    assert h.value is None


def test_valid_config_with_null_weights_is_rejected(lib):
    c = _tiny_config()
    w = B.mtp_weights()
    h = ctypes.c_void_p()
    assert lib.mtp_init_weights(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == B.MTP_ERR_INVALID_ARG


def test_verify_rejects_bad_sizes_before_the_device(lib):
    fake = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    assert lib.mtp_verify_greedy(fake, fake, 1, 1, 12, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_greedy(fake, fake, 0, 1, 16, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_greedy(fake, fake, 1, -1, 16, fake, fake, None) == B.MTP_ERR_INVALID_ARG


def test_verify_sample_rejects_bad_arguments_before_the_device(lib):
    fake = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    f = ctypes.c_float
    assert lib.mtp_verify_sample(None, fake, 1, 1, 16, f(1.0), fake, fake, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, fake, 1, 1, 12, f(1.0), fake, fake, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, fake, 1, 1, 16, f(-0.5), fake, fake, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, fake, 1, 1, 16, f(float("nan")), fake, fake, fake, fake,
                                 None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, fake, 1, 1, 16, f(float("inf")), fake, fake, fake, fake,
                                 None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, None, 1, 2, 16, f(1.0), fake, fake, fake, fake, None) == B.MTP_ERR_INVALID_ARG
    assert lib.mtp_verify_sample(fake, fake, 1, 1, 16, f(1.0), fake, None, fake, fake, None) == B.MTP_ERR_INVALID_ARG


def test_header_states_the_wide_activation_contract():
    # the boundary documents what the kernels and the oracle do: activations stay fp32 with
    # no intermediate rounding, and the carried hidden state is not rounded
    with open(os.path.join(ROOT, "include", "mtp.h")) as f:
        text = " ".join(f.read().split())
    assert "Activations are fp32 and are never rounded to a narrower type" in text
    assert "stays fp32 (unrounded)" in text
    for stale in ("is rounded to bf16 (bf16 models)", "rounded to the model dtype", "rounded to bf16 inside"):
        assert stale not in text, stale
    # nor does any kernel comment describe rounding activations to bf16
    csrc = os.path.join(ROOT, "mtp_speculative_decoding_gemma4_gb300", "csrc")
    for name in os.listdir(csrc):
        with open(os.path.join(csrc, name)) as f:
            src = " ".join(f.read().split())
        assert "rounded to bf16 inside" not in src and "Operand rounding of the precision contract" not in src, name
