"""GB300-native Gemma-4-assistant MTP drafter: the drafter step, draft block, centroid
head and greedy verify as hand-written sm_103a CUDA kernels behind the C ABI in
include/mtp.h (libmtp.so), with a thin Python binding.
"""
from . import binding  # noqa: F401
from .binding import EXPORTS, MtpError, load_library  # noqa: F401


def __getattr__(name):
    # The torch-facing layer is imported lazily so that the C ABI can be loaded without torch.
    if name in ("Drafter", "verify_greedy", "verify_sample", "make_config", "make_kv"):
        from . import drafter
        return getattr(drafter, name)
    raise AttributeError(name)
