"""C2KV composed-cache hot path for GB300 (sm_103a).

Compressed, composable, non-prefix KV-cache reuse (C2KV explainer,
paper-daily.com; arXiv 2607.17715): per-document compressed pre-RoPE K/V
segments live in a pinned host store; at request time they are streamed to
HBM, re-rotated at their composed positions and concatenated into one GQA
cache, over which the question is prefilled and the answer decoded.

The compute runs in libc2kv.so (include/c2kv.h); `binding` mirrors its C
names.  There is no CPU fallback: without the built library the binding
raises ImportError on first use.
"""
from .binding import *  # noqa: F401,F403
from .binding import C2KVError, load_library  # noqa: F401
from .pipeline import DecoderModel, RequestBatch, RequestSpec  # noqa: F401
