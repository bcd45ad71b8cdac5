"""Sparse MLA attention over a paged latent KV cache, for one GB300 (sm_103a).

The compute lives in libsvt.so (hand-written CUDA, C ABI declared in include/svt.h); the
binding in ``svt`` marshals torch tensors to it. ``workloads`` draws seeded synthetic
inputs. Importing the package does not load the library; the first call does, and fails
loudly if it has not been built.
"""

from .svt import (  # noqa: F401
    KV_BF16,
    KV_FP8_E4M3,
    KVCache,
    SvtError,
    Workspace,
    build_group_union,
    debug_pipeline_fault,
    gather_probe,
    merge_splits,
    resolve_topk_slots,
    sparse_mla_decode,
    sparse_mla_prefill_grouped,
    tensor_probe,
    topk_select,
)
