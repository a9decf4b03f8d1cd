"""GB300-native (sm_103a) single-token MLA decode with split-KV flash decoding.

The compute path is the C-ABI CUDA library declared in ``include/mla_decode.h`` (built
in-tree by ``build.build()``); the functions here only marshal arguments:

* ``decode`` / ``mla_decode`` -- contiguous cache, rows indexed by ``kv_indptr``;
* ``decode_paged`` / ``mla_decode_paged`` -- paged cache (page-level indptr, page indices,
  last-page lengths; pages of 8 to 128 rows);
* ``decode_paged_multi`` / ``mla_decode_paged_multi`` -- several query tokens per sequence
  (``qo_indptr``), each attending causally to its prefix of a paged cache.

``synth`` makes seeded synthetic inputs (``make_inputs``, ``to_paged``, ``make_queries``).
"""
from ._lib import (MLA_ERR_CUDA, MLA_ERR_INVALID_ARG, MLA_ERR_NO_MEMORY, MLA_ERR_TIMEOUT,  # noqa: F401
                   MLA_ERR_UNSUPPORTED, MLA_OK, MLAError, decode, decode_paged, decode_paged_multi, device_status,
                   load, mla_decode, mla_decode_paged, mla_decode_paged_multi, pick_splits, profile_begin,
                   profile_end, release_workspace, reserve_workspace, resolve_splits, set_test_stall,
                   set_wait_limit_ns, workspace_slots)

KV_BF16, KV_FP8, KV_MXFP4 = 0, 1, 2
