"""B300-native HashEvict decode step (pre-attention LSH eviction + attention over
the fixed-budget cache).

Python binding of ``libhashevict.so`` (C ABI in ``include/hashevict.h``):
argument marshalling only — every step of the decode path runs in the CUDA
kernels of the library.  There is no CPU fallback: importing the binding when
the library is missing raises.

Method: "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
Locality-Sensitive Hashing" (arXiv 2412.16187), abstract and technical
framework steps 1-5.
"""
from ._binding import (  # noqa: F401
    HE_DTYPE_BF16, HE_DTYPE_FP32, HE_ENGINE_FUSED, HE_ENGINE_PIPELINE, HE_TAU_FIXED,
    HE_TAU_MEDIAN, HE_VFMT_ELEM, HE_VFMT_FP8, HE_VFMT_INT8, HashEvict, HashEvictError, HeCfg,
    he_attend_noalloc, he_codes, he_create, he_destroy, he_fill, he_get_projection,
    he_last_evicted, he_launch_info, he_occupancy, he_profile_start, he_profile_stop,
    he_read_scores, he_read_state, he_read_thresholds, he_read_vscales, he_recompute_count,
    he_scores,
    he_set_alloc_limit, he_set_dist_log, he_set_evict_log, he_step, he_step_bytes, he_step_host,
    he_strerror, he_wait_probe, lib, lib_path,
)
from .shard import layer_shard, max_over_ranks  # noqa: F401
