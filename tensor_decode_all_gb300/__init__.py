"""Logical-rank all-reduce and allgather on one GB300 (sm_103a).

R logical ranks are concurrently resident kernels on their own non-blocking
streams of one GPU.  They exchange through double-buffered slots (mapped
pinned host memory or HBM) with per-block release/acquire flags, and sum in
fp32 in rank order with a single rounding.  The kernels live in
``libtda_ar.so`` (C ABI: include/ar.h); this package only binds it.
"""
from .ar import (AR_BF16, AR_C64, AR_F16, AR_SLOT_HBM, AR_SLOT_PINNED_HOST, ArError, Handle,  # noqa: F401
                 ar_allgather, ar_allreduce, ar_allreduce_noalloc, ar_noalloc_status, ar_choose_algo, ar_create, ar_destroy, ar_last_error, ar_plan_compute,
                 ar_plan_for, ar_probe_hbm_copy, ar_probe_host_link, ar_probe_host_link_latency, ar_query, ar_reset, ar_set_algo, ar_set_pdl, ar_set_timeout,
                 ar_status, ar_strerror, declared_symbols, lib, library_path, strerror)
from .builder import build  # noqa: F401
