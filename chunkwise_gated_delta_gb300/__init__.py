"""Chunkwise gated delta rule (KDA, GDN, DeltaNet, GLA) on GB300 / sm_103a.

The computation lives in the CUDA library ``_build/libkda.so`` (C ABI in
``include/kda.h``); :mod:`.api` is its Python binding.  Build the library with
:func:`.build.build`.
"""
from .api import (HostRunner, KdaError, deltanet_fwd, dplr_chunk_bwd, dplr_chunk_fwd, dplr_factor_norms,  # noqa: F401
                  gdn_fwd, gla_fwd, kda_chunk_bwd, kda_chunk_fwd, kda_chunk_fwd_noalloc, status_read)
