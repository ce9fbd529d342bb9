"""Kimi Delta Attention (KDA) for NVIDIA GB300 (sm_103a).

The compute lives in ``libkda.so`` (hand-written CUDA behind a C ABI,
``include/kda.h``); ``binding`` exposes its entry points to Python under the
same names. ``inputs`` draws seeded synthetic workloads.
"""
from .binding import (KDA_DEBUG_CHECK, KDA_DTYPE_BF16, KDA_DTYPE_F32, KDA_GATE_LOGITS,
                      KDA_QK_L2NORM, KdaError,
                      chunk_bwd, chunk_fwd, chunk_fwd_checkpoints, decode_step, kda_chunk_bwd,
                      kda_chunk_bwd_workspace_size, kda_chunk_fwd,
                      kda_chunk_fwd_checkpoints, kda_chunk_fwd_host,
                      kda_chunk_fwd_host_buffer_size, kda_chunk_fwd_noalloc,
                      kda_chunk_fwd_launches, kda_chunk_fwd_workspace_size,
                      kda_decode_step, kda_get_error, kda_last_error_string, kda_scan_combine,
                      kda_segment_summary, kda_segment_summary_workspace_size, kda_segmented_fwd,
                      kda_segmented_fwd_workspace_size, kda_trace_events,
                      kda_version, load,
                      scan_combine, segment_summary, segmented_fwd)

from .pipeline import HostPipeline  # noqa: E402

__all__ = [n for n in dir() if not n.startswith("_")]
