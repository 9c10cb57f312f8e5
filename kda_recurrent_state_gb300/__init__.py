"""kda_recurrent_state_gb300: Kimi Delta Attention forward (prefill + decode) for GB300.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA behind the C ABI
of ``include/kda.h``); ``binding`` marshals torch tensors into it.  Importing
the package does not load the library; the first call does, and it fails
loudly if the library has not been built.
"""
from .binding import (KDA_BF16, KDA_F32, KDA_GATE_CHANNEL, KDA_GATE_HEAD, KDA_GATE_NONE,  # noqa: F401
                      KDA_OP_BWD, KDA_OP_CHUNK, KDA_OP_CHUNK_BWD, KDA_OP_DECODE, KDA_OP_VARLEN, KdaError, kda_bwd, kda_chunk_fwd,
                      kda_chunk_fwd_host,
                      kda_decode_step, kda_decode_step_bf16state, kda_gdn_chunk_fwd, kda_gdn_decode_step,
                      kda_gdn_decode_step_bf16state,
                      kda_gdn_varlen_fwd, kda_get_device_status, kda_snapshot_count, kda_snapshot_lookup,
                      kda_snapshot_offsets, kda_status_string, kda_varlen_fwd, kda_varlen_fwd_pool,
                      kda_workspace_size)
