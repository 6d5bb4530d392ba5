"""CPR Gated DeltaNet for one GB300 GPU: a C-ABI CUDA library (sm_103a) and its binding.

Chunkwise-Parallel Recurrent evaluation of a Gated DeltaNet layer ("IsoExec:
Eliminating Trainer-Inference Mismatch in SkyRL", section "Chunkwise-Parallel
Recurrent (CPR) Gated DeltaNet"): boundary states by one fixed-order fp32 chunk update,
outputs by the token recurrence inside each chunk, decode by the same recurrence with a
resync every C tokens, so that prefill, training forward and decode agree bit for bit.
"""
from .binding import (  # noqa: F401
    CprError,
    Ring,
    cpr_gdn_backward,
    cpr_gdn_backward_supported,
    cpr_gdn_backward_workspace_size,
    cpr_gdn_decode,
    cpr_gdn_decode_workspace_size,
    cpr_gdn_device_status,
    cpr_gdn_num_chunks,
    cpr_gdn_prefill,
    cpr_gdn_prefill_continue,
    cpr_gdn_prefill_noalloc,
    cpr_gdn_prefill_noalloc_status,
    cpr_gdn_prefill_workspace_size,
    cpr_gdn_ring_from_prefill,
    cpr_gdn_set_profile_events,
    cpr_gdn_set_wait_test,
    cpr_gdn_strerror,
    cpr_gdn_supported,
    cpr_gdn_version,
    cpr_pik_combine,
    cpr_pik_gemm,
    cpr_pik_workspace_size,
    continue_chunks,
    load_library,
)
