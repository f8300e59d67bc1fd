"""GB300 (sm_103a) reuse-time MLA KV reconstruction: delta-rotated chunk reuse fused into
absorbed MLA attention, plus a standalone rotate+gather into a paged KV layout.

The compute path is libirm.so (C ABI in include/irm.h, CUDA kernels in csrc/); this
package holds its build script, a ctypes binding with the same entry-point names, and the
seeded synthetic workload generators.
"""
from .binding import (CDC_LOW_BITS, CDC_THRESHOLD, ROPE_INTERLEAVED, ROPE_NEOX, CdcParams,
                      ChunkTable, IrmError, Registry, Rope, cdc_sizes, cdc_slot_base, irm_cdc_chunk,
                      assemble_kv_workspace_size, decode_noalloc_status, decode_workspace_size,
                      device_status, irm_assemble_kv, irm_mla_attn_decode,
                      irm_mla_attn_decode_noalloc, irm_mla_attn_prefill, lib,
                      new_workspace, prefill_workspace_size, selftest_wait_timeout,
                      validate_chunks)

__all__ = ["Registry", "CDC_LOW_BITS", "CDC_THRESHOLD", "CdcParams", "cdc_sizes", "cdc_slot_base",
           "irm_cdc_chunk", "ROPE_INTERLEAVED", "ROPE_NEOX", "Rope", "ChunkTable", "IrmError",
           "assemble_kv_workspace_size", "decode_noalloc_status", "decode_workspace_size",
           "device_status", "irm_assemble_kv", "irm_mla_attn_decode", "irm_mla_attn_decode_noalloc",
           "irm_mla_attn_prefill",
           "lib", "new_workspace", "prefill_workspace_size", "selftest_wait_timeout", "validate_chunks"]
