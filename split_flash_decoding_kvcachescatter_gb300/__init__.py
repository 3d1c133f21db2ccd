"""GB300-native batched decode-step attention: KV-cache scatter + split-K
flash decoding under GQA, as hand-written sm_103a CUDA kernels behind a C ABI
(include/kvsdecode.h).  This package holds the kernels (csrc/), their build
script, the ctypes binding and the seeded synthetic workloads.
"""
from .binding import (EXPORTS, kvs_argmax, kvs_prefill_attention, KVS_SCHEDULE_AUTO, KVS_SCHEDULE_CLUSTER,  # noqa: F401
                      KVS_SCHEDULE_PERSISTENT, KvsError, StepGraph, kvs_choose_chunk_size,
                      kvs_decode_step, kvs_decode_step_host, kvs_decode_step_slots, kvs_flash_decode,
                      kvs_flash_decode_static, step_io,
                      kvs_flash_decode_workspace_bytes, kvs_get_schedule, kvs_kv_scatter,
                      kvs_prepare, kvs_schedule_for, prefill_workspace, kvs_set_schedule, kvs_step_graph_create, lib, strerror,
                      workspace)
