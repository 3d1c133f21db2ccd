"""GB300-native batched decode-step attention: KV-cache scatter + split-K
flash decoding under GQA, as hand-written sm_103a CUDA kernels behind a C ABI
(include/kvsdecode.h).  This package holds the kernels (csrc/), their build
script, the ctypes binding and the seeded synthetic workloads.
"""
from .binding import (EXPORTS, KvsError, kvs_choose_chunk_size, kvs_decode_step,  # noqa: F401
                      kvs_flash_decode, kvs_flash_decode_static,
                      kvs_flash_decode_workspace_bytes, kvs_kv_scatter, lib, strerror,
                      workspace)
