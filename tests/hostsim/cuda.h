/* Host-only stand-in for the CUDA driver header (see cuda_runtime.h here). */
#pragma once
typedef struct alignas(64) CUtensorMap_st {
  unsigned long long opaque[16];
} CUtensorMap;
