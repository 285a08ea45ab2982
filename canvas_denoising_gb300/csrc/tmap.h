// Cached bf16 tensor-map encoding (zero fill out of range).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace dg {
// dims / box innermost first; strides in bytes for dims 1..rank-1.
bool tmap_bf16_sw128(CUtensorMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box);
// Same without swizzle: the box lands in shared memory byte for byte as it is in
// global memory (for operands stored pre-swizzled).
bool tmap_bf16_plain(CUtensorMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box);
}  // namespace dg
