// Host-side tensor-map (TMA descriptor) encoding with a small cache.
//
// cuTensorMapEncodeTiled is a host call of a few microseconds; a denoising
// step issues several per call with the same pointers and shapes every step.
// The cache is keyed by every encode input (address, rank, extents, strides,
// box), so a hit returns exactly the descriptor a fresh encode would.
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "dg_common.cuh"
#include "tmap.h"

namespace dg {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

struct Key {
  const void* base;
  int rank;
  int swizzle;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
  bool operator==(const Key& o) const { return memcmp(this, &o, sizeof(Key)) == 0; }
};

constexpr int kSlots = 64;
struct Entry {
  Key key;
  CUtensorMap map;
  bool used;
};

std::mutex g_mu;
Entry g_cache[kSlots];
int g_next = 0;

bool encode(CUtensorMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
            const uint32_t* box, CUtensorMapSwizzle swizzle) {
  if (rank < 2 || rank > 5) return false;
  Key k;
  memset(&k, 0, sizeof(k));
  k.base = base;
  k.rank = rank;
  k.swizzle = (int)swizzle;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) k.strides[i] = strides[i];
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < kSlots; ++i)
      if (g_cache[i].used && g_cache[i].key == k) {
        *out = g_cache[i].map;
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(g_mu);
  g_cache[g_next].key = k;
  g_cache[g_next].map = m;
  g_cache[g_next].used = true;
  g_next = (g_next + 1) % kSlots;
  *out = m;
  return true;
}

}  // namespace

bool tmap_bf16_sw128(CUtensorMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box) {
  return encode(out, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_bf16_plain(CUtensorMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box) {
  return encode(out, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace dg
