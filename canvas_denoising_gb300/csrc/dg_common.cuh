// Shared device/host helpers of libdgcanvas (status codes, Philox, launch checks).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dg_canvas.h"

namespace dg {

// ---------------------------------------------------------------- status word
// Kernels latch the first fault they detect into a library-owned device int
// (its address is passed in as `status`). Never a trap.
__device__ __forceinline__ void latch(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

int* status_ptr();  // device address of the status word for the current device (api.cu)

// Host-side failure injection for tests (dg_debug_inject): the next launch of
// the named kernel withholds one arrival, so its peers' bounded waits expire.
enum { kInjectNone = 0, kInjectAttnArrival = 1, kInjectVocabReady = 2 };
struct Inject {
  int kind;
  long long wait_cycles;  // bound for that launch's waits (0: the default)
};
Inject take_inject(int kind);  // returns and clears the pending injection if it is `kind`

// Reports a failed CUDA call on stderr when DG_VERBOSE is set (defined in api.cu).
void report_cuda_error(cudaError_t e, const char* what, const char* file, int line);

#define DG_CUDA_TRY(expr)                                          \
  do {                                                             \
    cudaError_t e_ = (expr);                                       \
    if (e_ != cudaSuccess) {                                       \
      ::dg::report_cuda_error(e_, #expr, __FILE__, __LINE__);      \
      return DG_ERR_CUDA;                                          \
    }                                                              \
  } while (0)

#define DG_LAUNCH_CHECK() DG_CUDA_TRY(cudaGetLastError())

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- Philox4x64-10
// Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten
// rounds of two 64x64->128 multiplies with XOR/permute, key bumped by two
// Weyl constants between rounds.
struct u64x4 { uint64_t x, y, z, w; };

__device__ __forceinline__ u64x4 philox4x64_10(u64x4 c, uint64_t k0, uint64_t k1) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += W0; k1 += W1; }
    uint64_t lo0 = M0 * c.x, hi0 = __umul64hi(M0, c.x);
    uint64_t lo1 = M1 * c.z, hi1 = __umul64hi(M1, c.z);
    u64x4 n;
    n.x = hi1 ^ c.y ^ k0;
    n.y = lo1;
    n.z = hi0 ^ c.w ^ k1;
    n.w = lo0;
    c = n;
  }
  return c;
}

// Uniform id in [0, V): Lemire's multiply-shift of the high 32 bits of word 0.
__device__ __forceinline__ int32_t uniform_token(uint64_t seed, uint32_t step, int64_t abs_pos, uint32_t domain,
                                                 uint32_t V) {
  u64x4 c{(uint64_t)abs_pos, (uint64_t)step, (uint64_t)domain, 0ull};
  u64x4 o = philox4x64_10(c, seed, 0ull);
  return (int32_t)(((o.x >> 32) * (uint64_t)V) >> 32);
}

constexpr uint32_t kDomainRenoise = 0;
constexpr uint32_t kDomainInit = 1;

// ---------------------------------------------------------------- internal entry points
int attn_launch(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t P,
                const void* k_canvas, const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv,
                int hd, float scale, int dtype, int mask, void* ws, size_t ws_bytes, cudaStream_t s);
size_t attn_workspace(int C, int Hq, int Hkv, int hd, int64_t P, int dtype);
int attn_combine_launch(const float* part_o, const float* part_lse, __nv_bfloat16* out, float* lse, int C, int Hq,
                        int HD, int splits, cudaStream_t s);
void attn_tc_plan(int C, int Hq, int Hkv, int64_t P, int* splits, int* tiles_per_split);
int attn_tc_launch(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t P,
                   const void* k_canvas, const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv,
                   float scale, int mask, void* ws, size_t ws_bytes, cudaStream_t s,
                   const int64_t* P_dev = nullptr);
size_t attn_tc_workspace(int C, int Hq, int Hkv, int64_t P);

int vocab_simt_launch(const float* h, const float* emb, int C, int V, int d, int32_t* argmax, float* conf,
                      float* lse, float* selfcond, cudaStream_t s);

struct RenoiseArgs {  // threshold re-noise fused into the vocabulary step's last kernel
  int32_t* tokens;
  uint8_t* renoised;
  float threshold;
  uint64_t seed;
  uint32_t step;
  int64_t abs_pos0;
  const int64_t* abs_pos0_dev;  // if set, the position offset is read from device memory
};

size_t vocab_tc_workspace(int C, int V, int d);
int vocab_tc_plan(int C, int V, int d, int* out);
int vocab_tc_launch(const __nv_bfloat16* h, const __nv_bfloat16* emb, int C, int V, int d, int32_t* argmax,
                    float* conf, float* lse, __nv_bfloat16* selfcond, void* ws, size_t ws_bytes, cudaStream_t s,
                    const RenoiseArgs* rn = nullptr);

}  // namespace dg
