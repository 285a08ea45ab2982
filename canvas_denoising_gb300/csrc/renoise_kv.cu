// Threshold re-noise, canvas initialisation and the KV-cache append.
//
// Re-noise / init: DiffusionGemma explainer, "2. Uniform-state diffusion"
// (noise = a random vocabulary token; a token below the probability
// threshold is re-noised) and "The problem with autoregressive models" (the
// canvas starts as random vocabulary tokens). One thread per position; the
// canvas is 256 positions, so these launches are latency-bound.
//
// KV append: "Architecture: incremental prefill and denoising" / "Multi-canvas
// sampling": the finalised canvas's K/V rows go to cache rows [P, P+C).
// Pure 16-byte vector copy, one head block per blockIdx.y.
#include "dg_common.cuh"

namespace dg {

__global__ void renoise_kernel(int32_t* __restrict__ tokens, const int32_t* __restrict__ argmax,
                               const float* __restrict__ conf, int C, uint32_t V, float threshold, uint64_t seed,
                               uint32_t step, int64_t abs_pos0, uint8_t* __restrict__ renoised, int* status) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= C) return;
  float c = conf[i];
  int32_t a = argmax[i];
  bool low = c < threshold;
  int32_t t;
  if (low) {
    t = uniform_token(seed, step, abs_pos0 + i, kDomainRenoise, V);
  } else {
    if (a < 0 || (uint32_t)a >= V) latch(status, DG_ERR_DEVICE_BOUNDS);
    t = a;
  }
  tokens[i] = t;
  if (renoised) renoised[i] = low ? 1 : 0;
}

__global__ void canvas_init_kernel(int32_t* __restrict__ tokens, int C, uint32_t V, uint64_t seed,
                                   int64_t abs_pos0, const int64_t* __restrict__ abs_pos0_dev) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t p0 = abs_pos0_dev ? *abs_pos0_dev : abs_pos0;
  if (i < C) tokens[i] = uniform_token(seed, 0, p0 + i, kDomainInit, V);
}

// rows [P, P+C) of head blockIdx.y; `vec_per_head` 16-byte vectors per head block.
// With len_dev set, P is read from device memory (rows of `row_vecs` vectors)
// and a block that would end past `cap` copies nothing and latches a bounds error.
__global__ void kv_append_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc, const uint4* __restrict__ kn,
                                 const uint4* __restrict__ vn, int64_t cap_vecs_per_head, int64_t dst_off_vecs,
                                 int64_t vec_per_head, const int64_t* __restrict__ len_dev, int64_t row_vecs,
                                 int64_t C, int64_t cap, int* status) {
  if (len_dev) {
    const int64_t P = *len_dev;
    if (P < 0 || P + C > cap) {
      if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) latch(status, DG_ERR_DEVICE_BOUNDS);
      return;
    }
    dst_off_vecs = P * row_vecs;
  }
  const int64_t g = blockIdx.y;
  const uint4* ks = kn + g * vec_per_head;
  const uint4* vs = vn + g * vec_per_head;
  uint4* kd = kc + g * cap_vecs_per_head + dst_off_vecs;
  uint4* vd = vc + g * cap_vecs_per_head + dst_off_vecs;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < vec_per_head;
       j += (int64_t)gridDim.x * blockDim.x) {
    uint4 a = ks[j];
    uint4 b = vs[j];
    kd[j] = a;
    vd[j] = b;
  }
}

// *len += C after an append (same bounds rule as the copy, so both agree).
__global__ void len_advance_kernel(int64_t* len, int64_t C, int64_t cap) {
  const int64_t P = *len;
  if (P >= 0 && P + C <= cap) *len = P + C;
}

}  // namespace dg

using namespace dg;

extern "C" int dg_renoise(int32_t* tokens, const int32_t* argmax, const float* conf, int C, int V, float threshold,
                          uint64_t seed, uint32_t step, int64_t abs_pos0, uint8_t* renoised, void* stream) {
  if (!tokens || !argmax || !conf || C < 1 || V < 1 || abs_pos0 < 0) return DG_ERR_INVALID_ARG;
  if (threshold != threshold) return DG_ERR_INVALID_ARG;  // NaN
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  renoise_kernel<<<(C + 255) / 256, 256, 0, s>>>(tokens, argmax, conf, C, (uint32_t)V, threshold, seed, step,
                                                  abs_pos0, renoised, st);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_canvas_init(int32_t* tokens, int C, int V, uint64_t seed, int64_t abs_pos0, void* stream) {
  if (!tokens || C < 1 || V < 1 || abs_pos0 < 0) return DG_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  canvas_init_kernel<<<(C + 255) / 256, 256, 0, s>>>(tokens, C, (uint32_t)V, seed, abs_pos0, nullptr);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_kv_append(void* k_cache, void* v_cache, int64_t cap, int64_t* len, const void* k_new,
                            const void* v_new, int C, int Hkv, int hd, int dtype, const void* q_new, int Hq,
                            void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_cache || !v_cache || !len || !k_new || !v_new) return DG_ERR_INVALID_ARG;
  if (C < 1 || Hkv < 1 || cap < 1) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 && dtype != DG_F32) return DG_ERR_INVALID_ARG;
  if (hd != 32 && hd != 64 && hd != 128) return DG_ERR_UNSUPPORTED;
  const int64_t P = *len;
  if (P < 0 || P + C > cap) return DG_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return DG_ERR_INVALID_ARG;
  if (q_new) {
    if (!out || Hq < Hkv || Hq % Hkv) return DG_ERR_INVALID_ARG;
    if (workspace_bytes < attn_workspace(C, Hq, Hkv, hd, P, dtype)) return DG_ERR_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t esz = dtype == DG_BF16 ? 2 : 4;
  const int64_t row_vecs = (int64_t)hd * esz / 16;
  const int64_t vec_per_head = (int64_t)C * row_vecs;
  int gx = (int)((vec_per_head + 255) / 256);
  if (gx > 64) gx = 64;
  dim3 grid(gx, Hkv);
  kv_append_kernel<<<grid, 256, 0, s>>>((uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new,
                                        (const uint4*)v_new, cap * row_vecs, P * row_vecs, vec_per_head, nullptr,
                                        row_vecs, C, cap, nullptr);
  DG_LAUNCH_CHECK();
  if (q_new) {
    // The block's causal attention over the updated cache: keys [0, P) from the
    // cache and the block's own rows as the canvas keys.
    int rc = attn_launch(q_new, k_cache, v_cache, cap, P, k_new, v_new, out, lse, C, Hq, Hkv, hd, -1.0f, dtype,
                         DG_MASK_CAUSAL_BLOCK, workspace, workspace_bytes, s);
    if (rc != DG_OK) return rc;
  }
  *len = P + C;
  return DG_OK;
}

extern "C" int dg_canvas_init_devpos(int32_t* tokens, int C, int V, uint64_t seed, const int64_t* abs_pos0_dev,
                                     void* stream) {
  if (!tokens || !abs_pos0_dev || C < 1 || V < 1) return DG_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  canvas_init_kernel<<<(C + 255) / 256, 256, 0, s>>>(tokens, C, (uint32_t)V, seed, 0, abs_pos0_dev);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_kv_append_devlen(void* k_cache, void* v_cache, int64_t cap, int64_t* len_dev, const void* k_new,
                                   const void* v_new, int C, int Hkv, int hd, int dtype, void* stream) {
  if (!k_cache || !v_cache || !len_dev || !k_new || !v_new) return DG_ERR_INVALID_ARG;
  if (C < 1 || Hkv < 1 || cap < C) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 && dtype != DG_F32) return DG_ERR_INVALID_ARG;
  if (hd != 32 && hd != 64 && hd != 128) return DG_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return DG_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t esz = dtype == DG_BF16 ? 2 : 4;
  const int64_t row_vecs = (int64_t)hd * esz / 16;
  const int64_t vec_per_head = (int64_t)C * row_vecs;
  int gx = (int)((vec_per_head + 255) / 256);
  if (gx > 64) gx = 64;
  dim3 grid(gx, Hkv);
  kv_append_kernel<<<grid, 256, 0, s>>>((uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new,
                                        (const uint4*)v_new, cap * row_vecs, 0, vec_per_head, len_dev, row_vecs, C,
                                        cap, st);
  DG_LAUNCH_CHECK();
  len_advance_kernel<<<1, 1, 0, s>>>(len_dev, C, cap);
  DG_LAUNCH_CHECK();
  return DG_OK;
}
