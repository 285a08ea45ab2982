// Rows next to the denoising step: the self-conditioning input of the next
// step, the probability of the current canvas token, masked-diffusion
// unmasking with lock-in, canvas fill and a device-side flag count.
//
// DiffusionGemma explainer: "Self-conditioning" (the probabilities times the
// embedding table feed the next step), "2. Uniform-state diffusion" (a
// token's probability against a threshold), "1. Masked diffusion" ([MASK]
// tokens replaced once confident, then locked).
//
// All of these are memory- or latency-bound: one CTA per canvas row for the
// row-wise ones (16-byte vector loads along d), one thread per position for
// the rest.
#include "dg_common.cuh"

namespace dg {
namespace {

constexpr int kRowThreads = 128;

__device__ __forceinline__ void add8_bf16(const uint4& a, const uint4& b, uint4& o) {
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
  __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
    po[e] = __floats2bfloat162_rn(fa.x + fb.x, fa.y + fb.y);
  }
}

// x[i] = emb[tokens[i]] + selfcond[i]; bf16, 8 elements per 16-byte vector.
__global__ void __launch_bounds__(kRowThreads) selfcond_input_bf16(const int32_t* __restrict__ tokens,
                                                                   const uint4* __restrict__ emb,
                                                                   const uint4* __restrict__ sc, uint4* __restrict__ x,
                                                                   int V, int nvec, int* status) {
  const int i = blockIdx.x;
  const int tok = tokens[i];
  const bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) latch(status, DG_ERR_DEVICE_BOUNDS);
  const uint4* er = emb + (size_t)(ok ? tok : 0) * nvec;
  for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (ok) {
      const uint4 e = __ldg(er + v);
      if (sc) {
        add8_bf16(e, __ldg(sc + (size_t)i * nvec + v), o);
      } else {
        o = e;
      }
    }
    x[(size_t)i * nvec + v] = o;
  }
}

__global__ void __launch_bounds__(kRowThreads) selfcond_input_f32(const int32_t* __restrict__ tokens,
                                                                  const float4* __restrict__ emb,
                                                                  const float4* __restrict__ sc,
                                                                  float4* __restrict__ x, int V, int nvec,
                                                                  int* status) {
  const int i = blockIdx.x;
  const int tok = tokens[i];
  const bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) latch(status, DG_ERR_DEVICE_BOUNDS);
  const float4* er = emb + (size_t)(ok ? tok : 0) * nvec;
  for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
      o = __ldg(er + v);
      if (sc) {
        const float4 s = __ldg(sc + (size_t)i * nvec + v);
        o.x += s.x;
        o.y += s.y;
        o.z += s.z;
        o.w += s.w;
      }
    }
    x[(size_t)i * nvec + v] = o;
  }
}

__device__ __forceinline__ float block_sum(float v) {
  __shared__ float part[kRowThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += part[w];
  return t;
}

// prob[i] = exp(h[i] . emb[tokens[i]] - lse[i]), fp32 dot product.
template <bool kBf16>
__global__ void __launch_bounds__(kRowThreads) token_prob_kernel(const void* __restrict__ h,
                                                                 const void* __restrict__ emb,
                                                                 const int32_t* __restrict__ tokens,
                                                                 const float* __restrict__ lse, float* prob, int V,
                                                                 int nvec, int* status) {
  const int i = blockIdx.x;
  const int tok = tokens[i];
  const bool ok = tok >= 0 && tok < V;
  float acc = 0.f;
  if (ok) {
    if (kBf16) {
      const uint4* hr = reinterpret_cast<const uint4*>(h) + (size_t)i * nvec;
      const uint4* er = reinterpret_cast<const uint4*>(emb) + (size_t)tok * nvec;
      for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
        const uint4 a = __ldg(hr + v), b = __ldg(er + v);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
      }
    } else {
      const float4* hr = reinterpret_cast<const float4*>(h) + (size_t)i * nvec;
      const float4* er = reinterpret_cast<const float4*>(emb) + (size_t)tok * nvec;
      for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
        const float4 a = __ldg(hr + v), b = __ldg(er + v);
        acc = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
      }
    }
  }
  const float dot = block_sum(acc);
  if (threadIdx.x == 0) {
    if (!ok) latch(status, DG_ERR_DEVICE_BOUNDS);
    prob[i] = ok ? expf(dot - lse[i]) : 0.f;
  }
}

__global__ void unmask_kernel(int32_t* tokens, const int32_t* __restrict__ argmax, const float* __restrict__ conf,
                              int C, int32_t mask_id, float threshold, uint8_t* unmasked) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= C) return;
  const int32_t t = tokens[i];
  const bool take = t == mask_id && conf[i] >= threshold;
  if (take) tokens[i] = argmax[i];
  if (unmasked) unmasked[i] = take ? 1 : 0;
}

__global__ void fill_kernel(int32_t* tokens, int C, int32_t value) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < C) tokens[i] = value;
}

__global__ void __launch_bounds__(256) count_kernel(const uint8_t* __restrict__ flags, int C, int32_t* count) {
  int n = 0;
  for (int base = 0; base < C; base += 256) {
    const int i = base + (int)threadIdx.x;
    n += __syncthreads_count(i < C && flags[i] != 0);
  }
  if (threadIdx.x == 0) *count = n;
}

bool row_args_ok(int C, int V, int d, int dtype) {
  if (C < 1 || V < 1 || d < 1) return false;
  if (dtype == DG_BF16) return d % 8 == 0;
  if (dtype == DG_F32) return d % 4 == 0;
  return false;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" int dg_selfcond_input(const int32_t* tokens, const void* emb, const void* selfcond, void* x, int C, int V,
                                 int d, int dtype, void* stream) {
  if (!tokens || !emb || !x) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 && dtype != DG_F32) return DG_ERR_INVALID_ARG;
  if (!row_args_ok(C, V, d, dtype)) return DG_ERR_INVALID_ARG;
  if (!aligned16(emb) || !aligned16(x) || (selfcond && !aligned16(selfcond))) return DG_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == DG_BF16)
    selfcond_input_bf16<<<C, kRowThreads, 0, s>>>(tokens, (const uint4*)emb, (const uint4*)selfcond, (uint4*)x, V,
                                                   d / 8, st);
  else
    selfcond_input_f32<<<C, kRowThreads, 0, s>>>(tokens, (const float4*)emb, (const float4*)selfcond, (float4*)x, V,
                                                  d / 4, st);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_token_prob(const void* h, const void* emb, const int32_t* tokens, const float* lse, float* prob,
                             int C, int V, int d, int dtype, void* stream) {
  if (!h || !emb || !tokens || !lse || !prob) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 && dtype != DG_F32) return DG_ERR_INVALID_ARG;
  if (!row_args_ok(C, V, d, dtype)) return DG_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(emb)) return DG_ERR_INVALID_ARG;
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == DG_BF16)
    token_prob_kernel<true><<<C, kRowThreads, 0, s>>>(h, emb, tokens, lse, prob, V, d / 8, st);
  else
    token_prob_kernel<false><<<C, kRowThreads, 0, s>>>(h, emb, tokens, lse, prob, V, d / 4, st);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_unmask(int32_t* tokens, const int32_t* argmax, const float* conf, int C, int32_t mask_id,
                         float threshold, uint8_t* unmasked, void* stream) {
  if (!tokens || !argmax || !conf || C < 1 || threshold != threshold) return DG_ERR_INVALID_ARG;
  unmask_kernel<<<(C + 255) / 256, 256, 0, (cudaStream_t)stream>>>(tokens, argmax, conf, C, mask_id, threshold,
                                                                    unmasked);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_canvas_fill(int32_t* tokens, int C, int32_t value, void* stream) {
  if (!tokens || C < 1) return DG_ERR_INVALID_ARG;
  fill_kernel<<<(C + 255) / 256, 256, 0, (cudaStream_t)stream>>>(tokens, C, value);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

extern "C" int dg_count_flags(const uint8_t* flags, int C, int32_t* count, void* stream) {
  if (!flags || !count || C < 1) return DG_ERR_INVALID_ARG;
  count_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(flags, C, count);
  DG_LAUNCH_CHECK();
  return DG_OK;
}
