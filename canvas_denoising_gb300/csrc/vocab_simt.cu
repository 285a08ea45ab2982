// fp32 vocabulary step on CUDA cores, for small shapes (V <= 16384,
// d <= 1024). One CTA per canvas position: logits into shared memory,
// block max / first-index argmax / sum, then the self-conditioning row
// S_i = sum_v p_v E_v with threads over the model dimension.
//
// Explainer, "Self-conditioning" (probabilities times the embedding table)
// and "2. Uniform-state diffusion" (the probability compared with the
// re-noise threshold).
#include <math.h>

#include "dg_common.cuh"

namespace dg {
namespace {

constexpr int NT = 256;

__global__ void vocab_simt_kernel(const float* __restrict__ h, const float* __restrict__ emb, int V, int d,
                                  int32_t* argmax, float* conf, float* lse, float* selfcond) {
  extern __shared__ float sm[];
  float* logit = sm;       // [V]
  float* hrow = sm + V;    // [d]
  __shared__ float rv[NT / 32];
  __shared__ int ri[NT / 32];
  const int i = blockIdx.x, t = threadIdx.x;
  for (int k = t; k < d; k += NT) hrow[k] = h[(int64_t)i * d + k];
  __syncthreads();
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int v = t; v < V; v += NT) {
    const float* e = emb + (int64_t)v * d;
    float acc = 0.f;
    for (int k = 0; k < d; ++k) acc = fmaf(hrow[k], e[k], acc);
    logit[v] = acc;
    if (acc > best || (acc == best && v < bidx)) { best = acc; bidx = v; }
  }
  for (int o = 16; o; o >>= 1) {
    float ob = __shfl_xor_sync(0xffffffffu, best, o);
    int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
  }
  if ((t & 31) == 0) { rv[t >> 5] = best; ri[t >> 5] = bidx; }
  __syncthreads();
  best = rv[0];
  bidx = ri[0];
  for (int w = 1; w < NT / 32; ++w)
    if (rv[w] > best || (rv[w] == best && ri[w] < bidx)) { best = rv[w]; bidx = ri[w]; }
  __syncthreads();
  float z = 0.f;
  for (int v = t; v < V; v += NT) {
    float p = expf(logit[v] - best);
    logit[v] = p;
    z += p;
  }
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if ((t & 31) == 0) rv[t >> 5] = z;
  __syncthreads();
  z = 0.f;
  for (int w = 0; w < NT / 32; ++w) z += rv[w];
  const float inv = 1.f / z;
  if (t == 0) {
    argmax[i] = bidx;
    conf[i] = inv;
    if (lse) lse[i] = best + logf(z);
  }
  if (selfcond) {
    for (int k = t; k < d; k += NT) {
      float acc = 0.f;
      for (int v = 0; v < V; ++v) acc = fmaf(logit[v], emb[(int64_t)v * d + k], acc);
      selfcond[(int64_t)i * d + k] = acc * inv;
    }
  }
}

}  // namespace

int vocab_simt_launch(const float* h, const float* emb, int C, int V, int d, int32_t* argmax, float* conf, float* lse,
                      float* selfcond, cudaStream_t s) {
  size_t smem = (size_t)(V + d) * sizeof(float);
  DG_CUDA_TRY(cudaFuncSetAttribute(vocab_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  vocab_simt_kernel<<<C, NT, smem, s>>>(h, emb, V, d, argmax, conf, lse, selfcond);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

}  // namespace dg
