// C-ABI entry points that are not kernels' own files: status handling,
// argument validation and dispatch for dg_canvas_attn and dg_vocab_step.
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "dg_common.cuh"

namespace dg {

__device__ int g_status_word;

// One status word per device: its address, looked up once per device.
int* status_ptr() {
  static std::mutex mu;
  static int* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    addr[dev] = (int*)p;
  }
  return addr[dev];
}

namespace {
std::mutex g_inject_mu;
Inject g_inject{kInjectNone, 0};
}  // namespace

Inject take_inject(int kind) {
  std::lock_guard<std::mutex> lk(g_inject_mu);
  Inject r{kInjectNone, 0};
  if (g_inject.kind == kind) {
    r = g_inject;
    g_inject = Inject{kInjectNone, 0};
  }
  return r;
}

void report_cuda_error(cudaError_t e, const char* what, const char* file, int line) {
  static const bool verbose = [] {
    const char* v = getenv("DG_VERBOSE");
    return v && *v && *v != '0';
  }();
  if (verbose) fprintf(stderr, "libdgcanvas: %s failed: %s (%s:%d)\n", what, cudaGetErrorString(e), file, line);
}

}  // namespace dg

using namespace dg;

extern "C" const char* dg_status_string(int status) {
  switch (status) {
    case DG_OK: return "DG_OK";
    case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG: invalid argument";
    case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED: shape or dtype not supported";
    case DG_ERR_WORKSPACE: return "DG_ERR_WORKSPACE: workspace too small";
    case DG_ERR_CUDA: return "DG_ERR_CUDA: CUDA runtime error";
    case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT: a bounded device wait ran out";
    case DG_ERR_DEVICE_BOUNDS: return "DG_ERR_DEVICE_BOUNDS: device-side index out of range";
    default: return "unknown dg_status";
  }
}

extern "C" int dg_device_status(void* stream) {
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  DG_CUDA_TRY(cudaStreamSynchronize(s));
  int v = 0;
  DG_CUDA_TRY(cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost));
  if (v != 0) {
    int zero = 0;
    DG_CUDA_TRY(cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice));
  }
  return v;
}

extern "C" size_t dg_canvas_attn_workspace_size(int C, int Hq, int Hkv, int hd, int64_t prefix_len, int dtype) {
  if (C < 1 || Hq < 1 || Hkv < 1 || prefix_len < 0) return 0;
  return attn_workspace(C, Hq, Hkv, hd, prefix_len, dtype);
}

extern "C" int dg_canvas_attn(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                              int64_t prefix_len, const void* k_canvas, const void* v_canvas, void* out, float* lse,
                              int C, int Hq, int Hkv, int hd, float scale, int dtype, int mask, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!q || !k_canvas || !v_canvas || !out) return DG_ERR_INVALID_ARG;
  if (prefix_len > 0 && (!k_cache || !v_cache)) return DG_ERR_INVALID_ARG;
  if (C < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || prefix_len < 0 || prefix_len > cap) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 && dtype != DG_F32) return DG_ERR_INVALID_ARG;
  if (mask != DG_MASK_BIDIR && mask != DG_MASK_CAUSAL_BLOCK) return DG_ERR_INVALID_ARG;
  if (hd != 32 && hd != 64 && hd != 128) return DG_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_canvas) || !aligned16(v_canvas) || !aligned16(out)) return DG_ERR_INVALID_ARG;
  if (prefix_len > 0 && (!aligned16(k_cache) || !aligned16(v_cache))) return DG_ERR_INVALID_ARG;
  if (workspace_bytes < attn_workspace(C, Hq, Hkv, hd, prefix_len, dtype)) return DG_ERR_WORKSPACE;
  return attn_launch(q, k_cache, v_cache, cap, prefix_len, k_canvas, v_canvas, out, lse, C, Hq, Hkv, hd, scale,
                     dtype, mask, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" size_t dg_vocab_step_workspace_size(int C, int V, int d, int dtype) {
  if (dtype == DG_BF16 && C >= 1 && C <= 256 && V >= 1 && d >= 64 && d % 64 == 0 && d <= 8192)
    return vocab_tc_workspace(C, V, d);
  return 0;
}

extern "C" int dg_vocab_step(const void* h, const void* emb, int C, int V, int d, int dtype, int32_t* argmax,
                             float* conf, float* lse, void* selfcond, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!h || !emb || !argmax || !conf || C < 1 || V < 1 || d < 1) return DG_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == DG_F32) {
    if (V > 16384 || d > 1024) return DG_ERR_UNSUPPORTED;
    return vocab_simt_launch((const float*)h, (const float*)emb, C, V, d, argmax, conf, lse, (float*)selfcond, s);
  }
  if (dtype != DG_BF16) return DG_ERR_INVALID_ARG;
  if (C > 256 || d % 64 || d > 8192) return DG_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(emb) || (selfcond && !aligned16(selfcond))) return DG_ERR_INVALID_ARG;
  if (workspace_bytes < vocab_tc_workspace(C, V, d)) return DG_ERR_WORKSPACE;
  if (vocab_tc_workspace(C, V, d) && ((uintptr_t)workspace & 255u)) return DG_ERR_INVALID_ARG;
  return vocab_tc_launch((const __nv_bfloat16*)h, (const __nv_bfloat16*)emb, C, V, d, argmax, conf, lse,
                         (__nv_bfloat16*)selfcond, workspace, workspace_bytes, s);
}

extern "C" int dg_vocab_step_renoise(const void* h, const void* emb, int C, int V, int d, int dtype, int32_t* argmax,
                                     float* conf, float* lse, void* selfcond, int32_t* tokens, float threshold,
                                     uint64_t seed, uint32_t step, int64_t abs_pos0, uint8_t* renoised,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!tokens || abs_pos0 < 0 || threshold != threshold) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16) {
    // CUDA-core path: the two calls back to back
    const int rc = dg_vocab_step(h, emb, C, V, d, dtype, argmax, conf, lse, selfcond, workspace, workspace_bytes,
                                 stream);
    if (rc != DG_OK) return rc;
    return dg_renoise(tokens, argmax, conf, C, V, threshold, seed, step, abs_pos0, renoised, stream);
  }
  if (!h || !emb || !argmax || !conf || C < 1 || V < 1 || d < 1) return DG_ERR_INVALID_ARG;
  if (C > 256 || d % 64 || d > 8192) return DG_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(emb) || (selfcond && !aligned16(selfcond))) return DG_ERR_INVALID_ARG;
  if (workspace_bytes < vocab_tc_workspace(C, V, d)) return DG_ERR_WORKSPACE;
  if (vocab_tc_workspace(C, V, d) && ((uintptr_t)workspace & 255u)) return DG_ERR_INVALID_ARG;
  RenoiseArgs rn{tokens, renoised, threshold, seed, step, abs_pos0, nullptr};
  return vocab_tc_launch((const __nv_bfloat16*)h, (const __nv_bfloat16*)emb, C, V, d, argmax, conf, lse,
                         (__nv_bfloat16*)selfcond, workspace, workspace_bytes, (cudaStream_t)stream, &rn);
}

extern "C" int dg_vocab_step_plan(int C, int V, int d, int dtype, int32_t* plan) {
  if (!plan || dtype != DG_BF16 || C < 1 || C > 256 || V < 1 || d < 64 || d % 64 || d > 8192) return DG_ERR_INVALID_ARG;
  return vocab_tc_plan(C, V, d, plan);
}

extern "C" int dg_vocab_step_renoise_devpos(const void* h, const void* emb, int C, int V, int d, int dtype,
                                            int32_t* argmax, float* conf, float* lse, void* selfcond, int32_t* tokens,
                                            float threshold, uint64_t seed, uint32_t step,
                                            const int64_t* abs_pos0_dev, uint8_t* renoised, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  if (!tokens || !abs_pos0_dev || threshold != threshold) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16) return DG_ERR_UNSUPPORTED;
  if (!h || !emb || !argmax || !conf || C < 1 || V < 1 || d < 1) return DG_ERR_INVALID_ARG;
  if (C > 256 || d % 64 || d > 8192) return DG_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(emb) || (selfcond && !aligned16(selfcond))) return DG_ERR_INVALID_ARG;
  if (workspace_bytes < vocab_tc_workspace(C, V, d)) return DG_ERR_WORKSPACE;
  if (vocab_tc_workspace(C, V, d) && ((uintptr_t)workspace & 255u)) return DG_ERR_INVALID_ARG;
  RenoiseArgs rn{tokens, renoised, threshold, seed, step, 0, abs_pos0_dev};
  return vocab_tc_launch((const __nv_bfloat16*)h, (const __nv_bfloat16*)emb, C, V, d, argmax, conf, lse,
                         (__nv_bfloat16*)selfcond, workspace, workspace_bytes, (cudaStream_t)stream, &rn);
}

extern "C" int dg_canvas_attn_devlen(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                     const int64_t* prefix_len_dev, int64_t prefix_max, const void* k_canvas,
                                     const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv, int hd,
                                     float scale, int dtype, int mask, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (!q || !prefix_len_dev || !k_canvas || !v_canvas || !out) return DG_ERR_INVALID_ARG;
  if (prefix_max > 0 && (!k_cache || !v_cache)) return DG_ERR_INVALID_ARG;
  if (C < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || prefix_max < 0 || prefix_max > cap) return DG_ERR_INVALID_ARG;
  if (mask != DG_MASK_BIDIR && mask != DG_MASK_CAUSAL_BLOCK) return DG_ERR_INVALID_ARG;
  if (dtype != DG_BF16 || hd != 128) return DG_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_canvas) || !aligned16(v_canvas) || !aligned16(out)) return DG_ERR_INVALID_ARG;
  if (prefix_max > 0 && (!aligned16(k_cache) || !aligned16(v_cache))) return DG_ERR_INVALID_ARG;
  if (workspace_bytes < attn_workspace(C, Hq, Hkv, hd, prefix_max, dtype)) return DG_ERR_WORKSPACE;
  if (scale <= 0.f) scale = 1.0f / sqrtf((float)hd);
  return attn_tc_launch(q, k_cache, v_cache, cap, prefix_max, k_canvas, v_canvas, out, lse, C, Hq, Hkv, scale, mask,
                        workspace, workspace_bytes, (cudaStream_t)stream, prefix_len_dev);
}

extern "C" int dg_debug_inject(int kind, int wait_ms) {
  if (kind < kInjectNone || kind > kInjectVocabReady || wait_ms < 0 || wait_ms > 10000) return DG_ERR_INVALID_ARG;
  long long cycles = 0;
  if (kind != kInjectNone) {
    int dev = 0, khz = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess)
      return DG_ERR_CUDA;
    cycles = (long long)wait_ms * khz;  // kHz x ms = cycles
  }
  std::lock_guard<std::mutex> lk(g_inject_mu);
  g_inject = Inject{kind, cycles};
  return DG_OK;
}
