// Canvas attention: bidirectional (denoising) and causal-block (incremental
// prefill) grouped-query attention of the canvas queries over
// [KV-cache prefix ; canvas].
//
// DiffusionGemma explainer, "Architecture: incremental prefill and
// denoising": in denoising mode a canvas query sees every canvas token and
// the KV cache; in prefill mode attention is causal.
//
// bf16 path: flash-attention with split-KV. The Hq/Hkv query heads that read
// one KV head are stacked into one M = (Hq/Hkv) * C row block, so each K/V
// tile is loaded once per row block. Tiles of 64 queries x 64 keys, 4 warps,
// bf16 mma.sync with fp32 accumulation, online softmax in base 2, K/V double
// buffered with cp.async. Splits of the key range write fp32 partials (O,
// lse) that a second kernel merges by log-sum-exp.
// fp32 path: one CTA per (query, head), CUDA cores, online softmax over key
// tiles of 128 (for small shapes).
#include <math.h>

#include <mutex>

#include "dg_common.cuh"

namespace dg {

namespace {

constexpr int BM = 64, BN = 64, NW = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 152;
  }
  return n;
}

struct Plan {
  int splits;
  int64_t keys_per_split;  // multiple of BN
};

Plan make_plan(int C, int Hq, int Hkv, int64_t P) {
  const int64_t L = P + C;
  const int64_t M = (int64_t)(Hq / Hkv) * C;
  const int64_t base = ((M + BM - 1) / BM) * Hkv;
  const int64_t tiles = (L + BN - 1) / BN;
  int64_t want = (2 * num_sms() + base - 1) / base;
  int64_t maxs = tiles / 2 > 0 ? tiles / 2 : 1;
  if (want > maxs) want = maxs;
  if (want < 1) want = 1;
  if (want > 64) want = 64;
  int64_t tps = (tiles + want - 1) / want;
  int splits = (int)((tiles + tps - 1) / tps);
  return Plan{splits, tps * BN};
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Element offset of (row, 16-byte chunk) in a [rows][HD] bf16 tile with an
// XOR swizzle of the chunk index (conflict-free ldmatrix).
template <int HD>
__device__ __forceinline__ int swz(int row, int chunk) {
  constexpr int NCH = HD / 8;
  int f = NCH >= 8 ? (row & 7) : ((row >> 1) & (NCH - 1));
  return row * HD + ((chunk ^ f) << 3);
}

struct AttnArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const __nv_bfloat16* kn;
  const __nv_bfloat16* vn;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;    // [splits][C][Hq][HD] fp32 (splits > 1)
  float* part_lse;  // [splits][Hq][C]
  int64_t cap, P;
  int C, Hq, Hkv, grp;
  int64_t keys_per_split;
  int splits;
  float scale_log2;
  int causal;
};

template <int HD>
__global__ void __launch_bounds__(NW * 32) attn_fwd_bf16(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sK = sQ + BM * HD;       // [2][BN][HD]
  __nv_bfloat16* sV = sK + 2 * BN * HD;   // [2][BN][HD]
  constexpr int NCH = HD / 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, split = blockIdx.z;
  const int64_t M = (int64_t)a.grp * a.C;
  const int64_t row0 = (int64_t)blockIdx.x * BM;
  const int64_t L = a.P + a.C;
  const int64_t k_begin = (int64_t)split * a.keys_per_split;
  int64_t k_end = k_begin + a.keys_per_split;
  if (k_end > L) k_end = L;
  if (a.causal) {
    // the last visible key of this row block: P + i_max
    int64_t rmax = row0 + BM - 1;
    if (rmax > M - 1) rmax = M - 1;
    int64_t lim = a.P + rmax / a.grp + 1;
    if (k_end > lim) k_end = lim;
  }

  // ---- Q tile
  for (int c = tid; c < BM * NCH; c += NW * 32) {
    int r = c / NCH, ch = c % NCH;
    int64_t R = row0 + r;
    bool ok = R < M;
    int64_t i = ok ? R / a.grp : 0, j = ok ? R % a.grp : 0;
    const __nv_bfloat16* src = a.q + ((i * a.Hq + (int64_t)g * a.grp + j) * HD + ch * 8);
    cp_async16(smem_u32(sQ + swz<HD>(r, ch)), src, ok);
  }
  auto load_kv = [&](int buf, int64_t kt0) {
    for (int c = tid; c < BN * NCH; c += NW * 32) {
      int r = c / NCH, ch = c % NCH;
      int64_t key = kt0 + r;
      bool ok = key < k_end;
      const __nv_bfloat16 *ks, *vs;
      if (!ok) {
        ks = a.kn; vs = a.vn;
      } else if (key < a.P) {
        ks = a.kc + ((int64_t)g * a.cap + key) * HD + ch * 8;
        vs = a.vc + ((int64_t)g * a.cap + key) * HD + ch * 8;
      } else {
        ks = a.kn + ((int64_t)g * a.C + (key - a.P)) * HD + ch * 8;
        vs = a.vn + ((int64_t)g * a.C + (key - a.P)) * HD + ch * 8;
      }
      cp_async16(smem_u32(sK + buf * BN * HD + swz<HD>(r, ch)), ks, ok);
      cp_async16(smem_u32(sV + buf * BN * HD + swz<HD>(r, ch)), vs, ok);
    }
  };

  const int64_t ntiles = k_end > k_begin ? (k_end - k_begin + BN - 1) / BN : 0;
  if (ntiles > 0) load_kv(0, k_begin);
  cp_async_commit();

  // per-thread rows: warp*16 + lane/4 and +8
  const int r_lo = warp * 16 + (lane >> 2);
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  int64_t qpos[2];
  for (int h2 = 0; h2 < 2; ++h2) {
    int64_t R = row0 + r_lo + h2 * 8;
    qpos[h2] = R < M ? a.P + R / a.grp : -1;  // absolute position of the query (causal mask)
  }

  uint32_t qf[HD / 16][4];
  for (int64_t t = 0; t < ntiles; ++t) {
    const int buf = (int)(t & 1);
    if (t + 1 < ntiles) load_kv(buf ^ 1, k_begin + (t + 1) * BN);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        int r = warp * 16 + (lane & 15);
        int ch = kk * 2 + (lane >> 4);
        ldsm_x4(smem_u32(sQ + swz<HD>(r, ch)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const __nv_bfloat16* cK = sK + buf * BN * HD;
    const __nv_bfloat16* cV = sV + buf * BN * HD;
    float s[BN / 8][4];
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nb = 0; nb < BN / 16; ++nb) {
        int r = nb * 16 + ((lane >> 4) << 3) + (lane & 7);
        int ch = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(cK + swz<HD>(r, ch)), b0, b1, b2, b3);
        mma_bf16(s[2 * nb], qf[kk], b0, b1);
        mma_bf16(s[2 * nb + 1], qf[kk], b2, b3);
      }
    }
    // scale, mask, online softmax (base 2)
    const int64_t kt0 = k_begin + t * BN;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int64_t key = kt0 + n * 8 + 2 * (lane & 3) + (e & 1);
        int h2 = e >> 1;
        bool vis = key < k_end && qpos[h2] >= 0 && (!a.causal || key <= qpos[h2]);
        float v = vis ? s[n][e] * a.scale_log2 : -INFINITY;
        s[n][e] = v;
        mx[h2] = fmaxf(mx[h2], v);
      }
    }
    float corr[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
      mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
      float mnew = fmaxf(m_run[h2], mx[h2]);
      float ref = mnew == -INFINITY ? 0.f : mnew;
      corr[h2] = exp2f(m_run[h2] - ref);  // exp2(-inf) = 0 on the first tile
      m_run[h2] = mnew;
      mx[h2] = ref;
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pf[BN / 16][4];
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) {
      float p0 = exp2f(s[n][0] - mx[0]), p1 = exp2f(s[n][1] - mx[0]);
      float p2 = exp2f(s[n][2] - mx[1]), p3 = exp2f(s[n][3] - mx[1]);
      rs[0] += p0 + p1;
      rs[1] += p2 + p3;
      pf[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
      pf[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      rs[h2] += __shfl_xor_sync(0xffffffffu, rs[h2], 1);
      rs[h2] += __shfl_xor_sync(0xffffffffu, rs[h2], 2);
      l_run[h2] = l_run[h2] * corr[h2] + rs[h2];
    }
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      o[n][0] *= corr[0]; o[n][1] *= corr[0];
      o[n][2] *= corr[1]; o[n][3] *= corr[1];
    }
    // O += P V  (A = P from registers: k-block kb covers keys 16kb..16kb+15)
#pragma unroll
    for (int kb = 0; kb < BN / 16; ++kb) {
      uint32_t af[4] = {pf[kb][0], pf[kb][1], pf[kb][2], pf[kb][3]};
#pragma unroll
      for (int nb = 0; nb < HD / 16; ++nb) {
        int r = kb * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int ch = nb * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(cV + swz<HD>(r, ch)), b0, b1, b2, b3);
        mma_bf16(o[2 * nb], af, b0, b1);
        mma_bf16(o[2 * nb + 1], af, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- epilogue
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    int64_t R = row0 + r_lo + h2 * 8;
    if (R >= M) continue;
    int64_t i = R / a.grp, h = (int64_t)g * a.grp + R % a.grp;
    float inv = l_run[h2] > 0.f ? 1.f / l_run[h2] : 0.f;
    float lse_v = l_run[h2] > 0.f ? (m_run[h2] + log2f(l_run[h2])) * kLn2 : -INFINITY;
    if (a.splits == 1) {
      __nv_bfloat16* dst = a.out + (i * a.Hq + h) * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        int col = n * 8 + 2 * (lane & 3);
        *reinterpret_cast<__nv_bfloat162*>(dst + col) =
            __floats2bfloat162_rn(o[n][h2 * 2] * inv, o[n][h2 * 2 + 1] * inv);
      }
      if (a.lse && (lane & 3) == 0) a.lse[h * a.C + i] = lse_v;
    } else {
      float* dst = a.part_o + (((int64_t)split * a.C + i) * a.Hq + h) * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        int col = n * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(dst + col) = make_float2(o[n][h2 * 2] * inv, o[n][h2 * 2 + 1] * inv);
      }
      if ((lane & 3) == 0) a.part_lse[((int64_t)split * a.Hq + h) * a.C + i] = lse_v;
    }
  }
}

// fp32 path: one CTA (128 threads) per (query i, head h).
__global__ void attn_fwd_f32(const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc,
                             const float* __restrict__ kn, const float* __restrict__ vn, float* __restrict__ out,
                             float* lse, int64_t cap, int64_t P, int C, int Hq, int grp, int HD, float scale,
                             int causal) {
  __shared__ float sq[128];
  __shared__ float sp[128];
  __shared__ float red[4];
  const int i = blockIdx.x, h = blockIdx.y, g = h / grp, t = threadIdx.x;
  if (t < HD) sq[t] = q[((int64_t)i * Hq + h) * HD + t];
  __syncthreads();
  int64_t L = P + C;
  if (causal) L = P + i + 1;
  float m = -INFINITY, l = 0.f, acc = 0.f;
  for (int64_t k0 = 0; k0 < L; k0 += 128) {
    int64_t key = k0 + t;
    float sc = -INFINITY;
    if (key < L) {
      const float* kr = key < P ? kc + ((int64_t)g * cap + key) * HD : kn + ((int64_t)g * C + key - P) * HD;
      float dot = 0.f;
      for (int e = 0; e < HD; ++e) dot += sq[e] * kr[e];
      sc = dot * scale;
    }
    float tm = sc;
    for (int o = 16; o; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
    if ((t & 31) == 0) red[t >> 5] = tm;
    __syncthreads();
    tm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float mnew = fmaxf(m, tm);
    float p = key < L ? expf(sc - mnew) : 0.f;
    sp[t] = p;
    float ps = p;
    for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if ((t & 31) == 0) red[t >> 5] = ps;
    __syncthreads();
    ps = red[0] + red[1] + red[2] + red[3];
    float corr = expf(m - mnew);
    l = l * corr + ps;
    if (t < HD) {
      acc *= corr;
      int64_t nk = L - k0 < 128 ? L - k0 : 128;
      for (int64_t j = 0; j < nk; ++j) {
        int64_t kk = k0 + j;
        const float* vr = kk < P ? vc + ((int64_t)g * cap + kk) * HD : vn + ((int64_t)g * C + kk - P) * HD;
        acc += sp[j] * vr[t];
      }
    }
    m = mnew;
    __syncthreads();
  }
  if (t < HD) out[((int64_t)i * Hq + h) * HD + t] = acc / l;
  if (lse && t == 0) lse[(int64_t)h * C + i] = m + logf(l);
}

}  // namespace

// Merge split partials: lse = log sum_s exp(lse_s); O = sum_s exp(lse_s - lse) O_s.
// One warp per (position, head). Every lane reads all split lse values (the
// same addresses across the warp: broadcast loads) and forms the weights
// itself, so the column loop below is a chain of independent loads.
constexpr int kMaxSplits = 64;

template <typename OutT>
__global__ void __launch_bounds__(256) attn_combine(const float* __restrict__ part_o,
                                                    const float* __restrict__ part_lse, OutT* out, float* lse, int C,
                                                    int Hq, int HD, int splits) {
  // one warp per (position, head); split weights in shared memory (lanes
  // hold splits s = lane and lane + 32)
  __shared__ float s_w[256 / 32][kMaxSplits];
  const int wib = threadIdx.x >> 5;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)C * Hq) return;
  const int64_t i = w / Hq, h = w % Hq;
  float x0 = -INFINITY, x1 = -INFINITY;
  if (lane < splits) x0 = __ldg(part_lse + ((int64_t)lane * Hq + h) * C + i);
  if (lane + 32 < splits) x1 = __ldg(part_lse + ((int64_t)(lane + 32) * Hq + h) * C + i);
  float mx = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float ref = mx == -INFINITY ? 0.f : mx;
  const float e0 = lane < splits ? __expf(x0 - ref) : 0.f;
  const float e1 = lane + 32 < splits ? __expf(x1 - ref) : 0.f;
  float tot = e0 + e1;
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  s_w[wib][lane] = e0;
  s_w[wib][lane + 32] = e1;
  __syncwarp();
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  const float* base = part_o + (i * Hq + h) * HD;
  const int64_t sstride = (int64_t)C * Hq * HD;
  for (int c = lane * 4; c < HD; c += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < splits; ++s) {
      const float ws = s_w[wib][s];
      const float4 v = __ldg(reinterpret_cast<const float4*>(base + s * sstride + c));
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    OutT* o = out + (i * Hq + h) * HD + c;
    o[0] = (OutT)(acc.x * inv);
    o[1] = (OutT)(acc.y * inv);
    o[2] = (OutT)(acc.z * inv);
    o[3] = (OutT)(acc.w * inv);
  }
  if (lse && lane == 0) lse[h * C + i] = tot > 0.f ? ref + logf(tot) : -INFINITY;
}

int attn_combine_launch(const float* part_o, const float* part_lse, __nv_bfloat16* out, float* lse, int C, int Hq,
                        int HD, int splits, cudaStream_t s) {
  const int64_t warps = (int64_t)C * Hq;
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  attn_combine<__nv_bfloat16><<<blocks, 256, 0, s>>>(part_o, part_lse, out, lse, C, Hq, HD, splits);
  DG_LAUNCH_CHECK();
  return DG_OK;
}

size_t attn_workspace(int C, int Hq, int Hkv, int hd, int64_t P, int dtype) {
  if (dtype != DG_BF16 || C < 1 || Hkv < 1 || Hq % Hkv) return 0;
  if (hd == 128) return attn_tc_workspace(C, Hq, Hkv, P);
  // Sized for make_plan's split bound (non-decreasing in P) rather than this
  // P's split count, so a workspace sized for the largest prefix serves every
  // smaller one.
  const int64_t base = ((int64_t)(Hq / Hkv) * C + BM - 1) / BM * Hkv;
  const int64_t tiles = (P + C + BN - 1) / BN;
  int64_t want = (2 * num_sms() + base - 1) / base;
  const int64_t maxs = tiles / 2 > 0 ? tiles / 2 : 1;
  if (want > maxs) want = maxs;
  if (want > 64) want = 64;
  if (want <= 1) return 0;
  size_t o = (size_t)want * C * Hq * hd * sizeof(float);
  o = (o + 255) & ~(size_t)255;
  return o + (size_t)want * Hq * C * sizeof(float);
}

int attn_launch(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t P,
                const void* k_canvas, const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv, int hd,
                float scale, int dtype, int mask, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (scale <= 0.f) scale = 1.0f / sqrtf((float)hd);
  const int grp = Hq / Hkv;
  if (dtype == DG_F32) {
    dim3 grid(C, Hq);
    attn_fwd_f32<<<grid, 128, 0, s>>>((const float*)q, (const float*)k_cache, (const float*)v_cache,
                                      (const float*)k_canvas, (const float*)v_canvas, (float*)out, lse, cap, P, C,
                                      Hq, grp, hd, scale, mask == DG_MASK_CAUSAL_BLOCK);
    DG_LAUNCH_CHECK();
    return DG_OK;
  }
  if (hd == 128)
    return attn_tc_launch(q, k_cache, v_cache, cap, P, k_canvas, v_canvas, out, lse, C, Hq, Hkv, scale, mask, ws,
                          ws_bytes, s);
  Plan pl = make_plan(C, Hq, Hkv, P);
  AttnArgs a;
  a.q = (const __nv_bfloat16*)q;
  a.kc = (const __nv_bfloat16*)k_cache;
  a.vc = (const __nv_bfloat16*)v_cache;
  a.kn = (const __nv_bfloat16*)k_canvas;
  a.vn = (const __nv_bfloat16*)v_canvas;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  a.cap = cap;
  a.P = P;
  a.C = C;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = grp;
  a.keys_per_split = pl.keys_per_split;
  a.splits = pl.splits;
  a.scale_log2 = scale * kLog2e;
  a.causal = mask == DG_MASK_CAUSAL_BLOCK;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  if (pl.splits > 1) {
    size_t o = (size_t)pl.splits * C * Hq * hd * sizeof(float);
    o = (o + 255) & ~(size_t)255;
    if (ws_bytes < o + (size_t)pl.splits * Hq * C * sizeof(float)) return DG_ERR_WORKSPACE;
    a.part_o = (float*)ws;
    a.part_lse = (float*)((char*)ws + o);
  }
  const int64_t M = (int64_t)grp * C;
  dim3 grid((unsigned)((M + BM - 1) / BM), Hkv, pl.splits);
  size_t smem = (size_t)(BM + 4 * BN) * hd * sizeof(__nv_bfloat16);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const int m32 = (BM + 4 * BN) * 32 * 2, m64 = (BM + 4 * BN) * 64 * 2, m128 = (BM + 4 * BN) * 128 * 2;
    cudaError_t e1 = cudaFuncSetAttribute(attn_fwd_bf16<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, m32);
    cudaError_t e2 = cudaFuncSetAttribute(attn_fwd_bf16<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, m64);
    cudaError_t e3 = cudaFuncSetAttribute(attn_fwd_bf16<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, m128);
    attr_err = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3);
  });
  DG_CUDA_TRY(attr_err);
  switch (hd) {
    case 32:
      attn_fwd_bf16<32><<<grid, NW * 32, smem, s>>>(a);
      break;
    case 64:
      attn_fwd_bf16<64><<<grid, NW * 32, smem, s>>>(a);
      break;
    default:
      attn_fwd_bf16<128><<<grid, NW * 32, smem, s>>>(a);
      break;
  }
  DG_LAUNCH_CHECK();
  if (pl.splits > 1) return attn_combine_launch(a.part_o, a.part_lse, a.out, lse, C, Hq, hd, pl.splits, s);
  return DG_OK;
}

}  // namespace dg
