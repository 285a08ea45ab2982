// Canvas attention on the 5th-generation tensor cores (tcgen05), bf16,
// head_dim 128: bidirectional (denoising) and causal-block (incremental
// prefill) grouped-query attention of the canvas over [cache prefix ; canvas].
//
// DiffusionGemma explainer, "Architecture: incremental prefill and
// denoising": in denoising mode every canvas query sees every canvas token
// and the KV cache; in prefill mode attention is causal.
//
// One CTA per (256 query rows = two query tiles, KV head, key split). The
// Hq/Hkv query heads of one KV head are stacked (row = position * group +
// head-in-group), so a K/V tile feeds all of them. Keys come in tiles of 128:
// first the cache rows [0, P), then the canvas rows [0, C); tiles never
// straddle the two, and the tensor maps' row extents are exactly P and C, so
// rows past the end read as zeros. K and V tiles stream through a 3-slot TMA
// ring in the order K0 K1 V0 K2 V1 ..., keys one tile ahead of values. For each key tile and each query tile q:
//   S_q = Q_q K^T   tcgen05 into TMEM (128 columns per query tile)
//   softmax         4 warps per query tile, one row per thread: one 128-column
//                   TMEM load (after which S_q may be overwritten), row max, a
//                   per-row reference kept unless a tile's max exceeds it by
//                   2^8 (then O_q and the row sum are rescaled through TMEM),
//                   P = exp2(s - ref) in bf16 into shared memory in the
//                   128-byte-swizzled K-major operand layout
//   O_q += P_q V    tcgen05, V read MN-major, O_q accumulated in TMEM.
// The MMA warp issues S0(j+1) S1(j+1) PV0(j) PV1(j): both softmax groups
// work on tile j while the tensor core computes the next scores.
// Splits write fp32 partials (O, lse) merged by attn_combine.
// Every wait is bounded (about two seconds); on expiry the CTA latches
// DG_ERR_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>

#include <mutex>

#include "dg_common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace dg {

namespace {

using namespace sm100;

constexpr int kHD = 128;
constexpr int kBM = 256;  // two query tiles of 128 rows
constexpr int kBN = 128;
constexpr int kThreads = 320;  // warp 0: TMA, warp 1: MMA, warps 2..5 / 6..9: softmax of query tile 0 / 1
constexpr int kRing = 3;       // K/V tile slots (K0 V0 K1 V1 ... in order)
constexpr uint32_t kChunk = 16384;  // [128 rows x 64 bf16] swizzled block
constexpr uint32_t kTile = 2 * kChunk;
// shared memory: Q[2] | ring[3] | P[2]
constexpr uint32_t kOffQ = 0, kOffRing = 2 * kTile, kOffP = 5 * kTile, kSmem = 7 * kTile;
constexpr float kRescale = 8.f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kTimeoutCycles = 4000000000ll;

struct TcArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int C, Hq, Hkv, grp;
  int64_t P;
  int n_cache_tiles, n_tiles, tiles_per_split, splits;
  float scale_log2;
  int causal;
  int* status;
};

struct Ctl {
  volatile int* abort;
  int* status;
};

__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*c.abort) return false;
      if (clock64() - t0 > kTimeoutCycles) {
        *c.abort = 1;
        latch(c.status, DG_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Barrier over the 128 threads of softmax group q (named barrier 1 + q) that
// ORs a predicate, so the group takes the same branch after a bounded wait.
__device__ __forceinline__ bool grp_any(int q, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.red.or.pred po, %2, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + q)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int64_t min64(int64_t x, int64_t y) { return x < y ? x : y; }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc(const __grid_constant__ CUtensorMap tk_c, const __grid_constant__ CUtensorMap tv_c,
                const __grid_constant__ CUtensorMap tk_n, const __grid_constant__ CUtensorMap tv_n, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t ring_full[kRing], ring_empty[kRing], s_full[2], s_free[2], p_full[2], p_free[2],
      drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_addr(sm);
  const int mblk = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
  const int64_t M = (int64_t)a.grp * a.C;
  Ctl ctl{&abort_flag, a.status};

  // tiles of this CTA
  int T0 = split * a.tiles_per_split;
  int T1 = min(a.n_tiles, T0 + a.tiles_per_split);
  if (a.causal) {
    int64_t rmax = min64(M - 1, (int64_t)mblk * kBM + kBM - 1);
    int64_t imax = rmax / a.grp;  // last visible key: P + imax (a canvas row)
    int last = a.n_cache_tiles + (int)(imax / kBN);
    T1 = min(T1, last + 1);
  }
  const int n = T1 > T0 ? T1 - T0 : 0;

  // Ring items in load order K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), V(n-1): keys run
  // one tile ahead of values, so the slot a key tile needs frees a whole tile early.
  // Item index of K(j): 0 for j = 0, else 2j - 1. Item index of V(j): 2j + 2, or
  // 2n - 1 for the last tile.
  auto item_tile = [&](int it, bool& is_v) -> int {
    if (it == 0) { is_v = false; return 0; }
    if (it == 2 * n - 1) { is_v = true; return n - 1; }
    if (it & 1) { is_v = false; return (it + 1) >> 1; }
    is_v = true;
    return (it >> 1) - 1;
  };
  auto k_item = [&](int jj) { return jj == 0 ? 0 : 2 * jj - 1; };
  auto v_item = [&](int jj) { return jj == n - 1 ? 2 * n - 1 : 2 * jj + 2; };
  auto issue_item = [&](int it) {
    bool is_v;
    const int jj = item_tile(it, is_v), t = T0 + jj;
    const int slot = it % kRing;
    const bool cache = t < a.n_cache_tiles;
    const int y = cache ? t * kBN : (t - a.n_cache_tiles) * kBN;
    const CUtensorMap* mp = cache ? (is_v ? &tv_c : &tk_c) : (is_v ? &tv_n : &tk_n);
    mbar_expect_tx(smem_addr(&ring_full[slot]), kTile);
    tma_load_3d(sbase + kOffRing + slot * kTile, mp, 0, y, g, smem_addr(&ring_full[slot]));
    tma_load_3d(sbase + kOffRing + slot * kTile + kChunk, mp, 64, y, g, smem_addr(&ring_full[slot]));
  };
  const int n_pre = 2 * n < kRing ? 2 * n : kRing;  // ring items issued before Q is staged

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_addr(&ring_full[s]), 1);
      mbar_init(smem_addr(&ring_empty[s]), 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_addr(&s_full[q]), 1);
      mbar_init(smem_addr(&s_free[q]), 128);
      mbar_init(smem_addr(&p_full[q]), 128);
      mbar_init(smem_addr(&p_free[q]), 1);
    }
    mbar_init(smem_addr(&drain), 1);
    fence_mbar_init();
    // start the first K/V loads now, so they overlap the Q staging below
    for (int it = 0; it < n_pre; ++it) issue_item(it);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_slot), 512);
    tmem_relinquish();
  }
  // both Q tiles -> shared memory in the swizzled K-major layout (all threads)
  for (int idx = tid; idx < kBM * 16; idx += kThreads) {
    const int r = idx >> 4, ch = idx & 15;
    const int64_t R = (int64_t)mblk * kBM + r;
    const bool ok = R < M;
    const int64_t i = ok ? R / a.grp : 0, j = ok ? R % a.grp : 0;
    const __nv_bfloat16* src = a.q + ((i * a.Hq + (int64_t)g * a.grp + j) * kHD + ch * 8);
    const int qt = r >> 7, rr = r & 127;
    const uint32_t dst = sbase + kOffQ + qt * kTile + (ch >> 3) * kChunk + rr * 128 +
                         ((((uint32_t)ch & 7u) ^ ((uint32_t)rr & 7u)) << 4);
    const int sz = ok ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz) : "memory");
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: K0 K1 V0 K2 V1 ... through a 3-slot ring
    if (lane == 0 && n > 0) {
      bool issued[kRing] = {false, false, false};
      uint32_t par[kRing] = {0, 0, 0};
      for (int it = 0; it < n_pre; ++it) issued[it] = true;  // phase 0, issued during set-up
      for (int it = n_pre; it < 2 * n; ++it) {
        const int slot = it % kRing;
        const uint32_t ph = (uint32_t)(it / kRing) & 1u;
        if (!wait_bar(smem_addr(&ring_empty[slot]), ph ^ 1u, ctl)) break;
        issue_item(it);
        issued[slot] = true;
        par[slot] = ph;
      }
      for (int s = 0; s < kRing; ++s)
        if (issued[s]) wait_bar(smem_addr(&ring_full[s]), par[s], ctl);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // order: S0(0) S1(0) | S0(1) S1(1) PV0(0) PV1(0) | S0(2) S1(2) PV0(1) PV1(1) | ...
    // Each group's next S is issued as soon as that group has loaded its current
    // S, so both softmax groups work on a tile at the same time.
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kBN, 0, 0);
      const uint32_t id_o = idesc_bf16_f32(128, kHD, 0, 1);
      auto issue_s = [&](int q, int jj) -> bool {
        const int it = k_item(jj), slot = it % kRing;
        if (!wait_bar(smem_addr(&ring_full[slot]), (uint32_t)(it / kRing) & 1u, ctl)) return false;
        if (jj > 0 && !wait_bar(smem_addr(&s_free[q]), (uint32_t)(jj - 1) & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t kb = sbase + kOffRing + slot * kTile, qb = sbase + kOffQ + q * kTile;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(qb + (kk >> 2) * kChunk + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * kChunk + (kk & 3) * 32, 0, 1024);
          mma_bf16(tmem + q * 128, ad, bd, id_s, kk > 0);
        }
        mma_commit(smem_addr(&s_full[q]));
        if (q == 1) mma_commit(smem_addr(&ring_empty[slot]));  // K(jj) consumed by both tiles
        return true;
      };
      auto issue_pv = [&](int q, int jj) -> bool {
        const int it = v_item(jj), slot = it % kRing;
        if (!wait_bar(smem_addr(&ring_full[slot]), (uint32_t)(it / kRing) & 1u, ctl)) return false;
        if (!wait_bar(smem_addr(&p_full[q]), (uint32_t)jj & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t pb = sbase + kOffP + q * kTile, vb = sbase + kOffRing + slot * kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(pb + (kk >> 2) * kChunk + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, kChunk, 1024);
          mma_bf16(tmem + 256 + q * 128, ad, bd, id_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_addr(&p_free[q]));
        if (q == 1) mma_commit(smem_addr(&ring_empty[slot]));  // V(jj) consumed by both tiles
        return true;
      };
      bool ok = issue_s(0, 0) && issue_s(1, 0);
      for (int jj = 0; jj < n && ok; ++jj) {
        if (jj + 1 < n && !(issue_s(0, jj + 1) && issue_s(1, jj + 1))) break;
        if (!issue_pv(0, jj)) break;
        if (!issue_pv(1, jj)) break;
      }
      mma_commit(smem_addr(&drain));
      wait_bar(smem_addr(&drain), 0, ctl);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue: group q owns query tile q
    const int q = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t loff = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + q * 128, tO = tmem + 256 + q * 128;
    const int64_t R = (int64_t)mblk * kBM + q * 128 + r;
    const bool row_ok = R < M;
    const int64_t i = row_ok ? R / a.grp : 0;
    const int64_t h = (int64_t)g * a.grp + (row_ok ? R % a.grp : 0);
    float ref = -INFINITY, l = 0.f;
    bool ok = true;
    int done_tiles = 0;
    for (int jj = 0; jj < n; ++jj) {
      const int t = T0 + jj;
      int lim;
      if (t < a.n_cache_tiles) {
        lim = (int)min64(kBN, a.P - (int64_t)t * kBN);
      } else {
        const int64_t c0 = (int64_t)(t - a.n_cache_tiles) * kBN;
        lim = (int)min64(kBN, a.C - c0);
        if (a.causal) lim = (int)min64(lim, i - c0 + 1);
      }
      if (!row_ok || lim < 0) lim = 0;
      const bool got = wait_bar(smem_addr(&s_full[q]), (uint32_t)jj & 1u, ctl);
      if (grp_any(q, !got)) { ok = false; break; }
      tc_fence_after();
      float v[kBN];
      tmem_ld128(tS + loff, v);  // the whole S row of this tile, one load, one wait
      tc_fence_before();
      mbar_arrive(smem_addr(&s_free[q]));  // the MMA may overwrite S now
      if (lim < kBN) {
#pragma unroll
        for (int e = 0; e < kBN; ++e)
          if (e >= lim) v[e] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = v[e];
#pragma unroll
      for (int e = 8; e < kBN; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
      float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      mt *= a.scale_log2;  // scale > 0 keeps the order
      bool need = false;
      float factor = 1.f;
      if (mt > -INFINITY) {
        if (ref == -INFINITY) {
          ref = mt;  // first visible keys of this row: O and l are still zero
        } else if (mt > ref + kRescale) {
          need = true;
          factor = exp2f(ref - mt);
          ref = mt;
          l *= factor;
        }
      }
      // P row of this tile, packed to bf16 in registers while PV(jj-1) may still run
      const float rr = ref == -INFINITY ? 0.f : ref;
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        float p8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p8[e] = ex2_approx(fmaf(v[c * 8 + e], a.scale_log2, -rr));  // exp2(-inf) = 0 for masked keys
          sum8[e] += p8[e];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[c * 4 + e] = pack2(p8[2 * e], p8[2 * e + 1]);
      }
      // PV(jj-1) must be complete both before P is overwritten and before O is rescaled
      if (jj > 0) {
        const bool pf = wait_bar(smem_addr(&p_free[q]), (uint32_t)(jj - 1) & 1u, ctl);
        if (grp_any(q, !pf)) { ok = false; break; }
        tc_fence_after();
      }
      uint8_t* prow = sm + kOffP + q * kTile + r * 128;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        const int chunk = c >> 3, piece = c & 7;
        *reinterpret_cast<uint4*>(prow + chunk * kChunk + ((piece ^ (r & 7)) << 4)) =
            make_uint4(pk[c * 4], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      // O holds every PV issued so far (waited above); rescale it before PV(jj) adds to it.
      // Done after P is formed so the S row and the O chunk are never live together.
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tO + loff + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= factor;
          tmem_st32(tO + loff + c * 32, o);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(smem_addr(&p_full[q]));
      done_tiles = jj + 1;
    }
    // epilogue
    bool have = ok && done_tiles == n && n > 0;
    if (have) {
      const bool od = wait_bar(smem_addr(&p_free[q]), (uint32_t)(n - 1) & 1u, ctl);
      have = !grp_any(q, !od);
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (ref + log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
      if (have) {
        tmem_ld32(tO + loff + c * 32, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
      if (!row_ok) continue;
      if (a.splits == 1) {
        __nv_bfloat16* dst = a.out + (i * a.Hq + h) * kHD + c * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w = make_uint4(pack2(v[e] * inv, v[e + 1] * inv), pack2(v[e + 2] * inv, v[e + 3] * inv),
                               pack2(v[e + 4] * inv, v[e + 5] * inv), pack2(v[e + 6] * inv, v[e + 7] * inv));
          *reinterpret_cast<uint4*>(dst + e) = w;
        }
      } else {
        float* dst = a.part_o + (((int64_t)split * a.C + i) * a.Hq + h) * kHD + c * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + e) = make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
      }
    }
    if (row_ok) {
      if (a.splits == 1) {
        if (a.lse) a.lse[h * a.C + i] = lse_v;
      } else {
        a.part_lse[((int64_t)split * a.Hq + h) * a.C + i] = lse_v;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// [heads][rows][128] bf16 with `rows_alloc` rows per head in memory and
// `rows` valid ones; box [1][128 rows][64 columns], 128-byte swizzle.
bool make_kv_map(CUtensorMap* m, const void* base, int64_t rows, int64_t rows_alloc, int heads) {
  const uint64_t dims[3] = {(uint64_t)kHD, (uint64_t)rows, (uint64_t)heads};
  const uint64_t strides[2] = {(uint64_t)kHD * 2, (uint64_t)rows_alloc * kHD * 2};
  const uint32_t box[3] = {64, (uint32_t)kBN, 1};
  return tmap_bf16_sw128(m, base, 3, dims, strides, box);
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 152;
  }
  return n;
}

}  // namespace

// Split plan of the tensor-core path: one wave of CTAs (one per SM).
void attn_tc_plan(int C, int Hq, int Hkv, int64_t P, int* splits, int* tiles_per_split) {
  const int64_t M = (int64_t)(Hq / Hkv) * C;
  const int64_t base = ((M + kBM - 1) / kBM) * Hkv;
  const int nct = (int)((P + kBN - 1) / kBN), nvt = (C + kBN - 1) / kBN;
  const int tiles = nct + nvt;
  static const int env_splits = [] {
    const char* v = getenv("DG_ATTN_SPLITS");  // tuning knob: force the number of key splits
    const int x = v ? atoi(v) : 0;
    return x > 0 ? x : 0;
  }();
  int want = env_splits ? env_splits : (int)(num_sms() / base);
  if (want < 1) want = 1;
  if (want > tiles) want = tiles;
  if (want > 64) want = 64;
  const int tps = (tiles + want - 1) / want;
  if (tiles_per_split) *tiles_per_split = tps;
  *splits = (tiles + tps - 1) / tps;
}

int attn_tc_launch(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t P,
                   const void* k_canvas, const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv,
                   float scale, int mask, void* ws, size_t ws_bytes, cudaStream_t s) {
  int splits, tps;
  attn_tc_plan(C, Hq, Hkv, P, &splits, &tps);
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  CUtensorMap tk_c, tv_c, tk_n, tv_n;
  memset(&tk_c, 0, sizeof(tk_c));
  memset(&tv_c, 0, sizeof(tv_c));
  if (P > 0 && (!make_kv_map(&tk_c, k_cache, P, cap, Hkv) || !make_kv_map(&tv_c, v_cache, P, cap, Hkv)))
    return DG_ERR_CUDA;
  if (!make_kv_map(&tk_n, k_canvas, C, C, Hkv) || !make_kv_map(&tv_n, v_canvas, C, C, Hkv)) return DG_ERR_CUDA;
  TcArgs a;
  a.q = (const __nv_bfloat16*)q;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  a.C = C;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = Hq / Hkv;
  a.P = P;
  a.n_cache_tiles = (int)((P + kBN - 1) / kBN);
  a.n_tiles = a.n_cache_tiles + (C + kBN - 1) / kBN;
  a.tiles_per_split = tps;
  a.splits = splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = mask == DG_MASK_CAUSAL_BLOCK;
  a.status = st;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  if (splits > 1) {
    size_t o = (size_t)splits * C * Hq * kHD * sizeof(float);
    o = (o + 255) & ~(size_t)255;
    if (ws_bytes < o + (size_t)splits * Hq * C * sizeof(float)) return DG_ERR_WORKSPACE;
    a.part_o = (float*)ws;
    a.part_lse = (float*)((char*)ws + o);
  }
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem + 1024);
  });
  DG_CUDA_TRY(attr_err);
  const int64_t M = (int64_t)a.grp * C;
  dim3 grid((unsigned)((M + kBM - 1) / kBM), Hkv, splits);
  attn_fwd_tc<<<grid, kThreads, kSmem + 1024, s>>>(tk_c, tv_c, tk_n, tv_n, a);
  DG_LAUNCH_CHECK();
  if (splits > 1) return attn_combine_launch(a.part_o, a.part_lse, a.out, lse, C, Hq, kHD, splits, s);
  return DG_OK;
}

}  // namespace dg
