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
// rows past the end read as zeros (with the prefix length read from device
// memory the cache map spans its upper bound and rows past P are masked).
// Q arrives by TMA (a 4-D map whose box is 128 stacked rows); K and V tiles
// stream through a 4-slot TMA ring in the order K0 V0 K1 V1 ...
//
// Tensor memory (512 columns): S_q / P_q at 128 q, O_q at 256 + 128 q.
// For each key tile j and query tile q:
//   S_q = Q_q K^T     tcgen05, both operands in shared memory, fp32 in TMEM
//   softmax           4 warps per query tile, one row per thread: the row's
//                     max from one 128-column TMEM load, a per-row reference
//                     kept unless a tile's max exceeds it by 2^8 (then O_q and
//                     the row sum are rescaled in TMEM), then P = exp2(s - ref)
//                     from a second read in 32-column chunks, packed to bf16
//                     and written back over the first 64 columns of S_q. The
//                     softmax is bound by instruction issue: paired fp32
//                     FMA/add (f32x2) and a three-input max keep it short
//   O_q += P_q V      tcgen05 with A = P_q read from TMEM, V MN-major in smem
// The MMA warp issues PV_0(j) S_0(j+1) PV_1(j) S_1(j+1): while one softmax
// group works, the tensor core runs the other group's two products. Keeping P
// in TMEM leaves shared-memory bandwidth to the S operands and the TMA ring.
//
// Split merge (no second kernel; the grid is one wave, every CTA resident):
// CTA k of a (row block, KV head) group merges rows
// [k*rpc, (k+1)*rpc), rpc = ceil(256/splits). Each CTA writes its normalised
// O rows (bf16) and per-row lse into the workspace slices of the CTAs that
// merge them ([split][16-byte piece][row in slice], so a warp's stores are
// contiguous per piece) and arrives on the group's counter. Once all splits
// have arrived, CTA k fetches its whole slice with one bulk copy into shared
// memory and merges it with weights exp(lse_s - lse), writing the bf16 output
// and the final lse. With a single split the staged rows are the output and
// are copied straight out.
// The group counters are zeroed by a one-CTA kernel launched just before,
// whose programmatic dependent this launch is: the attention CTAs initialise
// their barriers and allocate TMEM while it runs, then wait for it
// (griddepcontrol.wait) before they read anything from memory.
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
constexpr int kRing = 4;       // K/V tile slots (K0 V0 K1 V1 ... in order)
constexpr int kMaxSplits = 64;
constexpr uint32_t kChunk = 16384;  // [128 rows x 64 bf16] swizzled block
constexpr uint32_t kTile = 2 * kChunk;
// shared memory: Q[2] | ring[4]; after the last MMA it holds the staged O rows
constexpr uint32_t kOffQ = 0, kOffRing = 2 * kTile, kSmem = kOffRing + kRing * kTile;
constexpr uint32_t kStageRow = kHD * 2;  // bf16 O row in the merge staging area
constexpr float kRescale = 8.f;          // log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kTimeoutCycles = 4000000000ll;

struct TcArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  int C, Hq, Hkv, grp;
  int64_t P;              // cache prefix (with P_dev: its upper bound)
  const int64_t* P_dev;   // device-side prefix length, or null
  int n_cache_tiles, n_tiles, tiles_per_split, splits;
  // Partial results, per group one slice for each merging CTA k (rows [k rpc, k rpc + rpc) of the
  // group): [split][16-byte piece][row in slice] (O / l, 8 bf16 each), then [split][row in slice]
  // lse; slice_bytes apart, so a merging CTA fetches its slice with one bulk copy.
  uint8_t* part;
  int rpc;
  uint32_t slice_bytes;
  int* arrived;  // [group] splits that have published their partial (zeroed before the launch)
  float scale_log2;
  int causal;
  int q_tma;  // Q tiles by TMA (the stacked rows of 128 / group positions form one box)
  int inject;  // test injection: split 0 withholds its arrival on the merge counter
  long long wait_cycles;
  int* status;
};

struct Ctl {
  volatile int* abort;
  int* status;
  long long wait_cycles;
};

__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*c.abort) return false;
      if (clock64() - t0 > c.wait_cycles) {
        *c.abort = 1;
        latch(c.status, DG_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Drain wait for this CTA's own TMA copies / MMAs before TMEM is freed: bounded
// by time only, not cut short by the abort flag.
__device__ void drain_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 255u) == 0 && clock64() - t0 > c.wait_cycles) {
      *c.abort = 1;
      latch(c.status, DG_ERR_TIMEOUT);
      return;
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

// Byte offset of 16-byte piece p (0..15, eight bf16) of staged O row `row`:
// rows of 256 B, pieces XOR-swizzled within each 128-byte half so that a warp
// writing 32 consecutive rows hits every bank equally.
__device__ __forceinline__ uint32_t stage_off(int row, int p) {
  return (uint32_t)row * kStageRow + (uint32_t)(p & 8) * 16u + ((uint32_t)((p & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ float2 unpack2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// The group arrival counters of the next attn_fwd_tc launch -> 0. It is
// itself a programmatic dependent of whatever precedes it on the stream: it
// lets its own dependent start at once, then waits for its predecessor to
// finish before it writes. The dependent's griddepcontrol.wait returns after
// this grid has finished and its stores are visible.
__global__ void attn_zero_arrivals(int* arrived, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < n; i += blockDim.x) arrived[i] = 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc(const __grid_constant__ CUtensorMap tk_c, const __grid_constant__ CUtensorMap tv_c,
                const __grid_constant__ CUtensorMap tk_n, const __grid_constant__ CUtensorMap tv_n,
                const __grid_constant__ CUtensorMap tq, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t ring_full[kRing], ring_empty[kRing], s_full[2], p_full[2], o_full[2], q_full, drain,
      mrg_full;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float s_lse[kBM];                  // per-row lse of this CTA's partial (natural log)
  __shared__ int s_go;                          // every split of the group has published

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_addr(sm);
  const int mblk = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
  const int64_t M = (int64_t)a.grp * a.C;
  Ctl ctl{&abort_flag, a.status, a.wait_cycles};

  // set-up that touches no global memory, ahead of the wait for the counter reset
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_addr(&ring_full[s]), 1);
      mbar_init(smem_addr(&ring_empty[s]), 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_addr(&s_full[q]), 1);
      mbar_init(smem_addr(&p_full[q]), 128);
      mbar_init(smem_addr(&o_full[q]), 1);
    }
    mbar_init(smem_addr(&q_full), 1);
    mbar_init(smem_addr(&drain), 1);
    mbar_init(smem_addr(&mrg_full), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_slot), 512);
    tmem_relinquish();
  }
  // a no-op unless launched as a programmatic dependent
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // key range: the cache prefix P (from device memory when P_dev is set; the
  // tensor maps then span P_max rows, and rows past P are masked below)
  int64_t P = a.P;
  int nct = a.n_cache_tiles, ntl = a.n_tiles, tps = a.tiles_per_split;
  if (a.P_dev) {
    int64_t pd = *a.P_dev;
    if (pd < 0 || pd > a.P) {
      if (tid == 0) latch(a.status, DG_ERR_DEVICE_BOUNDS);
      pd = pd < 0 ? 0 : a.P;
    }
    P = pd;
    nct = (int)((P + kBN - 1) / kBN);
    ntl = nct + (a.C + kBN - 1) / kBN;
    tps = (ntl + a.splits - 1) / a.splits;
  }

  // tiles of this CTA
  int T0 = split * tps;
  int T1 = min(ntl, T0 + tps);
  if (a.causal) {
    int64_t rmax = min64(M - 1, (int64_t)mblk * kBM + kBM - 1);
    int64_t imax = rmax / a.grp;  // last visible key: P + imax (a canvas row)
    int last = nct + (int)(imax / kBN);
    T1 = min(T1, last + 1);
  }
  const int n = T1 > T0 ? T1 - T0 : 0;

  // ring item it: tile it / 2, K for even it, V for odd it
  auto issue_item = [&](int it) {
    const bool is_v = it & 1;
    const int t = T0 + (it >> 1);
    const int slot = it % kRing;
    const bool cache = t < nct;
    const int y = cache ? t * kBN : (t - nct) * kBN;
    const CUtensorMap* mp = cache ? (is_v ? &tv_c : &tk_c) : (is_v ? &tv_n : &tk_n);
    mbar_expect_tx(smem_addr(&ring_full[slot]), kTile);
    tma_load_3d(sbase + kOffRing + slot * kTile, mp, 0, y, g, smem_addr(&ring_full[slot]));
    tma_load_3d(sbase + kOffRing + slot * kTile + kChunk, mp, 64, y, g, smem_addr(&ring_full[slot]));
  };
  const int n_pre = 2 * n < kRing ? 2 * n : kRing;  // ring items issued before Q is staged

  if (tid == 0) {
    if (a.q_tma && n > 0) {
      // Q tile qt = stacked rows [mblk*256 + qt*128, +128) = positions
      // [that / group, + 128 / group) x every head of the group: one box per 64 columns
      mbar_expect_tx(smem_addr(&q_full), 2 * kTile);
      for (int qt = 0; qt < 2; ++qt) {
        const int i0 = (mblk * kBM + qt * 128) / a.grp;
        for (int hf = 0; hf < 2; ++hf)
          tma_load_4d(sbase + kOffQ + qt * kTile + hf * kChunk, &tq, hf * 64, 0, g, i0, smem_addr(&q_full));
      }
    }
    // start the first K/V loads now, so they overlap the set-up below
    for (int it = 0; it < n_pre; ++it) issue_item(it);
  }
  // without the Q tensor map: both Q tiles -> shared memory in the swizzled K-major layout (all threads)
  for (int idx = tid; !a.q_tma && idx < kBM * 16; idx += kThreads) {
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
    // ------------------------------------------------ TMA producer: K0 V0 K1 V1 ... through a 4-slot ring
    if (lane == 0 && n > 0) {
      bool issued[kRing] = {false, false, false, false};
      uint32_t par[kRing] = {0, 0, 0, 0};
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
        if (issued[s]) drain_bar(smem_addr(&ring_full[s]), par[s], ctl);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) PV1(1) S1(2) | ...
    // S_q(j+1) overwrites the TMEM columns PV_q(j) reads P from; the tensor
    // core runs one thread's MMAs in issue order. Each s_full commit also
    // covers PV_q(j), so the softmax may rescale O_q as soon as S_q(j+1) lands.
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kBN, 0, 0);
      const uint32_t id_o = idesc_bf16_f32(128, kHD, 0, 1);
      auto item_ready = [&](int it) -> bool {
        return wait_bar(smem_addr(&ring_full[it % kRing]), (uint32_t)(it / kRing) & 1u, ctl);
      };
      auto mma_s = [&](int q, int slot) {
        const uint32_t kb = sbase + kOffRing + slot * kTile, qb = sbase + kOffQ + q * kTile;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(qb + (kk >> 2) * kChunk + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * kChunk + (kk & 3) * 32, 0, 1024);
          mma_bf16(tmem + q * 128, ad, bd, id_s, kk > 0);
        }
      };
      auto mma_pv = [&](int q, int slot, bool acc) {
        const uint32_t vb = sbase + kOffRing + slot * kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, kChunk, 1024);
          mma_bf16_ts(tmem + 256 + q * 128, tmem + q * 128 + kk * 8, bd, id_o, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = item_ready(0) && (!a.q_tma || wait_bar(smem_addr(&q_full), 0, ctl));
      if (ok) {
        mma_s(0, 0);
        mma_commit(smem_addr(&s_full[0]));
        mma_s(1, 0);
        mma_commit(smem_addr(&s_full[1]));
        mma_commit(smem_addr(&ring_empty[0]));  // K(0) consumed
      }
      for (int jj = 0; jj < n && ok; ++jj) {
        const int it_v = 2 * jj + 1, it_k = 2 * jj + 2;
        const int sv = it_v % kRing, sk = it_k % kRing;
        const bool more = jj + 1 < n;
        if (!item_ready(it_v)) break;
        if (!wait_bar(smem_addr(&p_full[0]), (uint32_t)jj & 1u, ctl)) break;
        tc_fence_after();
        mma_pv(0, sv, jj > 0);
        if (more) {
          if (!item_ready(it_k)) break;
          mma_s(0, sk);
          mma_commit(smem_addr(&s_full[0]));
        } else {
          mma_commit(smem_addr(&o_full[0]));
        }
        if (!wait_bar(smem_addr(&p_full[1]), (uint32_t)jj & 1u, ctl)) break;
        tc_fence_after();
        mma_pv(1, sv, jj > 0);
        mma_commit(smem_addr(&ring_empty[sv]));  // V(jj) consumed
        if (more) {
          mma_s(1, sk);
          mma_commit(smem_addr(&s_full[1]));
          mma_commit(smem_addr(&ring_empty[sk]));  // K(jj+1) consumed
        } else {
          mma_commit(smem_addr(&o_full[1]));
        }
      }
      mma_commit(smem_addr(&drain));
      drain_bar(smem_addr(&drain), 0, ctl);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue: group q owns query tile q
    const int q = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int rt = q * 128 + r;  // row within the CTA's 256
    const uint32_t loff = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + q * 128, tO = tmem + 256 + q * 128;
    const int64_t R = (int64_t)mblk * kBM + rt;
    const bool row_ok = R < M;
    const int64_t i = row_ok ? R / a.grp : 0;
    float ref = -INFINITY, l = 0.f;
    bool ok = true;
    int done_tiles = 0;
    for (int jj = 0; jj < n; ++jj) {
      const int t = T0 + jj;
      int lim;
      if (t < nct) {
        lim = (int)min64(kBN, P - (int64_t)t * kBN);
      } else {
        const int64_t c0 = (int64_t)(t - nct) * kBN;
        lim = (int)min64(kBN, a.C - c0);
        if (a.causal) lim = (int)min64(lim, i - c0 + 1);
      }
      if (!row_ok || lim < 0) lim = 0;
      const bool got = wait_bar(smem_addr(&s_full[q]), (uint32_t)jj & 1u, ctl);
      if (grp_any(q, !got)) { ok = false; break; }
      tc_fence_after();
      // The S row is read twice: all 128 columns for the row max (one load),
      // whose first 64 values then give the first half of P = exp2(s - ref);
      // the second half is read again (64 columns). P is packed to bf16x2 and
      // written over the first 64 columns of S_q, 16 at a time: P columns
      // [32h, 32h + 32) overwrite S elements [32h, 32h + 32), already read.
      float v[kBN];
      tmem_ld128(tS + loff, v);
      if (lim < kBN) {
#pragma unroll
        for (int e = 0; e < kBN; ++e)
          if (e >= lim) v[e] = -INFINITY;
      }
      float mx;
      {
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(v[e], v[120 + e]);
#pragma unroll
        for (int b = 8; b < 120; b += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = max3(m8[e], v[b + e], v[b + 8 + e]);
        mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      }
      const float mt = mx * a.scale_log2;  // scale > 0 keeps the order
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
      // O_q holds every PV_q issued so far (complete: covered by this tile's
      // s_full commit); rescale it before PV_q(jj) adds to it.
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
      const float rr = ref == -INFINITY ? 0.f : ref;
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
      const float sl2 = a.scale_log2, nrr = -rr;
      auto p_half = [&](const float* s64, int hf) {  // 64 S values -> 32 P columns
#pragma unroll
        for (int qt = 0; qt < 2; ++qt) {
          uint32_t pk[16];
#pragma unroll
          for (int g = 0; g < 16; ++g) {  // element pair (2g, 2g + 1) of the quarter
            float x0, x1;
            fma2(x0, x1, s64[qt * 32 + 2 * g], s64[qt * 32 + 2 * g + 1], sl2, sl2, nrr, nrr);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);  // exp2(-inf) = 0 for masked keys
            add2(sum8[2 * (g & 3)], sum8[2 * (g & 3) + 1], p0, p1);
            pk[g] = pack2(p0, p1);
          }
          tmem_st16_async(tS + loff + hf * 32 + qt * 16, pk);
        }
      };
      p_half(v, 0);
      {
        float s64[64];
        tmem_ld64(tS + loff + 64, s64);
        if (lim < kBN) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (64 + e >= lim) s64[e] = -INFINITY;
        }
        p_half(s64, 1);
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_addr(&p_full[q]));
      done_tiles = jj + 1;
    }
    // epilogue: O_q / l in bf16 and the row's lse. Several splits: written
    // straight to this split's slot of the workspace, piece-major ([16-byte
    // piece][row], so each warp store is 512 contiguous bytes). One split:
    // staged over the dead Q tiles (every S product is complete once
    // o_full[0] fires) for a coalesced copy to the output.
    bool have = ok && done_tiles == n && n > 0;
    if (have) {
      const bool od = wait_bar(smem_addr(&o_full[q]), 0, ctl);
      have = !grp_any(q, !od);
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = (have && l > 0.f) ? (ref + log2f(l)) * kLn2 : -INFINITY;
    float o[kHD];
    if (have) {
      tmem_ld128(tO + loff, o);
    } else {
#pragma unroll
      for (int e = 0; e < kHD; ++e) o[e] = 0.f;
    }
    // several splits: this row's pieces go to the slice of the CTA that merges it
    const int ks = rt / a.rpc, rs = rt % a.rpc;
    uint8_t* slice = a.splits > 1
                         ? a.part + ((size_t)(g * gridDim.x + mblk) * a.splits + ks) * a.slice_bytes
                         : nullptr;
    uint4* po = slice ? reinterpret_cast<uint4*>(slice) + (size_t)split * 16 * a.rpc + rs : nullptr;
#pragma unroll
    for (int pc = 0; pc < kHD / 8; ++pc) {
      const float* x = o + pc * 8;
      const uint4 w = make_uint4(pack2(x[0] * inv, x[1] * inv), pack2(x[2] * inv, x[3] * inv),
                                 pack2(x[4] * inv, x[5] * inv), pack2(x[6] * inv, x[7] * inv));
      if (po)
        po[pc * a.rpc] = w;
      else
        *reinterpret_cast<uint4*>(sm + stage_off(rt, pc)) = w;
    }
    const float lse_row = row_ok ? lse_v : -INFINITY;
    if (po) {
      reinterpret_cast<float*>(slice + (size_t)a.splits * 16 * a.rpc * 16)[split * a.rpc + rs] = lse_row;
      // this split's rows, before the arrival below (ordered by the barrier); the merging CTA reads
      // them with a bulk copy
      fence_proxy_async_global();
    } else {
      s_lse[rt] = lse_row;
    }
  }
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------ publish this split's partial, then merge
  const int grp_id = g * gridDim.x + mblk;
  const int cs = a.splits;
  constexpr int kRowPieces = kHD / 8;  // 16-byte pieces of a row
  bool merge = false;
  if (cs == 1) {
    // one split: the staged rows are the output (bf16 O / l); coalesced copy-out
    for (int item = tid; item < kBM * kRowPieces; item += kThreads) {
      const int row = item / kRowPieces, pc = item % kRowPieces;
      const int64_t R = (int64_t)mblk * kBM + row;
      if (R >= M) continue;
      const int64_t i = R / a.grp, h = (int64_t)g * a.grp + R % a.grp;
      *reinterpret_cast<uint4*>(a.out + (i * a.Hq + h) * kHD + pc * 8) =
          *reinterpret_cast<const uint4*>(sm + stage_off(row, pc));
      if (pc == 0 && a.lse) a.lse[h * a.C + i] = s_lse[row];
    }
  } else {
    if (tid == 0) {
      if (!(a.inject && split == 0)) red_release_add_gpu(a.arrived + grp_id, 1);
      bool go = true;
      const long long t0 = clock64();
      while ((int)ld_acquire_gpu(a.arrived + grp_id) < cs) {
        if (abort_flag || clock64() - t0 > a.wait_cycles) {
          latch(a.status, DG_ERR_TIMEOUT);
          go = false;
          break;
        }
        __nanosleep(32);
      }
      if (go) {
        // this CTA's slice of every split's rows -> shared memory (the ring area; every MMA has
        // completed), one bulk copy (async proxy, after the acquire above)
        fence_proxy_async_global();
        const uint8_t* src = a.part + ((size_t)grp_id * cs + split) * a.slice_bytes;
        mbar_expect_tx(smem_addr(&mrg_full), a.slice_bytes);
        bulk_load(sbase + kOffRing, src, a.slice_bytes, smem_addr(&mrg_full));
      }
      s_go = go;
    }
    __syncthreads();
    merge = s_go;
    if (merge) {
      const bool got = wait_bar(smem_addr(&mrg_full), 0, ctl);
      merge = __syncthreads_and(got);
    }
  }
  if (merge) {
    // Rows [r0, r0 + nr) of the group are merged by this CTA from its slice in shared memory, two
    // 16-byte pieces (16 columns) per item: the lse values and pieces of every split, combined with
    // weights exp(lse_s - max) (an online rescale joins batches of 9 splits).
    constexpr int kBatch = 9;
    constexpr int kItemsPerRow = kRowPieces / 2;
    const int rpc = a.rpc;
    const int r0 = split * rpc;
    const int nr = max(0, min(kBM, r0 + rpc) - r0);
    const uint4* pg = reinterpret_cast<const uint4*>(sm + kOffRing);  // [split][piece][row in slice]
    const float* pl = reinterpret_cast<const float*>(sm + kOffRing + (size_t)cs * 16 * rpc * 16);
    for (int item = tid; item < nr * kItemsPerRow; item += kThreads) {
      const int t = item / kItemsPerRow, pc = (item % kItemsPerRow) * 2;
      const int row = r0 + t;
      const int64_t R = (int64_t)mblk * kBM + row;
      if (R >= M) continue;
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
      float m = -INFINITY, tot = 0.f;
      for (int s0 = 0; s0 < cs; s0 += kBatch) {
        float lv[kBatch];
        uint4 x0[kBatch], x1[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          lv[u] = -INFINITY;
          if (s0 + u < cs) {
            const uint4* src0 = pg + ((size_t)(s0 + u) * 16 + pc) * rpc + t;
            lv[u] = pl[(s0 + u) * rpc + t];
            x0[u] = src0[0];
            x1[u] = src0[rpc];
          }
        }
        float bm = m;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, lv[u]);
        if (bm == -INFINITY) continue;
        const float f = __expf(m - bm);  // 0 while m = -inf
        tot *= f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] *= f;
        m = bm;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (s0 + u < cs && lv[u] > -INFINITY) {
            const float w = __expf(lv[u] - m);
            tot += w;
            const uint32_t wd[8] = {x0[u].x, x0[u].y, x0[u].z, x0[u].w, x1[u].x, x1[u].y, x1[u].z, x1[u].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 fv = unpack2(wd[e]);
              acc[2 * e] = fmaf(w, fv.x, acc[2 * e]);
              acc[2 * e + 1] = fmaf(w, fv.y, acc[2 * e + 1]);
            }
          }
        }
      }
      const float it = tot > 0.f ? 1.f / tot : 0.f;
      const int64_t i = R / a.grp, h = (int64_t)g * a.grp + R % a.grp;
      uint4* dst = reinterpret_cast<uint4*>(a.out + (i * a.Hq + h) * kHD + pc * 8);
      dst[0] = make_uint4(pack2(acc[0] * it, acc[1] * it), pack2(acc[2] * it, acc[3] * it),
                          pack2(acc[4] * it, acc[5] * it), pack2(acc[6] * it, acc[7] * it));
      dst[1] = make_uint4(pack2(acc[8] * it, acc[9] * it), pack2(acc[10] * it, acc[11] * it),
                          pack2(acc[12] * it, acc[13] * it), pack2(acc[14] * it, acc[15] * it));
      if (pc == 0 && a.lse) a.lse[h * a.C + i] = tot > 0.f ? m + logf(tot) : -INFINITY;
    }
  }
  // the bulk copy, if issued, has landed (bounded: nothing of this CTA in flight at exit)
  if (cs > 1 && tid == 0 && s_go) drain_bar(smem_addr(&mrg_full), 0, ctl);
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

// q [C][Hq][128] bf16 viewed as [C][Hkv][group][128]: box [128 / group positions]
// [1 KV head][group heads][64 columns], so one box is 128 stacked rows
// (position-major, head-in-group minor) of one KV head's queries.
bool make_q_map(CUtensorMap* m, const void* q, int C, int Hq, int Hkv) {
  const int grp = Hq / Hkv;
  const uint64_t dims[4] = {(uint64_t)kHD, (uint64_t)grp, (uint64_t)Hkv, (uint64_t)C};
  const uint64_t strides[3] = {(uint64_t)kHD * 2, (uint64_t)grp * kHD * 2, (uint64_t)Hq * kHD * 2};
  const uint32_t box[4] = {64, (uint32_t)grp, 1, (uint32_t)(128 / grp)};
  return tmap_bf16_sw128(m, q, 4, dims, strides, box);
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

// Kernel attribute (dynamic shared memory), set once.
cudaError_t prepare_kernel() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(attn_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem + 1024);
  });
  return err;
}

}  // namespace

// Split plan of the tensor-core path: one wave of CTAs, one per SM (the
// splits of a group wait for one another, so the grid must fit on the GPU at once).
namespace {
int key_tiles(int C, int64_t P) { return (int)((P + kBN - 1) / kBN) + (C + kBN - 1) / kBN; }

// Upper bound of the key splits for prefix P: non-decreasing in P, so a
// workspace sized for the largest prefix also serves every smaller one.
int max_splits(int C, int Hq, int Hkv, int64_t P) {
  const int64_t M = (int64_t)(Hq / Hkv) * C;
  const int64_t base = ((M + kBM - 1) / kBM) * Hkv;
  int want = (int)(num_sms() / base);
  const int tiles = key_tiles(C, P);
  if (want > tiles) want = tiles;
  if (want > kMaxSplits) want = kMaxSplits;
  return want < 1 ? 1 : want;
}
}  // namespace

void attn_tc_plan(int C, int Hq, int Hkv, int64_t P, int* splits, int* tiles_per_split) {
  const int tiles = key_tiles(C, P);
  const int want = max_splits(C, Hq, Hkv, P);
  const int tps = (tiles + want - 1) / want;
  if (tiles_per_split) *tiles_per_split = tps;
  *splits = (tiles + tps - 1) / tps;
}

// Workspace: one arrival counter per (row block, KV head) group (zeroed before
// each launch), then per group one slice per merging CTA ([split][16-byte
// piece][row in slice] O rows, then [split][row in slice] lse).
struct TcLayout {
  size_t counters, part, total;
  int64_t groups;
  int rpc;
  uint32_t slice_bytes;
};
uint32_t slice_bytes(int splits, int rpc) {
  return (uint32_t)(((size_t)splits * 16 * rpc * 16 + (size_t)splits * rpc * sizeof(float) + 15) & ~(size_t)15);
}
TcLayout tc_layout(int C, int Hq, int Hkv, int splits) {
  TcLayout L;
  const int64_t M = (int64_t)(Hq / Hkv) * C;
  L.groups = ((M + kBM - 1) / kBM) * Hkv;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.rpc = (kBM + splits - 1) / splits;
  L.slice_bytes = slice_bytes(splits, L.rpc);
  L.counters = 0;
  L.part = L.counters + al((size_t)L.groups * sizeof(int));
  L.total = splits > 1 ? L.part + al((size_t)L.groups * splits * L.slice_bytes) : 0;  // one split: nothing
  return L;
}

// Sized for every split count up to the plan's bound (non-decreasing in P), so a workspace sized
// for the largest prefix serves every smaller one.
size_t attn_tc_workspace(int C, int Hq, int Hkv, int64_t P) {
  if (C < 1 || Hkv < 1 || Hq % Hkv) return 0;
  size_t need = 0;
  for (int sp = 2; sp <= max_splits(C, Hq, Hkv, P); ++sp) {
    const size_t t = tc_layout(C, Hq, Hkv, sp).total;
    if (t > need) need = t;
  }
  return need;
}

int attn_tc_launch(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t P,
                   const void* k_canvas, const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv,
                   float scale, int mask, void* ws, size_t ws_bytes, cudaStream_t s, const int64_t* P_dev) {
  DG_CUDA_TRY(prepare_kernel());
  int splits, tps;
  attn_tc_plan(C, Hq, Hkv, P, &splits, &tps);
  const TcLayout L = tc_layout(C, Hq, Hkv, splits);
  if (splits > 1 && (!ws || ws_bytes < L.total || ((uintptr_t)ws & 255u))) return DG_ERR_WORKSPACE;
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  CUtensorMap tk_c, tv_c, tk_n, tv_n;
  memset(&tk_c, 0, sizeof(tk_c));
  memset(&tv_c, 0, sizeof(tv_c));
  if (P > 0 && (!make_kv_map(&tk_c, k_cache, P, cap, Hkv) || !make_kv_map(&tv_c, v_cache, P, cap, Hkv)))
    return DG_ERR_CUDA;
  if (!make_kv_map(&tk_n, k_canvas, C, C, Hkv) || !make_kv_map(&tv_n, v_canvas, C, C, Hkv)) return DG_ERR_CUDA;
  const int grp = Hq / Hkv;
  CUtensorMap tq;
  memset(&tq, 0, sizeof(tq));
  const bool q_tma = 128 % grp == 0 && make_q_map(&tq, q, C, Hq, Hkv);
  TcArgs a;
  a.q = (const __nv_bfloat16*)q;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  a.C = C;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = Hq / Hkv;
  a.P = P;
  a.P_dev = P_dev;
  a.n_cache_tiles = (int)((P + kBN - 1) / kBN);
  a.n_tiles = a.n_cache_tiles + (C + kBN - 1) / kBN;
  a.tiles_per_split = tps;
  a.splits = splits;
  a.part = splits > 1 ? (uint8_t*)ws + L.part : nullptr;
  a.rpc = L.rpc;
  a.slice_bytes = L.slice_bytes;
  a.arrived = splits > 1 ? (int*)((char*)ws + L.counters) : nullptr;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = mask == DG_MASK_CAUSAL_BLOCK;
  a.q_tma = q_tma;
  const Inject inj = take_inject(kInjectAttnArrival);
  a.inject = inj.kind != kInjectNone && splits > 1;
  a.wait_cycles = inj.wait_cycles > 0 ? inj.wait_cycles : kTimeoutCycles;
  a.status = st;
  const int64_t M = (int64_t)a.grp * C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + kBM - 1) / kBM), Hkv, splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem + 1024;
  cfg.stream = s;
  // Several splits meet on a counter, so every CTA must be resident: the grid
  // is one CTA per SM at most and every wait is bounded. By default the
  // counters are zeroed by attn_zero_arrivals and this launch is its
  // programmatic dependent (17.0 vs 20.0 us per call measured at 16q/8kv
  // heads, P = 4096, back to back; no change at P = 1024 or 32768).
  // attn_fwd_tc itself does not release its dependents early: a following
  // vocabulary step whose CTAs were placed while attention still held the SMs
  // ran slower (the whole step -2.5%). DG_ATTN_COOP=1 selects
  // a stream-ordered memset and a cooperative launch instead, which adds the
  // driver's guarantee of co-scheduling next to other work on the device.
  // Either way the counters start at zero on every call
  // (dg_canvas_attn_noalloc relies on this: its shared scratch keeps the
  // previous call's counts).
  static const bool coop = [] {
    const char* v = getenv("DG_ATTN_COOP");
    return v && v[0] == '1' && v[1] == 0;
  }();
  cudaLaunchAttribute at[1];
  if (coop) {
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
  } else {
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = at;
  cfg.numAttrs = splits > 1 ? 1 : 0;
  if (splits > 1) {
    if (coop) {
      DG_CUDA_TRY(cudaMemsetAsync(a.arrived, 0, (size_t)L.groups * sizeof(int), s));
    } else {
      cudaLaunchConfig_t zc = {};
      zc.gridDim = dim3(1);
      zc.blockDim = dim3(64);
      zc.stream = s;
      zc.attrs = at;  // programmatic dependent of the previous work on the stream as well
      zc.numAttrs = 1;
      DG_CUDA_TRY(cudaLaunchKernelEx(&zc, attn_zero_arrivals, a.arrived, (int)L.groups));
    }
  }
  DG_CUDA_TRY(cudaLaunchKernelEx(&cfg, attn_fwd_tc, tk_c, tv_c, tk_n, tv_n, tq, a));
  return DG_OK;
}

}  // namespace dg
