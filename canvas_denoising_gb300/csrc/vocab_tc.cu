// The fused vocabulary step on the 5th-generation tensor cores (tcgen05).
//
// What it computes (DiffusionGemma explainer, "Self-conditioning" and
// "2. Uniform-state diffusion"): for every canvas row i of H,
//   l_i = H_i E^T, p_i = softmax(l_i), argmax_i, conf_i = max p_i,
//   lse_i = log sum exp l_i, S_i = p_i E.
// The fp32 logits never reach memory: the softmax numerators exp(l - R) go
// in bf16 through a global ring (V x 512 bytes) to the CTAs that form S. E
// is streamed from HBM once for the logits; the S product reads each E tile
// again shortly after, from L2 where most of it is still resident (at V =
// 262144, d = 2816: 1.71 GB of DRAM reads per call for a 1.48 GB table).
//
// Design.
//  * Fixed per-row reference. softmax(l) = exp(l - R) / sum exp(l - R) for
//    any R. Each row gets one reference R_i shared by the whole grid, so
//    every P tile exp(l - R_i) is final the moment its logits exist: P.E
//    and the row sums accumulate linearly in any order, with no rescaling
//    of accumulators. R_i is the maximum over a sample of the vocabulary
//    (every producer's first tile, agreed on through one grid-wide count).
//    A row whose true maximum exceeds R_i + 40 (exp would leave the safe
//    fp32 range) is flagged and recomputed exactly by the combine kernel
//    with R = its true maximum.
//  * Two roles, all co-resident (one CTA per SM, the grid sized from the
//    device's occupancy; vocab_main by cooperative launch):
//    - producers make vocabulary tiles of 256 ids (round robin). GEMM1:
//      logits[rows x 256] = H . E_tile^T, K-loop over d in steps of 64
//      through a TMA ring. Eight epilogue warps read the logits from TMEM,
//      keep per-row running max / first argmax / sum of exp(l - R), and
//      write P = exp(l - R) in bf16 to a global ring, already in the
//      128-byte-swizzled K-major layout an MMA operand needs, then publish
//      the tile with a release flag. (Paired form: each warp assembles its
//      rows in a 4 KB shared-memory stage, so the ring is written in whole
//      128-byte lines.)
//    - consumers own a slice of S's columns and a residue class of
//      vocabulary tiles. GEMM2: S_slice += P_tile . E_tile[:, slice] with E
//      read MN-major (the rows producers just streamed, mostly from L2),
//      accumulating in TMEM over the whole vocabulary. Their fp32 partials
//      go to the workspace once, at the end.
//  * Two forms of those roles:
//    - vocab_pair (default): CTA pairs (clusters of two, cta_group::2). One
//      MMA of M = 256 spans the pair, so each SM reads half of the wide
//      operand from shared memory and holds 128 rows of the accumulator;
//      the producer accumulator is double-buffered in TMEM.
//    - vocab_main: one CTA per role unit (cta_group::1), M = 128 MMAs for
//      each row half; used where two-CTA clusters cannot be placed.
//  * A combine kernel merges producer statistics (max, lowest argmax, sums)
//    and consumer partials into argmax, conf, lse and S (bf16). After the
//    paired form it is a programmatic dependent launch.
//  * Cross-CTA hand-offs (reference count, tile flags): the CTA's threads
//    write, meet at a barrier, and one thread publishes with a release
//    add; the barrier orders the others' writes before that release, as in
//    a cooperative grid sync. One thread polls, with acquire loads, and a
//    barrier passes the outcome to the rest of the CTA.
// Every wait is bounded (about two seconds of clock); on expiry the kernel
// latches DG_ERR_TIMEOUT, raises a grid-wide abort flag, drains its own
// copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "dg_common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace dg {
namespace {

using namespace sm100;

constexpr int kStages = 3;
constexpr int kBK = 64;            // d elements per producer k-step (one 128-byte swizzle row)
constexpr int kVT = 256;           // vocabulary ids per tile
constexpr int kDT = 256;           // S columns per consumer CTA
constexpr int kThreads = 320;      // warp 0: TMA, warp 1: MMA, warps 2..9: epilogue
constexpr int kEpiThreads = 256;
constexpr uint32_t kStageBytes = 64u * 1024u;
constexpr uint32_t kEBytesA = 32768u;  // producer E block [256 ids x 64 d]
constexpr uint32_t kTileBytes = 16384u;  // [128 rows x 64 bf16], one swizzled operand block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 40.f;       // overflow margin above the reference, natural log
constexpr long long kTimeoutCycles = 4000000000ll;

struct Plan {
  int n_rh, n_dt, n_vt, ksplit, n_a, n_c;
};

// Optional integer override from the environment (tuning knobs, read once).
int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  long x = strtol(v, &end, 10);
  return (end && *end == 0 && x > 0 && x < (1 << 30)) ? (int)x : dflt;
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

Plan make_plan(int C, int V, int d) {
  Plan p;
  p.n_rh = (C + 127) / 128;
  p.n_dt = (d + kDT - 1) / kDT;
  p.n_vt = (V + kVT - 1) / kVT;
  const int sms = num_sms();
  const int tiles_c = p.n_dt;  // a consumer CTA covers every row for its d-slice
  int ks = (int)lround((double)(sms / 2) / tiles_c);
  if (ks < 1) ks = 1;
  if (ks > p.n_vt) ks = p.n_vt;
  while (ks > 1 && tiles_c * ks > sms - 1) --ks;
  p.ksplit = ks;
  p.n_c = tiles_c * ks;
  p.n_a = sms - p.n_c;
  if (p.n_a > p.n_vt) p.n_a = p.n_vt;
  if (p.n_a < 1) p.n_a = 1;
  return p;
}

struct Layout {
  size_t flags, smax, am, aa, az, cpart, pbuf, total;
  size_t flag_bytes;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t tile_words(int n_vt) { return ((size_t)n_vt + 3) / 4; }
constexpr size_t kFlagFixed = 4 + 4 + 256 + 1024;  // reference count, abort, overflow, row keys

Layout make_layout(const Plan& p, int d) {
  Layout L;
  size_t o = 0;
  L.flags = o;
  // Flags, zeroed before each launch (bytes): tile published counts [n_vt] (a byte per tile in
  // 32-bit words), reference count, abort, overflow [256] (a byte per row), row keys [256] (u32),
  // then the pacing counts [n_vt] (bytes in words; zeroed only when pacing is on). Kept small:
  // the one-CTA reset kernel writes them, and in the cooperative forms a memset of up to 4096
  // bytes costs ~1.2 us back to back, a larger one ~4.1 us.
  L.flag_bytes = 2 * tile_words(p.n_vt) * 4 + kFlagFixed;
  o += up256(L.flag_bytes);
  L.smax = o; o += up256((size_t)p.n_a * 256 * 4);
  L.am = o;   o += up256((size_t)p.n_a * 256 * 4);
  L.aa = o;   o += up256((size_t)p.n_a * 256 * 4);
  L.az = o;   o += up256((size_t)p.n_a * 256 * 4);
  L.cpart = o; o += up256((size_t)p.ksplit * 256 * d * 4);
  L.pbuf = o; o += (size_t)p.n_vt * 4 * p.n_rh * kTileBytes;
  L.total = o;
  return L;
}

struct Params {
  int C, V, d, n_rh, n_dt, n_vt, ksplit, n_a;
  unsigned* ready;  // tile published counts: tile t in byte t & 3 of word t >> 2
  int* ref_count;  // producers that have published their sample maxima
  int* abort_flag;
  uint8_t* overflow;  // [256]
  unsigned* rowkey;  // [256] paired form: running max of the sample, order-preserving key (0 = none)
  float* smax;     // [256][n_a] sample maxima (vocab_main; the paired form has rowkey)
  float* am;       // [256][n_a] running max
  int* aa;         // [256][n_a] first argmax
  float* az;       // [256][n_a] sum of exp(l - R)
  float* cpart;    // [ksplit][256][d]
  uint8_t* pbuf;   // [n_vt][4 sub-tiles of 64 ids][n_rh][16 KB]
  // optional fused threshold re-noise (tokens == nullptr: off)
  int32_t* rn_tokens;
  uint8_t* rn_flags;
  float rn_threshold;
  uint64_t rn_seed;
  uint32_t rn_step;
  int64_t rn_pos0;
  const int64_t* rn_pos0_dev;  // device-side position offset (or null)
  int inject;                  // test injection: tile 0's ready flag is never released
  long long wait_cycles;       // bound of every wait
  int* status;
  // paired form only: producer pairs, and the consumer pairs' d-slicing
  // (n_full slices of cw = 256 columns, then a remainder of `rem` columns; see consumer_slice)
  int n_pa, n_pc, n_full, rem, n_fullx, cw;
  int ring_bytes;  // paired form: operand ring per CTA (a multiple of 32 KB)
  // paired form, produce phase: consumer pair ci makes tile cb + ci in the first round; producer
  // pair a makes tile a, then pb + a + (j-1) n_pa for j >= 1 while below pe
  int cb, pb, pe;
  // paired form, pacing (lead > 0): a producer pair starts tile t (after its first) once the
  // consumer CTAs of tile t - lead have issued its loads (consumed[t - lead] == cons_per_tile), or
  // after pace_cycles: a soft wait that keeps the consumers' E re-reads within L2
  unsigned* consumed;  // tile t's count in byte t & 3 of word t >> 2
  int lead, cons_per_tile;
  long long pace_cycles;
};

__device__ __forceinline__ bool aborted(const int* f) { return *(volatile const int*)f != 0; }

__device__ __forceinline__ void raise_abort(const Params& p) {
  atomicExch(p.abort_flag, 1);
  latch(p.status, DG_ERR_TIMEOUT);
}

// Bounded mbarrier wait: false on timeout (abort raised) or if another CTA aborted.
__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Params& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (aborted(p.abort_flag)) return false;
      if (clock64() - t0 > p.wait_cycles) {
        raise_abort(p);
        return false;
      }
    }
  }
}

// Drain wait for this CTA's own TMA copies / MMAs before it frees TMEM or
// exits: bounded by time only (not cut short by an abort, so nothing of this
// CTA is in flight when it leaves); copies and MMAs already issued complete
// on their own.
__device__ void drain_bar(uint32_t bar, uint32_t parity, const Params& p) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 255u) == 0 && clock64() - t0 > p.wait_cycles) {
      raise_abort(p);
      return;
    }
  }
}

// Bounded wait until *flag >= target (acquire).
__device__ bool wait_flag(const int* flag, int target, const Params& p) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if ((int)ld_acquire_gpu(flag) >= target) return true;
    if (aborted(p.abort_flag)) return false;
    if (clock64() - t0 > p.wait_cycles) {
      raise_abort(p);
      return false;
    }
    __nanosleep(64);
  }
}

// Byte-per-tile counts in 32-bit words (every count stays below 256, and the word-wide adds below
// 2^31, so lanes never carry into each other).
__device__ __forceinline__ int tile_count(unsigned word, int t) { return (int)((word >> (8 * (t & 3))) & 0xffu); }
__device__ __forceinline__ void tile_add_release(unsigned* w, int t) {
  // word and lane computed inside the asm, where the compiler cannot hoist them into the loops
  asm volatile(
      "{\n .reg .u32 sh, v;\n .reg .u64 off, a;\n"
      " and.b32 sh, %1, 3;\n shl.b32 sh, sh, 3;\n shl.b32 v, 1, sh;\n"
      " shr.s32 sh, %1, 2;\n mul.wide.s32 off, sh, 4;\n add.u64 a, %0, off;\n"
      " red.release.gpu.global.add.u32 [a], v;\n}"
      ::"l"(w), "r"(t)
      : "memory");
}
// Bounded acquire wait until tile t's count reaches target. An acquire that reads a later add to
// the same word (another tile's) still synchronizes with this tile's release: adds extend the
// release sequence.
__device__ bool wait_tile(const unsigned* w, int t, int target, const Params& p) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (tile_count(ld_acquire_gpu(reinterpret_cast<const int*>(w + (t >> 2))), t) >= target) return true;
    if (aborted(p.abort_flag)) return false;
    if (clock64() - t0 > p.wait_cycles) {
      raise_abort(p);
      return false;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Barrier over the 256 epilogue threads that also ORs a predicate across them,
// so that every epilogue thread takes the same branch after a bounded wait.
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.red.or.pred po, 1, 256, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    vocab_main(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_ek,
               const __grid_constant__ CUtensorMap tm_emn, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages], bar_tfull, bar_tempty, bar_drain;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stages = (uint8_t*)(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
  const uint32_t s_base = smem_addr(stages);
  const bool is_a = (int)blockIdx.x < p.n_a;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bar_full[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
    }
    mbar_init(smem_addr(&bar_tfull), 1);
    mbar_init(smem_addr(&bar_tempty), kEpiThreads);
    mbar_init(smem_addr(&bar_drain), 1);
    fence_mbar_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_ek);
    prefetch_tmap(&tm_emn);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ksteps_d = p.d / kBK;

  if (is_a) {
    // ===================================================== producer role: GEMM1 + softmax epilogue
    const int a = blockIdx.x;
    const int n_my = a < p.n_vt ? (p.n_vt - a + p.n_a - 1) / p.n_a : 0;
    if (warp == 0) {
      if (lane == 0 && n_my > 0) {
        int stage = 0;
        uint32_t ph = 0;
        uint32_t issued_par[kStages];
        bool issued[kStages];
        for (int s = 0; s < kStages; ++s) issued[s] = false, issued_par[s] = 0;
        const uint32_t tx = (uint32_t)p.n_rh * kTileBytes + kEBytesA;
        const uint64_t pol_last = policy_evict_last();
        bool ok = true;
        for (int j = 0; j < n_my && ok; ++j) {
          const int t = a + j * p.n_a;
          for (int ks = 0; ks < ksteps_d; ++ks) {
            if (!wait_bar(smem_addr(&bar_empty[stage]), ph ^ 1, p)) { ok = false; break; }
            const uint32_t fb = smem_addr(&bar_full[stage]);
            const uint32_t sb = s_base + stage * kStageBytes;
            mbar_expect_tx(fb, tx);
            for (int h = 0; h < p.n_rh; ++h)
              tma_load_2d_hint(sb + h * kTileBytes, &tm_h, ks * kBK, h * 128, fb, pol_last);
            tma_load_2d_hint(sb + 2 * kTileBytes, &tm_ek, ks * kBK, t * kVT, fb, pol_last);
            issued[stage] = true;
            issued_par[stage] = ph;
            if (++stage == kStages) { stage = 0; ph ^= 1; }
          }
        }
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) drain_bar(smem_addr(&bar_full[s]), issued_par[s], p);
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0 && n_my > 0) {
        const uint32_t idesc = idesc_bf16_f32(128, kVT, 0, 0);
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; j < n_my && ok; ++j) {
          // single accumulator: the epilogue must have drained the previous tile
          if (!wait_bar(smem_addr(&bar_tempty), (uint32_t)(j & 1) ^ 1u, p)) break;
          tc_fence_after();
          for (int ks = 0; ks < ksteps_d; ++ks) {
            if (!wait_bar(smem_addr(&bar_full[stage]), ph, p)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sb = s_base + stage * kStageBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint64_t bdesc = sdesc_sw128(sb + 2 * kTileBytes + k * 32, 0, 1024);
              for (int h = 0; h < p.n_rh; ++h) {
                const uint64_t adesc = sdesc_sw128(sb + h * kTileBytes + k * 32, 0, 1024);
                mma_bf16(tmem + h * 256, adesc, bdesc, idesc, (ks | k) != 0);
              }
            }
            mma_commit(smem_addr(&bar_empty[stage]));
            if (++stage == kStages) { stage = 0; ph ^= 1; }
          }
          if (ok) mma_commit(smem_addr(&bar_tfull));
        }
        mma_commit(smem_addr(&bar_drain));
        drain_bar(smem_addr(&bar_drain), 0, p);
      }
      __syncwarp();
    } else {
      // epilogue warps 2..9: row half hh = (warp-2)/4, TMEM lane quarter q = warp % 4
      const int hh = (warp - 2) >> 2;
      const int q = warp & 3;
      const int r = q * 32 + lane;
      const int i = hh * 128 + r;
      const bool active = hh < p.n_rh;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + hh * 256;
      float R2 = 0.f, lim2 = 0.f;
      float m_run = -INFINITY, z_run = 0.f;
      int a_run = 0x7fffffff;
      bool ovf = false;
      bool ok = true;
      if (n_my == 0) {
        p.smax[(size_t)i * p.n_a + a] = -INFINITY;
        __threadfence();
        epi_sync();
        if (threadIdx.x == 64) red_release_add_gpu(p.ref_count, 1);
      }
      for (int j = 0; j < n_my && ok; ++j) {
        const int t = a + j * p.n_a;
        const bool got = wait_bar(smem_addr(&bar_tfull), (uint32_t)j & 1u, p);
        if (epi_any(!got)) { ok = false; break; }
        tc_fence_after();
        if (j == 0) {
          // sample maxima of this CTA's first tile -> grid-wide reference
          float mx = -INFINITY;
          if (active) {
            for (int c = 0; c < kVT / 128; ++c) {
              float v[128];
              tmem_ld128(taddr + c * 128, v);
              const int vb = t * kVT + c * 128;
#pragma unroll
              for (int e = 0; e < 128; ++e)
                if (vb + e < p.V) mx = fmaxf(mx, v[e]);
            }
          }
          p.smax[(size_t)i * p.n_a + a] = mx;
          __threadfence();
          epi_sync();
          if (threadIdx.x == 64) red_release_add_gpu(p.ref_count, 1);
          const bool refd = wait_flag(p.ref_count, p.n_a, p);
          if (epi_any(!refd)) { ok = false; break; }
          float R = -INFINITY;
          const float* sm_row = p.smax + (size_t)i * p.n_a;
          for (int aa = 0; aa < p.n_a; ++aa) R = fmaxf(R, __ldcg(sm_row + aa));
          R2 = R * kLog2e;
          lim2 = (R + kTau) * kLog2e;
        }
        if (!active) {
          tc_fence_before();
          mbar_arrive(smem_addr(&bar_tempty));
        }
        for (int c = 0; active && c < kVT / 128; ++c) {
          float v[128];
          tmem_ld128(taddr + c * 128, v);
          if (c == kVT / 128 - 1) {
            // every logit of this tile is in registers: hand TMEM back to the MMA warp now
            tc_fence_before();
            mbar_arrive(smem_addr(&bar_tempty));
          }
          const int vb = t * kVT + c * 128;
          if (vb + 128 > p.V) {
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (vb + e >= p.V) v[e] = -INFINITY;
          }
          // chunk max with 8 independent accumulators; the index is searched only
          // when the chunk beats the running max (first index attaining it)
          float bm[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) bm[e] = fmaxf(v[e], v[120 + e]);
#pragma unroll
          for (int b = 8; b < 120; b += 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) bm[e] = max3(bm[e], v[b + e], v[b + 8 + e]);
          const float cm = max3(max3(bm[0], bm[1], bm[2]), max3(bm[3], bm[4], bm[5]), fmaxf(bm[6], bm[7]));
          if (cm > m_run) {
            int ci = 127;
#pragma unroll
            for (int e = 127; e >= 0; --e)
              if (v[e] == cm) ci = e;
            m_run = cm;
            a_run = vb + ci;
          }
          if (cm * kLog2e > lim2) ovf = true;
          float zs[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) zs[e] = 0.f;
          uint8_t* prow = p.pbuf + ((size_t)((t * 4 + c * 2) * p.n_rh + hh)) * kTileBytes + (size_t)r * 128;
#pragma unroll
          for (int e8 = 0; e8 < 16; ++e8) {
            float pe[8];
#pragma unroll
            for (int f = 0; f < 8; f += 2) {  // paired fp32 instructions: the epilogue is issue-bound
              float x0, x1;
              fma2(x0, x1, v[e8 * 8 + f], v[e8 * 8 + f + 1], kLog2e, kLog2e, -R2, -R2);
              pe[f] = ex2_approx(x0);  // masked ids: exp2(-inf) = 0
              pe[f + 1] = ex2_approx(x1);
              add2(zs[f], zs[f + 1], pe[f], pe[f + 1]);
            }
            const int sub = e8 >> 3, piece = e8 & 7;
            uint8_t* dst = prow + (size_t)sub * p.n_rh * kTileBytes + ((piece ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) =
                make_uint4(pack2(pe[0], pe[1]), pack2(pe[2], pe[3]), pack2(pe[4], pe[5]), pack2(pe[6], pe[7]));
          }
          z_run += ((zs[0] + zs[1]) + (zs[2] + zs[3])) + ((zs[4] + zs[5]) + (zs[6] + zs[7]));
        }
        // publish the P tile to consumer CTAs (generic writes -> async-proxy reads elsewhere)
        fence_proxy_async_global();
        __threadfence();
        epi_sync();
        if (threadIdx.x == 64 && !(p.inject && t == 0)) tile_add_release(p.ready, t);
      }
      if (active && i < p.C) {
        p.am[(size_t)i * p.n_a + a] = m_run;
        p.aa[(size_t)i * p.n_a + a] = a_run;
        p.az[(size_t)i * p.n_a + a] = z_run;
        if (ovf) p.overflow[i] = 1;
      }
    }
  } else {
    // ===================================================== consumer role: GEMM2 (S += P . E)
    const int c = blockIdx.x - p.n_a;
    const int tau = c % p.n_dt;
    const int kap = c / p.n_dt;
    const int d0 = tau * kDT;
    const int nd = p.d - d0 < kDT ? p.d - d0 : kDT;
    const int nbox = nd / 64;
    const int n_my = kap < p.n_vt ? (p.n_vt - kap + p.ksplit - 1) / p.ksplit : 0;
    if (warp == 0) {
      if (lane == 0 && n_my > 0) {
        int stage = 0;
        uint32_t ph = 0;
        uint32_t issued_par[kStages];
        bool issued[kStages];
        for (int s = 0; s < kStages; ++s) issued[s] = false, issued_par[s] = 0;
        const uint32_t pbytes = (uint32_t)p.n_rh * kTileBytes;
        const uint32_t tx = pbytes + (uint32_t)nbox * 8192u;
        const uint64_t pol_first = policy_evict_first();
        bool ok = true;
        for (int j = 0; j < n_my && ok; ++j) {
          const int t = kap + j * p.ksplit;
          if (!wait_tile(p.ready, t, 1, p)) break;
          fence_proxy_async_global();
          for (int ks = 0; ks < kVT / 64; ++ks) {
            if (!wait_bar(smem_addr(&bar_empty[stage]), ph ^ 1, p)) { ok = false; break; }
            const uint32_t fb = smem_addr(&bar_full[stage]);
            const uint32_t sb = s_base + stage * kStageBytes;
            mbar_expect_tx(fb, tx);
            bulk_load_hint(sb, p.pbuf + (size_t)((t * 4 + ks) * p.n_rh) * kTileBytes, pbytes, fb, pol_first);
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d_hint(sb + 2 * kTileBytes + bx * 8192, &tm_emn, d0 + bx * 64, t * kVT + ks * 64, fb,
                               pol_first);
            issued[stage] = true;
            issued_par[stage] = ph;
            if (++stage == kStages) { stage = 0; ph ^= 1; }
          }
        }
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) drain_bar(smem_addr(&bar_full[s]), issued_par[s], p);
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0 && n_my > 0) {
        const uint32_t idesc = idesc_bf16_f32(128, nd, 0, 1);
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; j < n_my && ok; ++j) {
          for (int ks = 0; ks < kVT / 64; ++ks) {
            if (!wait_bar(smem_addr(&bar_full[stage]), ph, p)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sb = s_base + stage * kStageBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bdesc = sdesc_sw128(sb + 2 * kTileBytes + k * 2048, 8192, 1024);
              const uint32_t acc = (j | ks | k) != 0 ? 1u : 0u;
              for (int h = 0; h < p.n_rh; ++h) {
                const uint64_t adesc = sdesc_sw128(sb + h * kTileBytes + k * 32, 0, 1024);
                mma_bf16(tmem + h * 256, adesc, bdesc, idesc, acc);
              }
            }
            mma_commit(smem_addr(&bar_empty[stage]));
            if (++stage == kStages) { stage = 0; ph ^= 1; }
          }
        }
        mma_commit(smem_addr(&bar_tfull));
        drain_bar(smem_addr(&bar_tfull), 0, p);
      }
      __syncwarp();
    } else {
      const int hh = (warp - 2) >> 2;
      const int q = warp & 3;
      const int r = q * 32 + lane;
      const int i = hh * 128 + r;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + hh * 256;
      float* dst = p.cpart + ((size_t)kap * 256 + i) * p.d + d0;
      bool have = n_my > 0 && hh < p.n_rh;
      if (n_my > 0) {
        bool got = wait_bar(smem_addr(&bar_tfull), 0, p);
        got = __all_sync(0xffffffffu, got);  // tcgen05.ld below is warp-collective
        have = have && got;
        tc_fence_after();
      }
      for (int cc = 0; cc < nd / 32; ++cc) {
        float v[32];
        if (have) {
          tmem_ld32(taddr + cc * 32, v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (i < p.C) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + cc * 32 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
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

// ============================================================================ paired form
// The same two roles on CTA pairs (clusters of two, cta_group::2). One MMA of
// M = 256 covers all canvas rows: each CTA of the pair holds 128 rows of the A
// operand and half of the B operand's columns, so per unit of work each SM
// reads half as much B from shared memory as in vocab_main, and each CTA's
// accumulator holds only its own 128 rows.
//  * Producer pair: tile t of 256 ids; CTA r loads H rows [128r, 128r+128)
//    and E ids [256t + 128r, +128) per 64-deep k-step (32 KB per stage, six
//    stages). Its accumulator, 128 rows x 256 ids, is 256 TMEM columns, so
//    two buffers fit: the epilogue of tile j overlaps the MMAs of tile j+1.
//    Epilogue warp w reads one 128-id half (hc) of its row in one load and
//    keeps statistics per (pair, hc) slot.
//  * Consumer pair: a d-slice of 256 columns (one MMA of N = 256, each CTA
//    holding half of N) and one residue class of tiles; the pairs of a
//    narrow remainder slice take two residue classes each, so that every
//    consumer pair carries about the same work.
//  * First round: every pair, consumer pairs included, produces one tile
//    before anything is published, so consumers are not idle at the start;
//    a consumer pair then switches to GEMM2, reusing the ring with barriers
//    of its own once its GEMM1 MMAs have completed. For large vocabularies
//    the consumer pairs' first-round tiles are the last ones of the
//    vocabulary (consumed last), so that the consumers start with a backlog
//    of one producer wave instead of a whole round (see prod_tile).
// Loads of both CTAs complete on the even CTA's "full" barrier (it alone
// issues MMAs); commits arrive on both CTAs' barriers.
constexpr int kRingBytes = 196608;   // operand ring per CTA (6 producer stages; 7 measured no faster)
constexpr int kMaxRing = 6;
constexpr uint32_t kStageA2 = 32768u;  // producer stage per CTA: H [128 x 64] + E [128 ids x 64]
constexpr int kEpiWarps = 8;
// Per epilogue warp, after the ring: 32 rows x 128 bytes. The warp builds a 4 KB block of P
// (or 32 rows x 32 fp32 columns of its S partial) there and writes it to global memory in whole
// lines. With each thread storing its own row (16-byte pieces 128 bytes apart across the warp)
// a producer tile's exp-and-store pass took 3.3 instead of 2.3 us and the S partials 5 instead of
// 3.5 us (V = 32768, d = 1024: 55.5 against 52.9 us per call).
constexpr int kEpiStage = 4096;

// d-slice and residue classes of consumer pair c: n_fullx slices per residue
// class ra (n_full of cw columns, then possibly the remainder); pairs past
// ksplit * n_fullx serve a narrow remainder slice (rem <= cw/2 columns, next
// to full slices) for residues ra and rb = ra + 1 (rb = -1: none).
__device__ __forceinline__ void consumer_slice(const Params& p, int c, int& d0, int& nd, int& ra, int& rb) {
  const int n_res = p.ksplit * p.n_fullx;
  if (c < n_res) {
    const int sl = c % p.n_fullx;
    ra = c / p.n_fullx;
    rb = -1;
    d0 = sl * p.cw;
    nd = sl < p.n_full ? p.cw : p.rem;
  } else {
    const int h = c - n_res;
    ra = 2 * h;
    rb = 2 * h + 1 < p.ksplit ? 2 * h + 1 : -1;
    d0 = p.n_full * p.cw;
    nd = p.rem;
  }
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key; every
// key of a float is above 0, the key the workspace starts from).
__device__ __forceinline__ unsigned order_key(float x) {
  const unsigned b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ void red_max_u32(unsigned* a, unsigned v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// j-th tile a pair produces. Every pair takes part in the first round: producer
// pair a makes tile a, consumer pair ci tile cb + ci; producer pairs then
// continue with every n_pa-th tile from pb + a (below pe).
__device__ __forceinline__ int prod_tile(const Params& p, int pair, int j) {
  if (pair >= p.n_pa) return p.cb + (pair - p.n_pa);
  return j == 0 ? pair : p.pb + pair + (j - 1) * p.n_pa;
}


// u-th tile of a consumer pair (ascending; may exceed n_vt, which callers skip).
__device__ __forceinline__ int consumer_tile(int u, int ra, int rb, int ks) {
  return rb < 0 ? ra + u * ks : (u >> 1) * ks + ((u & 1) ? rb : ra);
}


// The flag words of the next vocab_pair launch -> 0. It is itself a
// programmatic dependent of whatever precedes it on the stream: it lets its
// own dependent start at once, then waits for its predecessor to finish
// before it writes. The dependent's griddepcontrol.wait returns after this
// grid has finished and its stores are visible.
__global__ void vocab_zero_flags(uint32_t* f, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < n; i += blockDim.x) f[i] = 0u;
}

__global__ void __launch_bounds__(kThreads, 1)
    vocab_pair(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_ek,
               const __grid_constant__ CUtensorMap tm_emn, const __grid_constant__ CUtensorMap tm_p, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  // ring barriers of the produce phase (full/empty) and of the consume phase (full2/empty2)
  __shared__ __align__(8) uint64_t bar_full[kMaxRing], bar_empty[kMaxRing], bar_full2[kMaxRing], bar_empty2[kMaxRing];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = (uint8_t*)(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
  const uint32_t s_base = smem_addr(ring);
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)(blockIdx.x >> 1);
  const bool is_a = pair < p.n_pa;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(smem_addr(&bar_full[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
      mbar_init(smem_addr(&bar_full2[s]), 1);
      mbar_init(smem_addr(&bar_empty2[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&bar_tfull[b]), 1);
      mbar_init(smem_addr(&bar_tempty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_addr(&bar_drain), 1);
    fence_mbar_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_ek);
    prefetch_tmap(&tm_emn);
    prefetch_tmap(&tm_p);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&tmem_slot), 512);
    tmem_relinquish_pair();
  }
  // the combine kernel may be scheduled from now on (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // nothing above reads global memory; below, the flags must be zero (a no-op unless launched as
  // the programmatic dependent of vocab_zero_flags)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int NP = p.n_pa + p.n_pc;
  const int ksteps_d = p.d / kBK;
  const int n_stages_a = p.ring_bytes / (int)kStageA2;
  // Produce phase (every pair takes part in the first round, see prod_tile).
  int n_prod;
  if (is_a) {
    n_prod = pair < p.n_vt ? 1 : 0;
    if (p.pb + pair < p.pe) n_prod += (p.pe - p.pb - pair + p.n_pa - 1) / p.n_pa;
  } else {
    n_prod = p.cb + (pair - p.n_pa) < p.n_vt ? 1 : 0;
  }
  // Consume phase (consumer pairs): a d-slice and residue class(es) of tiles.
  int d0 = 0, nd = 256, ra = 0, rb = -1;
  if (!is_a) consumer_slice(p, pair - p.n_pa, d0, nd, ra, rb);
  const int N0 = nd <= 128 ? 128 : 256;                          // MMA width of the slice
  const uint32_t stage_c = 16384u + (uint32_t)(N0 / 128) * 8192u;  // P block + E block
  const int n_stages_c = p.ring_bytes / (int)stage_c < kMaxRing ? p.ring_bytes / (int)stage_c : kMaxRing;
  const int cnt_a = !is_a && ra < p.n_vt ? (p.n_vt - ra + p.ksplit - 1) / p.ksplit : 0;
  const int cnt_b = !is_a && rb >= 0 && rb < p.n_vt ? (p.n_vt - rb + p.ksplit - 1) / p.ksplit : 0;
  const int n_iter = rb < 0 ? cnt_a : 2 * cnt_a;
  const int n_cons = cnt_a + cnt_b;

  if (warp == 0) {
    // ===================================================== TMA issue (both CTAs)
    if (lane == 0) {
      bool ok = true;
      if (n_prod > 0) {
        // L2 policies (measured: 0.540 ms with, 0.563 ms without at V = 262144): H and the producers'
        // E rows evict_last; P and the consumers' E rows evict_first
        const uint64_t pol_h = policy_evict_last(), pol_e = policy_evict_last();
        int stage = 0;
        uint32_t ph = 0;
        for (int j = 0; j < n_prod && ok; ++j) {
          const int t = prod_tile(p, pair, j);
          if (j > 0 && p.lead > 0 && t - p.lead >= 0) {
            const long long t0 = clock64();  // soft: never an error, only a delay of at most pace_cycles
            const int tl = t - p.lead;
            while (tile_count(*(volatile const unsigned*)(p.consumed + (tl >> 2)), tl) < p.cons_per_tile &&
                   !aborted(p.abort_flag) && clock64() - t0 < p.pace_cycles)
              __nanosleep(256);
          }
          for (int ks = 0; ks < ksteps_d; ++ks) {
            if (!wait_bar(smem_addr(&bar_empty[stage]), ph ^ 1, p)) { ok = false; break; }
            const uint32_t fb = smem_addr(&bar_full[stage]);
            const uint32_t fl = mapa_shared(fb, 0);
            const uint32_t sb = s_base + stage * kStageA2;
            if (leader) mbar_expect_tx(fb, 2 * kStageA2);
            tma_load_2d_pair_hint(sb, &tm_h, ks * kBK, (int)rank * 128, fl, pol_h);
            tma_load_2d_pair_hint(sb + 16384, &tm_ek, ks * kBK, t * kVT + (int)rank * 128, fl, pol_e);
            if (++stage == n_stages_a) { stage = 0; ph ^= 1; }
          }
        }
      }
      if (ok && n_cons > 0) {
        // the ring is reused with its own barriers: the produce phase's MMAs must have read it
        if (n_prod > 0 && !wait_bar(smem_addr(&bar_tfull[0]), 0, p)) ok = false;
        const uint64_t pol_p = policy_evict_first(), pol_e = policy_evict_first();
        int stage = 0;
        uint32_t ph = 0;
        for (int u = 0; u < n_iter && ok; ++u) {
          const int t = consumer_tile(u, ra, rb, p.ksplit);
          if (t >= p.n_vt) continue;
          if (!wait_tile(p.ready, t, 2, p)) break;
          fence_proxy_async_global();
          for (int ks = 0; ks < kVT / 64; ++ks) {
            if (!wait_bar(smem_addr(&bar_empty2[stage]), ph ^ 1, p)) { ok = false; break; }
            const uint32_t fb = smem_addr(&bar_full2[stage]);
            const uint32_t fl = mapa_shared(fb, 0);
            const uint32_t sb = s_base + stage * stage_c;
            if (leader) mbar_expect_tx(fb, 2 * stage_c);
            tma_load_2d_pair_hint(sb, &tm_p, 0, ((t * 4 + ks) * 2 + (int)rank) * 128, fl, pol_p);
            for (int bx = 0; bx < N0 / 128; ++bx)
              tma_load_2d_pair_hint(sb + 16384 + bx * 8192, &tm_emn, d0 + (int)rank * (N0 / 2) + bx * 64,
                                    t * kVT + ks * 64, fl, pol_e);
            if (++stage == n_stages_c) { stage = 0; ph ^= 1; }
          }
          if (ok && p.lead > 0)  // pacing hint for the producers
            red_add_relaxed_gpu(reinterpret_cast<int*>(p.consumed + (t >> 2)), 1 << (8 * (t & 3)));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================================================== MMA issue (even CTA)
    if (leader && lane == 0) {
      bool ok = true;
      if (n_prod > 0) {
        // GEMM1: logits of a tile into accumulator j & 1 (128 rows x 256 ids per CTA)
        const uint32_t idesc = idesc_bf16_f32(256, kVT, 0, 0);
        int stage = 0;
        uint32_t ph = 0;
        for (int j = 0; j < n_prod && ok; ++j) {
          const int b = j & 1;
          // accumulator b must have been read out (tile j-2) by both CTAs' epilogues
          if (!wait_bar(smem_addr(&bar_tempty[b]), ((uint32_t)(j >> 1) & 1u) ^ 1u, p)) { ok = false; break; }
          tc_fence_after();
          for (int ks = 0; ks < ksteps_d; ++ks) {
            if (!wait_bar(smem_addr(&bar_full[stage]), ph, p)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sb = s_base + stage * kStageA2;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_pair(tmem + b * 256, sdesc_sw128(sb + k * 32, 0, 1024), sdesc_sw128(sb + 16384 + k * 32, 0, 1024),
                            idesc, (ks | k) != 0);
            mma_commit_pair_mc(smem_addr(&bar_empty[stage]), 3);
            if (++stage == n_stages_a) { stage = 0; ph ^= 1; }
          }
          if (ok) mma_commit_pair_mc(smem_addr(&bar_tfull[b]), 3);
        }
      }
      if (ok && n_cons > 0) {
        // GEMM2: S_slice += P . E into the accumulator at column 0, over buffer 0 of the produce
        // phase: both CTAs' epilogues must have read that tile's logits
        if (n_prod > 0 && !wait_bar(smem_addr(&bar_tempty[0]), 0, p)) ok = false;
        tc_fence_after();
        const uint32_t id0 = idesc_bf16_f32(256, N0, 0, 1);
        int stage = 0;
        uint32_t ph = 0;
        bool first = true;
        for (int u = 0; u < n_iter && ok; ++u) {
          const int t = consumer_tile(u, ra, rb, p.ksplit);
          if (t >= p.n_vt) continue;
          for (int ks = 0; ks < kVT / 64; ++ks) {
            if (!wait_bar(smem_addr(&bar_full2[stage]), ph, p)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sb = s_base + stage * stage_c;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = (first && ks == 0 && k == 0) ? 0u : 1u;
              const uint64_t adesc = sdesc_sw128(sb + k * 32, 0, 1024);
              mma_bf16_pair(tmem, adesc, sdesc_sw128(sb + 16384 + k * 2048, 8192, 1024), id0, acc);
            }
            mma_commit_pair_mc(smem_addr(&bar_empty2[stage]), 3);
            if (++stage == n_stages_c) { stage = 0; ph ^= 1; }
          }
          first = false;
        }
        mma_commit_pair_mc(smem_addr(&bar_tfull[1]), 3);
      }
      if (n_prod > 0 || n_cons > 0) {
        mma_commit_pair_mc(smem_addr(&bar_drain), 1);
        drain_bar(smem_addr(&bar_drain), 0, p);
      }
    }
    __syncwarp();
  } else {
    // ===================================================== epilogue warps 2..9
    // Produce phase: id half hc of the tile, TMEM lane quarter q; one row per thread.
    const int hc = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row within this CTA's half = TMEM lane
    const int i = (int)rank * 128 + r;
    const int slot = pair * 2 + hc;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + hc * 128;
    uint8_t* stg = ring + p.ring_bytes + (warp - 2) * kEpiStage;  // this warp's 4 KB stage
    float R2 = 0.f, lim2 = 0.f;
    float m_run = -INFINITY, z_run = 0.f;
    int a_run = 0x7fffffff;
    bool ovf = false;
    bool ok = true;
    if (n_prod == 0) {
      epi_sync();
      if (threadIdx.x == 64) red_release_add_gpu(p.ref_count, 1);
    }
    for (int j = 0; j < n_prod && ok; ++j) {
      const int t = prod_tile(p, pair, j);
      const int b = j & 1;
      const bool got = wait_bar(smem_addr(&bar_tfull[b]), (uint32_t)(j >> 1) & 1u, p);
      if (epi_any(!got)) { ok = false; break; }
      tc_fence_after();
      float v[128];
      tmem_ld128(tl + b * 256, v);
      // every logit of this half-tile is in registers: hand the buffer back
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(&bar_tempty[b]), 0));
      const int vb = t * kVT + hc * 128;
      if (vb + 128 > p.V) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (vb + e >= p.V) v[e] = -INFINITY;
      }
      float bm[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) bm[e] = fmaxf(v[e], v[120 + e]);
#pragma unroll
      for (int bb = 8; bb < 120; bb += 16)
#pragma unroll
        for (int e = 0; e < 8; ++e) bm[e] = max3(bm[e], v[bb + e], v[bb + 8 + e]);
      const float cm = max3(max3(bm[0], bm[1], bm[2]), max3(bm[3], bm[4], bm[5]), fmaxf(bm[6], bm[7]));
      if (j == 0) {
        // this slot's first half-tile is its sample -> grid-wide reference: one
        // atomic max per row, read back once every CTA has contributed
        red_max_u32(p.rowkey + i, order_key(cm));
        // the barrier orders every thread's contribution before thread 64's release; thread 64
        // alone polls for the other CTAs' and the barrier below passes the outcome on
        epi_sync();
        bool refd = true;
        if (threadIdx.x == 64) {
          red_release_add_gpu(p.ref_count, 1);
          refd = wait_flag(p.ref_count, 2 * NP, p);
        }
        if (epi_any(!refd)) { ok = false; break; }
        const float R = from_order_key(__ldcg(p.rowkey + i));
        R2 = R * kLog2e;
        lim2 = (R + kTau) * kLog2e;
      }
      if (cm > m_run) {
        int ci = 127;
#pragma unroll
        for (int e = 127; e >= 0; --e)
          if (v[e] == cm) ci = e;
        m_run = cm;
        a_run = vb + ci;
      }
      if (cm * kLog2e > lim2) ovf = true;
      float zs[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) zs[e] = 0.f;
      // P blocks [t][sub-tile of 64 ids][row half = rank], pre-swizzled K-major. The warp's 32
      // rows of a block are 4 KB of contiguous memory: each row's 128 bytes are built in the
      // warp's shared-memory stage in their final (swizzled) order, then the 4 KB go out in
      // 512-byte coalesced stores.
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
#pragma unroll
        for (int piece = 0; piece < 8; ++piece) {
          const int e8 = sub * 8 + piece;
          float pe[8];
#pragma unroll
          for (int f = 0; f < 8; f += 2) {
            float x0, x1;
            fma2(x0, x1, v[e8 * 8 + f], v[e8 * 8 + f + 1], kLog2e, kLog2e, -R2, -R2);
            pe[f] = ex2_approx(x0);  // masked ids: exp2(-inf) = 0
            pe[f + 1] = ex2_approx(x1);
            add2(zs[f], zs[f + 1], pe[f], pe[f + 1]);
          }
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((piece ^ (lane & 7)) << 4)) =
              make_uint4(pack2(pe[0], pe[1]), pack2(pe[2], pe[3]), pack2(pe[4], pe[5]), pack2(pe[6], pe[7]));
        }
        __syncwarp();
        uint8_t* blk = p.pbuf + ((size_t)((t * 4 + hc * 2 + sub) * 2 + (int)rank)) * kTileBytes + (size_t)q * 4096;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(blk + k * 512 + lane * 16) =
              *reinterpret_cast<const uint4*>(stg + k * 512 + lane * 16);
        __syncwarp();
      }
      z_run += ((zs[0] + zs[1]) + (zs[2] + zs[3])) + ((zs[4] + zs[5]) + (zs[6] + zs[7]));
      // publish this CTA's half of the P tile (consumers wait for both halves)
      fence_proxy_async_global();
      epi_sync();
      if (threadIdx.x == 64 && !(p.inject && t == 0)) tile_add_release(p.ready, t);
    }
    if (i < p.C) {
      p.am[(size_t)i * p.n_a + slot] = m_run;
      p.aa[(size_t)i * p.n_a + slot] = a_run;
      p.az[(size_t)i * p.n_a + slot] = z_run;
      if (ovf) p.overflow[i] = 1;
    }
    // Consume phase: the warps of id half hc read columns [hc N0/2, (hc + 1) N0/2) of the
    // accumulator for their lane quarter.
    if (!is_a) {
      bool have = n_cons > 0 && ok;
      if (n_cons > 0) {
        bool got = wait_bar(smem_addr(&bar_tfull[1]), 0, p);
        got = __all_sync(0xffffffffu, got);  // tcgen05.ld below is warp-collective
        have = have && got;
        tc_fence_after();
      }
      have = __all_sync(0xffffffffu, have);
      const int cend = d0 + nd;
      // Each thread holds 32 columns of its row; through the warp's stage, 8 lanes then
      // write each row's 128 bytes together (4 rows per store instruction).
      const int rr0 = lane >> 3, pc = lane & 7;
      for (int cc = hc * (N0 / 64); cc < (hc + 1) * (N0 / 64); ++cc) {
        const int col = d0 + cc * 32;
        float v[32];
        if (have) {
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + cc * 32, v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (col >= cend) continue;  // warp-uniform
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4)
          *reinterpret_cast<float4*>(stg + lane * 128 + ((e4 ^ (lane & 7)) << 4)) =
              make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + rr0;
          const int ir = (int)rank * 128 + q * 32 + rr;
          if (ir < p.C) {
            const float4 x = *reinterpret_cast<const float4*>(stg + rr * 128 + ((pc ^ (rr & 7)) << 4));
            *reinterpret_cast<float4*>(p.cpart + ((size_t)ra * 256 + ir) * p.d + col + 4 * pc) = x;
            if (rb >= 0)
              *reinterpret_cast<float4*>(p.cpart + ((size_t)rb * 256 + ir) * p.d + col + 4 * pc) =
                  make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        __syncwarp();
      }
    }
  }
  // After a timeout or abort, loads this CTA issued may still be landing (their
  // barrier is the even CTA's): give them time before the pair's shared memory
  // is released.
  if (warp == 0 && lane == 0 && aborted(p.abort_flag)) {
    const long long t0 = clock64();
    while (clock64() - t0 < 4000000ll) {
    }
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync();  // the even CTA's MMAs have finished with both CTAs' shared memory and TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Merge producer statistics and consumer partials for one canvas row and one
// slice of kCombineCols columns of S. Row statistics are contiguous per row
// ([row][producer]); S partials are read once, coalesced. A row flagged by the
// producers is recomputed here from scratch with its true maximum as the
// reference (fp32, CUDA cores; slow, only for rows whose logits exceed the
// sampled reference by more than the safe margin).
// kMaxSplitRegs: residue classes whose partials a thread holds in registers
// (8: 64 registers, four CTAs per SM; 16, for small d_model where the plan
// takes up to 16 classes: 128 registers, two CTAs per SM). Launched after the
// paired kernel as a programmatic dependent, so that its launch overlaps that
// kernel's last CTAs; griddepcontrol.wait returns once the paired kernel has
// completed and its writes are visible (at once after vocab_main).
constexpr int kCombineCols = 1024;  // columns of S per combine CTA (4 per thread)

template <int kMaxSplitRegs, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks)
    vocab_combine(const Params p, const __nv_bfloat16* __restrict__ h, const __nv_bfloat16* __restrict__ emb,
                  int32_t* argmax, float* conf, float* lse, __nv_bfloat16* selfcond) {
  extern __shared__ float hrow[];  // [d] (recompute path only)
  __shared__ float s_m[8], s_z[8], s_r[8], s_pv[256];
  __shared__ int s_a[8];
  const int i = blockIdx.x, slice = blockIdx.y, t = threadIdx.x, lane = t & 31, w = t >> 5;
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Issue this thread's partial-S loads first (4 columns x every split), so
  // they are in flight while the row statistics are reduced below.
  const int jc = slice * kCombineCols + 4 * t;
  const bool has_cols = selfcond && jc < p.d && p.ksplit <= kMaxSplitRegs;
  float4 part[kMaxSplitRegs];
  if (has_cols) {
    const float* src = p.cpart + (size_t)i * p.d + jc;
    const size_t kstride = (size_t)256 * p.d;
#pragma unroll
    for (int k = 0; k < kMaxSplitRegs; ++k)
      if (k < p.ksplit) part[k] = __ldcg(reinterpret_cast<const float4*>(src + k * kstride));
  }
  const bool ovf = __ldcg(p.overflow + i) != 0;  // with the loads above, not after the reductions
  const unsigned rkey = p.n_pa > 0 ? __ldcg(p.rowkey + i) : 0u;
  float m = -INFINITY, z = 0.f, R = -INFINITY;
  int ai = 0x7fffffff;
  const size_t rb = (size_t)i * p.n_a;
  for (int a = t; a < p.n_a; a += 256) {
    const float ma = p.am[rb + a];
    const int aa = p.aa[rb + a];
    z += p.az[rb + a];
    if (p.n_pa == 0) R = fmaxf(R, p.smax[rb + a]);
    if (ma > m || (ma == m && aa < ai)) { m = ma; ai = aa; }
  }
  for (int o = 16; o; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oa = __shfl_xor_sync(0xffffffffu, ai, o);
    if (om > m || (om == m && oa < ai)) { m = om; ai = oa; }
    z += __shfl_xor_sync(0xffffffffu, z, o);
    R = fmaxf(R, __shfl_xor_sync(0xffffffffu, R, o));
  }
  if (p.n_pa > 0) R = from_order_key(rkey);
  if (lane == 0) { s_m[w] = m; s_a[w] = ai; s_z[w] = z; s_r[w] = R; }
  __syncthreads();
  m = s_m[0]; ai = s_a[0]; z = s_z[0]; R = s_r[0];
  for (int k = 1; k < 8; ++k) {
    if (s_m[k] > m || (s_m[k] == m && s_a[k] < ai)) { m = s_m[k]; ai = s_a[k]; }
    z += s_z[k];
    R = fmaxf(R, s_r[k]);
  }
  __syncthreads();
  const int c0 = slice * kCombineCols;
  const int c1 = min(p.d, c0 + kCombineCols);
  float out_conf, out_lse;
  if (!ovf) {
    out_conf = expf(m - R) / z;
    out_lse = R + logf(z);
    if (selfcond) {
      const float inv = 1.f / z;
      if (has_cols) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kMaxSplitRegs; ++k)
          if (k < p.ksplit) {
            acc.x += part[k].x;
            acc.y += part[k].y;
            acc.z += part[k].z;
            acc.w += part[k].w;
          }
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(selfcond + (size_t)i * p.d + jc);
        o[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        o[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      } else if (p.ksplit > kMaxSplitRegs) {
        for (int j = c0 + 2 * t; j < c1; j += 512) {
          float2 acc = make_float2(0.f, 0.f);
          for (int k = 0; k < p.ksplit; ++k) {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(p.cpart + ((size_t)k * 256 + i) * p.d + j));
            acc.x += v.x;
            acc.y += v.y;
          }
          *reinterpret_cast<__nv_bfloat162*>(selfcond + (size_t)i * p.d + j) =
              __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        }
      }
    }
  } else {
    // exact recompute with R = m (the row's true maximum)
    for (int k = t; k < p.d; k += 256) hrow[k] = __bfloat162float(h[(size_t)i * p.d + k]);
    __syncthreads();
    constexpr int kPer = kCombineCols / 256;
    float zp = 0.f, acc[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) acc[q] = 0.f;
    for (int v0 = 0; v0 < p.V; v0 += 256) {
      for (int vv = w * 32; vv < w * 32 + 32; ++vv) {
        const int v = v0 + vv;
        float dot = 0.f;
        if (v < p.V)
          for (int k = lane; k < p.d; k += 32) dot = fmaf(hrow[k], __bfloat162float(emb[(size_t)v * p.d + k]), dot);
        for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) s_pv[vv] = v < p.V ? expf(dot - m) : 0.f;
      }
      __syncthreads();
      zp += s_pv[t];
      const int nv = p.V - v0 < 256 ? p.V - v0 : 256;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int j = c0 + q * 256 + t;
        if (j < c1)
          for (int vv = 0; vv < nv; ++vv)
            acc[q] = fmaf(s_pv[vv], __bfloat162float(emb[(size_t)(v0 + vv) * p.d + j]), acc[q]);
      }
      __syncthreads();
    }
    for (int o = 16; o; o >>= 1) zp += __shfl_xor_sync(0xffffffffu, zp, o);
    if (lane == 0) s_z[w] = zp;
    __syncthreads();
    zp = 0.f;
    for (int k = 0; k < 8; ++k) zp += s_z[k];
    out_conf = 1.f / zp;
    out_lse = m + logf(zp);
    if (selfcond) {
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int j = c0 + q * 256 + t;
        if (j < c1) selfcond[(size_t)i * p.d + j] = __float2bfloat16_rn(acc[q] / zp);
      }
    }
  }
  if (slice == 0 && t == 0) {
    argmax[i] = ai;
    conf[i] = out_conf;
    if (lse) lse[i] = out_lse;
    if (p.rn_tokens) {
      // threshold re-noise of this position (same rule and draw as dg_renoise)
      const bool low = out_conf < p.rn_threshold;
      const int64_t pos0 = p.rn_pos0_dev ? *p.rn_pos0_dev : p.rn_pos0;
      p.rn_tokens[i] = low ? uniform_token(p.rn_seed, p.rn_step, pos0 + i, kDomainRenoise, (uint32_t)p.V) : ai;
      if (p.rn_flags) p.rn_flags[i] = low ? 1 : 0;
    }
  }
}

// 2D bf16 map over a row-major [rows][cols] matrix, box [box_rows][64], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return tmap_bf16_sw128(m, base, 2, dims, strides, box);
}

// ---------------------------------------------------------------- paired form: plan
// Clusters of two vocab_pair CTAs that fit on the device at once (0: none).
// Without a device (a host-only plan query) the plan assumes every SM pairs up.
int pair_capacity() {
  static std::once_flag once;
  static int cap = 0;
  std::call_once(once, [] {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) {
      cudaGetLastError();
      cap = num_sms() / 2;
      return;
    }
    const size_t smem = (size_t)kRingBytes + kEpiWarps * kEpiStage + 1024;
    if (cudaFuncSetAttribute(vocab_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (nsm / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, vocab_pair, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cap = n;
  });
  return cap;
}

struct PairPlan {
  int n_vt, n_pa, n_pc, ksplit, n_full, rem, n_fullx, cw;
};

// Splits the pairs between the roles and picks the number of vocabulary residue
// classes (ksplit) that minimises the step's length, in units of one producer
// pair's tile time. In the first round every pair makes one tile; the
// producer pairs then make the remaining n_vt - (n_pa + n_pc) tiles in
// ceil(remaining / n_pa) rounds. A consumer pair of width w takes each of the
// ceil(n_vt / ksplit) tiles of its class in w / d of a producer tile's time at
// `rate` of its speed (remainder pairs, serving two classes, 2 ceil(n_vt /
// ksplit) tiles of width rem). The length is the larger of the two; ties go to
// the higher steady-state tile rate min(n_pa, rate ksplit d / w). False if no
// split fits.
//
// The consumer rate is measured, not derived. With a table larger than L2 a
// consumer re-reads a share of its E rows from DRAM and runs at 0.73 of the
// MMA rate: at V = 262144, d = 2816 (512-column slices) the step took 0.597 /
// 0.536 / 0.598 ms with 37 / 32 / 26 producer pairs, and with 256-column
// slices 0.651 / 0.536 / 0.704 ms with 43 / 32 / 26. A table that fits in L2
// is re-read from there and consumers run at the full rate: at V = 32768,
// d = 1024 the step took 49.3 / 47.2 / 46.8 / 45.2 / 45.9 / 46.7 us with 9-14
// residue classes, the model's order (12 first).
constexpr double kConsumerRate = 0.73;

size_t l2_bytes() {
  static size_t n = 0;
  if (!n) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess &&
        v > 0)
      n = (size_t)v;
    else {
      cudaGetLastError();
      n = (size_t)126 << 20;  // no device: the GB300's L2
    }
  }
  return n;
}

bool make_pair_plan(int V, int d, PairPlan* q) {
  static const char* single = getenv("DG_VOCAB_SINGLE_SM");
  if (single && single[0] == '1') return false;
  const int pairs = pair_capacity() < num_sms() / 2 ? pair_capacity() : num_sms() / 2;
  // consumer slice width: 256 columns (one MMA of N = 256 per k-slice; 512 columns, two MMAs
  // sharing the P operand, measured 0.5-1% slower at d = 2816)
  q->cw = 256;
  q->n_vt = (V + kVT - 1) / kVT;
  q->n_full = d / q->cw;
  q->rem = d % q->cw;
  // A remainder of at most cw/2 columns next to full slices gets pairs that serve
  // two residue classes; otherwise the remainder is one more per-class slice.
  const bool half = q->rem > 0 && q->rem <= q->cw / 2 && q->n_full > 0;
  q->n_fullx = q->n_full + (q->rem > 0 && !half ? 1 : 0);
  const double wmax = q->n_full > 0 ? (double)q->cw : (double)q->rem;
  const double rate = (double)V * d * 2.0 <= (double)l2_bytes() ? 1.0 : kConsumerRate;
  double best_len = 1e300, best_rate = -1.0;
  for (int ks = 1; ks <= 32 && ks <= q->n_vt; ++ks) {
    const int n_pc = ks * q->n_fullx + (half ? (ks + 1) / 2 : 0);
    if (n_pc >= pairs) break;
    const int n_pa = pairs - n_pc < q->n_vt ? pairs - n_pc : q->n_vt;
    const int rest = q->n_vt - (n_pa + n_pc) > 0 ? q->n_vt - (n_pa + n_pc) : 0;
    const int per_class = (q->n_vt + ks - 1) / ks;
    double len = (double)((rest + n_pa - 1) / n_pa);
    double cons = 1e30;
    if (q->n_fullx > 0) {
      len = fmax(len, per_class * wmax / d / rate);
      cons = fmin(cons, rate * ks * (double)d / wmax);
    }
    if (half) {
      len = fmax(len, 2.0 * per_class * q->rem / d / rate);
      cons = fmin(cons, rate * ks * (double)d / (2.0 * q->rem));
    }
    const double tile_rate = fmin((double)n_pa, cons);
    if (len < best_len - 1e-9 || (len < best_len + 1e-9 && tile_rate > best_rate + 1e-9)) {
      best_len = len;
      best_rate = tile_rate;
      q->ksplit = ks;
      q->n_pc = n_pc;
      q->n_pa = n_pa;
    }
  }
  return best_rate > 0.0;
}

// The single-SM plan's fields that size the workspace, for the paired form.
Plan as_plan(const PairPlan& q) {
  Plan p = {};
  p.n_rh = 2;
  p.n_vt = q.n_vt;
  p.ksplit = q.ksplit;
  p.n_a = 2 * (q.n_pa + q.n_pc);  // statistics slots: (pair, id half); every pair produces a tile
  p.n_c = 2 * q.n_pc;
  p.n_dt = 0;
  return p;
}

}  // namespace

int vocab_tc_plan(int C, int V, int d, int* out) {
  PairPlan q;
  if (make_pair_plan(V, d, &q)) {
    out[0] = 2 * q.n_pa;
    out[1] = 2 * q.n_pc;
    out[2] = q.ksplit;
    out[3] = 1;  // CTA pairs (clusters of two)
    out[4] = 2 * (q.n_pa + q.n_pc);
    out[5] = q.n_vt;
    return DG_OK;
  }
  const Plan pl = make_plan(C, V, d);
  out[0] = pl.n_a;
  out[1] = pl.n_c;
  out[2] = pl.ksplit;
  out[3] = 0;  // producers are independent CTAs
  out[4] = pl.n_a + pl.n_c;
  out[5] = pl.n_vt;
  return DG_OK;
}

size_t vocab_tc_workspace(int C, int V, int d) {
  PairPlan q;
  if (make_pair_plan(V, d, &q)) return make_layout(as_plan(q), d).total;
  Plan pl = make_plan(C, V, d);
  return make_layout(pl, d).total;
}

int vocab_tc_launch(const __nv_bfloat16* h, const __nv_bfloat16* emb, int C, int V, int d, int32_t* argmax,
                    float* conf, float* lse, __nv_bfloat16* selfcond, void* ws, size_t ws_bytes, cudaStream_t s,
                    const RenoiseArgs* rn) {
  PairPlan pq;
  const bool pairs = make_pair_plan(V, d, &pq);
  const Plan pl = pairs ? as_plan(pq) : make_plan(C, V, d);
  const Layout L = make_layout(pl, d);
  if (ws_bytes < L.total) return DG_ERR_WORKSPACE;
  int* st = status_ptr();
  if (!st) return DG_ERR_CUDA;
  CUtensorMap tm_h, tm_ek, tm_emn, tm_p;
  if (!make_map(&tm_h, h, d, C, 128) || !make_map(&tm_ek, emb, d, V, pairs ? 128 : kVT) ||
      !make_map(&tm_emn, emb, d, V, 64))
    return DG_ERR_CUDA;
  if (pairs) {
    // the P ring as rows of 64 bf16: one box = one pre-swizzled 16 KB block
    const uint64_t dims[2] = {64, (uint64_t)pl.n_vt * 4 * 2 * 128};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {64, 128};
    if (!tmap_bf16_plain(&tm_p, (uint8_t*)ws + L.pbuf, 2, dims, strides, box)) return DG_ERR_CUDA;
  }
  uint8_t* w = (uint8_t*)ws;
  Params p;
  p.C = C; p.V = V; p.d = d;
  p.n_rh = pl.n_rh; p.n_dt = pl.n_dt; p.n_vt = pl.n_vt; p.ksplit = pl.ksplit; p.n_a = pl.n_a;
  p.n_pa = pairs ? pq.n_pa : 0;
  p.n_pc = pairs ? pq.n_pc : 0;
  p.n_full = pairs ? pq.n_full : 0;
  p.rem = pairs ? pq.rem : 0;
  p.n_fullx = pairs ? pq.n_fullx : 0;
  p.cw = pairs ? pq.cw : 0;
  p.ring_bytes = kRingBytes;
  if (pairs) {
    // Large vocabularies: the consumer pairs' first-round tiles are the last ones (consumed last),
    // so that consumers do not start with a backlog of a whole round; in steady state a consumer
    // then reads a tile's E rows about one producer tile-time after the producer streamed them,
    // more of them still in L2 (measured at V = 262144, d = 2816: DRAM reads 2.44 instead of
    // 2.64 GB per call, same time). Small ones (fewer than four tiles per pair): consumer pair ci
    // makes tile n_pa + ci, since there the deferred tiles would be consumed after everything
    // else with nothing left to overlap them (V = 32768, d = 1024: 0.0609 against 0.0597 ms).
    const int NP = pq.n_pa + pq.n_pc;
    if (pl.n_vt >= 4 * NP) {
      int n_def = pl.n_vt - pq.n_pa;
      if (n_def > pq.n_pc) n_def = pq.n_pc;
      if (n_def < 0) n_def = 0;
      p.cb = pl.n_vt - n_def;
      p.pb = pq.n_pa;
      p.pe = pl.n_vt - n_def;
    } else {
      p.cb = pq.n_pa;
      p.pb = NP;
      p.pe = pl.n_vt;
    }
  } else {
    p.cb = p.pb = p.pe = 0;
  }
  int* flags = (int*)(w + L.flags);
  const size_t tw = tile_words(pl.n_vt);
  p.ready = reinterpret_cast<unsigned*>(flags);
  p.ref_count = flags + tw;
  p.abort_flag = flags + tw + 1;
  p.overflow = reinterpret_cast<uint8_t*>(flags + tw + 2);
  p.rowkey = reinterpret_cast<unsigned*>(flags + tw + 2 + 64);
  p.consumed = reinterpret_cast<unsigned*>(flags + tw + 2 + 64 + 256);
  p.lead = 0;
  p.cons_per_tile = 0;
  p.pace_cycles = 40000;  // ~20 us
  if (pairs && pl.n_vt >= 4 * (pq.n_pa + pq.n_pc) && d >= 2048) {
    // Pacing, for large tables with large d: producers stay at most two waves (2 n_pa tiles)
    // ahead of the consumers, so more of the E rows the consumers re-read are still in L2.
    // Measured per call, off / on: V = 262144, d = 2816 0.5056 / 0.5006 ms (DRAM reads -10%);
    // V = 131072, d = 2816 0.2698 / 0.2673; V = 152064, d = 3584 0.3852 / 0.3749; V = 262144,
    // d = 4096 0.7759 / 0.7674. Not used at d = 1024 (15-20% slower there) nor with the
    // small-vocabulary order (V = 65536, d = 2816: 2% slower); leads of 1 / 1.5 / 3 waves at the
    // headline size: 0.665 / 0.520 / 0.4976 ms.
    p.lead = 2 * pq.n_pa;
    const bool half = pq.rem > 0 && pq.rem <= pq.cw / 2 && pq.n_full > 0;
    p.cons_per_tile = 2 * (pq.n_fullx + (half ? 1 : 0));  // both CTAs of each pair serving the tile's class
  }
  p.smax = (float*)(w + L.smax);
  p.am = (float*)(w + L.am);
  p.aa = (int*)(w + L.aa);
  p.az = (float*)(w + L.az);
  p.cpart = (float*)(w + L.cpart);
  p.pbuf = w + L.pbuf;
  p.status = st;
  p.rn_tokens = rn ? rn->tokens : nullptr;
  p.rn_flags = rn ? rn->renoised : nullptr;
  p.rn_threshold = rn ? rn->threshold : 0.f;
  p.rn_seed = rn ? rn->seed : 0;
  p.rn_step = rn ? rn->step : 0;
  p.rn_pos0 = rn ? rn->abs_pos0 : 0;
  p.rn_pos0_dev = rn ? rn->abs_pos0_dev : nullptr;
  const Inject inj = take_inject(kInjectVocabReady);
  p.inject = inj.kind != kInjectNone;
  p.wait_cycles = inj.wait_cycles > 0 ? inj.wait_cycles : kTimeoutCycles;
  // the pacing counts are zeroed only when pacing reads them
  const size_t zero_bytes = L.flag_bytes - (p.lead > 0 ? 0 : tw * 4);
  // Paired form: a one-CTA kernel zeroes the flags and vocab_pair is its programmatic dependent,
  // so the pairs set up barriers and TMEM while it runs (V = 32768, d = 1024: 43.6-43.8 vs
  // 44.9-45.2 us per call after a memset; about 1 us less at the larger tables). The cooperative
  // launches keep the memset.
  static const int coop = env_int("DG_VOCAB_COOP", 0);
  const bool reset_kernel = pairs && coop != 1;
  if (reset_kernel) {
    cudaLaunchAttribute za[1];
    za[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    za[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t zc = {};
    zc.gridDim = dim3(1);
    zc.blockDim = dim3(256);
    zc.stream = s;
    zc.attrs = za;
    zc.numAttrs = 1;
    DG_CUDA_TRY(cudaLaunchKernelEx(&zc, vocab_zero_flags, (uint32_t*)flags, (int)(zero_bytes / 4)));
  } else {
    DG_CUDA_TRY(cudaMemsetAsync(flags, 0, zero_bytes, s));
  }

  if (pairs) {
    const size_t psmem = (size_t)p.ring_bytes + kEpiWarps * kEpiStage + 1024;  // attribute (the maximum) set by pair_capacity()
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (pq.n_pa + pq.n_pc));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = psmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[2].val.programmaticStreamSerializationAllowed = 1;
    // The grid is sized from the device's cluster occupancy (one CTA per SM), so every CTA is
    // resident at once on an otherwise idle GPU, and every cross-CTA wait is bounded. The
    // cooperative attribute adds the driver's guarantee of co-scheduling next to other work on
    // the device; it is opt-in (DG_VOCAB_COOP=1) because Nsight Compute cannot replay a
    // cooperative launch of two-CTA clusters (it refuses the launch), and it measured no faster.
    // The default launch is the programmatic dependent of the flag reset above.
    cfg.attrs = coop == 1 ? attr : attr + 1;
    cfg.numAttrs = 2;
    DG_CUDA_TRY(cudaLaunchKernelEx(&cfg, vocab_pair, tm_h, tm_ek, tm_emn, tm_p, p));
  } else {
  const size_t smem = (size_t)kStages * kStageBytes + 1024;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(vocab_main, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  DG_CUDA_TRY(attr_err);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.n_a + pl.n_c);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  DG_CUDA_TRY(cudaLaunchKernelEx(&cfg, vocab_main, tm_h, tm_ek, tm_emn, p));
  }

  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(C, (d + kCombineCols - 1) / kCombineCols);
  ccfg.blockDim = dim3(256);
  ccfg.dynamicSmemBytes = (size_t)d * sizeof(float);
  ccfg.stream = s;
  cudaLaunchAttribute cattr[1];
  cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cattr[0].val.programmaticStreamSerializationAllowed = 1;
  ccfg.attrs = cattr;
  ccfg.numAttrs = pairs ? 1 : 0;
  if (p.ksplit <= 8)
    DG_CUDA_TRY(cudaLaunchKernelEx(&ccfg, vocab_combine<8, 4>, p, h, emb, argmax, conf, lse, selfcond));
  else
    DG_CUDA_TRY(cudaLaunchKernelEx(&ccfg, vocab_combine<16, 2>, p, h, emb, argmax, conf, lse, selfcond));
  return DG_OK;
}

}  // namespace dg
