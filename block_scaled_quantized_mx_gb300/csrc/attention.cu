// attention.cu -- O = softmax(Q K^T * scale) V in one kernel, fp16 / bf16
// operands, fp32 accumulation, the scores and probabilities never leaving
// the SM.
//
// What is computed follows WWDC26 session 330, "Building advanced ops"
// (10:27-12:33): per block of keys, S = Q x K^T; a row-max reduction; the
// exponentials; the product with V, the probabilities fed to that second
// matmul without a round trip through memory -- FlashAttention.  The running
// maximum, the running sum and the final division that make the blockwise
// form equal softmax over all keys are FlashAttention's online softmax.
//
// Design (one CTA per (head, 256 queries), 12 warps in three warpgroups, two
// query tiles of 128 that take turns on the tensor core):
//   * warp 0: TMA -- both Q tiles once, then K and V blocks of 128 keys
//     through a two-deep ring (3-D tensor maps, so no box crosses heads);
//   * warp 1: tensor-memory allocation; the whole warp runs the issue loop
//     (so its descriptors stay warp-uniform) and one elected lane issues, per
//     key block j and tile t, O_t += P_t,{j-1} V_{j-1} and then
//     S_t,j = Q_t K_j^T (tcgen05.mma kind::f16, M = 128): while one tile's
//     softmax warps work, the tensor core runs the other tile's two products;
//   * warps 2, 3: idle (they complete warpgroup 0, whose registers go to the
//     softmax warpgroups);
//   * warps 4..7 (tile 0) and 8..11 (tile 1): softmax, one thread per query
//     row: the row's 128 scores from TMEM into registers; their maximum in
//     log2 units (for a full key block taken on the raw scores and scaled
//     once, the scale then folded into the exponent's FMA); p = 2^(x - m)
//     rounded to the operand type (the running sum adds the fp32 values:
//     each output is then within the rounding unit of the operand type,
//     relative to sum_j w_j |v_j|, of the exact one), written back over the
//     scores as the packed A operand of
//     the P V product, which reads it from tensor memory -- the
//     probabilities never touch shared memory.  The exponentials' reference
//     point moves only when a row's maximum outgrows it by more than 2^8;
//     then the row's O is rescaled in TMEM first.  At the end O / sum.
// Ordering: the MMA lane issues P_{j-1} V before S_j, and a commit covers
// every earlier operation of its thread, so once S_t,j is complete so is
// the previous product that read P_t and accumulated into O_t: the softmax
// warps may then rescale O_t and overwrite P_t without another wait.
// Tensor memory: tile t's S (and P) in columns [256 t, 256 t + 128), its O
// in [256 t + 128, 256 t + 128 + d).
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_attn and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

__device__ unsigned int g_status_attn = 0;

constexpr int AT_BQ = 128;          // queries per tile (two tiles per CTA)
constexpr int AT_BK = 128;          // keys per block
constexpr int AT_THREADS = 384;     // warpgroup 0 (TMA, MMA, 2 idle), two softmax warpgroups
// Registers: launched at 168 per thread (384 threads); warpgroup 0 gives its
// share down to 80 and the softmax warpgroups take theirs up to 208:
// 80 * 128 + 208 * 256 = 63488 <= 384 * 168 = 64512, the launch's
// allocation, so the increase never waits on registers that do not exist.
// (56 / 224 made the MMA warp spill; 80 / 208 spills nowhere.)
constexpr int AT_REGS_LOW = 80;
constexpr int AT_REGS_HIGH = 208;
constexpr int AT_TMEM_COLS = 512;
constexpr float AT_LAZY = 8.0f;     // slack of the exponentials' reference point

template <int D>
struct AtSmem {
  static constexpr int REGION = 128 * 128;          // 128 rows x 128 bytes
  static constexpr int Q_BYTES = (D / 64) * REGION; // one tile
  static constexpr int K_BYTES = (D / 64) * REGION;
  static constexpr int V_BYTES = 2 * (D / 64) * 8192; // 2 halves of 64 keys
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + 2 * K_BYTES;
  static constexpr int BAR_OFF = V_OFF + 2 * V_BYTES;
  // q_full, k_full[2], v_full[2], k_empty[2], v_empty[2], s_full[2],
  // p_full[2 tiles][2 halves], o_done[2]
  static constexpr int MISC_OFF = BAR_OFF + 17 * 8;
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
};

__device__ __forceinline__ void at_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_attn, STATUS_TIMEOUT | site);
}

// kind::f16 instruction descriptor: D f32, A / B f16 or bf16, A K-major,
// B K-major (b_mn = 0) or MN-major (1), N >> 3 at bit 17, M = 128.
__device__ __forceinline__ uint32_t at_idesc(bool bf16, uint32_t n, uint32_t b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | (b_mn << 16) |
         ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// The MMA warp runs its loop with all 32 lanes, so that the descriptors and
// addresses it computes are warp-uniform; one elected lane (always the same
// one: the lowest) issues each tcgen05 operation.
__device__ __forceinline__ void mma_ts_elect(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ss_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// Packed fp32 pairs (sm_100 and later): one instruction does two fp32
// operations, each rounded as the scalar one is, so results are the same
// per element and the softmax issues half as many instructions for them.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// three-input maximum / minimum (sm_100 and later): two comparisons in one
// instruction, NaN inputs ignored as fmaxf / fminf ignore them
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two probabilities -> a packed pair of the operand type.
__device__ __forceinline__ uint32_t pack_p(float a, float b, bool bf16) {
  return bf16 ? cvt_bf16x2(a, b) : cvt_f16x2(a, b);
}

// The work of one launch: units are (head, 256 queries), head-major.  Units
// [0, whole) run whole; each later unit is cut into `split` parts along the
// key blocks, and a part writes its un-normalised O together with each row's
// reference point m and sum l to the workspace (part r of the split units at
// ws + r * 256 * (D + 2) floats: O 256 x D row-major, then m[256], l[256]).
struct AtWork {
  int units_per_head;   // ceil(Lq / 256)
  int whole;
  int split;
  float* ws;
};

template <int D, bool BF>
__global__ void __launch_bounds__(AT_THREADS, 1)
attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, void* __restrict__ Optr, int o_dtype,
                 int Lq, int Lk, float scale_log2e, AtWork work) {
  using L = AtSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t bar_q = base + L::BAR_OFF;
  const uint32_t bar_k = bar_q + 8;            // [2] ring stage
  const uint32_t bar_v = bar_k + 16;           // [2] ring stage
  const uint32_t bar_k_empty = bar_v + 16;     // [2] ring stage
  const uint32_t bar_v_empty = bar_k_empty + 16;   // [2] ring stage
  const uint32_t bar_s_full = bar_v_empty + 16;    // [2] tile
  const uint32_t bar_p_full = bar_s_full + 16;     // [2] tile x [2] half of the keys
  const uint32_t bar_o_done = bar_p_full + 32;     // [2] tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb_all = (Lk + AT_BK - 1) / AT_BK;
  const int item = blockIdx.x;
  int unit = item, kb0 = 0, nkb = nkb_all, part_slot = -1;
  if (item >= work.whole) {
    const int r = item - work.whole;
    const int part = r % work.split;
    unit = work.whole + r / work.split;
    kb0 = static_cast<int>(static_cast<int64_t>(part) * nkb_all / work.split);
    nkb = static_cast<int>(static_cast<int64_t>(part + 1) * nkb_all / work.split) - kb0;
    part_slot = r;
  }
  const int head = unit / work.units_per_head;
  const int q0 = (unit % work.units_per_head) * 2 * AT_BQ;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_k + 8 * i, 1);
      mbar_init(bar_v + 8 * i, 1);
      mbar_init(bar_k_empty + 8 * i, 1);
      mbar_init(bar_v_empty + 8 * i, 1);
      mbar_init(bar_s_full + 8 * i, 1);
      mbar_init(bar_p_full + 16 * i, 4);
      mbar_init(bar_p_full + 16 * i + 8, 4);
      mbar_init(bar_o_done + 8 * i, 1);
    }
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) tmem_alloc_cg<1>(smem_u32(tmem_slot), AT_TMEM_COLS);
  __syncwarp();   // reconverge before the aligned barrier (one-lane setup)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Each role's code sits inside the branch that sets its register count,
  // so the compiler allots each its own budget; every warp of a warpgroup
  // executes the same setmaxnreg.
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_REGS_LOW));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, 2 * L::Q_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int r = 0; r < D / 64; ++r)
          tma_load_3d(base + L::Q_OFF + t * L::Q_BYTES + r * L::REGION, &tmQ, bar_q, 64 * r,
                      q0 + AT_BQ * t, head);
      // K_j and V_j have separate slots: K_j's is free once both tiles'
      // S_j are done, V_j's only after both P_j V_j products
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1u;
        const int k0 = (kb0 + j) * AT_BK;
        bool okp = mbar_wait(bar_k_empty + 8 * st, ph ^ 1u, abort);
        if (okp) {
          ++k_issued;
          mbar_arrive_expect_tx(bar_k + 8 * st, L::K_BYTES);
          for (int r = 0; r < D / 64; ++r)
            tma_load_3d(base + L::K_OFF + st * L::K_BYTES + r * L::REGION, &tmK, bar_k + 8 * st,
                        64 * r, k0, head);
          okp = mbar_wait(bar_v_empty + 8 * st, ph ^ 1u, abort);
        }
        if (!okp) {
          at_timeout(abort, 0x31);
          // let the copies already issued land before the CTA retires
          const long long t0 = clock64();
          while (!mbar_try_wait(bar_q, 0) && clock64() - t0 < MXK_WAIT_LIMIT_CYCLES) {
          }
          for (int i = k_issued >= 2 ? k_issued - 2 : 0; i < k_issued; ++i) {
            const long long t1 = clock64();
            while (!mbar_try_wait(bar_k + 8 * (i & 1), (i >> 1) & 1u) &&
                   clock64() - t1 < MXK_WAIT_LIMIT_CYCLES) {
            }
          }
          for (int i = v_issued >= 2 ? v_issued - 2 : 0; i < v_issued; ++i) {
            const long long t1 = clock64();
            while (!mbar_try_wait(bar_v + 8 * (i & 1), (i >> 1) & 1u) &&
                   clock64() - t1 < MXK_WAIT_LIMIT_CYCLES) {
            }
          }
          break;
        }
        ++v_issued;
        mbar_arrive_expect_tx(bar_v + 8 * st, L::V_BYTES);
        for (int h = 0; h < 2; ++h)
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(base + L::V_OFF + st * L::V_BYTES + h * (D / 64) * 8192 + a * 8192, &tmV,
                        bar_v + 8 * st, 64 * a, k0 + 64 * h, head);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {
      const uint32_t id_qk = at_idesc(BF, AT_BK, 0);
      const uint32_t id_pv = at_idesc(BF, D, 1);
      // descriptors of the operand regions; an MMA adds its offset (16-byte units)
      const uint64_t dq0 = smem_desc(base + L::Q_OFF, 16, 1024, 2);
      const uint64_t dk0 = smem_desc(base + L::K_OFF, 16, 1024, 2);
      const uint64_t dv0 = smem_desc(base + L::V_OFF, 8192, 1024, 2);
      bool ok = mbar_wait(bar_q, 0, abort);
      if (!ok) at_timeout(abort, 0x32);
      tc_fence_after();
      for (int j = 0; j <= nkb && ok; ++j) {
        for (int t = 0; t < 2 && ok; ++t) {
          const uint32_t s_t = tmem_base + 256 * t;            // S_t, then P_t
          const uint32_t o_t = s_t + 128;
          if (j >= 1) {
            // O_t += P_t,{j-1} V_{j-1}, P read from tensor memory
            const int jj = j - 1, st = jj & 1;
            // P arrives in two halves of 64 keys: the product with the first
            // half runs while the softmax warps compute the second
            if (!mbar_wait(bar_p_full + 16 * t, jj & 1, abort) ||
                !mbar_wait(bar_v + 8 * st, (jj >> 1) & 1u, abort)) {
              at_timeout(abort, 0x34);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < AT_BK / 16; ++kk) {
              if (kk == AT_BK / 32) {
                if (!mbar_wait(bar_p_full + 16 * t + 8, jj & 1, abort)) {
                  at_timeout(abort, 0x36);
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              const uint32_t boff = (kk >> 2) * (D / 64) * 8192 + (kk & 3) * 2048;
              mma_ts_elect(o_t, s_t + 8 * kk,
                           dv0 + static_cast<uint64_t>((st * L::V_BYTES + boff) >> 4),
                           id_pv, (jj > 0 || kk > 0) ? 1u : 0u);
            }
            if (!ok) break;
            // both tiles' products with V_{j-1} issued: its slot frees when they end
            if (t == 1) commit_elect(bar_v_empty + 8 * st);
          }
          if (j < nkb) {
            // S_t,j = Q_t K_j^T, after the product that read P_t
            const int st = j & 1;
            if (!mbar_wait(bar_k + 8 * st, (j >> 1) & 1u, abort)) {
              at_timeout(abort, 0x33);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * L::REGION + (kk & 3) * 32;
              mma_ss_elect(s_t, dq0 + static_cast<uint64_t>((t * L::Q_BYTES + off) >> 4),
                           dk0 + static_cast<uint64_t>((st * L::K_BYTES + off) >> 4), id_qk,
                           kk > 0 ? 1u : 0u);
            }
            commit_elect(bar_s_full + 8 * t);
            // both tiles' S_j issued: K_j's slot frees when they end
            if (t == 1) commit_elect(bar_k_empty + 8 * st);
          } else {
            commit_elect(bar_o_done + 8 * t);
          }
        }
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_HIGH));
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;                          // query tile
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;                    // row in the tile
    const uint32_t lane_addr =
        tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + 256 * t;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      if (!mbar_wait(bar_s_full + 8 * t, j & 1, abort)) {
        at_timeout(abort, 0x35);
        ok = false;
        break;
      }
      tc_fence_after();
      const int valid = Lk - (kb0 + j) * AT_BK;              // keys in this block
      // the row's 128 scores, four loads in flight, scaled to log2 units
      uint32_t sv[AT_BK];
#pragma unroll
      for (int c = 0; c < AT_BK / 32; ++c)
        tmem_ld_32x32b_x32(lane_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
      tmem_wait_ld();
      // row maximum over eight independent partial maxima (short chains)
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
      float s_eff = 1.0f;
      if (valid >= AT_BK) {
        // a full block: the scale goes into the exponent's FMA instead of a
        // multiply per score; the largest scaled score is the scale times
        // the largest raw score (the smallest, for a negative scale) --
        // rounding is monotonic, so this is exactly the maximum of the
        // rounded products.  A partial block scales and masks as below.
        s_eff = scale_log2e;
        if (scale_log2e >= 0.0f) {
#pragma unroll
          for (int e = 0; e < AT_BK; e += 2)
            mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], __uint_as_float(sv[e]),
                                      __uint_as_float(sv[e + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = INFINITY;
#pragma unroll
          for (int e = 0; e < AT_BK; e += 2)
            mx8[(e >> 1) & 7] = min3f(mx8[(e >> 1) & 7], __uint_as_float(sv[e]),
                                      __uint_as_float(sv[e + 1]));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] *= scale_log2e;
      } else {
#pragma unroll
        for (int e = 0; e < AT_BK; ++e) {
          const float x = e < valid ? __uint_as_float(sv[e]) * scale_log2e : -INFINITY;
          sv[e] = __float_as_uint(x);
          mx8[e & 7] = fmaxf(mx8[e & 7], x);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // The reference point m of the exponentials moves only when the block's
      // maximum exceeds it by more than AT_LAZY (log2 units): every p stays
      // <= 2^AT_LAZY, exact in fp32 and in the 16-bit operand types, and O / l
      // does not depend on which m was used, so the O rescale (a round trip
      // of the row's O through registers) is skipped for almost every block.
      const float m_new = (mx > m + AT_LAZY) ? mx : m;
      const float alpha = ex2_approx(m - m_new);             // 0 on the first block
      // O_t rescale when a row's reference moved; the product that last
      // wrote O_t completed before this block's scores did
      if (j >= 1 && __any_sync(0xFFFFFFFFu, m_new != m)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(lane_addr + 128 + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_32x32b_x32(lane_addr + 128 + 32 * c, o);
        }
      }
      // p = 2^(x - m), rounded to the operand type, written back as packed P
      // over the scores (already in registers): chunk c of P is columns
      // 16 c .. 16 c + 15; keys beyond Lk have x = -inf, p = 0
      // pairs of scores: x = s s_eff - m and the running sums as packed fp32
      const uint64_t se2 = f2_pack(s_eff, s_eff), nm2 = f2_pack(-m_new, -m_new);
      uint64_t sum2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
      for (int c = 0; c < AT_BK / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[32 * c + 2 * e]),
                                   __uint_as_float(sv[32 * c + 2 * e + 1])),
                           se2, nm2),
                    x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          pk[e] = pack_p(p0, p1, BF);
          sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
        }
        tmem_st_32x32b_x16(lane_addr + 16 * c, pk);
        if (c == AT_BK / 64 - 1 || c == AT_BK / 32 - 1) {
          // half of P (64 keys) written: the product with it may start
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p_full + 16 * t + (c == AT_BK / 32 - 1 ? 8 : 0));
        }
      }
      float s0, s1, s2, s3;
      f2_unpack(sum2[0], s0, s1);
      f2_unpack(sum2[1], s2, s3);
      l = l * alpha + ((s0 + s2) + (s1 + s3));
      m = m_new;
    }
    if (ok) {
      if (!mbar_wait(bar_o_done + 8 * t, 0, abort)) {
        at_timeout(abort, 0x38);
      } else {
        tc_fence_after();
        const int qrow = q0 + AT_BQ * t + row;
        const float inv = 1.0f / l;
        const int64_t obase = (static_cast<int64_t>(head) * Lq + qrow) * D;
        if (part_slot >= 0) {
          // a part: un-normalised O, m and l of every row of the unit
          float* ws = work.ws + static_cast<int64_t>(part_slot) * (2 * AT_BQ) * (D + 2);
          const int urow = AT_BQ * t + row;
          float* dst0 = ws + static_cast<int64_t>(urow) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(lane_addr + 128 + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<float4*>(dst0 + 32 * c + 4 * v) =
                  make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                              __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
          }
          ws[(2 * AT_BQ) * D + urow] = m;
          ws[(2 * AT_BQ) * (D + 1) + urow] = l;
        } else {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(lane_addr + 128 + 32 * c, o);
          tmem_wait_ld();
          if (qrow < Lq) {
            if (o_dtype == DT_F32) {
              float* dst = reinterpret_cast<float*>(Optr) + obase + 32 * c;
#pragma unroll
              for (int v = 0; v < 8; ++v)
                *reinterpret_cast<float4*>(dst + 4 * v) =
                    make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                __uint_as_float(o[4 * v + 2]) * inv,
                                __uint_as_float(o[4 * v + 3]) * inv);
            } else {
              uint16_t* dst = reinterpret_cast<uint16_t*>(Optr) + obase + 32 * c;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float a = __uint_as_float(o[8 * v + 2 * e]) * inv;
                  const float b = __uint_as_float(o[8 * v + 2 * e + 1]) * inv;
                  w[e] = (o_dtype == DT_BF16) ? cvt_bf16x2(a, b) : cvt_f16x2(a, b);
                }
                *reinterpret_cast<uint4*>(dst + 8 * v) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
        }
      }
    }
  }

  __syncwarp();   // reconverge before the aligned barrier (one-lane roles)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<1>(tmem_base, AT_TMEM_COLS);
  }
}

// Merge the parts of the split units: per row, M = max over parts of m_p,
// O = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p, parts in a fixed order.
// One thread per (split unit, row, four columns).
template <int D>
__global__ void __launch_bounds__(256)
attention_merge_kernel(const float* __restrict__ ws, void* __restrict__ Optr, int o_dtype, int Lq,
                       AtWork work, int64_t n_threads) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_threads) return;
  constexpr int G = D / 4;
  const int g = static_cast<int>(gid % G);
  const int urow = static_cast<int>((gid / G) % (2 * AT_BQ));
  const int su = static_cast<int>(gid / (G * 2 * AT_BQ));
  const int unit = work.whole + su;
  const int head = unit / work.units_per_head;
  const int qrow = (unit % work.units_per_head) * 2 * AT_BQ + urow;
  if (qrow >= Lq) return;
  constexpr int64_t PART = (2 * AT_BQ) * (D + 2);
  const float* base = ws + static_cast<int64_t>(su) * work.split * PART;
  float M = -INFINITY;
  for (int p = 0; p < work.split; ++p) M = fmaxf(M, base[p * PART + (2 * AT_BQ) * D + urow]);
  float l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int p = 0; p < work.split; ++p) {
    const float* part = base + p * PART;
    const float w = ex2_approx(part[(2 * AT_BQ) * D + urow] - M);
    l = fmaf(w, part[(2 * AT_BQ) * (D + 1) + urow], l);
    const float4 o = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(urow) * D + 4 * g);
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
  }
  const float inv = 1.0f / l;
  const int64_t obase = (static_cast<int64_t>(head) * Lq + qrow) * D + 4 * g;
  if (o_dtype == DT_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(Optr) + obase) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  } else {
    const bool bf = o_dtype == DT_BF16;
    const uint32_t w0 = bf ? cvt_bf16x2(acc.x * inv, acc.y * inv) : cvt_f16x2(acc.x * inv, acc.y * inv);
    const uint32_t w1 = bf ? cvt_bf16x2(acc.z * inv, acc.w * inv) : cvt_f16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(Optr) + obase) = make_uint2(w0, w1);
  }
}

template <int D, bool BF>
cudaError_t at_run(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* O,
                   int o_dtype, const AtWork& work, int64_t items, int Lq, int Lk,
                   float scale_log2e, cudaStream_t st) {
  using L = AtSmem<D>;
  auto kern = attention_kernel<D, BF>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the registers it asks for are free: it can
    // only complete if the launch allocated at least what the two splits
    // add up to.  Refuse to launch otherwise instead of waiting forever.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * AT_THREADS < AT_REGS_LOW * 128 + AT_REGS_HIGH * 256)
      return cudaErrorInvalidConfiguration;
    if (dev < 64) attr_set[dev] = true;
  }
  kern<<<static_cast<unsigned>(items), AT_THREADS, L::ALLOC, st>>>(tq, tk, tv, O, o_dtype, Lq, Lk,
                                                                   scale_log2e, work);
  e = cudaGetLastError();
  if (e != cudaSuccess || work.split <= 1) return e;
  const int64_t split_units = (items - work.whole) / work.split;
  const int64_t n = split_units * (2 * AT_BQ) * (D / 4);
  attention_merge_kernel<D><<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
      work.ws, O, o_dtype, Lq, work, n);
  return cudaGetLastError();
}

int at_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

struct AtPlan {
  int64_t units, whole, split, items;
  size_t ws_bytes;
};

// Whole units fill whole waves of one CTA per SM; the units of a last partial
// wave (all units, when there are fewer than SMs) are split along the key
// blocks over the idle SMs: parts of at least two blocks, at most 16 parts.
AtPlan at_plan(int64_t BH, int64_t Lq, int64_t Lk, int64_t d, bool use_split) {
  AtPlan p{};
  const int64_t uph = (Lq + 2 * AT_BQ - 1) / (2 * AT_BQ);
  p.units = BH * uph;
  p.whole = p.units;
  p.split = 1;
  p.items = p.units;
  const int64_t sms = at_sm_count();
  const int64_t nkb = (Lk + AT_BK - 1) / AT_BK;
  if (!use_split || sms <= 0 || p.units == 0) return p;
  const int64_t tail = p.units % sms;
  if (tail == 0) return p;
  const int64_t split = std::min<int64_t>(std::min<int64_t>(sms / tail, nkb / 2), 16);
  if (split < 2) return p;
  p.whole = p.units - tail;
  p.split = split;
  p.items = p.whole + tail * split;
  p.ws_bytes = static_cast<size_t>(tail * split) * (2 * AT_BQ) * (d + 2) * sizeof(float);
  return p;
}

}  // namespace

size_t attention_workspace_bytes(int64_t BH, int64_t Lq, int64_t Lk, int64_t d) {
  return at_plan(BH, Lq, Lk, d, true).ws_bytes;
}

cudaError_t launch_attention(int dtype, const void* Q, const void* K, const void* V, void* O,
                             int o_dtype, int64_t BH, int64_t Lq, int64_t Lk, int64_t d,
                             float scale, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (BH == 0 || Lq == 0) return cudaSuccess;
  AtPlan plan = at_plan(BH, Lq, Lk, d, ws != nullptr);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes) plan = at_plan(BH, Lq, Lk, d, false);
  if (plan.items > 0x7FFFFFFF) return cudaErrorInvalidValue;
  AtWork work;
  work.units_per_head = static_cast<int>((Lq + 2 * AT_BQ - 1) / (2 * AT_BQ));
  work.whole = static_cast<int>(plan.whole);
  work.split = static_cast<int>(plan.split);
  work.ws = static_cast<float*>(ws);
  const CUtensorMapDataType dt = (dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  auto enc = [&](CUtensorMap* m, const void* p, uint64_t L, uint32_t by) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(L * d) * 2};
    cuuint32_t box[3] = {64, by, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode_tiled(m, dt, 3, p, dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  CUtensorMap tq, tk, tv;
  if (!enc(&tq, Q, Lq, 128) || !enc(&tk, K, Lk, 128) || !enc(&tv, V, Lk, 64))
    return cudaErrorInvalidValue;
  const float sl2 = scale * 1.4426950408889634f;
  const bool bf = dtype == DT_BF16;
  const int lq = static_cast<int>(Lq), lk = static_cast<int>(Lk);
  const int64_t it = plan.items;
  if (d == 64)
    return bf ? at_run<64, true>(tq, tk, tv, O, o_dtype, work, it, lq, lk, sl2, st)
              : at_run<64, false>(tq, tk, tv, O, o_dtype, work, it, lq, lk, sl2, st);
  return bf ? at_run<128, true>(tq, tk, tv, O, o_dtype, work, it, lq, lk, sl2, st)
            : at_run<128, false>(tq, tk, tv, O, o_dtype, work, it, lq, lk, sl2, st);
}

unsigned fetch_and_clear_status_attn(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_attn, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_attn, &z, sizeof(z));
  return v;
}

}  // namespace mxk
