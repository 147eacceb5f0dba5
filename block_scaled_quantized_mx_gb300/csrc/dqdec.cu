// dqdec.cu -- the dequantizing GEMM for decode-shaped products: a few rows of
// 16-bit activations A (M <= 128 tokens) times an MX weight tensor B (N x K)
// of any element format (E4M3, E5M2, E2M1, int8, int4, int2).
//
// What is computed is what dqgemm.cu computes, C = A * dequant(B)^T (WWDC26
// session 330, "Quantized matrix multiplication": dequantize a chunk of the
// quantized data to 16 bits, then multiply), with fp32 accumulation.  The
// shape is different: with a few tokens the product is a stream over the
// weights, bound by the HBM bytes of B's codes, and a 128-row tile of tokens
// would be mostly padding.  So the roles are turned around: the kernel forms
// C^T = dequant(B) * A^T, the weights' 128-row blocks being the MMA's M and
// the tokens (padded to NT = 64 or 128) its N.
//
// Design:
//   * work: the (128-row weight block, 64-K chunk) units are cut into one
//     contiguous range per CTA, over every SM, so that all SMs stream codes.
//     A weight block whose chunks span several CTAs is summed by the last of
//     them to finish (a tagged arrival counter in the workspace), in CTA
//     order, so the result does not depend on timing.  Without a workspace
//     each CTA takes whole weight blocks.
//   * warp 0: TMA producer -- per chunk the weight block's codes (128 rows x
//     64 K, raw bytes), its scale atom and the tokens' 64-K slice (NT rows,
//     128-byte swizzle) into a ring as deep as shared memory allows (up to 16
//     stages: 64 KB of int4 codes in flight per SM);
//   * warps 2..: dequantizers, in groups of four (one warp per TMEM lane
//     quarter) that take the chunks in turn, one weight row per thread, both
//     32-element blocks of it per chunk: codes x scale -> 16-bit values
//     written straight into tensor memory (tcgen05.st) in one of four slots
//     per group, never through shared memory;
//   * warp 1: tensor-memory allocation and the MMA loop (one elected lane
//     issues): per chunk four kind::f16 MMAs, M = 128 weight rows, N = NT
//     tokens, K = 16, A read from the tensor-memory slot, B (the tokens) from
//     shared memory; per range of a weight block, a commit of the accumulator
//     (two buffers, alternating) to the epilogue;
//   * the last four warps: epilogue, one weight row per thread and 32 tokens at a
//     time: bias and activation, C[m][n] stored for every token m (a warp's
//     32 rows are 32 consecutive columns of C), or the range's fp32 partial
//     to the workspace.
// Tensor memory: accumulators in columns [0, 2 NT), weight slots from 256.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_dqd and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>

#include "common.cuh"
#include "dq_common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

using namespace dq;

__device__ unsigned int g_status_dqd = 0;

constexpr int WR = 128;                  // weight rows per block (MMA M)
constexpr int KC = 64;                   // K per chunk (one ring stage)
constexpr int A_COL0 = 256;              // first tensor-memory slot column
constexpr int MAX_STAGES = 16;
constexpr int MAX_SLOTS = 8;
constexpr int DQ_W0 = 2;                 // first dequantizer warp
constexpr int NUM_EPI = 4;
constexpr int SMEM_BUDGET = 200 * 1024;  // ring bytes

// Warp layout per token width NT.  Dequantizers come in groups of four
// warps, one per TMEM lane quarter (a warp reaches the quarter warp % 4);
// with two groups they take the chunks in turn, which hides one chunk's
// conversion and tensor-memory store behind the other's (the chain of one
// group set the pace: one chunk per ~0.45 us).  Then four epilogue warps.
// Two groups make 14 warps, so 128 registers a thread (a sub-partition
// holds 4 warps): enough for NT = 64; NT = 128, whose epilogue needs more,
// keeps one group (10 warps, 3 per sub-partition, 170 registers).
template <int NT>
struct Lay {
  static constexpr int DQG = (NT == 64) ? 2 : 1;
  static constexpr int NUM_DQ = 4 * DQG;
  static constexpr int A_SLOTS = 4 * DQG;   // tensor-memory slots of dequantized weights
  static constexpr int EPI_W0 = DQ_W0 + NUM_DQ;
  static constexpr int THREADS = 32 * (EPI_W0 + NUM_EPI);
  static_assert(A_SLOTS <= MAX_SLOTS, "slot barriers");
  static_assert(2 * NT <= A_COL0 && A_COL0 + 32 * A_SLOTS <= 512, "tensor-memory columns");
};

// barriers: full[16], empty[16], a_ready[8], a_free[8], acc_full[2],
// acc_empty[2], part_written, decided
constexpr int NBAR = 2 * MAX_STAGES + 2 * MAX_SLOTS + 4 + 2;

struct DecArgs {
  void* C;
  int64_t ldc;
  int M, N, K;
  int fmt;              // B's element format
  int a_bf16;           // A (and the dequantized weights) bf16, else f16
  int stages;           // ring depth
  int code_row_bytes;   // bytes of one weight row's 64 K codes
  int x_bytes;          // bytes of one stage's token slice (NT x 128)
  int stage_bytes;      // ring stride: token slice + codes + scale atom, 1024-aligned
  int whole;            // 1: whole weight blocks per CTA (no workspace)
  float* ws;            // partial tiles: CTA c's first range at slot 2c, last at 2c + 1
  unsigned long long* ctr;   // one arrival counter per weight block
  unsigned long long tag;
  EpiArgs epi;
};

__device__ __forceinline__ void dqd_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_dqd, STATUS_TIMEOUT | site);
}

// The contiguous unit range [u0, u1) of CTA c: units are (weight block nb,
// chunk kc) in the order nb * kch + kc.
struct Ranges {
  int64_t T;      // units
  int G;          // CTAs
  int kch;        // chunks per weight block
  int nb_count;   // weight blocks
  int whole;
  __host__ __device__ int64_t begin(int c) const {
    if (whole) return (static_cast<int64_t>(c) * nb_count / G) * kch;
    return static_cast<int64_t>(c) * T / G;
  }
  // the CTA whose range holds unit x (the ranges are contiguous and cover
  // [0, T) in CTA order; begin(c) <= x < begin(c + 1))
  __host__ __device__ int owner(int64_t x) const {
    if (whole) {
      const int64_t nb = x / kch;
      return static_cast<int>(((nb + 1) * G - 1) / nb_count);
    }
    return static_cast<int>(((x + 1) * G - 1) / T);
  }
};

// Same counter protocol as the GEMM's K-split: tag << 16 | count, another
// tag counts as zero, the completing arrival writes zero.
__device__ __forceinline__ int dqd_arrive(unsigned long long* ctr, unsigned long long tag,
                                          int target) {
  unsigned long long v = 0ull;
  for (int i = 0; i < (1 << 16); ++i) {
    const unsigned long long cnt = ((v >> 16) == tag) ? (v & 0xFFFFull) : 0ull;
    const unsigned long long nv =
        (cnt + 1 == static_cast<unsigned long long>(target)) ? 0ull : (tag << 16) | (cnt + 1);
    const unsigned long long old = atomicCAS(ctr, v, nv);
    if (old == v) return static_cast<int>(cnt + 1);
    v = old;
  }
  return -1;
}

// kind::f16 instruction descriptor: D f32, A and B f16 (0) or bf16 (1), both
// K-major (A from tensor memory), N>>3 at bit 17, M = 128 (>>4 at bit 24).
template <int NT>
__device__ __forceinline__ uint32_t idesc_dec(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(NT >> 3) << 17) | (static_cast<uint32_t>(WR >> 4) << 24);
}

// One dequantizer warp's part of every chunk of this CTA: weight row
// 32 q + lane, both 32-element blocks of the chunk.
template <int FMT, int DQG>
__device__ __forceinline__ void dequant_loop(const DecArgs& a, const Ranges& rg, int c,
                                             uint32_t base, uint32_t tmem_base, uint32_t bar_full,
                                             uint32_t bar_empty, uint32_t bar_a_ready,
                                             uint32_t bar_a_free, int q, int g, int lane,
                                             volatile int* abort) {
  constexpr int A_SLOTS = 4 * DQG;
  const int row = 32 * q + lane;
  const bool bf16 = a.a_bf16 != 0;
  constexpr int BB = block_code_bytes<FMT>();
  const int u0 = static_cast<int>(rg.begin(c)), u1 = static_cast<int>(rg.begin(c + 1));
  // the loop's counters advance by one: no divisions inside it (a 64-bit
  // or runtime-divisor division is a long instruction sequence)
  int kc = u0 % rg.kch, s = 0;
  uint32_t ph = 0, ci = 0;
  for (int u = u0; u < u1; ++u, ++ci) {
    // this group's chunks only (the counters advance over every chunk)
    if (DQG > 1 && static_cast<int>(ci % DQG) != g) {
      if (++kc == rg.kch) kc = 0;
      if (++s == a.stages) {
        s = 0;
        ph ^= 1u;
      }
      continue;
    }
    const int slot = static_cast<int>(ci & (A_SLOTS - 1));
    const uint32_t sph = (ci / A_SLOTS) & 1u;
    if (!mbar_wait_short(bar_full + 8 * s, ph, abort)) {
      dqd_timeout(abort, 21);
      return;
    }
    const uint32_t st = base + static_cast<uint32_t>(s) * a.stage_bytes;
    const uint8_t* codes = reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(
        st + a.x_bytes + row * a.code_row_bytes));
    const uint8_t* atom = reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(
        st + a.x_bytes + WR * a.code_row_bytes));
    uint32_t w0[8], w1[8];
    load_block_codes<FMT>(codes, w0);
    load_block_codes<FMT>(codes + BB, w1);
    const uint32_t sc0 = atom[sf_in_atom(row, (kc & 1) * 2)];
    const uint32_t sc1 = atom[sf_in_atom(row, (kc & 1) * 2 + 1)];
    uint32_t o0[16], o1[16];
    dq_block_regs<FMT>(w0, sc0, bf16, o0);
    dq_block_regs<FMT>(w1, sc1, bf16, o1);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // codes and scales consumed
    if (!mbar_wait_short(bar_a_free + 8 * slot, sph ^ 1u, abort)) {
      dqd_timeout(abort, 22);
      return;
    }
    tc_fence_after();
    const uint32_t ta = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + A_COL0 + slot * 32;
    tmem_st_32x32b_x16(ta, o0);
    tmem_st_32x32b_x16(ta + 16, o1);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_a_ready + 8 * slot);
    if (++kc == rg.kch) kc = 0;
    if (++s == a.stages) {
      s = 0;
      ph ^= 1u;
    }
  }
}

// bias + activation on 32 values of weight row n (one column of C)
__device__ __forceinline__ void dec_epi(float (&v)[32], const EpiArgs& e, int n, int N) {
  if (e.bias != nullptr) {
    const float b = (n < N) ? __ldg(e.bias + n) : 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += b;
  }
  if (e.act == ACT_GELU) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_exact(v[i]);
  } else if (e.act == ACT_GELU_TANH) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
  }
}

// C[m][n] for the 32 tokens m = m0 .. m0 + 31 of weight row n.
template <int OUT>
__device__ __forceinline__ void dec_store(const float (&v)[32], void* C, int64_t ldc, int m0,
                                          int n, int M, int N) {
  if (n >= N) return;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int m = m0 + i;
    if (m < M) {
      if (OUT == OUT_BF16)
        reinterpret_cast<uint16_t*>(C)[static_cast<int64_t>(m) * ldc + n] =
            static_cast<uint16_t>(cvt_bf16x2(v[i], 0.f) & 0xFFFFu);
      else
        reinterpret_cast<float*>(C)[static_cast<int64_t>(m) * ldc + n] = v[i];
    }
  }
}

template <int NT, int OUT>
__global__ void __launch_bounds__(Lay<NT>::THREADS, 1)
dqdec_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
             const __grid_constant__ CUtensorMap tmSF, const DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + static_cast<uint32_t>(a.stages) * a.stage_bytes;
  const uint32_t bar_full = bars;
  const uint32_t bar_empty = bar_full + 8 * MAX_STAGES;
  const uint32_t bar_a_ready = bar_empty + 8 * MAX_STAGES;
  using LY = Lay<NT>;
  constexpr int A_SLOTS = LY::A_SLOTS;
  constexpr int EPI_W0 = LY::EPI_W0;
  const uint32_t bar_a_free = bar_a_ready + 8 * MAX_SLOTS;
  const uint32_t bar_acc_full = bar_a_free + 8 * MAX_SLOTS;
  const uint32_t bar_acc_empty = bar_acc_full + 16;
  const uint32_t bar_written = bar_acc_empty + 16;
  const uint32_t bar_decided = bar_written + 8;
  uint8_t* misc = gbase + (bars - base) + 8 * NBAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  Ranges rg;
  rg.kch = a.K / KC;
  rg.nb_count = (a.N + WR - 1) / WR;
  rg.T = static_cast<int64_t>(rg.nb_count) * rg.kch;
  rg.G = gridDim.x;
  rg.whole = a.whole;
  const int64_t u0 = rg.begin(c), u1 = rg.begin(c + 1);

  if (warp == 0) {
    for (int i = lane; i < NBAR; i += 32) {
      uint32_t count = 1;
      // one group of four dequantizer warps handles each chunk
      if (i >= MAX_STAGES && i < 2 * MAX_STAGES) count = 1 + 4;               // empty
      else if (i >= 2 * MAX_STAGES && i < 2 * MAX_STAGES + MAX_SLOTS) count = 4;  // a_ready
      else if (i >= 2 * MAX_STAGES + 2 * MAX_SLOTS + 2 &&
               i < 2 * MAX_STAGES + 2 * MAX_SLOTS + 4) count = NUM_EPI;       // acc_empty
      else if (i == 2 * MAX_STAGES + 2 * MAX_SLOTS + 4) count = NUM_EPI;      // written
      mbar_init(bar_full + 8 * i, count);
    }
    fence_mbar_init();
    if (lane == 0) {
      *abort = 0;
      *last_flag = 0;
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmSF);
    }
  }
  if (warp == 1) tmem_alloc_cg<1>(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int k_atoms = (a.K + 127) / 128;
      const uint32_t tx = static_cast<uint32_t>(a.x_bytes + WR * a.code_row_bytes + 512);
      int nb = static_cast<int>(u0 / rg.kch), kc = static_cast<int>(u0 % rg.kch), s = 0;
      uint32_t ph = 0;
      for (int64_t u = u0; u < u1; ++u) {
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) {
          dqd_timeout(abort, 20);
          break;
        }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, tx);
        const uint32_t st = base + static_cast<uint32_t>(s) * a.stage_bytes;
        tma_load_2d(st, &tmX, full, kc * KC, 0);
        tma_load_2d(st + a.x_bytes, &tmW, full, kc * a.code_row_bytes, nb * WR);
        tma_load_2d(st + a.x_bytes + WR * a.code_row_bytes, &tmSF, full, 0,
                    nb * k_atoms + (kc >> 1));
        if (++kc == rg.kch) {
          kc = 0;
          ++nb;
        }
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool issuer = elect_one();
    const uint32_t id = idesc_dec<NT>(a.a_bf16 != 0);
    uint32_t ci = 0, si = 0, ph = 0;
    int s = 0, nb = static_cast<int>(u0 / rg.kch);
    bool ok = true;
    for (int64_t u = u0; u < u1 && ok; ++si, ++nb) {
      const int64_t seg_end = min(u1, static_cast<int64_t>(nb + 1) * rg.kch);
      const uint32_t buf = si & 1u, use = si >> 1;
      if (!mbar_wait_spin(bar_acc_empty + 8 * buf, (use & 1u) ^ 1u, abort)) {
        dqd_timeout(abort, 23);
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + buf * NT;
      bool first = true;
      for (; u < seg_end; ++u, ++ci) {
        const int slot = static_cast<int>(ci & (A_SLOTS - 1));
        const uint32_t sph = (ci / A_SLOTS) & 1u;
        // the MMA warp's waits are on the critical path and usually find
        // the slot not yet written: spin rather than sleep through a wake-up
        if (!mbar_wait_spin(bar_a_ready + 8 * slot, sph, abort) ||
            !mbar_wait_spin(bar_full + 8 * s, ph, abort)) {
          dqd_timeout(abort, 24);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t xd = smem_desc(base + static_cast<uint32_t>(s) * a.stage_bytes, 16, 1024, 2);
        if (issuer) {
#pragma unroll
          for (int kk = 0; kk < KC / 16; ++kk)
            mma_f16_ts(d, tmem_base + A_COL0 + slot * 32 + kk * 8, xd + 2 * kk, id,
                       (first && kk == 0) ? 0u : 1u);
          tc_commit(bar_empty + 8 * s);
          tc_commit(bar_a_free + 8 * slot);
        }
        __syncwarp();
        first = false;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (issuer) tc_commit(bar_acc_full + 8 * buf);
      __syncwarp();
    }
  } else if (warp >= DQ_W0 && warp < EPI_W0) {
    // ------------------------------------------------------------ dequantizers
    const int q = warp & 3, g = (warp - DQ_W0) >> 2;
    switch (a.fmt) {
      case FMT_INT4:
        dequant_loop<FMT_INT4, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
      case FMT_INT8:
        dequant_loop<FMT_INT8, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
      case FMT_INT2:
        dequant_loop<FMT_INT2, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
      case FMT_E2M1:
        dequant_loop<FMT_E2M1, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
      case FMT_E5M2:
        dequant_loop<FMT_E5M2, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
      default:
        dequant_loop<FMT_E4M3, LY::DQG>(a, rg, c, base, tmem_base, bar_full, bar_empty,
                               bar_a_ready, bar_a_free, q, g, lane, abort);
        break;
    }
  } else if (warp >= EPI_W0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t si = 0, n_split = 0;
    int nb = static_cast<int>(u0 / rg.kch);
    for (int64_t u = u0; u < u1; ++si, ++nb) {
      const int64_t blk0 = static_cast<int64_t>(nb) * rg.kch;
      const int64_t seg_end = min(u1, blk0 + rg.kch);
      const bool whole = (u == blk0 && seg_end == blk0 + rg.kch);
      const bool first_seg = (u == u0);
      u = seg_end;
      const uint32_t buf = si & 1u, use = si >> 1;
      if (!mbar_wait(bar_acc_full + 8 * buf, use & 1u, abort)) {
        dqd_timeout(abort, 25);
        break;
      }
      tc_fence_after();
      const int n = nb * WR + 32 * q + lane;   // weight row = column of C
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * NT;
      if (whole) {
#pragma unroll 1
        for (int cc = 0; cc < NT / 32; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + 32 * cc, r);
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          dec_epi(v, a.epi, n, a.N);
          dec_store<OUT>(v, a.C, a.ldc, 32 * cc, n, a.M, a.N);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
        continue;
      }
      // a range of a weight block that other CTAs share: its fp32 partial
      // to this CTA's slot (thread-major: each warp store writes 512
      // contiguous bytes), one arrival on the block's counter; the CTA that
      // completes the count sums the block's ranges in CTA order
      constexpr int CH = NT / 4;                       // float4 chunks per thread
      const size_t slice = static_cast<size_t>(WR) * NT;
      const size_t mine = (static_cast<size_t>(q) * CH * 32 + lane) * 4;
      float* own = a.ws + (static_cast<size_t>(c) * 2 + (first_seg ? 0 : 1)) * slice + mine;
#pragma unroll 1
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + 32 * cc, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(own + (8 * cc + j) * 128) =
              make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                          __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_written);
      const uint32_t par = n_split & 1u;
      ++n_split;
      const int c_first = rg.owner(blk0);
      const int c_last = rg.owner(blk0 + rg.kch - 1);
      if (warp == EPI_W0 && lane == 0) {
        int last = 0;
        if (mbar_wait_spin(bar_written, par, abort)) {
          __threadfence();
          const int cnt = dqd_arrive(a.ctr + nb, a.tag, c_last - c_first + 1);
          if (cnt < 0) dqd_timeout(abort, 27);
          last = (cnt == c_last - c_first + 1);
          __threadfence();
        } else {
          dqd_timeout(abort, 26);
        }
        *last_flag = last;
        mbar_arrive(bar_decided);
      }
      __syncwarp();
      if (!mbar_wait_spin(bar_decided, par, abort)) {
        dqd_timeout(abort, 28);
        break;
      }
      if (!*last_flag) continue;
      __threadfence();
      // CTA cp holds this block in its first slot when its range starts
      // inside the block, else (the block is where its range ends) in its
      // second
#pragma unroll 1
      for (int cc = 0; cc < NT / 32; ++cc) {
        float v[32];
        for (int cp = c_first; cp <= c_last; ++cp) {
          const int sl = (rg.begin(cp) >= blk0) ? 0 : 1;
          const float* src = a.ws + (static_cast<size_t>(cp) * 2 + sl) * slice + mine;
          float4 x[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = ld_global_cg_f4(src + (8 * cc + j) * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (cp == c_first) {
              v[4 * j] = x[j].x;
              v[4 * j + 1] = x[j].y;
              v[4 * j + 2] = x[j].z;
              v[4 * j + 3] = x[j].w;
            } else {
              v[4 * j] += x[j].x;
              v[4 * j + 1] += x[j].y;
              v[4 * j + 2] += x[j].z;
              v[4 * j + 3] += x[j].w;
            }
          }
        }
        dec_epi(v, a.epi, n, a.N);
        dec_store<OUT>(v, a.C, a.ldc, 32 * cc, n, a.M, a.N);
      }
    }
  }

  __syncwarp();   // reconverge before the aligned barrier (one-lane roles)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<1>(tmem_base, 512);
  }
}

int dqd_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cache[dev] = n;
  return n;
}

unsigned long long dqd_tag() {
  static std::atomic<unsigned long long> count{0};
  static const unsigned long long start = [] {
    unsigned long long z =
        static_cast<unsigned long long>(
            std::chrono::steady_clock::now().time_since_epoch().count()) ^
        (reinterpret_cast<uintptr_t>(&count) << 9);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
  }();
  for (;;) {
    const unsigned long long t = (start + count.fetch_add(1)) & ((1ull << 48) - 1);
    if (t != 0) return t;
  }
}

// Ranges over every SM (T units over G = min(SMs, T) CTAs); the workspace
// holds two partial slots per CTA and one counter per weight block.
size_t dqd_ws_bytes(int64_t M, int64_t N, int64_t K, int* grid) {
  const int nt = (M <= 64) ? 64 : 128;
  const int64_t nbk = (N + WR - 1) / WR, T = nbk * (K / KC);
  const int G = static_cast<int>(T < dqd_sm_count() ? T : dqd_sm_count());
  if (grid) *grid = G;
  return static_cast<size_t>(G) * 2 * WR * nt * sizeof(float) +
         static_cast<size_t>(nbk) * sizeof(unsigned long long);
}

template <int NT, int OUT>
cudaError_t dqd_run(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& tsf,
                    const DecArgs& a, int grid, cudaStream_t st) {
  auto kern = dqdec_kernel<NT, OUT>;
  const int smem = a.stages * a.stage_bytes + 8 * NBAR + 16 + 1024;
  static int attr_smem[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || attr_smem[dev] < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_smem[dev] = smem;
  }
  kern<<<grid, Lay<NT>::THREADS, smem, st>>>(tx, tw, tsf, a);
  return cudaGetLastError();
}

}  // namespace

// Whether the decode kernel takes this product (a few tokens, a plain or
// bias / activation output).
bool dequant_decode_applies(int64_t M, const Epilogue& epi) {
  return M >= 1 && M <= 128 && epi.q_fmt == 0;
}

// The kernel counts (weight block, chunk) units in 32 bits.
static bool dqd_units_fit(int64_t N, int64_t K) {
  return ((N + WR - 1) / WR) * (K / KC) < (int64_t{1} << 31);
}

size_t dequant_decode_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > 128 || N <= 0 || K <= 0 || K % KC) return 0;
  return dqd_ws_bytes(M, N, K, nullptr);
}

cudaError_t launch_gemm_dequant_decode(int a_dtype, const void* A, int64_t lda, int fmt_b,
                                       const void* b_data, const uint8_t* b_sf, void* C,
                                       int c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                       const Epilogue& epi, void* ws, size_t ws_bytes,
                                       cudaStream_t st) {
  if (!dqd_units_fit(N, K)) return cudaErrorInvalidValue;
  const int nt = (M <= 64) ? 64 : 128;
  int grid = 0;
  const size_t need = dqd_ws_bytes(M, N, K, &grid);
  DecArgs a{};
  a.C = C;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.fmt = fmt_b;
  a.a_bf16 = (a_dtype == DT_BF16) ? 1 : 0;
  a.code_row_bytes = KC * code_bits(fmt_b) / 8;
  a.x_bytes = nt * 128;
  a.stage_bytes = (a.x_bytes + WR * a.code_row_bytes + 512 + 1023) / 1024 * 1024;
  a.stages = SMEM_BUDGET / a.stage_bytes;
  if (a.stages > MAX_STAGES) a.stages = MAX_STAGES;
  a.epi.bias = epi.bias;
  a.epi.act = epi.act;
  a.epi.q_fmt = 0;
  a.epi.q_sf = nullptr;
  a.epi.q_k_atoms = 0;
  a.epi.q_row_atoms = 0;
  if (ws != nullptr && ws_bytes >= need) {
    a.whole = 0;
    a.ws = static_cast<float*>(ws);
    a.ctr = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + need -
                                                  ((N + WR - 1) / WR) * sizeof(unsigned long long));
    a.tag = dqd_tag();
  } else {
    // whole weight blocks per CTA: one CTA per block, up to one per SM
    const int64_t nbk = (N + WR - 1) / WR;
    grid = static_cast<int>(nbk < dqd_sm_count() ? nbk : dqd_sm_count());
    a.whole = 1;
  }
  const CUtensorMapDataType dt = (a_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t row_bytes = static_cast<uint64_t>(K) * code_bits(fmt_b) / 8;
  const uint64_t atoms = static_cast<uint64_t>(sf_row_atoms(N) * sf_k_atoms(K));
  CUtensorMap tx, tw, tsf;
  if (!make_tmap(&tx, A, dt, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(lda), 64, static_cast<uint32_t>(nt),
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tw, b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, row_bytes,
                 static_cast<uint64_t>(N), row_bytes, static_cast<uint32_t>(a.code_row_bytes), WR,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tmap(&tsf, b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128, atoms, 128, 128, 1,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const bool bf = (c_dtype == DT_BF16);
  if (nt == 64)
    return bf ? dqd_run<64, OUT_BF16>(tx, tw, tsf, a, grid, st)
              : dqd_run<64, OUT_F32>(tx, tw, tsf, a, grid, st);
  return bf ? dqd_run<128, OUT_BF16>(tx, tw, tsf, a, grid, st)
            : dqd_run<128, OUT_F32>(tx, tw, tsf, a, grid, st);
}

unsigned fetch_and_clear_status_dqd(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_dqd, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_dqd, &z, sizeof(z));
  return v;
}

}  // namespace mxk
