// gemm_kernel.cuh -- the persistent, warp-specialised tcgen05 GEMM kernel for
// sm_103a and its launch, shared by the translation units that instantiate it
// for each kind of operand (gemm_mxf8.cu, gemm_mxf4.cu, gemm_f16.cu); gemm.cu
// holds the host entry points and picks the configuration.
//
// What is computed: C = A * B with fp32 accumulation (dicastech tutorial
// "Treinar LLM em Swift", Passo 4-6: tiled matmul, FP16 variant); for the MX
// kinds the operands are quantized tensors (data plane + UE8M0 scale plane,
// one scale per 32 K) and the dequantization happens inside the matmul
// (WWDC26 session 330, "Quantized matrix multiplication", 7:19 listing):
// here the tensor core applies the two scales per 32-wide K block itself.
//
// Kinds: kind::f16 (fp16 / bf16 operands), kind::mxf8f6f4 block-scaled
// E4M3 / E5M2 (either operand may instead be E2M1, which TMA unpacks into the
// 8-bit shared-memory layout) and kind::mxf4 block-scaled packed E2M1 on both
// sides; fp32 accumulation in tensor memory.
//
// Configurations (template arguments): CG = 2, a cluster of two CTAs on two
// SMs sharing one (256 x TBN) tile through tcgen05 cta_group::2, each CTA
// staging its own 128 rows of A and its TBN / 2 rows of B; CG = 1, one CTA
// and a 128 x TBN tile.  TBN = 256, or 128 for problems whose 256-wide tiles
// leave SMs idle (measured: N = 128 runs the MMA at the full per-clock rate
// in both CTA-group forms, N = 64 at two thirds).
//
//   * persistent: each cluster walks its work items (whole tiles in a grouped
//     raster order, then the K ranges of split tiles) so that co-running
//     clusters share A and B tiles in L2;
//   * warp 0: TMA producer -- A, B (128-byte swizzle, 128 bytes of K per row
//     per stage) and the stage's scale atoms, into a STAGES-deep ring; in a
//     pair, both CTAs' copies complete on the leader's "full" barrier;
//   * warp 1: tensor-memory allocation; in the leader, the whole warp runs
//     the MMA loop and one elected lane issues 4 MMAs per stage, commits each
//     stage back to both producers and, per item, the accumulator to both
//     epilogues;
//   * warp 10 (MX kinds): copies each landed stage's scale atoms into tensor
//     memory (tcgen05.cp) and commits them to the stage's sf_ready barrier;
//   * warps 2..9: epilogue -- each warp drains TBN / 2 accumulator columns of
//     its 32-lane quarter into registers and hands the accumulator back at
//     once.  A K range of a split tile goes to the workspace; the last of a
//     tile's ranges to finish sums them all in a fixed order.  Whole (or
//     summed) tiles get bias and activation when asked (the fused GEMM + bias
//     + GELU of the RIGEL summary, Main findings section 4) and are stored as
//     fp32, bf16 (RNE), or quantized to an MX tensor for the next layer.
//     A CTA's last tile, whose store no main loop hides, is staged in the
//     (then idle) operand ring and written by TMA stores; earlier tiles are
//     stored from registers while the next tile's main loop runs.
// Tensor memory: accumulator(s) in columns [0, 256) -- one of 256 columns, or
// two of 128 taken by alternate tiles; per-stage scales from column 256.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in the translation unit's status word and the CTA shuts down in
// order.
#pragma once
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "mx_rule.cuh"
#include "ptx.cuh"

namespace mxk {
namespace gemm {

// One status word per translation unit that instantiates the kernel (no
// relocatable device code): gemm.cu reads and clears each of them.
static __device__ unsigned int g_status = 0;

enum Kind : int { KIND_F16 = 0, KIND_BF16 = 1, KIND_MXF8 = 2, KIND_MXF4 = 3 };

constexpr int TMEM_COLS = 512;
constexpr int SF_TMEM_BASE = 256;
constexpr int MMAS_PER_STAGE = 4;    // 4 x 32 bytes of K per 128-byte stage row
// warp roles
constexpr int EPI_WARP0 = 2;         // warps 2..9: epilogue
constexpr int NUM_EPI_WARPS = 8;
constexpr int SF_WARP = EPI_WARP0 + NUM_EPI_WARPS;    // warp 10: scale-factor copies
constexpr int NUM_THREADS = 32 * (SF_WARP + 1);       // 352

// A stage holds 128 bytes of K per operand row (one 128-byte-swizzled
// region); 4 MMAs per stage.
template <int KIND>
struct KT {
  static constexpr bool MX = (KIND == KIND_MXF8 || KIND == KIND_MXF4);
  static constexpr int KPS = (KIND == KIND_MXF4) ? 256 : (MX ? 128 : 64);   // K per stage
  static constexpr int MMA_K = KPS / MMAS_PER_STAGE;
  static constexpr int CK = MX ? KPS / 128 : 0;   // scale atoms (128 K each) per stage
};

template <int KIND, int CG, int TBN, int STAGES>
struct Smem {
  static constexpr int A_BYTES = BM * 128;                // this CTA's 128 rows of A
  static constexpr int B_BYTES = (TBN / CG) * 128;        // this CTA's part of B
  static constexpr int SFA_BYTES = KT<KIND>::CK * 512;    // this CTA's 128 rows
  static constexpr int SFB_BYTES = (TBN / 128) * KT<KIND>::CK * 512;   // all TBN rows
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int SFA_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + STAGES * SFA_BYTES;
  static constexpr int BAR_OFF = (SFB_OFF + STAGES * SFB_BYTES + 7) / 8 * 8;
  // accumulator buffers in tensor memory: two for 128-wide tiles, so that
  // the MMAs of the next tile never wait for the epilogue's drain
  static constexpr int ACC_BUFS = (TBN == 128) ? 2 : 1;
  // full[STAGES], empty[STAGES], sf_ready[STAGES], acc_full[ACC_BUFS],
  // acc_empty[ACC_BUFS], part_written, decided
  static constexpr int MISC_OFF = BAR_OFF + (3 * STAGES + 2 * ACC_BUFS + 2) * 8;
  static constexpr int TOTAL = MISC_OFF + 16;   // tmem slot, abort flag, last flag
  static constexpr int ALLOC = TOTAL + 1024;    // slack to align the base to 1024
  // TMEM columns of scale factors per stage: A then B
  static constexpr int SF_COLS = KT<KIND>::CK * 4 * (1 + TBN / 128);
  // accumulator columns each epilogue warp drains (two warps per lane quarter)
  static constexpr int EPI_COLS = TBN / (NUM_EPI_WARPS / 4);
  // one epilogue warp's staging region for a TMA-stored tile: 32 rows of
  // EPI_COLS fp32 values, as boxes of 32 rows x 128 bytes
  static constexpr int STAGE_C_BYTES = 32 * EPI_COLS * 4;
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(ACC_BUFS * TBN <= SF_TMEM_BASE, "accumulators must fit below the scales");
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(NUM_EPI_WARPS * STAGE_C_BYTES <= STAGES * (A_BYTES + B_BYTES),
                "the last tile's staging fits in the operand ring");
};

// Instruction descriptor, kind::f16: D f32, A/B f16 or bf16, A K-major,
// B MN-major, N>>3 at bit 17, M>>4 at bit 24 (M = 128 per CTA of the group).
template <int KIND, int CG, int TBN>
__host__ __device__ constexpr uint32_t idesc_f16() {
  return (1u << 4) | ((KIND == KIND_BF16 ? 1u : 0u) << 7) |
         ((KIND == KIND_BF16 ? 1u : 0u) << 10) | (0u << 15) | (1u << 16) |
         (static_cast<uint32_t>(TBN >> 3) << 17) |
         (static_cast<uint32_t>((BM * CG) >> 4) << 24);
}

// Instruction descriptor, block-scaled kinds: both operands K-major, N>>3 at
// bit 17, scale type UE8M0 (bit 23), M>>4 at bit 24.  The A / B element
// formats (bits 7-9 / 10-12) are E2M1 = 1 for mxf4; for mxf8f6f4 they are a
// launch argument (fmt_field), and the scale-factor byte selectors (bits 4-5
// for B, 29-30 for A) are filled in per MMA.
template <int KIND, int CG, int TBN>
__host__ __device__ constexpr uint32_t idesc_mx() {
  return ((KIND == KIND_MXF4 ? 1u : 0u) << 7) | ((KIND == KIND_MXF4 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(TBN >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>((BM * CG) >> 4) << 24);
}

// Work items: [0, full_tiles) are whole tiles in raster order; the remaining
// tiles (the last, partial wave) are each split into `split` K ranges, one
// work item per range.  Each range's fp32 partial tile goes to the workspace;
// the last range of a tile to finish sums them.
struct WorkList {
  TileSched sched;
  int num_kb;
  int full_tiles;
  int split;
  int total;
  __host__ __device__ void init(int num_m, int num_n, int kb, int full, int sp, int group) {
    sched.num_m = num_m;
    sched.num_n = num_n;
    sched.total = num_m * num_n;
    sched.group = group;
    num_kb = kb;
    full_tiles = full;
    split = sp;
    total = full + (sched.total - full) * sp;
  }
  // unit < 0: a whole tile; else the range's index among the split ranges
  // (split tile unit / split, range unit % split)
  __host__ __device__ __forceinline__ void item(int w, int& mb, int& nb, int& kb0, int& kb1,
                                                int& unit) const {
    if (w < full_tiles) {
      sched.tile(w, mb, nb);
      kb0 = 0;
      kb1 = num_kb;
      unit = -1;
    } else {
      const int u = w - full_tiles;
      const int sp = u % split;
      sched.tile(full_tiles + u / split, mb, nb);
      kb0 = sp * num_kb / split;
      kb1 = (sp + 1) * num_kb / split;
      unit = u;
    }
  }
};

// Kernel arguments besides the tensor maps.
struct Args {
  void* C;
  int64_t ldc;
  int M, N, K;
  float* ws;                  // partial tiles of the split ranges
  unsigned long long* ctr;    // one arrival counter per (split tile, CTA of the group)
  unsigned long long tag;     // this launch's 48-bit counter tag (non-zero)
  int full_tiles;
  int split;
  int group;                  // raster group height in tile rows
  uint32_t ab_fmt;
  EpiArgs epi;
};

__device__ __forceinline__ void record_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status, STATUS_TIMEOUT | site);
}

// Count one arrival on a split tile's counter and return the count including
// this one, or -1 if the update did not go through.  The word holds
// tag << 16 | count; a word carrying another tag (whatever the caller's
// workspace held) counts as zero, so a fresh workspace needs no clearing.
// The arrival that completes the count (`target`) writes zero instead, so
// every completed launch leaves its counters at zero: a launch replayed from
// a CUDA graph, which reuses its tag, counts from zero again.
__device__ __forceinline__ int tagged_arrive(unsigned long long* ctr, unsigned long long tag,
                                             int target) {
  // first guess zero, what a completed launch leaves: the first arrival then
  // takes one atomic round trip instead of a read and an atomic
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

// Stage one epilogue warp's 32 rows x NC values (fp32 or bf16) in shared
// memory as boxes of 32 rows x 128 bytes with the 128-byte swizzle (16-byte
// chunk c of row r at chunk position c ^ (r % 8): eight consecutive lanes
// hit eight different bank groups), then write them with TMA stores, which
// clip the rows beyond M and columns beyond N of a box that starts inside C
// (boxes that start outside are not issued).  Lane = row.  Returns once the
// stores have read the staging buffer (the CTA's last use of it); their
// writes complete before the grid does.
template <int OUT, int NC>
__device__ __forceinline__ void store_tile_tma(const uint32_t (&r)[NC], uint32_t stage,
                                               const CUtensorMap* tmC, int x0, int y0, int M,
                                               int N, int lane) {
  constexpr int BOX_COLS = (OUT == OUT_BF16) ? 64 : 32;
  constexpr int NBOX = NC / BOX_COLS;
  static_assert(NC % BOX_COLS == 0, "whole boxes per warp");
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sw = static_cast<uint32_t>(lane & 7);
#pragma unroll
  for (int b = 0; b < NBOX; ++b) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w0, w1, w2, w3;
      if (OUT == OUT_BF16) {
        const int e = b * 64 + 8 * c;
        w0 = cvt_bf16x2(__uint_as_float(r[e + 0]), __uint_as_float(r[e + 1]));
        w1 = cvt_bf16x2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        w2 = cvt_bf16x2(__uint_as_float(r[e + 4]), __uint_as_float(r[e + 5]));
        w3 = cvt_bf16x2(__uint_as_float(r[e + 6]), __uint_as_float(r[e + 7]));
      } else {
        const int e = b * 32 + 4 * c;
        w0 = r[e + 0];
        w1 = r[e + 1];
        w2 = r[e + 2];
        w3 = r[e + 3];
      }
      st_shared_v4(row + b * 4096u + ((static_cast<uint32_t>(c) ^ sw) << 4), w0, w1, w2, w3);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && y0 < M) {
#pragma unroll
    for (int b = 0; b < NBOX; ++b)
      if (x0 + b * BOX_COLS < N) tma_store_2d(tmC, stage + b * 4096u, x0 + b * BOX_COLS, y0);
    bulk_commit();
    bulk_wait_read();
  }
  __syncwarp();
}

template <int KIND, int CG, int TBN, int STAGES, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmSFA,
            const __grid_constant__ CUtensorMap tmSFB,
            const __grid_constant__ CUtensorMap tmC, const Args args) {
  using T = KT<KIND>;
  using L = Smem<KIND, CG, TBN, STAGES>;
  constexpr int EPI_COLS = L::EPI_COLS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t bar_full = base + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_sf_ready = bar_empty + 8 * STAGES;
  const uint32_t bar_acc_full = bar_sf_ready + 8 * STAGES;        // [ACC_BUFS]
  const uint32_t bar_acc_empty = bar_acc_full + 8 * L::ACC_BUFS;   // [ACC_BUFS]
  const uint32_t bar_written = bar_acc_empty + 8 * L::ACC_BUFS;
  const uint32_t bar_decided = bar_written + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  const int M = args.M, N = args.N, K = args.K;

  const int num_kb = (K + T::KPS - 1) / T::KPS;
  const int k_atoms = (K + 127) / 128;
  WorkList work;
  work.init((M + BM * CG - 1) / (BM * CG), (N + TBN - 1) / TBN, num_kb, args.full_tiles,
            args.split, args.group);
  // MMAs in a tile's last (possibly partial) stage
  const int last_nmma = min(MMAS_PER_STAGE,
                            (K - (num_kb - 1) * T::KPS + T::MMA_K - 1) / T::MMA_K);

  if (warp == 0) {
    // one barrier per lane (the barriers are consecutive 8-byte words):
    // full, empty, sf_ready per stage, then acc_full, acc_empty per
    // accumulator, then part_written and decided
    constexpr int NBAR = 3 * STAGES + 2 * L::ACC_BUFS + 2;
    static_assert(NBAR <= 32, "one barrier per lane");
    if (lane < NBAR) {
      uint32_t count = 1;
      if (lane >= 3 * STAGES + L::ACC_BUFS && lane < 3 * STAGES + 2 * L::ACC_BUFS)
        count = CG * NUM_EPI_WARPS;                              // acc_empty
      else if (lane == 3 * STAGES + 2 * L::ACC_BUFS)
        count = NUM_EPI_WARPS;                                   // part_written
      mbar_init(bar_full + 8 * lane, count);
      fence_mbar_init();
    }
    if (lane == 0) {
      *abort = 0;
      *last_flag = 0;
    }
    // the descriptors' first use is on the critical path: fetch them now
    if (lane == 0) prefetch_tmap(&tmA);
    if (lane == 1) prefetch_tmap(&tmB);
    if (lane == 2 && (OUT == OUT_F32 || OUT == OUT_BF16)) prefetch_tmap(&tmC);
    if (T::MX && lane == 3) prefetch_tmap(&tmSFA);
    if (T::MX && lane == 4) prefetch_tmap(&tmSFB);
  }
  if (warp == 1) tmem_alloc_cg<CG>(smem_u32(tmem_slot), TMEM_COLS);
  __syncwarp();   // reconverge before the aligned barrier (lane-dependent setup)
  tc_fence_before();
  if (CG == 2)
    cluster_sync();   // peers' barriers are initialised before any remote use
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // all copies of the group complete on the leader's full barrier
      const uint32_t full0 = (CG == 2) ? map_to_cta(bar_full, 0) : bar_full;
      uint32_t it = 0;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // Bytes one stage's copies complete on the full barrier.  TMA counts an
      // E2M1 operand that it unpacks for the FP8-rate kernel at its packed
      // size, half of what it occupies in shared memory.
      uint32_t stage_tx = L::STAGE_TX;
      if (KIND == KIND_MXF8) {
        if (((args.ab_fmt >> 7) & 7u) == 5u) stage_tx -= L::A_BYTES / 2;
        if (((args.ab_fmt >> 10) & 7u) == 5u) stage_tx -= L::B_BYTES / 2;
      }
      for (int w = cluster_id; w < work.total && ok; w += num_clusters) {
        int mb, nb, kb0, kb1, unit;
        work.item(w, mb, nb, kb0, kb1, unit);
        const int m0 = mb * BM * CG + static_cast<int>(rank) * BM;   // this CTA's rows
        const int nb_cta = nb * TBN + static_cast<int>(rank) * (TBN / CG);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) {
            record_timeout(abort, 1);
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, CG * stage_tx);
          const uint32_t full = full0 + 8 * s;
          const uint32_t a_dst = base + L::A_OFF + s * L::A_BYTES;
          const uint32_t b_dst = base + L::B_OFF + s * L::B_BYTES;
          if (T::MX) {
            // data planes are byte matrices: x counts bytes of K
            const int kx = kb * 128;
            tma_load_2d_cg<CG>(a_dst, &tmA, full, kx, m0);
            tma_load_2d_cg<CG>(b_dst, &tmB, full, kx, nb_cta);
            // scale planes viewed as [atoms][128 x u32]: one box = CK atoms;
            // each CTA takes the atoms of its own A rows and of all TBN rows
            tma_load_2d_cg<CG>(base + L::SFA_OFF + s * L::SFA_BYTES, &tmSFA, full, 0,
                               (m0 / 128) * k_atoms + kb * T::CK);
            for (int h = 0; h < TBN / 128; ++h)
              tma_load_2d_cg<CG>(base + L::SFB_OFF + s * L::SFB_BYTES + h * T::CK * 512,
                                 &tmSFB, full, 0,
                                 (nb * (TBN / 128) + h) * k_atoms + kb * T::CK);
          } else {
            const int k0 = kb * T::KPS;
            tma_load_2d_cg<CG>(a_dst, &tmA, full, k0, m0);
            // B is K x N row-major: boxes of 64 (N) x 64 (K rows)
            for (int j = 0; j < TBN / CG / 64; ++j)
              tma_load_2d_cg<CG>(b_dst + j * 64 * 128, &tmB, full, nb_cta + 64 * j, k0);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // let copies already issued land before the CTA retires
        const uint32_t first = it >= STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) {
          const uint32_t b = bar_full + 8 * (i % STAGES);
          const long long t0 = clock64();
          while (!mbar_try_wait(b, (i / STAGES) & 1u) &&
                 clock64() - t0 < MXK_WAIT_LIMIT_CYCLES) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One lane of the leader issues every MMA of the group.  The issuing
    // thread is the critical path (each tcgen05.mma occupies it for about as
    // long as the tensor core takes to run it), so it does nothing else per
    // stage: one wait, the stage's MMAs, one commit.  The whole warp runs the
    // loop, so that its descriptors and addresses are warp-uniform, and the
    // elected lane issues (measured: MXFP4 8192^3 0.191 -> 0.164 ms, MXFP8
    // 0.331 -> 0.322 ms against the same loop in lane 0 alone).  Scale
    // factors are copied into tensor memory by the scale-copy warp.
    if (leader) {
      const bool issuer = elect_one();
      const uint64_t a_desc0 = smem_desc(base + L::A_OFF, 16, 1024, 2);
      const uint64_t b_desc0 = T::MX ? smem_desc(base + L::B_OFF, 16, 1024, 2)
                                     : smem_desc(base + L::B_OFF, 64 * 128, 1024, 2);
      // per MMA: A advances 32 bytes of K; B 32 bytes (K-major) or 16 K rows
      // of 128 bytes (MN-major); descriptors count 16-byte units
      constexpr uint32_t A_STEP = 32 >> 4;
      constexpr uint32_t B_STEP = (T::MX ? 32 : 2048) >> 4;
      int s = 0;
      uint32_t ph = 0;
      uint32_t tc = 0;
      bool ok = true;
      for (int w = cluster_id; w < work.total && ok; w += num_clusters, ++tc) {
        int mb, nb, kb0, kb1, unit;
        work.item(w, mb, nb, kb0, kb1, unit);
        // the hand-off is short and on the critical path: spin
        const uint32_t buf = tc % L::ACC_BUFS, use = tc / L::ACC_BUFS;
        if (!mbar_wait_spin(bar_acc_empty + 8 * buf, (use & 1u) ^ 1u, abort)) {
          record_timeout(abort, 2);
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem_base + buf * TBN;
        for (int kb = kb0; kb < kb1; ++kb) {
          // MX: the scale copy of this stage is done (which implies its data
          // has landed); 16-bit kinds: the data has landed
          const uint32_t ready = (T::MX ? bar_sf_ready : bar_full) + 8 * s;
          if (!mbar_wait(ready, ph, abort)) {
            record_timeout(abort, 3);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_d = a_desc0 + static_cast<uint64_t>((s * L::A_BYTES) >> 4);
          const uint64_t b_d = b_desc0 + static_cast<uint64_t>((s * L::B_BYTES) >> 4);
          const uint32_t sfa_t = tmem_base + SF_TMEM_BASE + s * L::SF_COLS;
          const uint32_t sfb_t = sfa_t + T::CK * 4;
          const int nmma = (kb + 1 < num_kb) ? MMAS_PER_STAGE : last_nmma;
#pragma unroll
          for (int m = 0; m < MMAS_PER_STAGE; ++m) {
            if (m < nmma) {
              const uint32_t acc = (kb > kb0 || m > 0) ? 1u : 0u;
              const uint64_t ad = a_d + m * A_STEP;
              const uint64_t bd = b_d + m * B_STEP;
              if (!issuer) {
              } else if (KIND == KIND_F16 || KIND == KIND_BF16) {
                mma_f16_cg<CG>(d_acc, ad, bd, idesc_f16<KIND, CG, TBN>(), acc);
              } else if (KIND == KIND_MXF8) {
                // one scale atom (4 blocks) per stage; byte m of it
                constexpr uint32_t ID = idesc_mx<KIND, CG, TBN>();
                mma_mxf8_cg<CG>(d_acc, ad, bd,
                                ID | args.ab_fmt | (static_cast<uint32_t>(m) << 4) |
                                    (static_cast<uint32_t>(m) << 29),
                                sfa_t, sfb_t, acc);
              } else {
                // two scale atoms per stage, two MMAs per atom; bytes {0,1}
                // or {2,3} of it
                constexpr uint32_t ID = idesc_mx<KIND, CG, TBN>();
                const int c = m >> 1;
                const uint32_t sf_id = static_cast<uint32_t>((m & 1) * 2);
                mma_mxf4_cg<CG>(d_acc, ad, bd, ID | (sf_id << 4) | (sf_id << 29),
                                sfa_t + 4 * c, sfb_t + c * 4 * (TBN / 128), acc);
              }
            }
          }
          if (issuer) tc_commit_cg<CG>(bar_empty + 8 * s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (issuer) tc_commit_cg<CG>(bar_acc_full + 8 * buf);
      }
    }
  } else if (warp < SF_WARP) {
    // ------------------------------------------------------------ epilogue
    const int we = warp - EPI_WARP0;                 // 0..7
    const int q = warp & 3;                          // TMEM lane quarter
    const int cg_ = we >> 2;                         // which EPI_COLS columns
    uint32_t tc = 0;
    uint32_t n_split = 0;   // split ranges this warp has handled (barrier parity)
    for (int w = cluster_id; w < work.total; w += num_clusters, ++tc) {
      int mb, nb, kb0, kb1, unit;
      work.item(w, mb, nb, kb0, kb1, unit);
      const uint32_t buf = tc % L::ACC_BUFS, use = tc / L::ACC_BUFS;
      if (!mbar_wait(bar_acc_full + 8 * buf, use & 1u, abort)) {
        record_timeout(abort, 4);
        break;
      }
      tc_fence_after();
      uint32_t r[EPI_COLS];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(buf * TBN + cg_ * EPI_COLS);
#pragma unroll
      for (int i = 0; i < EPI_COLS / 32; ++i)
        tmem_ld_32x32b_x32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_cluster(map_to_cta(bar_acc_empty + 8 * buf, 0));
        else
          mbar_arrive(bar_acc_empty + 8 * buf);
      }

      if constexpr (TBN == 256) {
        // 256-wide tiles are never split (the host plans splits on 128-wide
        // tiles, whose 64 values per thread leave registers for the sum)
        if (unit >= 0) {
          record_timeout(abort, 9);
          break;
        }
      } else if (unit >= 0) {
        // One K range of a split tile.  Its fp32 partial goes to the
        // workspace in a thread-major layout (each warp store writes 512
        // contiguous bytes, and the same thread of whichever CTA finishes the
        // tile reads it back the same way); then one arrival on the tile's
        // counter.  The CTA that completes the count sums the ranges in range
        // order -- the same order whichever CTA that is, so the result does
        // not depend on timing -- and stores the tile.
        const int tile = unit / args.split;
        constexpr int CHUNKS = EPI_COLS / 4;
        const size_t slice = static_cast<size_t>(BM) * TBN;   // floats per partial
        const size_t mine = (static_cast<size_t>(we) * CHUNKS * 32 + lane) * 4;
        float* own = args.ws + (static_cast<size_t>(unit) * CG + rank) * slice + mine;
#pragma unroll
        for (int v = 0; v < CHUNKS; ++v)
          *reinterpret_cast<float4*>(own + v * 128) =
              make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                          __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_written);
        const uint32_t par = n_split & 1u;
        ++n_split;
        // both hand-offs are short and on the tile's critical path: spin
        if (warp == EPI_WARP0 && lane == 0) {
          int last = 0;
          if (mbar_wait_spin(bar_written, par, abort)) {
            __threadfence();
            const int cnt = tagged_arrive(args.ctr + static_cast<size_t>(tile) * CG + rank,
                                          args.tag, args.split);
            if (cnt < 0) record_timeout(abort, 7);
            last = (cnt == args.split);
            __threadfence();
          } else {
            record_timeout(abort, 6);
          }
          *last_flag = last;
          mbar_arrive(bar_decided);
        }
        __syncwarp();
        if (!mbar_wait_spin(bar_decided, par, abort)) {
          record_timeout(abort, 8);
          break;
        }
        if (!*last_flag) continue;
        __threadfence();
        const float* tile_ws = args.ws + (static_cast<size_t>(tile) * args.split * CG + rank) *
                                             slice + mine;
        // Every range's partial, this CTA's own included, is in the
        // workspace: reload them in range order, each range's CHUNKS loads
        // issued together (one L2 round trip per range), and add them in
        // that order into r (indexed by constants only).
        for (int p = 0; p < args.split; ++p) {
          const float* src = tile_ws + static_cast<size_t>(p) * CG * slice;
          float4 x[CHUNKS];
#pragma unroll
          for (int v = 0; v < CHUNKS; ++v) x[v] = ld_global_cg_f4(src + v * 128);
#pragma unroll
          for (int v = 0; v < CHUNKS; ++v) {
            if (p == 0) {
              r[4 * v] = __float_as_uint(x[v].x);
              r[4 * v + 1] = __float_as_uint(x[v].y);
              r[4 * v + 2] = __float_as_uint(x[v].z);
              r[4 * v + 3] = __float_as_uint(x[v].w);
            } else {
              r[4 * v] = __float_as_uint(__uint_as_float(r[4 * v]) + x[v].x);
              r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + x[v].y);
              r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + x[v].z);
              r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + x[v].w);
            }
          }
        }
      }
      const int64_t row0 = static_cast<int64_t>(mb) * BM * CG + rank * BM + 32 * q;
      const int64_t row = row0 + lane;
      const int col0 = nb * TBN + cg_ * EPI_COLS;
      if (args.epi.bias != nullptr || args.epi.act != ACT_NONE)
        apply_bias_act(r, args.epi, col0, N);
      if constexpr (OUT == OUT_MX8 || OUT == OUT_MX4) {
        store_mx_row<OUT>(r, args.epi, static_cast<uint8_t*>(args.C), row, col0, M, N);
      } else if (w + num_clusters >= work.total) {
        // this CTA's last item: every MMA has completed and no load is
        // pending, so the operand ring is free to stage the tile
        store_tile_tma<OUT, EPI_COLS>(r, base + L::A_OFF + we * L::STAGE_C_BYTES, &tmC, col0,
                                      static_cast<int>(row0), M, N, lane);
      } else if (row < M) {
        store_row_segment<OUT, EPI_COLS>(r, args.C, args.ldc, row, col0, N);
      }
    }
  } else if (T::MX) {
    // ------------------------------------------------------------ scale copies
    // For every stage: once its data (and scale atoms) have landed, copy the
    // scale atoms into that stage's tensor-memory slot with tcgen05.cp (each
    // 512-byte atom -> 4 columns of every lane quarter), then commit the copies
    // to the stage's sf_ready barrier, which the MMA issuer waits on.  The
    // slot is free: the stage was refilled only after the MMAs that last read
    // it had completed.
    if (leader) {
      const bool issuer = elect_one();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int w = cluster_id; w < work.total && ok; w += num_clusters) {
        int mb, nb, kb0, kb1, unit;
        work.item(w, mb, nb, kb0, kb1, unit);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(bar_full + 8 * s, ph, abort)) {
            record_timeout(abort, 5);
            ok = false;
            break;
          }
          tc_fence_after();
          const int nmma = (kb + 1 < num_kb) ? MMAS_PER_STAGE : last_nmma;
          const int ck_used = (nmma * T::MMA_K + 127) / 128;
          const uint32_t sfa_t = tmem_base + SF_TMEM_BASE + s * L::SF_COLS;
          const uint32_t sfb_t = sfa_t + T::CK * 4;
          const uint32_t sfa_s = base + L::SFA_OFF + s * L::SFA_BYTES;
          const uint32_t sfb_s = base + L::SFB_OFF + s * L::SFB_BYTES;
          for (int c = 0; c < ck_used && issuer; ++c) {
            tc_cp_32x128b_x4_cg<CG>(sfa_t + 4 * c, smem_desc(sfa_s + c * 512, 0, 128, 0));
#pragma unroll
            for (int h = 0; h < TBN / 128; ++h)
              tc_cp_32x128b_x4_cg<CG>(sfb_t + c * 4 * (TBN / 128) + 4 * h,
                                      smem_desc(sfb_s + (h * T::CK + c) * 512, 0, 128, 0));
          }
          if (issuer) tc_commit_leader<CG>(bar_sf_ready + 8 * s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  }

  // Reconverge the warp first: some roles ran on one lane (the producer),
  // and an aligned block or cluster barrier must be reached by every lane of
  // a warp together.
  __syncwarp();
  tc_fence_before();
  if (CG == 2)
    cluster_sync();   // no CTA of the pair retires while the other may use it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<CG>(tmem_base, TMEM_COLS);
  }
}

// Everything one launch needs besides the configuration.
struct Launch {
  const CUtensorMap* ta;
  const CUtensorMap* tb;
  const CUtensorMap* tsa;
  const CUtensorMap* tsb;
  const CUtensorMap* tc;
  int clusters;
  Args args;
  cudaStream_t st;
};

template <int KIND, int CG, int TBN, int STAGES, int OUT>
cudaError_t run(const Launch& l) {
  using L = Smem<KIND, CG, TBN, STAGES>;
  auto kern = gemm_kernel<KIND, CG, TBN, STAGES, OUT>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.clusters * CG), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = l.st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *l.ta, *l.tb, *l.tsa, *l.tsb, *l.tc, l.args);
}

// Ring depth of each (CTA group, tile width): the deepest ring that fits
// shared memory.
template <int CG, int TBN>
struct Depth {
  static constexpr int STAGES = (CG == 2) ? (TBN == 256 ? 6 : 8) : (TBN == 256 ? 4 : 6);
};

// Launch the kernel of one kind for a configuration picked at run time:
// cg (1 or 2), tbn (128 or 256), out (OUT_*).  Only tbn = 256 carries the
// MX-quantized outputs (one thread must hold four whole 32-column blocks).
// Defined by the translation unit of each kind.
cudaError_t launch_mxf8(int cg, int tbn, int out, const Launch& l);
cudaError_t launch_mxf4(int cg, int tbn, int out, const Launch& l);
cudaError_t launch_f16(int kind, int cg, int tbn, const Launch& l);
unsigned fetch_and_clear_status_mxf8(cudaError_t* err);
unsigned fetch_and_clear_status_mxf4(cudaError_t* err);
unsigned fetch_and_clear_status_f16(cudaError_t* err);

// Dispatch over the configurations for one kind (used by those units).
template <int KIND, int OUT>
cudaError_t launch_cfg(int cg, int tbn, const Launch& l) {
  if (cg == 2) {
    if (tbn == 256) return run<KIND, 2, 256, Depth<2, 256>::STAGES, OUT>(l);
    if constexpr (OUT == OUT_F32 || OUT == OUT_BF16)
      return run<KIND, 2, 128, Depth<2, 128>::STAGES, OUT>(l);
  } else {
    if (tbn == 256) return run<KIND, 1, 256, Depth<1, 256>::STAGES, OUT>(l);
    if constexpr (OUT == OUT_F32 || OUT == OUT_BF16)
      return run<KIND, 1, 128, Depth<1, 128>::STAGES, OUT>(l);
  }
  return cudaErrorInvalidValue;
}

inline unsigned fetch_and_clear_status_tu(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status, &z, sizeof(z));
  return v;
}

}  // namespace gemm
}  // namespace mxk
