// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   kind::f16 (fp16 / bf16 operands), kind::mxf8f6f4 block-scaled E4M3 / E5M2
//   (either operand may instead be E2M1, which TMA unpacks into the 8-bit
//   shared-memory layout) and kind::mxf4 block-scaled packed E2M1 on both
//   sides, fp32 accumulation in tensor memory.
//
// What is computed: C = A * B with fp32 accumulation (dicastech tutorial
// "Treinar LLM em Swift", Passo 4-6: tiled matmul, FP16 variant); for the MX
// kinds the operands are quantized tensors (data plane + UE8M0 scale plane,
// one scale per 32 K) and the dequantization happens inside the matmul
// (WWDC26 session 330, "Quantized matrix multiplication", 7:19 listing):
// here the tensor core applies the two scales per 32-wide K block itself.
//
// Design (GB300-first, not the pages' threadgroup-tile design):
//   * CG = 2 (default): a cluster of two CTAs on two SMs shares one
//     256 (M) x 256 (N) MMA tile (tcgen05 cta_group::2).  Each CTA stages its
//     own 128 rows of A and its own 128-row half of B, so per SM a stage is
//     32 KB of operands for 256 x 256 x (128 bytes of K) of work; the leader
//     CTA (rank 0) issues the MMAs for both.  CG = 1: one CTA, 128 x 256.
//   * persistent: each cluster walks the tiles in a grouped raster order so
//     that co-running clusters share A and B tiles in L2;
//   * warp 0: TMA producer -- A, B (128-byte swizzle, 128 bytes of K per row
//     per stage) and the stage's scale atoms, into a STAGES-deep ring; in a
//     pair, both CTAs' copies complete on the leader's "full" barrier;
//   * warp 1: tensor-memory allocation; in the leader, one thread issues the
//     scale-factor copies (tcgen05.cp) and 4 MMAs per stage, commits each
//     stage back to both producers and, per tile, the accumulator to both
//     epilogues;
//   * warps 2..9: epilogue -- each warp drains 128 accumulator columns of its
//     32-lane quarter into registers, hands the accumulator back to the MMA
//     issuer at once, then, while the next tile's main loop runs, adds the
//     bias and applies the activation when asked (the fused GEMM + bias +
//     GELU kernel of the RIGEL summary, Main findings section 4) and stores
//     fp32, bf16 (RNE), or C quantized to an MX tensor for the next layer:
//     one thread holds one row's 128 columns, i.e. four whole 32-blocks.
// Tensor memory: accumulator in columns [0, BN); per-stage scales from 256.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_gemm and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "mx_rule.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

__device__ unsigned int g_status_gemm = 0;

enum Kind : int { KIND_F16 = 0, KIND_BF16 = 1, KIND_MXF8 = 2, KIND_MXF4 = 3 };

constexpr int TMEM_COLS = 512;
constexpr int SF_TMEM_BASE = 256;
constexpr int MMAS_PER_SUB = 4;      // 4 x 32 bytes of K per 128-byte sub-tile
// warp roles
constexpr int EPI_WARP0 = 2;         // warps 2..9: epilogue, EPI_COLS columns each
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_COLS = BN / (NUM_EPI_WARPS / 4);
constexpr int SF_WARP = EPI_WARP0 + NUM_EPI_WARPS;    // warp 10: scale-factor copies
constexpr int NUM_THREADS = 32 * (SF_WARP + 1);       // 352

// A stage holds KSUB sub-tiles of 128 bytes of K per operand row (each its
// own 128-byte-swizzled region); 4 MMAs per sub-tile.
template <int KIND, int KSUB>
struct KT {
  static constexpr bool MX = (KIND == KIND_MXF8 || KIND == KIND_MXF4);
  // K elements per 128-byte sub-tile, and per stage
  static constexpr int KPSUB = (KIND == KIND_MXF4) ? 256 : (MX ? 128 : 64);
  static constexpr int KPS = KPSUB * KSUB;
  static constexpr int MMAS_PER_STAGE = MMAS_PER_SUB * KSUB;
  static constexpr int MMA_K = KPSUB / MMAS_PER_SUB;
  // scale atoms (128 K each) per stage along K
  static constexpr int CK = MX ? KPS / 128 : 0;
};

template <int KIND, int CG, int STAGES, int KSUB>
struct Smem {
  static constexpr int A_SUB = BM * 128;                // one sub-tile of A
  static constexpr int B_SUB = (BN / CG) * 128;         // this CTA's part of B
  static constexpr int A_BYTES = A_SUB * KSUB;
  static constexpr int B_BYTES = B_SUB * KSUB;
  static constexpr int SFA_BYTES = KT<KIND, KSUB>::CK * 512;  // this CTA's 128 rows
  static constexpr int SFB_BYTES = (BN / 128) * KT<KIND, KSUB>::CK * 512;  // all of BN
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int SFA_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + STAGES * SFA_BYTES;
  static constexpr int BAR_OFF = (SFB_OFF + STAGES * SFB_BYTES + 7) / 8 * 8;
  // full[STAGES], empty[STAGES], sf_ready[STAGES], acc_full, acc_empty
  static constexpr int MISC_OFF = BAR_OFF + (3 * STAGES + 2) * 8;
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;   // slack to align the base to 1024
  // TMEM columns of scale factors per stage: A then B
  static constexpr int SF_COLS = KT<KIND, KSUB>::CK * 4 * (1 + BN / 128);
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(BN <= SF_TMEM_BASE, "accumulator must fit below the scales");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Instruction descriptor, kind::f16: D f32, A/B f16 or bf16, A K-major,
// B MN-major, N>>3 at bit 17, M>>4 at bit 24 (M = 128 per CTA of the group).
template <int KIND, int CG>
__host__ __device__ constexpr uint32_t idesc_f16() {
  return (1u << 4) | ((KIND == KIND_BF16 ? 1u : 0u) << 7) |
         ((KIND == KIND_BF16 ? 1u : 0u) << 10) | (0u << 15) | (1u << 16) |
         (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>((BM * CG) >> 4) << 24);
}

// Instruction descriptor, block-scaled kinds: both operands K-major, N>>3 at
// bit 17, scale type UE8M0 (bit 23), M>>4 at bit 24.  The A / B element
// formats (bits 7-9 / 10-12) are E2M1 = 1 for mxf4; for mxf8f6f4 they are a
// launch argument (fmt_field), and the scale-factor byte selectors (bits 4-5
// for B, 29-30 for A) are filled in per MMA.
template <int KIND, int CG>
__host__ __device__ constexpr uint32_t idesc_mx() {
  return ((KIND == KIND_MXF4 ? 1u : 0u) << 7) | ((KIND == KIND_MXF4 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>((BM * CG) >> 4) << 24);
}

// Work items: [0, full_tiles) are whole tiles in raster order; the remaining
// tiles (the last, partial wave) are each split into `split` K ranges, one
// work item per range, whose fp32 partial tiles go to the workspace and are
// summed by reduce_partials_kernel.
struct WorkList {
  TileSched sched;
  int num_kb;
  int full_tiles;
  int split;
  int total;
  __host__ __device__ void init(int num_m, int num_n, int kb, int full, int sp) {
    sched.num_m = num_m;
    sched.num_n = num_n;
    sched.total = num_m * num_n;
    num_kb = kb;
    full_tiles = full;
    split = sp;
    total = full + (sched.total - full) * sp;
  }
  // unit < 0: a whole tile (write C); else index of the partial in the workspace
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

__device__ __forceinline__ void record_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_gemm, STATUS_TIMEOUT | site);
}

template <int KIND, int CG, int STAGES, int KSUB, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmSFA,
            const __grid_constant__ CUtensorMap tmSFB, void* __restrict__ Cptr,
            int64_t ldc, int M, int N, int K, float* __restrict__ ws, int full_tiles,
            int split, uint32_t ab_fmt, EpiArgs epi) {
  using T = KT<KIND, KSUB>;
  using L = Smem<KIND, CG, STAGES, KSUB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t bar_full = base + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_sf_ready = bar_empty + 8 * STAGES;
  const uint32_t bar_acc_full = bar_sf_ready + 8 * STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;

  const int num_kb = (K + T::KPS - 1) / T::KPS;
  const int k_atoms = (K + 127) / 128;
  WorkList work;
  work.init((M + BM * CG - 1) / (BM * CG), (N + BN - 1) / BN, num_kb, full_tiles, split);
  // MMAs in a tile's last (possibly partial) stage
  const int last_nmma = min(T::MMAS_PER_STAGE,
                            (K - (num_kb - 1) * T::KPS + T::MMA_K - 1) / T::MMA_K);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sf_ready + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, CG * NUM_EPI_WARPS);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (T::MX) {
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) tmem_alloc_cg<CG>(smem_u32(tmem_slot), TMEM_COLS);
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
        if (((ab_fmt >> 7) & 7u) == 5u) stage_tx -= L::A_BYTES / 2;
        if (((ab_fmt >> 10) & 7u) == 5u) stage_tx -= L::B_BYTES / 2;
      }
      for (int w = cluster_id; w < work.total && ok; w += num_clusters) {
        int mb, nb, kb0, kb1, unit;
        work.item(w, mb, nb, kb0, kb1, unit);
        const int m0 = mb * BM * CG + static_cast<int>(rank) * BM;   // this CTA's rows
        const int nb_cta = nb * BN + static_cast<int>(rank) * (BN / CG);
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
#pragma unroll
            for (int u = 0; u < KSUB; ++u) {
              const int kx = (kb * KSUB + u) * 128;
              tma_load_2d_cg<CG>(a_dst + u * L::A_SUB, &tmA, full, kx, m0);
              tma_load_2d_cg<CG>(b_dst + u * L::B_SUB, &tmB, full, kx, nb_cta);
            }
            // scale planes viewed as [atoms][128 x u32]: one box = CK atoms;
            // each CTA takes the atoms of its own A rows and of all BN rows
            tma_load_2d_cg<CG>(base + L::SFA_OFF + s * L::SFA_BYTES, &tmSFA, full, 0,
                               (m0 / 128) * k_atoms + kb * T::CK);
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d_cg<CG>(base + L::SFB_OFF + s * L::SFB_BYTES + h * T::CK * 512,
                                 &tmSFB, full, 0,
                                 (nb * (BN / 128) + h) * k_atoms + kb * T::CK);
          } else {
#pragma unroll
            for (int u = 0; u < KSUB; ++u) {
              const int k0 = kb * T::KPS + u * 64;
              tma_load_2d_cg<CG>(a_dst + u * L::A_SUB, &tmA, full, k0, m0);
              // B is K x N row-major: boxes of 64 (N) x 64 (K rows)
              for (int j = 0; j < BN / CG / 64; ++j)
                tma_load_2d_cg<CG>(b_dst + u * L::B_SUB + j * 64 * 128, &tmB, full,
                                   nb_cta + 64 * j, k0);
            }
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
        if (!mbar_wait_spin(bar_acc_empty, (tc & 1u) ^ 1u, abort)) {
          record_timeout(abort, 2);
          break;
        }
        tc_fence_after();
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
          const int nmma = (kb + 1 < num_kb) ? T::MMAS_PER_STAGE : last_nmma;
#pragma unroll
          for (int m = 0; m < T::MMAS_PER_STAGE; ++m) {
            if (m < nmma) {
              const uint32_t acc = (kb > kb0 || m > 0) ? 1u : 0u;
              const int u = m / MMAS_PER_SUB, mm = m % MMAS_PER_SUB;
              const uint64_t ad = a_d + ((u * L::A_SUB) >> 4) + mm * A_STEP;
              const uint64_t bd = b_d + ((u * L::B_SUB) >> 4) + mm * B_STEP;
              if (!issuer) {
              } else if (KIND == KIND_F16 || KIND == KIND_BF16) {
                mma_f16_cg<CG>(tmem_base, ad, bd, idesc_f16<KIND, CG>(), acc);
              } else if (KIND == KIND_MXF8) {
                // one scale atom (4 blocks) per sub-tile; byte mm of it
                constexpr uint32_t ID = idesc_mx<KIND, CG>();
                mma_mxf8_cg<CG>(tmem_base, ad, bd,
                                ID | ab_fmt | (static_cast<uint32_t>(mm) << 4) |
                                    (static_cast<uint32_t>(mm) << 29),
                                sfa_t + 4 * u, sfb_t + u * 4 * (BN / 128), acc);
              } else {
                // two scale atoms per sub-tile, two MMAs per atom; bytes
                // {0,1} or {2,3} of it
                constexpr uint32_t ID = idesc_mx<KIND, CG>();
                const int c = m >> 1;
                const uint32_t sf_id = static_cast<uint32_t>((m & 1) * 2);
                mma_mxf4_cg<CG>(tmem_base, ad, bd, ID | (sf_id << 4) | (sf_id << 29),
                                sfa_t + 4 * c, sfb_t + c * 4 * (BN / 128), acc);
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
        if (issuer) tc_commit_cg<CG>(bar_acc_full);
      }
    }
  } else if (warp < SF_WARP) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                          // TMEM lane quarter
    const int cg_ = (warp - EPI_WARP0) >> 2;         // which EPI_COLS columns
    const uint32_t acc_empty0 = (CG == 2) ? map_to_cta(bar_acc_empty, 0) : bar_acc_empty;
    uint32_t tc = 0;
    for (int w = cluster_id; w < work.total; w += num_clusters, ++tc) {
      int mb, nb, kb0, kb1, unit;
      work.item(w, mb, nb, kb0, kb1, unit);
      if (!mbar_wait(bar_acc_full, tc & 1u, abort)) {
        record_timeout(abort, 4);
        break;
      }
      tc_fence_after();
      uint32_t r[EPI_COLS];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(cg_ * EPI_COLS);
#pragma unroll
      for (int i = 0; i < EPI_COLS / 32; ++i)
        tmem_ld_32x32b_x32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_cluster(acc_empty0);
        else
          mbar_arrive(bar_acc_empty);
      }

      if (unit >= 0) {
        // partial of a split tile: the whole fp32 accumulator row segment to
        // the workspace (rows beyond M are left out, columns beyond N
        // included: the reduction reads neither)
        if (static_cast<int64_t>(mb) * BM * CG + rank * BM + 32 * q + lane < M) {
          float* wrow = ws + static_cast<int64_t>(unit) * (BM * CG * BN) +
                        static_cast<int64_t>(rank * BM + 32 * q + lane) * BN + cg_ * EPI_COLS;
          const bool wide = (reinterpret_cast<uintptr_t>(wrow) & 31u) == 0;
#pragma unroll
          for (int v = 0; v < EPI_COLS / 8; ++v)
            store_32B(wrow + 8 * v, *reinterpret_cast<const uint32_t(*)[8]>(r + 8 * v), wide);
        }
        continue;
      }
      const int64_t row = static_cast<int64_t>(mb) * BM * CG + rank * BM + 32 * q + lane;
      const int col0 = nb * BN + cg_ * EPI_COLS;
      if (epi.bias != nullptr || epi.act != ACT_NONE) apply_bias_act(r, epi, col0, N);
      if (OUT == OUT_MX8 || OUT == OUT_MX4) {
        store_mx_row<OUT>(r, epi, static_cast<uint8_t*>(Cptr), row, col0, M, N);
        continue;
      }
      if (row < M) store_row_segment<OUT, EPI_COLS>(r, Cptr, ldc, row, col0, N);
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
        const int nmma = (kb + 1 < num_kb) ? T::MMAS_PER_STAGE : last_nmma;
        const int ck_used = (nmma * T::MMA_K + 127) / 128;
        const uint32_t sfa_t = tmem_base + SF_TMEM_BASE + s * L::SF_COLS;
        const uint32_t sfb_t = sfa_t + T::CK * 4;
        const uint32_t sfa_s = base + L::SFA_OFF + s * L::SFA_BYTES;
        const uint32_t sfb_s = base + L::SFB_OFF + s * L::SFB_BYTES;
        for (int c = 0; c < ck_used && issuer; ++c) {
          tc_cp_32x128b_x4_cg<CG>(sfa_t + 4 * c, smem_desc(sfa_s + c * 512, 0, 128, 0));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tc_cp_32x128b_x4_cg<CG>(sfb_t + c * 4 * (BN / 128) + 4 * h,
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

// Sum the `split` fp32 partials of each split tile in a fixed order (so the
// result does not depend on timing) and write C.  CTA = (split tile r,
// group of 4 tile rows); each thread owns 4 consecutive columns.
template <int OUT>
__global__ void __launch_bounds__(256)
reduce_partials_kernel(const float* __restrict__ ws, void* __restrict__ Cptr, int64_t ldc,
                       int M, int N, WorkList work, int tile_rows) {
  const int r = blockIdx.x;
  int mb, nb;
  work.sched.tile(work.full_tiles + r, mb, nb);
  const int i = blockIdx.y * 4 + (threadIdx.x >> 6);          // row in tile
  const int c = (threadIdx.x & 63) * 4;                       // column in tile
  const int64_t row = static_cast<int64_t>(mb) * tile_rows + i;
  const int col = nb * BN + c;
  if (row >= M || col >= N) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < work.split; ++sp) {
    const float4 v = *reinterpret_cast<const float4*>(
        ws + (static_cast<int64_t>(r * work.split + sp) * tile_rows + i) * BN + c);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const float a[4] = {acc.x, acc.y, acc.z, acc.w};
  if (OUT == OUT_BF16) {
    uint16_t* crow = reinterpret_cast<uint16_t*>(Cptr) + row * ldc;
    const uint32_t lo = cvt_bf16x2(a[0], a[1]), hi = cvt_bf16x2(a[2], a[3]);
    if (col + 3 < N) {
      *reinterpret_cast<uint2*>(crow + col) = make_uint2(lo, hi);
    } else {
      const uint32_t w[2] = {lo, hi};
      for (int e = 0; e < 4 && col + e < N; ++e)
        crow[col + e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
    }
  } else {
    float* crow = reinterpret_cast<float*>(Cptr) + row * ldc;
    if (col + 3 < N) {
      *reinterpret_cast<float4*>(crow + col) = acc;
    } else {
      for (int e = 0; e < 4 && col + e < N; ++e) crow[col + e] = a[e];
    }
  }
}

// ---------------------------------------------------------------- host side


// The scale plane as rows of 512-byte atoms (128 x u32); one box = ck atoms.
bool make_sf_tmap(CUtensorMap* m, const uint8_t* sf, int64_t outer, int64_t K, int ck) {
  const uint64_t atoms = static_cast<uint64_t>(sf_row_atoms(outer) * sf_k_atoms(K));
  return make_tmap(m, sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128, atoms, 128, 128,
                   static_cast<uint32_t>(ck), CU_TENSOR_MAP_SWIZZLE_NONE);
}

int sm_count() {
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

// How the tiles of one GEMM are laid on the clusters.  Whole waves of tiles
// run as whole tiles; the tiles of a last, partial wave (or of a problem with
// fewer tiles than clusters) are split into `split` K ranges so that the idle
// clusters share their work, provided a workspace for the fp32 partials is
// given.  split = 1: no splitting.
struct SplitPlan {
  int clusters, full_tiles, split, rem;
  size_t ws_bytes;
};

SplitPlan plan_split(int64_t M, int64_t N, int64_t K, int kps, bool use_split) {
  const int cg = (M > BM) ? 2 : 1;
  const int64_t tiles = ((M + BM * cg - 1) / (BM * cg)) * ((N + BN - 1) / BN);
  const int maxc = sm_count() / cg;
  const int num_kb = static_cast<int>((K + kps - 1) / kps);
  SplitPlan p{static_cast<int>(tiles < maxc ? tiles : maxc), static_cast<int>(tiles), 1, 0, 0};
  if (!use_split || tiles == 0) return p;
  const int64_t full = (tiles / maxc) * maxc;
  const int rem = static_cast<int>(tiles - full);
  int sp = rem ? maxc / rem : 1;
  if (sp > 4) sp = 4;                          // bound the partial traffic
  if (sp > num_kb / 2) sp = num_kb / 2;        // at least 2 stages per range
  if (sp < 2) return p;
  p.clusters = maxc;
  p.full_tiles = static_cast<int>(full);
  p.split = sp;
  p.rem = rem;
  p.ws_bytes = static_cast<size_t>(rem) * sp * (BM * cg) * BN * sizeof(float);
  return p;
}

template <int KIND, int CG, int STAGES, int KSUB, int OUT>
cudaError_t run(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                const CUtensorMap& tsb, void* C, int64_t ldc, int M, int N, int K,
                const SplitPlan& plan, float* ws, uint32_t ab_fmt, const EpiArgs& epi,
                cudaStream_t st) {
  using L = Smem<KIND, CG, STAGES, KSUB>;
  auto kern = gemm_kernel<KIND, CG, STAGES, KSUB, OUT>;
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
  cfg.gridDim = dim3(static_cast<unsigned>(plan.clusters * CG), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, C, ldc, M, N, K, ws, plan.full_tiles,
                         plan.split, ab_fmt, epi);
  // a split problem is a plain one (no epilogue work, fp32 or bf16 C)
  if (e != cudaSuccess || plan.split < 2 || OUT == OUT_MX8 || OUT == OUT_MX4) return e;
  WorkList work;
  work.init((M + BM * CG - 1) / (BM * CG), (N + BN - 1) / BN,
            (K + KT<KIND, KSUB>::KPS - 1) / KT<KIND, KSUB>::KPS, plan.full_tiles, plan.split);
  dim3 grid(static_cast<unsigned>(plan.rem), BM * CG / 4);
  constexpr int ROUT = (OUT == OUT_BF16) ? OUT_BF16 : OUT_F32;
  reduce_partials_kernel<ROUT><<<grid, 256, 0, st>>>(ws, C, ldc, M, N, work, BM * CG);
  return cudaGetLastError();
}

// K sub-tiles per stage and ring depth; the ring holds the same bytes either
// way, more K per stage means fewer waits and commits per MMA
constexpr int KSUB_CG2 = 1;
constexpr int STAGES_CG2 = 6 / KSUB_CG2;
constexpr int KSUB_CG1 = 1;
constexpr int STAGES_CG1 = 4;

template <int KIND, int OUT>
cudaError_t dispatch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                     const CUtensorMap& tsb, void* C, int64_t ldc, int M, int N, int K,
                     const SplitPlan& plan, float* ws, uint32_t ab_fmt, const EpiArgs& epi,
                     cudaStream_t st) {
  if (M > BM)
    return run<KIND, 2, STAGES_CG2, KSUB_CG2, OUT>(ta, tb, tsa, tsb, C, ldc, M, N, K, plan, ws,
                                                  ab_fmt, epi, st);
  return run<KIND, 1, STAGES_CG1, KSUB_CG1, OUT>(ta, tb, tsa, tsb, C, ldc, M, N, K, plan, ws,
                                                ab_fmt, epi, st);
}

EpiArgs epi_args(const Epilogue& e, int64_t M, int64_t N) {
  EpiArgs a;
  a.bias = e.bias;
  a.act = e.act;
  a.q_fmt = e.q_fmt;
  a.q_sf = e.q_sf;
  a.q_k_atoms = sf_k_atoms(N);
  a.q_row_atoms = sf_row_atoms(M);
  return a;
}

bool plain_epilogue(const Epilogue& e) {
  return e.bias == nullptr && e.act == ACT_NONE && e.q_fmt == 0;
}

// K elements per stage of each kind (KSUB is the same for both CTA groups)
int stage_k(int kind) {
  static_assert(KSUB_CG1 == KSUB_CG2, "one K per stage for both CTA groups");
  return kind == KIND_MXF4 ? KT<KIND_MXF4, KSUB_CG2>::KPS
                           : kind == KIND_MXF8 ? KT<KIND_MXF8, KSUB_CG2>::KPS
                                               : KT<KIND_F16, KSUB_CG2>::KPS;
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D tensor map, row-major rows x cols (cols contiguous).
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  const cuuint32_t* estr, CUtensorMapSwizzle swz) {
  auto enc = get_encode();
  if (!enc) return false;
  return enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int elem_bytes,
               uint64_t cols, uint64_t rows, uint64_t ld_elems, uint32_t box_cols,
               uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t gemm_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const int k = (kind == FMT_E4M3 || kind == FMT_E5M2) ? KIND_MXF8
                : (kind == FMT_E2M1)                  ? KIND_MXF4
                                                      : KIND_F16;
  return plan_split(M, N, K, stage_k(k), true).ws_bytes;
}

namespace {

// The tensor map of one operand's data plane: rows x K codes, a box of 128 K
// by box_rows rows.  8-bit codes are copied as bytes.  Packed E2M1 codes for
// the FP4-rate kernel are copied as bytes too (128 bytes = 256 codes); for
// the FP8-rate kernel TMA unpacks them (16U4_ALIGN16B) into the 8-bit
// layout, 16 codes in 8 bytes followed by an 8-byte gap, so that the tile in
// shared memory is laid out exactly as an E4M3 tile is.
bool make_data_tmap(CUtensorMap* m, const void* data, int fmt, bool fp4_kind, int64_t rows,
                    int64_t K, uint32_t box_rows) {
  if (fmt != FMT_E2M1)
    return make_tmap(m, data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, rows, K, 128, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (fp4_kind)
    return make_tmap(m, data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, K / 2, 128,
                     box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(data), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Element-format field of the mxf8f6f4 instruction descriptor.
uint32_t f8f6f4_code(int fmt) { return fmt == FMT_E5M2 ? 1u : fmt == FMT_E2M1 ? 5u : 0u; }

}  // namespace

cudaError_t launch_gemm_mx(int fmt_a, int fmt_b, const void* a_data, const uint8_t* a_sf,
                           const void* b_data, const uint8_t* b_sf, void* C,
                           int c_dtype, int64_t ldc, int64_t M, int64_t N,
                           int64_t K, void* ws, size_t ws_bytes, const Epilogue& epi,
                           cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const bool plain = plain_epilogue(epi);
  const int eb = (c_dtype == DT_BF16) ? 2 : 4;
  if (K == 0) {
    if (!plain) return cudaErrorInvalidValue;   // the fused calls need K > 0
    return launch_zero_fill(C, M, N, ldc, eb, st);
  }
  const bool fp4 = (fmt_a == FMT_E2M1 && fmt_b == FMT_E2M1);
  const int kind = fp4 ? KIND_MXF4 : KIND_MXF8;
  // the K-split is for plain products only: the partials' reduction has no
  // epilogue
  SplitPlan plan = plan_split(M, N, K, stage_k(kind), ws != nullptr && plain);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes) plan = plan_split(M, N, K, stage_k(kind), false);
  // scale atoms per stage of the configuration dispatch() picks
  const bool pair = M > BM;
  const int ck = !fp4 ? (pair ? KT<KIND_MXF8, KSUB_CG2>::CK : KT<KIND_MXF8, KSUB_CG1>::CK)
                      : (pair ? KT<KIND_MXF4, KSUB_CG2>::CK : KT<KIND_MXF4, KSUB_CG1>::CK);
  // one TMA box of B is this CTA's half of the N tile when M > BM
  const uint32_t b_rows = pair ? BN / 2 : BN;
  CUtensorMap ta, tb, tsa, tsb;
  if (!make_data_tmap(&ta, a_data, fmt_a, fp4, M, K, BM) ||
      !make_data_tmap(&tb, b_data, fmt_b, fp4, N, K, b_rows) ||
      !make_sf_tmap(&tsa, a_sf, M, K, ck) || !make_sf_tmap(&tsb, b_sf, N, K, ck))
    return cudaErrorInvalidValue;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  float* w = static_cast<float*>(ws);
  const EpiArgs ea = epi_args(epi, M, N);
  const int out = epi.q_fmt == FMT_E2M1 ? OUT_MX4
                  : epi.q_fmt != 0      ? OUT_MX8
                  : c_dtype == DT_BF16  ? OUT_BF16
                                        : OUT_F32;
  if (!fp4) {
    const uint32_t f = (f8f6f4_code(fmt_a) << 7) | (f8f6f4_code(fmt_b) << 10);
    switch (out) {
      case OUT_BF16:
        return dispatch<KIND_MXF8, OUT_BF16>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, f, ea, st);
      case OUT_MX8:
        return dispatch<KIND_MXF8, OUT_MX8>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, f, ea, st);
      case OUT_MX4:
        return dispatch<KIND_MXF8, OUT_MX4>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, f, ea, st);
      default:
        return dispatch<KIND_MXF8, OUT_F32>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, f, ea, st);
    }
  }
  switch (out) {
    case OUT_BF16:
      return dispatch<KIND_MXF4, OUT_BF16>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, 0u, ea, st);
    case OUT_MX8:
      return dispatch<KIND_MXF4, OUT_MX8>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, 0u, ea, st);
    case OUT_MX4:
      return dispatch<KIND_MXF4, OUT_MX4>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, 0u, ea, st);
    default:
      return dispatch<KIND_MXF4, OUT_F32>(ta, tb, tsa, tsb, C, ldc, m, n, k, plan, w, 0u, ea, st);
  }
}

cudaError_t launch_gemm_f16(int ab_dtype, const void* A, const void* B, float* C,
                            int64_t M, int64_t N, int64_t K, int64_t lda,
                            int64_t ldb, int64_t ldc, void* ws, size_t ws_bytes,
                            const Epilogue& epi, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const bool plain = plain_epilogue(epi);
  if (epi.q_fmt != 0) return cudaErrorInvalidValue;     // fp32 C only
  if (K == 0) {
    if (!plain) return cudaErrorInvalidValue;
    return launch_zero_fill(C, M, N, ldc, 4, st);
  }
  SplitPlan plan = plan_split(M, N, K, stage_k(KIND_F16), ws != nullptr && plain);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes)
    plan = plan_split(M, N, K, stage_k(KIND_F16), false);
  const CUtensorMapDataType dt = (ab_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A, dt, 2, K, M, lda, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tb, B, dt, 2, N, K, ldb, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  float* w = static_cast<float*>(ws);
  const EpiArgs ea = epi_args(epi, M, N);
  // the scale maps are unused by the 16-bit kinds
  if (ab_dtype == DT_BF16)
    return dispatch<KIND_BF16, OUT_F32>(ta, tb, ta, tb, C, ldc, m, n, k, plan, w, 0u, ea, st);
  return dispatch<KIND_F16, OUT_F32>(ta, tb, ta, tb, C, ldc, m, n, k, plan, w, 0u, ea, st);
}

unsigned fetch_and_clear_status_gemm(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_gemm, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_gemm, &z, sizeof(z));
  return v;
}

}  // namespace mxk
