// dqgemm.cu -- C = A * dequant(B)^T: a row-major fp16 / bf16 A (M x K) times
// an MX tensor B (N x K) of any element format -- E4M3, E5M2, E2M1 or the
// integer formats int8 / int4 / int2 -- on the 16-bit tensor cores.
//
// What is computed follows WWDC26 session 330, "Quantized matrix
// multiplication": when a quantized format has no matmul of its own, load a
// chunk of the quantized data, dequantize it to f16 in threadgroup memory and
// multiply that.  Here "threadgroup memory" is the shared memory of the CTA
// pair, and the multiply is tcgen05.mma kind::f16.
//
// Design:
//   * CG = 2 (M > 128): a cluster of two CTAs shares one 256 x 256 tile
//     (cta_group::2, M = 256, N = 256, K = 16 per MMA); each CTA stages its
//     own 128 rows of A and dequantizes its own 128-row half of B.  CG = 1:
//     one CTA, a 128 x 256 tile, all 256 rows of B.
//   * 64 K per stage (one 128-byte swizzled row of 16-bit values).
//   * warp 0: TMA producer -- A's tile into the operand ring; B's codes (raw
//     bytes) and the stage's scale atom into a staging ring;
//   * warp 1: tensor-memory allocation; the leader's warp runs the issue
//     loop and one elected lane issues the MMAs, four per stage;
//   * warps 2..5: epilogue, one per TMEM lane quarter, draining both
//     128-column halves of a double-buffered accumulator 32 columns at a
//     time while the next tile accumulates into the other buffer;
//   * warps 6..29: dequantizers, three groups of eight that take the stages
//     in turn.  A group has three stages' time for each of its own, which
//     hides the latency of one stage's conversion chain (W4A16 8192^3: 0.94
//     ms with one group, 0.70 with two, 0.67 with three).  In a group, one
//     thread per 32-element block of a row of B (one scale): codes and scale
//     to 16-bit values, written in the 128-byte-swizzled K-major layout the
//     MMA reads, then a proxy fence and an arrive on the leader's barrier.
//     int4 / int2 codes against a bf16 A are spread to bytes with masks and
//     byte permutes and scaled two at a time with a packed bf16 FMA.
// Tensor memory: accumulators in columns [0, 256) and [256, 512).
//
// Exactness: a code times its scale is exact in fp32 (integers by an exact
// fused multiply-add on a magic-number float, or for scales beyond the
// constant's range by an exact subtraction and product; 8- and 4-bit floats
// by the hardware conversion to f16x2), and exact in the 16-bit type
// whenever the value lies in its range.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_dq and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "dq_common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

using namespace dq;

__device__ unsigned int g_status_dq = 0;

constexpr int DQ_KPS = 64;                 // K per stage
constexpr int TMEM_COLS_DQ = 512;          // two 256-column accumulators
constexpr int DQ_EPI_WARP0 = 2;            // warps 2..5
constexpr int DQ_NUM_EPI = 4;
constexpr int DQ_WARP0 = DQ_EPI_WARP0 + DQ_NUM_EPI;   // warps 6..29
constexpr int DQ_NUM_DQ = 8;                // dequantizer warps per stage
constexpr int DQ_GROUPS = 3;                // groups taking turns on the stages
constexpr int DQ_THREADS = 32 * (DQ_WARP0 + DQ_GROUPS * DQ_NUM_DQ);   // 960
constexpr int DQ_CODE_MAX = 128 * 64;      // code bytes per stage and 128 rows (8-bit)

template <int CG>
struct DqSmem {
  static constexpr int STAGES = (CG == 2) ? 5 : 3;
  static constexpr int B_ROWS = BN / CG;                 // rows of B this CTA holds
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = B_ROWS * 128;
  static constexpr int CODE_BYTES = (B_ROWS / 128) * DQ_CODE_MAX;
  static constexpr int SF_BYTES = (B_ROWS / 128) * SF_ATOM_BYTES;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int CODE_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int SF_OFF = CODE_OFF + STAGES * CODE_BYTES;
  static constexpr int BAR_OFF = SF_OFF + STAGES * SF_BYTES;
  // a_full, dq_full, codes_full, empty [STAGES]; acc_full[2], acc_empty[2]
  static constexpr int MISC_OFF = BAR_OFF + (4 * STAGES + 4) * 8;
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(B_ROWS % 128 == 0, "dequantizer rows");
};

// kind::f16 instruction descriptor: D f32, A and B f16 (0) or bf16 (1), both
// K-major, N>>3 at bit 17, M>>4 at bit 24.
template <int CG>
__host__ __device__ constexpr uint32_t idesc_dq(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>((BM * CG) >> 4) << 24);
}

__device__ __forceinline__ void dq_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_dq, STATUS_TIMEOUT | site);
}

// Dequantize one 32-element block of one row of B (its codes at `codes`, its
// scale code sc) into 16-byte chunks 4 h .. 4 h + 3 of row `row` of the B
// tile (chunk c of row r sits at chunk c ^ (r % 8): the 128-byte swizzle the
// MMA descriptor names).
template <int FMT>
__device__ __forceinline__ void dq_block(const uint8_t* codes, uint32_t sc, bool bf16,
                                         uint8_t* dst_row, int row, int h) {
  uint32_t w[8];
  load_block_codes<FMT>(codes, w);
  uint32_t o[16];
  dq_block_regs<FMT>(w, sc, bf16, o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = 4 * h + j;
    *reinterpret_cast<uint4*>(dst_row + ((c ^ (row & 7)) << 4)) =
        make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
  }
}

// Work items: tile t of the raster, K range `part` of `split` (split = 1:
// whole tiles).  Item w = t * split + part, so the parts of a tile are
// neighbours; a split item writes its fp32 partial tile to the workspace and
// dq_reduce_kernel adds the parts.
struct DqWork {
  TileSched sched;
  int num_kb, split, total;
  __device__ __forceinline__ void item(int w, int& mb, int& nb, int& kb0, int& kb1) const {
    const int t = w / split, part = w - t * split;
    sched.tile(t, mb, nb);
    kb0 = part * num_kb / split;
    kb1 = (part + 1) * num_kb / split;
  }
};

template <int CG, int OUT>
__global__ void __launch_bounds__(DQ_THREADS, 1)
dqgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmSF, void* __restrict__ Cptr, int64_t ldc,
              int M, int N, int K, int fmt_b, int a_bf16, EpiArgs epi, float* __restrict__ ws,
              int split) {
  using L = DqSmem<CG>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t bar_a_full = base + L::BAR_OFF;
  const uint32_t bar_dq_full = bar_a_full + 8 * L::STAGES;
  const uint32_t bar_codes = bar_dq_full + 8 * L::STAGES;
  const uint32_t bar_empty = bar_codes + 8 * L::STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * L::STAGES;    // [2]
  const uint32_t bar_acc_empty = bar_acc_full + 16;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  const int num_kb = K / DQ_KPS;                       // K % 64 == 0 (host check)
  const int k_atoms = (K + 127) / 128;
  const int row_bytes = (fmt_b == FMT_INT2) ? 16 : (fmt_b == FMT_INT4 || fmt_b == FMT_E2M1) ? 32 : 64;
  DqWork work;
  work.sched.num_m = (M + BM * CG - 1) / (BM * CG);
  work.sched.num_n = (N + BN - 1) / BN;
  work.sched.total = work.sched.num_m * work.sched.num_n;
  work.num_kb = num_kb;
  work.split = split;
  work.total = work.sched.total * split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar_a_full + 8 * s, 1);
      mbar_init(bar_dq_full + 8 * s, CG * DQ_NUM_DQ);
      mbar_init(bar_codes + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, CG * DQ_NUM_EPI);
    }
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSF);
  }
  if (warp == 1) tmem_alloc_cg<CG>(smem_u32(tmem_slot), TMEM_COLS_DQ);
  __syncwarp();   // reconverge before the aligned barrier (one-lane setup)
  tc_fence_before();
  if (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t a_full0 = (CG == 2) ? map_to_cta(bar_a_full, 0) : bar_a_full;
      uint32_t it = 0;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      const uint32_t code_tx = static_cast<uint32_t>((L::B_ROWS / 128) * 128 * row_bytes + L::SF_BYTES);
      for (int w = cluster_id; w < work.total && ok; w += num_clusters) {
        int mb, nb, kb0, kb1;
        work.item(w, mb, nb, kb0, kb1);
        const int m0 = mb * BM * CG + static_cast<int>(rank) * BM;
        const int n0 = nb * BN + static_cast<int>(rank) * L::B_ROWS;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) {
            dq_timeout(abort, 0x21);
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_a_full + 8 * s, CG * L::A_BYTES);
          tma_load_2d_cg<CG>(base + L::A_OFF + s * L::A_BYTES, &tmA, a_full0 + 8 * s,
                             kb * DQ_KPS, m0);
          mbar_arrive_expect_tx(bar_codes + 8 * s, code_tx);
#pragma unroll
          for (int g = 0; g < L::B_ROWS / 128; ++g) {
            tma_load_2d(base + L::CODE_OFF + s * L::CODE_BYTES + g * 128 * row_bytes, &tmB,
                        bar_codes + 8 * s, kb * row_bytes, n0 + 128 * g);
            tma_load_2d(base + L::SF_OFF + s * L::SF_BYTES + g * SF_ATOM_BYTES, &tmSF,
                        bar_codes + 8 * s, 0, ((n0 + 128 * g) / 128) * k_atoms + kb / 2);
          }
          if (++s == L::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA retires
        const uint32_t first = it >= L::STAGES ? it - L::STAGES : 0;
        for (uint32_t i = first; i < it; ++i) {
          const long long t0 = clock64();
          while (!mbar_try_wait(bar_codes + 8 * (i % L::STAGES), (i / L::STAGES) & 1u) &&
                 clock64() - t0 < MXK_WAIT_LIMIT_CYCLES) {
          }
          if (leader) {
            const long long t1 = clock64();
            while (!mbar_try_wait(bar_a_full + 8 * (i % L::STAGES), (i / L::STAGES) & 1u) &&
                   clock64() - t1 < MXK_WAIT_LIMIT_CYCLES) {
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the loop (warp-uniform descriptors); one elected
    // lane issues
    if (leader) {
      const bool issuer = elect_one();
      const uint64_t a_desc0 = smem_desc(base + L::A_OFF, 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(base + L::B_OFF, 16, 1024, 2);
      const uint32_t id = idesc_dq<CG>(a_bf16 != 0);
      int s = 0;
      uint32_t ph = 0;
      uint32_t tc = 0;
      bool ok = true;
      for (int w = cluster_id; w < work.total && ok; w += num_clusters, ++tc) {
        int mb, nb, kb0, kb1;
        work.item(w, mb, nb, kb0, kb1);
        const uint32_t b = tc & 1u;
        const uint32_t acc = tmem_base + b * BN;
        if (!mbar_wait_spin(bar_acc_empty + 8 * b, ((tc >> 1) & 1u) ^ 1u, abort)) {
          dq_timeout(abort, 0x22);
          break;
        }
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(bar_a_full + 8 * s, ph, abort) ||
              !mbar_wait(bar_dq_full + 8 * s, ph, abort)) {
            dq_timeout(abort, 0x23);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_d = a_desc0 + static_cast<uint64_t>((s * L::A_BYTES) >> 4);
          const uint64_t b_d = b_desc0 + static_cast<uint64_t>((s * L::B_BYTES) >> 4);
          if (issuer) {
#pragma unroll
            for (int m = 0; m < 4; ++m)    // 4 x 16 K = 64 K; 32 bytes per step
              mma_f16_cg<CG>(acc, a_d + 2 * m, b_d + 2 * m, id, (kb > kb0 || m > 0) ? 1u : 0u);
            tc_commit_cg<CG>(bar_empty + 8 * s);
          }
          if (++s == L::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (issuer) tc_commit_cg<CG>(bar_acc_full + 8 * b);
      }
    }
  } else if (warp < DQ_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                          // TMEM lane quarter
    uint32_t tc = 0;
    for (int w = cluster_id; w < work.total; w += num_clusters, ++tc) {
      int mb, nb, kb0, kb1;
      work.item(w, mb, nb, kb0, kb1);
      const uint32_t b = tc & 1u;
      if (!mbar_wait(bar_acc_full + 8 * b, (tc >> 1) & 1u, abort)) {
        dq_timeout(abort, 0x24);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(mb) * BM * CG + rank * BM + 32 * q + lane;
#pragma unroll 1
      for (int cg_ = 0; cg_ < BN / 128; ++cg_) {
      const int col0 = nb * BN + cg_ * 128;
      uint32_t sf_word = 0;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * BN +
                               static_cast<uint32_t>(cg_ * 128 + 32 * i),
                           r);
        tmem_wait_ld();
        const int c = col0 + 32 * i;
        if (split > 1) {
          // a part of a split tile: the raw fp32 accumulator to the workspace
          // (rows beyond M are left out, columns beyond N included: the
          // reduction reads neither)
          if (row < M) {
            float* wrow = ws + static_cast<int64_t>(w) * (BM * CG * BN) +
                          static_cast<int64_t>(rank * BM + 32 * q + lane) * BN + cg_ * 128 +
                          32 * i;
            const bool wide = (reinterpret_cast<uintptr_t>(wrow) & 31u) == 0;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              store_32B(wrow + 8 * v, *reinterpret_cast<const uint32_t(*)[8]>(r + 8 * v), wide);
          }
          continue;
        }
        if (epi.bias != nullptr || epi.act != ACT_NONE) apply_bias_act(r, epi, c, N);
        if (OUT == OUT_MX8 || OUT == OUT_MX4) {
          if (row < M && c < N)
            sf_word |= quantize_block_row<OUT>(r, epi, static_cast<uint8_t*>(Cptr), row, c, N)
                       << (8 * i);
        } else if (row < M) {
          store_row_segment<OUT, 32>(r, Cptr, ldc, row, c, N);
        }
      }
      if ((OUT == OUT_MX8 || OUT == OUT_MX4) && split == 1)
        store_mx_scales(sf_word, epi, row, col0, N);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_cluster(map_to_cta(bar_acc_empty + 8 * b, 0));
        else
          mbar_arrive(bar_acc_empty + 8 * b);
      }
    }
  } else {
    // ------------------------------------------------------------ dequantizers
    // Group grp takes the stages with it % DQ_GROUPS == grp.  In a group,
    // unit u = thread + 256 i (i < 2 / CG) is block u % 2 of row u / 2 of this
    // CTA's rows of B: 32 codes and one scale.
    const int tg = threadIdx.x - 32 * DQ_WARP0;
    const int t = tg % (32 * DQ_NUM_DQ);
    const uint32_t grp = static_cast<uint32_t>(tg / (32 * DQ_NUM_DQ));
    uint32_t it = 0;
    const uint32_t dq_full0 = (CG == 2) ? map_to_cta(bar_dq_full, 0) : bar_dq_full;
    const int block_bytes = row_bytes / 2;
    int s = 0;
    uint32_t ph = 0;
    const bool bf = a_bf16 != 0;
    for (int w = cluster_id; w < work.total; w += num_clusters) {
      int mb, nb, kb0, kb1;
      work.item(w, mb, nb, kb0, kb1);
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        // the groups take the stages in turn
        if ((it++ % DQ_GROUPS) != grp) {
          if (++s == L::STAGES) {
            s = 0;
            ph ^= 1u;
          }
          continue;
        }
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort) ||
            !mbar_wait(bar_codes + 8 * s, ph, abort)) {
          dq_timeout(abort, 0x25);
          ok = false;
          break;
        }
        const uint8_t* codes = gbase + L::CODE_OFF + s * L::CODE_BYTES;
        const uint8_t* sf = gbase + L::SF_OFF + s * L::SF_BYTES;
        uint8_t* btile = gbase + L::B_OFF + s * L::B_BYTES;
#pragma unroll
        for (int i = 0; i < 2 / CG; ++i) {
          const int u = t + 32 * DQ_NUM_DQ * i;
          const int r = u >> 1, h = u & 1;
          // the block's scale: block 2 kb + h of the row, byte 2 (kb % 2) + h
          // of the row's group in atom kb / 2 of its row group
          const uint32_t sc =
              sf[(r >> 7) * SF_ATOM_BYTES + sf_in_atom(r & 127, 2 * (kb & 1) + h)];
          const uint8_t* cr = codes + r * row_bytes + h * block_bytes;
          uint8_t* dst = btile + r * 128;
          switch (fmt_b) {
            case FMT_INT8: dq_block<FMT_INT8>(cr, sc, bf, dst, r, h); break;
            case FMT_INT4: dq_block<FMT_INT4>(cr, sc, bf, dst, r, h); break;
            case FMT_INT2: dq_block<FMT_INT2>(cr, sc, bf, dst, r, h); break;
            case FMT_E2M1: dq_block<FMT_E2M1>(cr, sc, bf, dst, r, h); break;
            case FMT_E5M2: dq_block<FMT_E5M2>(cr, sc, bf, dst, r, h); break;
            default: dq_block<FMT_E4M3>(cr, sc, bf, dst, r, h); break;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2 && !leader)
            mbar_arrive_remote(dq_full0 + 8 * s);
          else
            mbar_arrive(bar_dq_full + 8 * s);
        }
        if (++s == L::STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  __syncwarp();   // reconverge before the aligned barrier (one-lane roles)
  tc_fence_before();
  if (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<CG>(tmem_base, TMEM_COLS_DQ);
  }
}

// Sum the `split` fp32 partials of each tile in a fixed order (results do not
// depend on timing), apply the epilogue's bias and activation, write C (fp32
// or bf16).  CTA = (tile, group of 4 tile rows); a thread owns 4 columns.
template <int OUT>
__global__ void __launch_bounds__(256)
dq_reduce_kernel(const float* __restrict__ ws, void* __restrict__ Cptr, int64_t ldc, int M,
                 int N, TileSched sched, int split, int tile_rows, EpiArgs epi) {
  const int t = blockIdx.x;
  int mb, nb;
  sched.tile(t, mb, nb);
  const int i = blockIdx.y * 4 + (threadIdx.x >> 6);
  const int c = (threadIdx.x & 63) * 4;
  const int64_t row = static_cast<int64_t>(mb) * tile_rows + i;
  const int col = nb * BN + c;
  if (row >= M || col >= N) return;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  for (int p = 0; p < split; ++p) {
    const float4 v = *reinterpret_cast<const float4*>(
        ws + (static_cast<int64_t>(t * split + p) * tile_rows + i) * BN + c);
    a[0] += v.x;
    a[1] += v.y;
    a[2] += v.z;
    a[3] += v.w;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (epi.bias != nullptr && col + e < N) a[e] += __ldg(epi.bias + col + e);
    if (epi.act == ACT_GELU) a[e] = gelu_exact(a[e]);
    else if (epi.act == ACT_GELU_TANH) a[e] = gelu_tanh(a[e]);
  }
  if (OUT == OUT_BF16) {
    uint16_t* crow = reinterpret_cast<uint16_t*>(Cptr) + row * ldc;
    const uint32_t w[2] = {cvt_bf16x2(a[0], a[1]), cvt_bf16x2(a[2], a[3])};
    for (int e = 0; e < 4 && col + e < N; ++e)
      crow[col + e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
  } else {
    float* crow = reinterpret_cast<float*>(Cptr) + row * ldc;
    for (int e = 0; e < 4 && col + e < N; ++e) crow[col + e] = a[e];
  }
}

int dq_sm_count() {
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

// K-split plan: when the tiles leave clusters idle, each tile's K range is
// cut into `split` parts (at least 4 stages each, at most 16) over the idle
// clusters.
struct DqPlan {
  int split;
  size_t ws_bytes;
};

DqPlan dq_plan(int64_t M, int64_t N, int64_t K, bool use_split) {
  DqPlan p{1, 0};
  const int cg = (M > BM) ? 2 : 1;
  const int64_t tiles = ((M + BM * cg - 1) / (BM * cg)) * ((N + BN - 1) / BN);
  const int64_t clusters = dq_sm_count() / cg;
  const int64_t nkb = K / DQ_KPS;
  if (!use_split || tiles >= clusters || nkb < 8) return p;
  int64_t sp = clusters / tiles;
  if (sp > nkb / 4) sp = nkb / 4;
  if (sp > 16) sp = 16;
  if (sp < 2) return p;
  p.split = static_cast<int>(sp);
  p.ws_bytes = static_cast<size_t>(tiles * sp) * (BM * cg) * BN * sizeof(float);
  return p;
}

template <int CG, int OUT>
cudaError_t dq_run(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsf, void* C,
                   int64_t ldc, int M, int N, int K, int fmt_b, int a_bf16, const EpiArgs& ea,
                   float* ws, int split, cudaStream_t st) {
  using L = DqSmem<CG>;
  auto kern = dqgemm_kernel<CG, OUT>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev] = true;
  }
  TileSched sched;
  sched.num_m = (M + BM * CG - 1) / (BM * CG);
  sched.num_n = (N + BN - 1) / BN;
  sched.total = sched.num_m * sched.num_n;
  const int items = sched.total * split;
  int clusters = dq_sm_count() / CG;
  if (clusters > items) clusters = items;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CG), 1, 1);
  cfg.blockDim = dim3(DQ_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsf, C, ldc, M, N, K, fmt_b, a_bf16, ea, ws, split);
  if (e != cudaSuccess || split < 2) return e;
  if constexpr (OUT == OUT_F32 || OUT == OUT_BF16) {
    dim3 grid(static_cast<unsigned>(sched.total), BM * CG / 4);
    dq_reduce_kernel<OUT><<<grid, 256, 0, st>>>(ws, C, ldc, M, N, sched, split, BM * CG, ea);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

template <int OUT>
cudaError_t dq_dispatch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsf,
                        void* C, int64_t ldc, int M, int N, int K, int fmt_b, int a_bf16,
                        const EpiArgs& ea, float* ws, int split, cudaStream_t st) {
  if (M > BM) return dq_run<2, OUT>(ta, tb, tsf, C, ldc, M, N, K, fmt_b, a_bf16, ea, ws, split, st);
  return dq_run<1, OUT>(ta, tb, tsf, C, ldc, M, N, K, fmt_b, a_bf16, ea, ws, split, st);
}

}  // namespace

cudaError_t launch_gemm_dequant(int a_dtype, const void* A, int64_t lda, int fmt_b,
                                const void* b_data, const uint8_t* b_sf, void* C, int c_dtype,
                                int64_t ldc, int64_t M, int64_t N, int64_t K, const Epilogue& epi,
                                void* ws, size_t ws_bytes, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0 || K % DQ_KPS) return cudaErrorInvalidValue;
  // one token of a bf16 A, 4- or 2-bit weights: CUDA-core dot products
  // streaming B (dqgemv.cu)
  if (dequant_gemv_applies(M, a_dtype, fmt_b, epi))
    return launch_gemm_dequant_gemv(A, fmt_b, b_data, b_sf, C, c_dtype, N, K, epi, st);
  // a few tokens: the weights-as-M decode kernel (dqdec.cu)
  if (dequant_decode_applies(M, epi))
    return launch_gemm_dequant_decode(a_dtype, A, lda, fmt_b, b_data, b_sf, C, c_dtype, ldc, M,
                                      N, K, epi, st);
  DqPlan plan = dq_plan(M, N, K, ws != nullptr && epi.q_fmt == 0);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes) plan = DqPlan{1, 0};
  float* w = static_cast<float*>(ws);
  const int sp = plan.split;
  const int bits = (fmt_b == FMT_INT2) ? 2 : (fmt_b == FMT_INT4 || fmt_b == FMT_E2M1) ? 4 : 8;
  const uint64_t row_bytes = static_cast<uint64_t>(K) * bits / 8;
  const bool pair = M > BM;
  const uint32_t b_rows = pair ? BN / 2 : BN;
  const CUtensorMapDataType dt = (a_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb, tsf;
  const uint64_t atoms = static_cast<uint64_t>(sf_row_atoms(N) * sf_k_atoms(K));
  if (!make_tmap(&ta, A, dt, 2, K, M, lda, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tb, b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, row_bytes, N, row_bytes,
                static_cast<uint32_t>(DQ_KPS * bits / 8), 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tmap(&tsf, b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128, atoms, 128, 128, 1,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  (void)b_rows;
  EpiArgs ea;
  ea.bias = epi.bias;
  ea.act = epi.act;
  ea.q_fmt = epi.q_fmt;
  ea.q_sf = epi.q_sf;
  ea.q_k_atoms = sf_k_atoms(N);
  ea.q_row_atoms = sf_row_atoms(M);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int bf = (a_dtype == DT_BF16) ? 1 : 0;
  const int out = epi.q_fmt == FMT_E2M1 ? OUT_MX4
                  : epi.q_fmt != 0      ? OUT_MX8
                  : c_dtype == DT_BF16  ? OUT_BF16
                                        : OUT_F32;
  switch (out) {
    case OUT_BF16:
      return dq_dispatch<OUT_BF16>(ta, tb, tsf, C, ldc, m, n, k, fmt_b, bf, ea, w, sp, st);
    case OUT_MX8:
      return dq_dispatch<OUT_MX8>(ta, tb, tsf, C, ldc, m, n, k, fmt_b, bf, ea, w, 1, st);
    case OUT_MX4:
      return dq_dispatch<OUT_MX4>(ta, tb, tsf, C, ldc, m, n, k, fmt_b, bf, ea, w, 1, st);
    default:
      return dq_dispatch<OUT_F32>(ta, tb, tsf, C, ldc, m, n, k, fmt_b, bf, ea, w, sp, st);
  }
}

size_t dequant_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % DQ_KPS) return 0;
  if (dequant_decode_applies(M, Epilogue{})) return dequant_decode_workspace_bytes(M, N, K);
  return dq_plan(M, N, K, true).ws_bytes;
}

unsigned fetch_and_clear_status_dq(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_dq, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_dq, &z, sizeof(z));
  return v;
}

}  // namespace mxk
