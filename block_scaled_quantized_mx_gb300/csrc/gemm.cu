// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   kind::f16 (fp16 / bf16 operands), kind::mxf8f6f4 block-scaled E4M3 and
//   kind::mxf4 block-scaled packed E2M1, fp32 accumulation in tensor memory.
//
// What is computed: C = A * B with fp32 accumulation (dicastech tutorial
// "Treinar LLM em Swift", Passo 4-6: tiled matmul, FP16 variant); for the MX
// kinds the operands are quantized tensors (data plane + UE8M0 scale plane,
// one scale per 32 K) and the dequantization happens inside the matmul
// (WWDC26 session 330, "Quantized matrix multiplication", 7:19 listing):
// here the tensor core applies the two scales per 32-wide K block itself.
//
// Design (GB300-first, not the pages' threadgroup-tile design):
//   * tile 128 (M) x BN (N), BN = 256; one CTA per SM, persistent over tiles
//     in a grouped raster order so that concurrently running CTAs share A and
//     B tiles in L2;
//   * warp 0: TMA producer -- A and B tiles (128-byte swizzled, 128 bytes of K
//     per row per stage) plus the stage's scale atoms by bulk copy, into a
//     STAGES-deep shared-memory ring guarded by mbarriers;
//   * warp 1: allocates tensor memory and issues, from one thread, the
//     scale-factor copies (tcgen05.cp, shared -> tensor memory) and 4 MMAs
//     per stage (32 bytes of K each), then commits the stage back to the
//     producer; after the last stage it commits the accumulator to the
//     epilogue;
//   * warps 2..9: epilogue -- each warp drains 128 accumulator columns of its
//     32-lane quarter into registers (tcgen05.ld), hands the accumulator back
//     to the MMA warp at once, then converts (fp32 or bf16, RNE) and stores
//     while the next tile's main loop already runs.
// Tensor memory: accumulator in columns [0, BN); per-stage scale factors from
// column 256 on.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_gemm and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

__device__ unsigned int g_status_gemm = 0;

enum Kind : int { KIND_F16 = 0, KIND_BF16 = 1, KIND_MXF8 = 2, KIND_MXF4 = 3 };

constexpr int BM = 128;
constexpr int NUM_THREADS = 320;    // 10 warps
constexpr int EPI_WARP0 = 2;
constexpr int NUM_EPI_THREADS = 256;
constexpr int TMEM_COLS = 512;
constexpr int SF_TMEM_BASE = 256;
constexpr int MMAS_PER_STAGE = 4;   // 4 x 32 bytes of K per 128-byte row
constexpr int GROUP_M = 16;         // raster group height in M tiles

template <int KIND>
struct KT {
  static constexpr bool MX = (KIND == KIND_MXF8 || KIND == KIND_MXF4);
  // K elements per stage (128 bytes of K per operand row)
  static constexpr int KPS = (KIND == KIND_MXF4) ? 256 : (MX ? 128 : 64);
  static constexpr int MMA_K = KPS / MMAS_PER_STAGE;
  // scale atoms (128 K each) per stage along K
  static constexpr int CK = MX ? KPS / 128 : 0;
};

template <int KIND, int BN, int STAGES>
struct Smem {
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SFA_BYTES = KT<KIND>::CK * 512;
  static constexpr int SFB_BYTES = (BN / 128) * KT<KIND>::CK * 512;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int SFA_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + STAGES * SFA_BYTES;
  static constexpr int BAR_OFF = (SFB_OFF + STAGES * SFB_BYTES + 7) / 8 * 8;
  // full[STAGES], empty[STAGES], acc_full, acc_empty
  static constexpr int MISC_OFF = BAR_OFF + (2 * STAGES + 2) * 8;
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;   // slack to align the base to 1024
  // TMEM columns of scale factors per stage: A then B
  static constexpr int SF_COLS = KT<KIND>::CK * 4 * (1 + BN / 128);
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(BN <= SF_TMEM_BASE, "accumulator must fit below the scales");
};

// Instruction descriptor, kind::f16: D f32, A/B f16 or bf16, A K-major,
// B MN-major, N>>3 at bit 17, M>>4 at bit 24.
template <int KIND, int BN>
__host__ __device__ constexpr uint32_t idesc_f16() {
  return (1u << 4) |                                   // D = f32
         ((KIND == KIND_BF16 ? 1u : 0u) << 7) |        // A type
         ((KIND == KIND_BF16 ? 1u : 0u) << 10) |       // B type
         (0u << 15) |                                  // A K-major
         (1u << 16) |                                  // B MN-major
         (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// Instruction descriptor, block-scaled kinds: A/B format (E4M3 = 0 for
// mxf8f6f4, E2M1 = 1 for mxf4), both K-major, N>>3 at bit 17, scale type
// UE8M0 (bit 23), M>>4 at bit 24; scale-factor byte selectors at bits 4-5 (B)
// and 29-30 (A) are filled in per MMA.
template <int KIND, int BN>
__host__ __device__ constexpr uint32_t idesc_mx() {
  return ((KIND == KIND_MXF4 ? 1u : 0u) << 7) | ((KIND == KIND_MXF4 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

struct TileSched {
  int num_m, num_n, total;
  __device__ __forceinline__ void tile(int t, int& mb, int& nb) const {
    const int per_group = GROUP_M * num_n;
    const int g = t / per_group;
    const int first_m = g * GROUP_M;
    const int gsz = min(num_m - first_m, GROUP_M);
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
  }
};

__device__ __forceinline__ void record_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_gemm, STATUS_TIMEOUT | site);
}

template <int KIND, int BN, int STAGES, int OUT_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const uint8_t* __restrict__ sfA, const uint8_t* __restrict__ sfB,
            void* __restrict__ Cptr, int64_t ldc, int M, int N, int K) {
  using T = KT<KIND>;
  using L = Smem<KIND, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t bar_full = base + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  TileSched sched;
  sched.num_m = (M + BM - 1) / BM;
  sched.num_n = (N + BN - 1) / BN;
  sched.total = sched.num_m * sched.num_n;
  const int num_kb = (K + T::KPS - 1) / T::KPS;
  const int k_atoms = (K + 127) / 128;
  const int n_row_atoms = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, NUM_EPI_THREADS);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < sched.total && ok; t += gridDim.x) {
        int mb, nb;
        sched.tile(t, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = static_cast<int>(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort)) {
            record_timeout(abort, 1);
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * s;
          uint32_t bytes = L::A_BYTES + L::B_BYTES;
          int ck_valid = 0;
          if (T::MX) {
            ck_valid = min(T::CK, k_atoms - kb * T::CK);
            int nh = 0;
            for (int h = 0; h < BN / 128; ++h)
              if (nb * (BN / 128) + h < n_row_atoms) ++nh;
            bytes += static_cast<uint32_t>(ck_valid * 512 * (1 + nh));
          }
          mbar_arrive_expect_tx(full, bytes);
          const uint32_t a_dst = base + L::A_OFF + s * L::A_BYTES;
          const uint32_t b_dst = base + L::B_OFF + s * L::B_BYTES;
          if (T::MX) {
            // data planes are byte matrices: x counts bytes of K
            tma_load_2d(a_dst, &tmA, full, kb * 128, mb * BM);
            tma_load_2d(b_dst, &tmB, full, kb * 128, nb * BN);
            const uint32_t sfa_dst = base + L::SFA_OFF + s * L::SFA_BYTES;
            bulk_load(sfa_dst, sfA + (static_cast<int64_t>(mb) * k_atoms + kb * T::CK) * 512,
                      ck_valid * 512, full);
            const uint32_t sfb_dst = base + L::SFB_OFF + s * L::SFB_BYTES;
            for (int h = 0; h < BN / 128; ++h) {
              const int ra = nb * (BN / 128) + h;
              if (ra < n_row_atoms)
                bulk_load(sfb_dst + h * T::CK * 512,
                          sfB + (static_cast<int64_t>(ra) * k_atoms + kb * T::CK) * 512,
                          ck_valid * 512, full);
            }
          } else {
            tma_load_2d(a_dst, &tmA, full, kb * 64, mb * BM);
            // B is K x N row-major: BN/64 boxes of 64 (N) x 64 (K rows)
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_dst + j * 64 * 128, &tmB, full, nb * BN + 64 * j, kb * 64);
          }
        }
      }
      if (!ok) {
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
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < sched.total && ok; t += gridDim.x, ++tc) {
        if (!mbar_wait(bar_acc_empty, (tc & 1u) ^ 1u, abort)) {
          record_timeout(abort, 2);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = static_cast<int>(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort)) {
            record_timeout(abort, 3);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_s = base + L::A_OFF + s * L::A_BYTES;
          const uint32_t b_s = base + L::B_OFF + s * L::B_BYTES;
          const uint32_t sfa_t = tmem_base + SF_TMEM_BASE + s * L::SF_COLS;
          const uint32_t sfb_t = sfa_t + T::CK * 4;
          const int k_left = K - kb * T::KPS;
          const int nmma = min(MMAS_PER_STAGE, (k_left + T::MMA_K - 1) / T::MMA_K);
          if (T::MX) {
            const int ck_valid = min(T::CK, k_atoms - kb * T::CK);
            const uint32_t sfa_s = base + L::SFA_OFF + s * L::SFA_BYTES;
            const uint32_t sfb_s = base + L::SFB_OFF + s * L::SFB_BYTES;
            for (int c = 0; c < ck_valid; ++c) {
              tc_cp_32x128b_x4(sfa_t + 4 * c, smem_desc(sfa_s + c * 512, 0, 128, 0));
              for (int h = 0; h < BN / 128; ++h)
                tc_cp_32x128b_x4(sfb_t + c * 4 * (BN / 128) + 4 * h,
                                 smem_desc(sfb_s + (h * T::CK + c) * 512, 0, 128, 0));
            }
          }
          for (int m = 0; m < nmma; ++m) {
            const uint32_t acc = (kb > 0 || m > 0) ? 1u : 0u;
            const uint64_t a_desc = smem_desc(a_s + 32 * m, 16, 1024, 2);
            if (KIND == KIND_F16 || KIND == KIND_BF16) {
              // B MN-major: 64-wide N chunks LBO = 64 K rows * 128 B apart,
              // 8-row K groups SBO = 1024 B apart; 16 K rows per MMA
              const uint64_t b_desc = smem_desc(b_s + 2048 * m, 64 * 128, 1024, 2);
              mma_f16(tmem_base, a_desc, b_desc, idesc_f16<KIND, BN>(), acc);
            } else if (KIND == KIND_MXF8) {
              const uint64_t b_desc = smem_desc(b_s + 32 * m, 16, 1024, 2);
              const uint32_t id = idesc_mx<KIND, BN>() | (static_cast<uint32_t>(m) << 4) |
                                  (static_cast<uint32_t>(m) << 29);
              mma_mxf8(tmem_base, a_desc, b_desc, id, sfa_t, sfb_t, acc);
            } else {
              const uint64_t b_desc = smem_desc(b_s + 32 * m, 16, 1024, 2);
              const int c = m >> 1;                       // scale atom along K
              const uint32_t sf_id = static_cast<uint32_t>((m & 1) * 2);
              const uint32_t id = idesc_mx<KIND, BN>() | (sf_id << 4) | (sf_id << 29);
              mma_mxf4(tmem_base, a_desc, b_desc, id, sfa_t + 4 * c,
                       sfb_t + c * 4 * (BN / 128), acc);
            }
          }
          tc_commit(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                        // TMEM lane quarter
    const int half = (warp - EPI_WARP0) >> 2;      // which BN/2 columns
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < sched.total; t += gridDim.x, ++tc) {
      int mb, nb;
      sched.tile(t, mb, nb);
      if (!mbar_wait(bar_acc_full, tc & 1u, abort)) {
        record_timeout(abort, 4);
        break;
      }
      tc_fence_after();
      uint32_t r[BN / 2];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(half * (BN / 2));
#pragma unroll
      for (int i = 0; i < BN / 64; ++i)
        tmem_ld_32x32b_x32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_acc_empty);

      const int64_t row = static_cast<int64_t>(mb) * BM + 32 * q + lane;
      const int col0 = nb * BN + half * (BN / 2);
      if (row < M) {
        if (OUT_BF16) {
          uint16_t* crow = reinterpret_cast<uint16_t*>(Cptr) + row * ldc;
#pragma unroll
          for (int v = 0; v < BN / 16; ++v) {       // 8 columns per vector
            const int c = col0 + 8 * v;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = cvt_bf16x2(__uint_as_float(r[8 * v + 2 * e]),
                                __uint_as_float(r[8 * v + 2 * e + 1]));
            if (c + 7 < N) {
              *reinterpret_cast<uint4*>(crow + c) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (c + e < N)
                  crow[c + e] =
                      static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
            }
          }
        } else {
          float* crow = reinterpret_cast<float*>(Cptr) + row * ldc;
#pragma unroll
          for (int v = 0; v < BN / 8; ++v) {        // 4 columns per vector
            const int c = col0 + 4 * v;
            if (c + 3 < N) {
              *reinterpret_cast<uint4*>(crow + c) =
                  make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (c + e < N) crow[c + e] = __uint_as_float(r[4 * v + e]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// 2-D tensor map, row-major rows x cols (cols contiguous), 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int elem_bytes,
               uint64_t cols, uint64_t rows, uint64_t ld_elems, uint32_t box_cols,
               uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
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

template <int KIND, int BN, int STAGES, int OUT_BF16>
cudaError_t run(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* sfa,
                const uint8_t* sfb, void* C, int64_t ldc, int M, int N, int K,
                cudaStream_t st) {
  using L = Smem<KIND, BN, STAGES>;
  auto kern = gemm_kernel<KIND, BN, STAGES, OUT_BF16>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev] = true;
  }
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  kern<<<grid, NUM_THREADS, L::ALLOC, st>>>(ta, tb, sfa, sfb, C, ldc, M, N, K);
  return cudaGetLastError();
}

constexpr int BN_DEF = 256;
constexpr int STAGES_DEF = 4;

}  // namespace

cudaError_t launch_gemm_mx(int fmt, const void* a_data, const uint8_t* a_sf,
                           const void* b_data, const uint8_t* b_sf, void* C,
                           int c_dtype, int64_t ldc, int64_t M, int64_t N,
                           int64_t K, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int eb = (c_dtype == DT_BF16) ? 2 : 4;
  if (K == 0) return launch_zero_fill(C, M, N, ldc, eb, st);
  const uint64_t kbytes = (fmt == FMT_E4M3) ? K : K / 2;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, M, kbytes, 128, BM) ||
      !make_tmap(&tb, b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, N, kbytes, 128,
                 BN_DEF))
    return cudaErrorInvalidValue;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (fmt == FMT_E4M3) {
    if (c_dtype == DT_BF16)
      return run<KIND_MXF8, BN_DEF, STAGES_DEF, 1>(ta, tb, a_sf, b_sf, C, ldc, m, n, k, st);
    return run<KIND_MXF8, BN_DEF, STAGES_DEF, 0>(ta, tb, a_sf, b_sf, C, ldc, m, n, k, st);
  }
  if (c_dtype == DT_BF16)
    return run<KIND_MXF4, BN_DEF, STAGES_DEF, 1>(ta, tb, a_sf, b_sf, C, ldc, m, n, k, st);
  return run<KIND_MXF4, BN_DEF, STAGES_DEF, 0>(ta, tb, a_sf, b_sf, C, ldc, m, n, k, st);
}

cudaError_t launch_gemm_f16(int ab_dtype, const void* A, const void* B, float* C,
                            int64_t M, int64_t N, int64_t K, int64_t lda,
                            int64_t ldb, int64_t ldc, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return launch_zero_fill(C, M, N, ldc, 4, st);
  const CUtensorMapDataType dt = (ab_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A, dt, 2, K, M, lda, 64, BM) ||
      !make_tmap(&tb, B, dt, 2, N, K, ldb, 64, 64))
    return cudaErrorInvalidValue;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (ab_dtype == DT_BF16)
    return run<KIND_BF16, BN_DEF, STAGES_DEF, 0>(ta, tb, nullptr, nullptr, C, ldc, m, n, k, st);
  return run<KIND_F16, BN_DEF, STAGES_DEF, 0>(ta, tb, nullptr, nullptr, C, ldc, m, n, k, st);
}

unsigned fetch_and_clear_status_gemm(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_gemm, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_gemm, &z, sizeof(z));
  return v;
}

}  // namespace mxk
