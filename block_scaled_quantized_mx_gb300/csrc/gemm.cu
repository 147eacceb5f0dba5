// gemm.cu -- host side of the tcgen05 GEMM (the kernel is in gemm_kernel.cuh,
// instantiated per kind in gemm_mxf8.cu, gemm_mxf4.cu and gemm_f16.cu): the
// operands' tensor maps, the configuration and K-split plan of each shape,
// the split's workspace layout and counter tags, and the status words.
#include <atomic>
#include <chrono>

#include "gemm_kernel.cuh"

namespace mxk {

namespace {

using gemm::KIND_BF16;
using gemm::KIND_F16;
using gemm::KIND_MXF4;
using gemm::KIND_MXF8;
using gemm::KT;

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

// How one GEMM is laid on the SMs.
//  * cg: CTA pairs (256-row tiles) when M > 128, else single CTAs;
//  * tbn: tile width 256 or 128 (N = 128 runs the MMA at the full per-clock
//    rate; 128-wide tiles alternate two accumulators in tensor memory);
//  * split (128-wide tiles, with a workspace): the tiles of a last partial
//    wave (or of a problem with fewer tiles than clusters) are split into
//    `split` K ranges so that idle clusters share their work; the partial
//    tiles go to the workspace and the last range of each tile to finish
//    sums them.
// The plan with the smallest estimated time is taken.  A 256-wide tile's
// main loop takes about kStageUs per stage of K (four MMAs of 128 clk at
// ~1.9 GHz, the same for every kind: each kind's stage holds the K its rate
// covers in that time); a 128-wide tile takes kNarrowCost of that per stage
// (measured on GB300 with several tiles per cluster: 1.33-1.49x the half
// tile's share -- more operand bytes per flop and two tiles' hand-offs); the
// split adds kSplitUs for writing, counting and summing the partial tiles
// (measured: the chain of partial store and fence, counter, reload and store
// costs 5-6 us over a direct store, so the split pays for long K only: bf16
// 128 x 2048 x 8192 37.5 -> 23.6 us, MXFP8 256 x 256 x 8192 25.3 -> 19.7 us,
// bf16 1024^3 13.0 -> 17.3 us).
struct Plan {
  int cg, tbn;
  int clusters, full_tiles, split, rem;
  size_t part_bytes;   // workspace bytes of the partial tiles
  size_t ws_bytes;     // partial tiles + one counter per (split tile, CTA)
};

constexpr double kStageUs = 0.27;
constexpr double kNarrowCost = 0.70;   // 128-wide tile per stage / 256-wide
constexpr double kSplitUs = 5.0;

Plan make_plan(int64_t M, int64_t N, int64_t K, int kps, bool use_split, bool narrow_ok,
               int force_tbn = 0) {
  const int cg = (M > BM) ? 2 : 1;
  const int maxc = sm_count() / cg;
  const int64_t rows = (M + BM * cg - 1) / (BM * cg);
  const int num_kb = static_cast<int>((K + kps - 1) / kps);
  const double tile_us = num_kb * kStageUs;   // one 256-wide tile, all of K
  auto whole = [&](int tbn, double* cost) {
    const int64_t t = rows * ((N + tbn - 1) / tbn);
    Plan p{};
    p.cg = cg;
    p.tbn = tbn;
    p.clusters = static_cast<int>(t < maxc ? t : maxc);
    p.full_tiles = static_cast<int>(t);
    p.split = 1;
    *cost = static_cast<double>((t + maxc - 1) / maxc) * tile_us *
            (tbn == 128 ? kNarrowCost : 1.0);
    return p;
  };
  double c256 = 0, c128 = 0;
  Plan best = whole(256, &c256);
  double best_cost = c256;
  if (narrow_ok && force_tbn != 256) {
    Plan p = whole(128, &c128);
    if (force_tbn == 128 || c128 < best_cost) {
      best = p;
      best_cost = c128;
    }
    if (use_split) {
      // the split, on 128-wide tiles
      const int64_t t = rows * ((N + 127) / 128);
      const int64_t full = (t / maxc) * maxc;
      const int rem = static_cast<int>(t - full);
      int sp = rem ? maxc / rem : 1;
      if (sp > 4) sp = 4;                          // bound the partial traffic
      if (sp > num_kb / 2) sp = num_kb / 2;        // at least 2 stages per range
      const double cs =
          (static_cast<double>(full / maxc) + 1.0 / sp) * tile_us * kNarrowCost + kSplitUs;
      // a forced 128 width splits whenever the tiles leave a partial wave
      if (sp >= 2 && (force_tbn == 128 || cs < best_cost)) {
        Plan q{};
        q.cg = cg;
        q.tbn = 128;
        q.full_tiles = static_cast<int>(full);
        q.split = sp;
        q.rem = rem;
        const int64_t items = full + static_cast<int64_t>(rem) * sp;
        q.clusters = static_cast<int>(items < maxc ? items : maxc);
        q.part_bytes = static_cast<size_t>(rem) * sp * cg * BM * 128 * sizeof(float);
        q.ws_bytes = q.part_bytes + static_cast<size_t>(rem) * cg * sizeof(unsigned long long);
        best = q;
        best_cost = cs;
      }
    }
  }
  return best;
}

// K elements per stage of each kind.
int stage_k(int kind) {
  return kind == KIND_MXF4 ? KT<KIND_MXF4>::KPS
                           : kind == KIND_MXF8 ? KT<KIND_MXF8>::KPS : KT<KIND_F16>::KPS;
}

// A split launch's counter tag: 48 bits, non-zero, different for every launch
// of the process (a per-process random start plus a launch count), so that
// whatever the caller's workspace held -- or a counter an aborted launch left
// behind -- does not count as an arrival of this one.  (Completed launches
// leave their counters at zero.)
unsigned long long next_tag() {
  static std::atomic<unsigned long long> count{0};
  static const unsigned long long start = [] {
    unsigned long long z =
        static_cast<unsigned long long>(
            std::chrono::steady_clock::now().time_since_epoch().count()) ^
        (reinterpret_cast<uintptr_t>(&count) << 7);
    // splitmix64 finaliser
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
  }();
  for (;;) {
    const unsigned long long t = (start + count.fetch_add(1)) & ((1ull << 48) - 1);
    if (t != 0) return t;
  }
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

// Tensor map of any rank.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  const cuuint32_t* estr, CUtensorMapSwizzle swz) {
  auto enc = get_encode();
  if (!enc) return false;
  return enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map, row-major rows x cols (cols contiguous).
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

// Tile width override (mx_set_tile_width): 0 picks per shape.
static std::atomic<int> g_force_tbn{0};
void gemm_force_tile_width(int tbn) { g_force_tbn.store(tbn); }

size_t gemm_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const int k = (kind == FMT_E4M3 || kind == FMT_E5M2) ? KIND_MXF8
                : (kind == FMT_E2M1)                  ? KIND_MXF4
                                                      : KIND_F16;
  // the split entry points store a plain C: 128-wide tiles are allowed
  return make_plan(M, N, K, stage_k(k), true, true, g_force_tbn.load()).ws_bytes;
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

// The tensor map through which the epilogue's TMA stores write a plain C:
// boxes of 32 rows x 128 bytes (32 fp32 or 64 bf16 values), 128-byte swizzle.
bool make_c_tmap(CUtensorMap* m, void* C, bool bf16, int64_t M, int64_t N, int64_t ldc) {
  return make_tmap(m, C, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   bf16 ? 2 : 4, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(ldc), bf16 ? 64 : 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Element-format field of the mxf8f6f4 instruction descriptor.
uint32_t f8f6f4_code(int fmt) { return fmt == FMT_E5M2 ? 1u : fmt == FMT_E2M1 ? 5u : 0u; }

// Raster group height: as many tile rows as keep the group's band of A
// (tile rows x K x bytes per A element) within 32 MB of L2, next to the
// columns of B the co-running clusters read and the C they write, so that B
// streams from DRAM once per group.  Measured on 8192^3 MXFP8 (DRAM bytes
// read per launch): 4 rows 527 MB, 8 rows 358 MB, 16 rows 278 MB, 32 rows
// 726 MB -- about 50-60 MB of the 126 MB L2 hold a band across the waves of
// a group; 16 rows (the 32 MB budget) read least and ran fastest.
int raster_group(int64_t M, int64_t K, int cg, double a_bytes_per_elem) {
  const int64_t num_m = (M + BM * cg - 1) / (BM * cg);
  const double band_row = static_cast<double>(BM * cg) * static_cast<double>(K) * a_bytes_per_elem;
  int64_t g = static_cast<int64_t>((32.0 * (1 << 20)) / (band_row > 1.0 ? band_row : 1.0));
  if (g < 1) g = 1;
  if (g > num_m) g = num_m;
  return static_cast<int>(g);
}

// Fill the split fields of a launch from its plan and the caller's workspace.
void set_split(gemm::Args& a, const Plan& p, void* ws) {
  a.full_tiles = p.full_tiles;
  a.split = p.split;
  a.ws = static_cast<float*>(ws);
  a.ctr = p.split > 1 ? reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) +
                                                              p.part_bytes)
                      : nullptr;
  a.tag = p.split > 1 ? next_tag() : 0;
}

}  // namespace

namespace {

Plan plan_for(int64_t M, int64_t N, int64_t K, int kind, bool use_split, bool narrow_ok) {
  return make_plan(M, N, K, stage_k(kind), use_split, narrow_ok, g_force_tbn.load());
}

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
  const int out = epi.q_fmt == FMT_E2M1 ? OUT_MX4
                  : epi.q_fmt != 0      ? OUT_MX8
                  : c_dtype == DT_BF16  ? OUT_BF16
                                        : OUT_F32;
  const bool narrow_ok = (out == OUT_F32 || out == OUT_BF16);
  Plan plan = plan_for(M, N, K, kind, ws != nullptr, narrow_ok);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes) plan = plan_for(M, N, K, kind, false, narrow_ok);
  const int ck = fp4 ? KT<KIND_MXF4>::CK : KT<KIND_MXF8>::CK;
  // one TMA box of B is this CTA's part of the tile's columns
  const uint32_t b_rows = static_cast<uint32_t>(plan.tbn / plan.cg);
  CUtensorMap ta, tb, tsa, tsb, tc;
  if (!make_data_tmap(&ta, a_data, fmt_a, fp4, M, K, BM) ||
      !make_data_tmap(&tb, b_data, fmt_b, fp4, N, K, b_rows) ||
      !make_sf_tmap(&tsa, a_sf, M, K, ck) || !make_sf_tmap(&tsb, b_sf, N, K, ck))
    return cudaErrorInvalidValue;
  if (narrow_ok) {
    if (!make_c_tmap(&tc, C, out == OUT_BF16, M, N, ldc)) return cudaErrorInvalidValue;
  } else {
    tc = ta;   // not read: an MX-quantized C is stored from registers
  }
  gemm::Launch l{&ta, &tb, &tsa, &tsb, &tc, plan.clusters, {}, st};
  l.args.C = C;
  l.args.ldc = ldc;
  l.args.M = static_cast<int>(M);
  l.args.N = static_cast<int>(N);
  l.args.K = static_cast<int>(K);
  l.args.ab_fmt = fp4 ? 0u : (f8f6f4_code(fmt_a) << 7) | (f8f6f4_code(fmt_b) << 10);
  l.args.group = raster_group(M, K, plan.cg, fmt_a == FMT_E2M1 ? 0.5 : 1.0);
  l.args.epi = epi_args(epi, M, N);
  set_split(l.args, plan, ws);
  return fp4 ? gemm::launch_mxf4(plan.cg, plan.tbn, out, l)
             : gemm::launch_mxf8(plan.cg, plan.tbn, out, l);
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
  Plan plan = plan_for(M, N, K, KIND_F16, ws != nullptr, true);
  if (plan.split > 1 && ws_bytes < plan.ws_bytes) plan = plan_for(M, N, K, KIND_F16, false, true);
  const CUtensorMapDataType dt = (ab_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb, tc;
  if (!make_tmap(&ta, A, dt, 2, K, M, lda, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tb, B, dt, 2, N, K, ldb, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_c_tmap(&tc, C, false, M, N, ldc))
    return cudaErrorInvalidValue;
  // the scale maps are unused by the 16-bit kinds
  gemm::Launch l{&ta, &tb, &ta, &tb, &tc, plan.clusters, {}, st};
  l.args.C = C;
  l.args.ldc = ldc;
  l.args.M = static_cast<int>(M);
  l.args.N = static_cast<int>(N);
  l.args.K = static_cast<int>(K);
  l.args.ab_fmt = 0;
  l.args.group = raster_group(M, K, plan.cg, 2.0);
  l.args.epi = epi_args(epi, M, N);
  set_split(l.args, plan, ws);
  return gemm::launch_f16(ab_dtype == DT_BF16 ? KIND_BF16 : KIND_F16, plan.cg, plan.tbn, l);
}

unsigned fetch_and_clear_status_gemm(cudaError_t* err) {
  cudaError_t e1 = cudaSuccess, e2 = cudaSuccess, e3 = cudaSuccess;
  const unsigned v = gemm::fetch_and_clear_status_mxf8(&e1) |
                     gemm::fetch_and_clear_status_mxf4(&e2) |
                     gemm::fetch_and_clear_status_f16(&e3);
  *err = e1 != cudaSuccess ? e1 : e2 != cudaSuccess ? e2 : e3;
  return v;
}

}  // namespace mxk
