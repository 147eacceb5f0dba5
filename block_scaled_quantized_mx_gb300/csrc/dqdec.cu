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
// Design.  The unit of work is a quad: one 128-row weight block times 256 K
// (four 64-K steps of four K = 16 MMAs each).  Every per-quad cost is paid
// once per quad, because a copy issue (~190 clocks of the issuing thread)
// or a tcgen05.commit (~100-170) per 64-K step would cap the stream well
// below HBM speed (measured on GB300: one copy + one commit per step held a
// CTA at ~0.3 us per 64 K, whatever the copy's size).
//   * work: with a few weight blocks (up to half as many as SMs) each
//     block's quads are split over a thread-block cluster of S CTAs (S a
//     power of two, up to 8, so that the clusters fill the SMs); the S fp32
//     partial accumulators are summed through distributed shared memory, in
//     rank order, so the result does not depend on timing, and no workspace
//     is needed.  With more blocks each CTA takes whole blocks in turn.
//   * warp 0: code producer -- per quad one copy of the block's codes (128
//     rows x 256 K: 128-byte rows in the 128-byte swizzle; 8-bit codes as two
//     such boxes, 2-bit codes as 64-byte rows in the 64-byte swizzle) and
//     its two scale atoms, into a ring as deep as shared memory allows;
//   * the last warp: token producer -- per quad one three-dimensional copy of
//     the tokens' 256-K slice (NT rows x 4 x 64 K, 128-byte swizzle), into
//     the quad's slot;
//   * warps 2..: dequantizers, in groups of four (one warp per tensor-memory
//     lane quarter) that take the quads in turn, one weight row per thread:
//     codes x scale -> 16-bit values written straight into the quad's
//     tensor-memory slot (tcgen05.st, 32 columns per 64 K), never through
//     shared memory; one arrival per quad.  With a single weight block per
//     CTA (as in every cluster) the four epilogue warps, idle until the
//     last MMA, join as one more group;
//   * warp 1: tensor-memory allocation and the MMA loop (one elected lane
//     issues): per quad up to 16 kind::f16 MMAs, M = 128 weight rows, N = NT
//     tokens, A read from the slot, B (the tokens) from shared memory, then
//     ONE commit that frees both the slot and the token slice; per range of
//     a weight block a commit of the accumulator (two buffers) to the
//     epilogue;
//   * four epilogue warps, one weight row per thread and 32 tokens at a
//     time: bias and activation, C[m][n] stored for every token m (a warp's
//     32 rows are 32 consecutive columns of C).  In a cluster, rank r owns
//     rows [128 r / S, 128 (r + 1) / S) of the block: after every rank's
//     MMAs are done, each thread sends its row's accumulator to the row's
//     owner (shared memory of that CTA), and the owners add the S parts in
//     rank order before the epilogue.
// Tensor memory: accumulators in columns [0, 2 NT), then the quad slots of
// 128 columns (three for NT = 64, two for NT = 128).
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records a
// timeout in g_status_dqd and the CTA shuts down in order.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "dq_common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

using namespace dq;

__device__ unsigned int g_status_dqd = 0;

constexpr int WR = 128;                  // weight rows per block (MMA M)
constexpr int KC = 64;                   // K per step (four K = 16 MMAs)
constexpr int QU = 4;                    // steps per quad
constexpr int MAX_CS = 8;                // code ring stages
constexpr int MAX_SLOTS = 3;
constexpr int NUM_EPI = 4;
constexpr int SMEM_BUDGET = 200 * 1024;  // token slots + code ring

// Warp layout per token width NT: code producer, MMA, dequantizer groups of
// four warps (one per tensor-memory lane quarter; a warp reaches the
// quarter warp % 4), four epilogue warps, token producer.  Two groups take
// the quads in turn for NT = 64 (one quad's conversion and stores overlap
// the other's); NT = 128, whose accumulators leave room for two slots and
// whose epilogue needs more registers, keeps one group.  The epilogue warps
// add a group when the CTA has one block (3 for NT = 64, 2 for NT = 128:
// one per slot).
template <int NT>
struct Lay {
  static constexpr int DQG = (NT == 64) ? 2 : 1;
  static constexpr int SLOTS = (NT == 64) ? 3 : 2;
  static constexpr int DQ_W0 = 2;
  static constexpr int EPI_W0 = DQ_W0 + 4 * DQG;
  static constexpr int XW = EPI_W0 + NUM_EPI;
  static constexpr int THREADS = 32 * (XW + 1);
  static constexpr int SLOT_COL0 = 2 * NT;
  static constexpr int X_BYTES = QU * NT * 128;   // one quad's token slice
  static_assert(SLOTS <= MAX_SLOTS, "slot barriers");
  static_assert(SLOT_COL0 + 128 * SLOTS <= 512, "tensor-memory columns");
};

constexpr int MAX_CLUSTER = 8;

// barriers: code_full[8], code_empty[8], x_full[3], slot_free[3],
// a_ready[3], acc_full[2], acc_empty[2]
constexpr int NBAR = 2 * MAX_CS + 3 * MAX_SLOTS + 4;
constexpr int MISC_BYTES = 16;   // tensor-memory address, abort flag
// everything, with the 1024-byte alignment slack, within a CTA's 227 KB
static_assert(SMEM_BUDGET + 8 * NBAR + MISC_BYTES + 1024 <= 227 * 1024, "shared memory");

struct DecArgs {
  void* C;
  int64_t ldc;
  int M, N, K;
  int fmt;              // B's element format
  int a_bf16;           // A (and the dequantized weights) bf16, else f16
  int cs;               // code ring depth
  int cs_bytes;         // code ring stride: codes + two scale atoms, 1024-aligned
  int qb;               // bytes of one weight row's codes per quad (256 K)
  int S;                // cluster size: the ranks that split one block's quads
  EpiArgs epi;
};

// One outcome of a wait for a whole warp: the tensor-memory instructions
// after the warp-wide waits are warp-collective, so no lane may go on while
// another gives up.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xFFFFFFFFu, ok); }

__device__ __forceinline__ void dqd_timeout(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_status_dqd, STATUS_TIMEOUT | site);
}

// This CTA's work: jobs (weight block nb, quads [qa, qb) of it), in the
// order nb = nb0, nb0 + nb_step, ...; quad i of the CTA's sequence is
// quad qa + i % jq of job i / jq.
struct Work {
  int kq;        // quads per weight block
  int kch;       // 64-K steps per weight block
  int nb0, nb_step, n_jobs, qa, jq;
  __device__ int nq() const { return n_jobs * jq; }
};

// kind::f16 instruction descriptor: D f32, A and B f16 (0) or bf16 (1), both
// K-major (A from tensor memory), N>>3 at bit 17, M = 128 (>>4 at bit 24).
template <int NT>
__device__ __forceinline__ uint32_t idesc_dec(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(NT >> 3) << 17) | (static_cast<uint32_t>(WR >> 4) << 24);
}

// The 16-byte chunk c of weight row r of a code box, as TMA placed it:
// 128-byte rows in the 128-byte swizzle (chunk c ^ (r % 8)), or 64-byte rows
// (2-bit codes) in the 64-byte swizzle (chunk c ^ ((r / 2) % 4)).
template <int BITS>
__device__ __forceinline__ uint4 code_chunk(uint32_t box, int r, int c) {
  if (BITS == 2)
    return ld_shared_v4(box + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
  return ld_shared_v4(box + r * 128 + ((c ^ (r & 7)) << 4));
}

// One 64-K step of weight row r from a quad's code stage: its two 32-element
// blocks' codes in w0, w1 (words as dq_block_regs reads them).
template <int FMT>
__device__ __forceinline__ void step_codes(uint32_t st, int r, int j, uint32_t (&w0)[8],
                                           uint32_t (&w1)[8]) {
  constexpr int BITS = (FMT == FMT_INT2) ? 2 : (FMT == FMT_INT4 || FMT == FMT_E2M1) ? 4 : 8;
  if (BITS == 8) {
    // step j: box j / 2, bytes 64 (j % 2) .. of the 128-byte row
    const uint32_t box = st + (j >> 1) * (WR * 128);
    const int c0 = (j & 1) * 4;
    const uint4 a = code_chunk<8>(box, r, c0), b = code_chunk<8>(box, r, c0 + 1);
    const uint4 c = code_chunk<8>(box, r, c0 + 2), d = code_chunk<8>(box, r, c0 + 3);
    w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
    w0[4] = b.x; w0[5] = b.y; w0[6] = b.z; w0[7] = b.w;
    w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w;
    w1[4] = d.x; w1[5] = d.y; w1[6] = d.z; w1[7] = d.w;
  } else if (BITS == 4) {
    const uint4 a = code_chunk<4>(st, r, 2 * j), b = code_chunk<4>(st, r, 2 * j + 1);
    w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
    w1[0] = b.x; w1[1] = b.y; w1[2] = b.z; w1[3] = b.w;
  } else {
    const uint4 a = code_chunk<2>(st, r, j);
    w0[0] = a.x; w0[1] = a.y;
    w1[0] = a.z; w1[1] = a.w;
  }
}

// One dequantizer warp's part of this CTA's quads (those of its group):
// weight row 32 q + lane, every 64-K step of the quad into the quad's slot.
template <int FMT, int NT>
__device__ __forceinline__ void dequant_loop(const DecArgs& a, const Work& wk,
                                             uint32_t code_base, uint32_t tmem_base,
                                             uint32_t bar_code_full, uint32_t bar_code_empty,
                                             uint32_t bar_slot_free, uint32_t bar_a_ready, int q,
                                             int g, int ngroups, int lane, volatile int* abort) {
  using LY = Lay<NT>;
  const int row = 32 * q + lane;
  const bool bf16 = a.a_bf16 != 0;
  const uint32_t qrow = static_cast<uint32_t>(32 * q) << 16;
  // the scale word of this row in a scale atom: blocks 0..3 of the atom
  const uint32_t sf_word = 16 * (row & 31) + 4 * ((row >> 5) & 3);
  const int nq = wk.nq();
  for (int i = g; i < nq; i += ngroups) {
    const int qi = wk.qa + i % wk.jq;
    const int nu = min(QU, wk.kch - QU * qi);
    const int s = i % a.cs;
    if (!warp_all(mbar_wait_short(bar_code_full + 8 * s, (i / a.cs) & 1, abort))) {
      dqd_timeout(abort, 21);
      return;
    }
    const int slot = i % LY::SLOTS;
    if (!warp_all(mbar_wait_short(bar_slot_free + 8 * slot, ((i / LY::SLOTS) & 1) ^ 1, abort))) {
      dqd_timeout(abort, 22);
      return;
    }
    tc_fence_after();
    const uint32_t st = code_base + static_cast<uint32_t>(s) * a.cs_bytes;
    const uint32_t sf0 = st + WR * a.qb;
    const uint32_t scw0 = ld_shared_u32(sf0 + sf_word), scw1 = ld_shared_u32(sf0 + 512 + sf_word);
    const uint32_t ta = tmem_base + qrow + LY::SLOT_COL0 + slot * 128;
    // two 64-K steps per pass (both in one scale atom): all their code loads
    // first, then both conversions, so that one step's latency overlaps the
    // other's work
    int j = 0;
#pragma unroll 1
    for (; j + 2 <= nu; j += 2) {
      uint32_t w0[8], w1[8], w2[8], w3[8];
      step_codes<FMT>(st, row, j, w0, w1);
      step_codes<FMT>(st, row, j + 1, w2, w3);
      const uint32_t sw = (j >> 1) ? scw1 : scw0;
      uint32_t o0[16], o1[16], o2[16], o3[16];
      dq_block_regs<FMT>(w0, sw & 0xFFu, bf16, o0);
      dq_block_regs<FMT>(w1, (sw >> 8) & 0xFFu, bf16, o1);
      dq_block_regs<FMT>(w2, (sw >> 16) & 0xFFu, bf16, o2);
      dq_block_regs<FMT>(w3, sw >> 24, bf16, o3);
      uint32_t o[32], p[32];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        o[k] = o0[k];
        o[16 + k] = o1[k];
        p[k] = o2[k];
        p[16 + k] = o3[k];
      }
      tmem_st_32x32b_x32(ta + 32 * j, o);
      tmem_st_32x32b_x32(ta + 32 * (j + 1), p);
    }
    if (j < nu) {   // an odd last step (the end of K)
      uint32_t w0[8], w1[8];
      step_codes<FMT>(st, row, j, w0, w1);
      const uint32_t sw = ((j >> 1) ? scw1 : scw0) >> (16 * (j & 1));
      uint32_t o0[16], o1[16], o[32];
      dq_block_regs<FMT>(w0, sw & 0xFFu, bf16, o0);
      dq_block_regs<FMT>(w1, (sw >> 8) & 0xFFu, bf16, o1);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        o[k] = o0[k];
        o[16 + k] = o1[k];
      }
      tmem_st_32x32b_x32(ta + 32 * j, o);
    }
    // codes and scales consumed (the stores above read registers only)
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_code_empty + 8 * s);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_a_ready + 8 * slot);
  }
}

// dequant_loop for B's element format.
template <int NT>
__device__ __forceinline__ void dequant_any(const DecArgs& a, const Work& wk, uint32_t code_base,
                                            uint32_t tmem_base, uint32_t bar_code_full,
                                            uint32_t bar_code_empty, uint32_t bar_slot_free,
                                            uint32_t bar_a_ready, int q, int g, int ngroups,
                                            int lane, volatile int* abort) {
#define MXK_DQD_LOOP(F)                                                                   \
  dequant_loop<F, NT>(a, wk, code_base, tmem_base, bar_code_full, bar_code_empty,         \
                      bar_slot_free, bar_a_ready, q, g, ngroups, lane, abort)
  switch (a.fmt) {
    case FMT_INT4: MXK_DQD_LOOP(FMT_INT4); break;
    case FMT_INT8: MXK_DQD_LOOP(FMT_INT8); break;
    case FMT_INT2: MXK_DQD_LOOP(FMT_INT2); break;
    case FMT_E2M1: MXK_DQD_LOOP(FMT_E2M1); break;
    case FMT_E5M2: MXK_DQD_LOOP(FMT_E5M2); break;
    default: MXK_DQD_LOOP(FMT_E4M3); break;
  }
#undef MXK_DQD_LOOP
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
  using LY = Lay<NT>;
  constexpr int SLOTS = LY::SLOTS;
  constexpr int EPI_W0 = LY::EPI_W0;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  // [token slots][code ring][barriers][misc]
  const uint32_t x_base = base;
  const uint32_t code_base = x_base + SLOTS * LY::X_BYTES;
  const uint32_t bars = code_base + static_cast<uint32_t>(a.cs) * a.cs_bytes;
  const uint32_t bar_code_full = bars;
  const uint32_t bar_code_empty = bar_code_full + 8 * MAX_CS;
  const uint32_t bar_x_full = bar_code_empty + 8 * MAX_CS;
  const uint32_t bar_slot_free = bar_x_full + 8 * MAX_SLOTS;
  const uint32_t bar_a_ready = bar_slot_free + 8 * MAX_SLOTS;
  const uint32_t bar_acc_full = bar_a_ready + 8 * MAX_SLOTS;
  const uint32_t bar_acc_empty = bar_acc_full + 16;
  uint8_t* misc = gbase + (bars - base) + 8 * NBAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = reinterpret_cast<volatile int*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.S;
  const int rank = (S > 1) ? static_cast<int>(cluster_ctarank()) : 0;
  Work wk;
  wk.kch = a.K / KC;
  wk.kq = (wk.kch + QU - 1) / QU;
  {
    const int nbk = (a.N + WR - 1) / WR;
    if (S > 1) {   // one block per cluster, its quads split over the ranks
      wk.nb0 = blockIdx.x / S;
      wk.nb_step = 1;
      wk.n_jobs = 1;
      wk.qa = rank * wk.kq / S;
      wk.jq = (rank + 1) * wk.kq / S - wk.qa;
    } else {       // whole blocks, in turn
      wk.nb0 = blockIdx.x;
      wk.nb_step = gridDim.x;
      wk.n_jobs = (nbk - wk.nb0 + gridDim.x - 1) / gridDim.x;
      wk.qa = 0;
      wk.jq = wk.kq;
    }
  }
  const int nq = wk.nq();
  // dequantizer groups: the epilogue warps join as one more when this CTA
  // has a single block (every slot then has its own group)
  const int ngroups = (wk.n_jobs == 1) ? LY::DQG + 1 : LY::DQG;

  if (warp == 0) {
    constexpr int N0 = 2 * MAX_CS, N1 = N0 + 3 * MAX_SLOTS;
    for (int i = lane; i < NBAR; i += 32) {
      uint32_t count = 1;   // code_full, x_full, slot_free, acc_full
      if (i >= MAX_CS && i < N0) count = 4;                              // code_empty
      else if (i >= N0 + 2 * MAX_SLOTS && i < N1) count = 4;             // a_ready
      else if (i >= N1 + 2) count = NUM_EPI;                            // acc_empty
      mbar_init(bar_code_full + 8 * i, count);
    }
    fence_mbar_init();
    if (lane == 0) {
      *abort = 0;
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmSF);
    }
  }
  if (warp == 1) tmem_alloc_cg<1>(smem_u32(tmem_slot), 512);
  __syncwarp();   // reconverge before the aligned barrier (lane-dependent setup)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------- code producer
    if (lane == 0) {
      const int k_atoms = (a.K + 127) / 128;
      const uint32_t tx = static_cast<uint32_t>(WR * a.qb + 2 * 512);
      const bool two_boxes = a.qb > 128;   // 8-bit codes: two 128-byte boxes
      int nb = wk.nb0, qi = wk.qa, jr = 0;
      for (int i = 0; i < nq; ++i) {
        const int s = i % a.cs;
        if (!mbar_wait(bar_code_empty + 8 * s, ((i / a.cs) & 1) ^ 1, abort)) {
          dqd_timeout(abort, 20);
          break;
        }
        const uint32_t full = bar_code_full + 8 * s;
        const uint32_t st = code_base + static_cast<uint32_t>(s) * a.cs_bytes;
        mbar_arrive_expect_tx(full, tx);
        tma_load_2d(st, &tmW, full, qi * a.qb, nb * WR);
        if (two_boxes) tma_load_2d(st + WR * 128, &tmW, full, qi * a.qb + 128, nb * WR);
        tma_load_2d(st + WR * a.qb, &tmSF, full, 0, nb * k_atoms + 2 * qi);
        ++qi;
        if (++jr == wk.jq) {
          jr = 0;
          qi = wk.qa;
          nb += wk.nb_step;
        }
      }
    }
  } else if (warp == LY::XW) {
    // ------------------------------------------------------ token producer
    if (lane == 0) {
      int qi = wk.qa, jr = 0;
      for (int i = 0; i < nq; ++i) {
        const int slot = i % SLOTS;
        if (!mbar_wait(bar_slot_free + 8 * slot, ((i / SLOTS) & 1) ^ 1, abort)) {
          dqd_timeout(abort, 29);
          break;
        }
        const uint32_t full = bar_x_full + 8 * slot;
        mbar_arrive_expect_tx(full, static_cast<uint32_t>(LY::X_BYTES));
        tma_load_3d(x_base + slot * LY::X_BYTES, &tmX, full, 0, 0, QU * qi);
        ++qi;
        if (++jr == wk.jq) {
          jr = 0;
          qi = wk.qa;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool issuer = elect_one();
    const uint32_t id = idesc_dec<NT>(a.a_bf16 != 0);
    int i = 0;
    bool ok = true;
    for (int job = 0; job < wk.n_jobs && ok; ++job) {
      const uint32_t buf = job & 1, use = job >> 1;
      if (!warp_all(mbar_wait_spin(bar_acc_empty + 8 * buf, (use & 1u) ^ 1u, abort))) {
        dqd_timeout(abort, 23);
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + buf * NT;
      for (int jr = 0; jr < wk.jq; ++jr, ++i) {
        const int slot = i % SLOTS;
        const uint32_t sph = (i / SLOTS) & 1u;
        // the MMA warp's waits are on the critical path: spin rather than
        // sleep through a wake-up
        if (!warp_all(mbar_wait_spin(bar_a_ready + 8 * slot, sph, abort) &&
                      mbar_wait_spin(bar_x_full + 8 * slot, sph, abort))) {
          dqd_timeout(abort, 24);
          ok = false;
          break;
        }
        tc_fence_after();
        const int nu = min(QU, wk.kch - QU * (wk.qa + jr));
        if (issuer) {
          const uint32_t xs = x_base + slot * LY::X_BYTES;
          const uint32_t as = tmem_base + LY::SLOT_COL0 + slot * 128;
          for (int j = 0; j < nu; ++j) {
            const uint64_t xd = smem_desc(xs + j * (NT * 128), 16, 1024, 2);
#pragma unroll
            for (int kk = 0; kk < KC / 16; ++kk)
              mma_f16_ts(d, as + 32 * j + 8 * kk, xd + 2 * kk, id,
                         (jr == 0 && j == 0 && kk == 0) ? 0u : 1u);
          }
          tc_commit(bar_slot_free + 8 * slot);   // the slot and the token slice
        }
        __syncwarp();
      }
      if (!ok) break;
      if (issuer) tc_commit(bar_acc_full + 8 * buf);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ dequantizers
    // One call site for every group, so the conversion loop exists once in
    // the code and in the instruction cache.  With a single block the
    // epilogue warps have nothing to do until the last MMA: they convert
    // quads meanwhile, as one more group.
    const bool epi_warp = warp >= EPI_W0;
    if (!epi_warp || ngroups > LY::DQG)
      dequant_any<NT>(a, wk, code_base, tmem_base, bar_code_full, bar_code_empty, bar_slot_free,
                      bar_a_ready, warp & 3, epi_warp ? LY::DQG : (warp - LY::DQ_W0) >> 2,
                      ngroups, lane, abort);
  }
  if (warp >= EPI_W0 && warp < EPI_W0 + NUM_EPI) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    for (int job = 0; job < wk.n_jobs; ++job) {
      const uint32_t buf = job & 1, use = job >> 1;
      if (!warp_all(mbar_wait(bar_acc_full + 8 * buf, use & 1u, abort))) {
        dqd_timeout(abort, 25);
        break;
      }
      tc_fence_after();
      if (S > 1) break;   // a cluster's block is summed below, after every rank's MMAs
      const int nb = wk.nb0 + job * wk.nb_step;
      const int n = nb * WR + 32 * q + lane;   // weight row = column of C
#pragma unroll 1
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tq + buf * NT + 32 * cc, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
        dec_epi(v, a.epi, n, a.N);
        dec_store<OUT>(v, a.C, a.ldc, 32 * cc, n, a.M, a.N);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
    }
  }

  __syncwarp();   // reconverge before the aligned barriers (one-lane roles)
  tc_fence_before();
  if (S > 1) {
    // Every rank's MMAs are done (its epilogue waited for them) and its
    // token slots are free: they receive the other ranks' rows.  Rank r's
    // rows [r R, r R + R), R = 128 / S, arrive from rank s at
    // x_base + s (R NT 4) bytes, float4 (row lr, tokens 4 c4 .. 4 c4 + 3) at
    // (c4 R + lr) 16: consecutive lanes write consecutive 16 bytes.
    cluster_sync();
    tc_fence_after();
    const int R = WR / S;
    const bool epi = warp >= EPI_W0 && warp < EPI_W0 + NUM_EPI;
    const int q = warp & 3, row = 32 * q + lane, owner = row / R, lr = row - owner * R;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    if (epi) {
      const uint32_t dst = map_to_cta(x_base, static_cast<uint32_t>(owner)) +
                           static_cast<uint32_t>(rank * R * NT * 4 + lr * 16);
#pragma unroll 1
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tq + 32 * cc, r);
        tmem_wait_ld();
        if (owner != rank) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_cluster_v4(dst + static_cast<uint32_t>((8 * cc + j) * R * 16),
                          __uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                          __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
        __syncwarp();   // converged for the next warp-wide load
      }
    }
    __syncwarp();
    cluster_sync();
    if (epi) {
      // the S parts of this row, in rank order (the tensor-memory loads are
      // warp-wide; with S = 8 a warp's rows have two owners)
      const int n = wk.nb0 * WR + row;
#pragma unroll 1
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tq + 32 * cc, r);
        tmem_wait_ld();
        if (owner == rank) {
          float v[32];
          for (int sr = 0; sr < S; ++sr) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float4 x;
              if (sr == rank) {
                x = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
              } else {
                const uint4 u = ld_shared_v4(x_base + static_cast<uint32_t>(
                                                          sr * R * NT * 4 + lr * 16 +
                                                          (8 * cc + j) * R * 16));
                x = make_float4(__uint_as_float(u.x), __uint_as_float(u.y),
                                __uint_as_float(u.z), __uint_as_float(u.w));
              }
              if (sr == 0) {
                v[4 * j] = x.x;
                v[4 * j + 1] = x.y;
                v[4 * j + 2] = x.z;
                v[4 * j + 3] = x.w;
              } else {
                v[4 * j] += x.x;
                v[4 * j + 1] += x.y;
                v[4 * j + 2] += x.z;
                v[4 * j + 3] += x.w;
              }
            }
          }
          dec_epi(v, a.epi, n, a.N);
          dec_store<OUT>(v, a.C, a.ldc, 32 * cc, n, a.M, a.N);
        }
        __syncwarp();   // converged for the next warp-wide load
      }
    }
    __syncwarp();
    tc_fence_before();
  }
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

// The cluster size S for a product with nbk weight blocks of kq quads: the
// largest power of two (up to 8) with nbk S <= SMs and S <= kq; 1 (whole
// blocks per CTA, no reduction) once the blocks alone fill half the SMs.
int dqd_cluster(int64_t nbk, int64_t kq) {
  const int64_t sms = dqd_sm_count();
  if (2 * nbk > sms) return 1;
  int S = 1;
  while (2 * S <= MAX_CLUSTER && nbk * 2 * S <= sms && 2 * S <= kq) S *= 2;
  return S;
}

template <int NT, int OUT>
cudaError_t dqd_run(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& tsf,
                    DecArgs a, int grid, cudaStream_t st) {
  using LY = Lay<NT>;
  const int ring = SMEM_BUDGET - LY::SLOTS * LY::X_BYTES;
  a.cs = ring / a.cs_bytes;
  if (a.cs > MAX_CS) a.cs = MAX_CS;
  if (a.cs < 2) return cudaErrorInvalidValue;
  // the token slots take the other ranks' rows at the end: S x (128 / S) x NT fp32
  static_assert(LY::SLOTS * LY::X_BYTES >= WR * NT * 4, "reduction buffer");
  auto kern = dqdec_kernel<NT, OUT>;
  const int smem = LY::SLOTS * LY::X_BYTES + a.cs * a.cs_bytes + 8 * NBAR + MISC_BYTES + 1024;
  static int attr_smem[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || attr_smem[dev] < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_smem[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(LY::THREADS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx, tw, tsf, a);
}

}  // namespace

// Whether the decode kernel takes this product (a few tokens, a plain or
// bias / activation output).
bool dequant_decode_applies(int64_t M, const Epilogue& epi) {
  return M >= 1 && M <= 128 && epi.q_fmt == 0;
}

// The decode kernel needs no workspace: its K split stays inside a cluster.
size_t dequant_decode_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_gemm_dequant_decode(int a_dtype, const void* A, int64_t lda, int fmt_b,
                                       const void* b_data, const uint8_t* b_sf, void* C,
                                       int c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                       const Epilogue& epi, cudaStream_t st) {
  const int64_t nbk = (N + WR - 1) / WR, kq = (K / KC + QU - 1) / QU;
  if (nbk * kq >= (int64_t{1} << 31)) return cudaErrorInvalidValue;   // 32-bit quad counts
  const int nt = (M <= 64) ? 64 : 128;
  const int bits = code_bits(fmt_b);
  DecArgs a{};
  a.C = C;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.fmt = fmt_b;
  a.a_bf16 = (a_dtype == DT_BF16) ? 1 : 0;
  a.qb = QU * KC * bits / 8;                       // 256, 128 or 64 bytes
  a.cs_bytes = (WR * a.qb + 2 * 512 + 1023) / 1024 * 1024;
  a.S = dqd_cluster(nbk, kq);
  a.epi.bias = epi.bias;
  a.epi.act = epi.act;
  a.epi.q_fmt = 0;
  a.epi.q_sf = nullptr;
  a.epi.q_k_atoms = 0;
  a.epi.q_row_atoms = 0;
  const int64_t sms = dqd_sm_count();
  const int grid = static_cast<int>(a.S > 1 ? nbk * a.S : (nbk < sms ? nbk : sms));
  const CUtensorMapDataType dt = (a_dtype == DT_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t row_bytes = static_cast<uint64_t>(K) * bits / 8;
  const uint64_t atoms = static_cast<uint64_t>(sf_row_atoms(N) * sf_k_atoms(K));
  // the tokens as [K / 64][M][64]: one box is a quad's four 64-K slices of
  // NT rows, each slice 128-byte rows in the 128-byte swizzle
  const cuuint64_t xdims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
  const cuuint64_t xstrides[2] = {static_cast<cuuint64_t>(lda) * 2, 128};
  const cuuint32_t xbox[3] = {64, static_cast<cuuint32_t>(nt), QU};
  const cuuint32_t xestr[3] = {1, 1, 1};
  const uint32_t wbox = a.qb > 128 ? 128u : static_cast<uint32_t>(a.qb);
  CUtensorMap tx, tw, tsf;
  if (!encode_tiled(&tx, dt, 3, A, xdims, xstrides, xbox, xestr, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tw, b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, row_bytes,
                 static_cast<uint64_t>(N), row_bytes, wbox, WR,
                 wbox == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tsf, b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128, atoms, 128, 128, 2,
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
