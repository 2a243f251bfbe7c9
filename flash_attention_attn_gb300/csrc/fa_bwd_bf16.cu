// fa_bwd_bf16.cu -- attention backward for sm_103a (tcgen05 + TMA).
//
// Two kernels, each recomputing P block by block from the forward's LSE:
//
// dK/dV: one CTA per (b, kv head g, 128-row KV block).  It keeps K and V in
//   shared memory and dK, dV in TMEM for its whole life, and visits every
//   query head of the group and every 128-row query block that sees the KV
//   block.  Accumulation is private to the CTA: no atomics.
//     S^T  = K Q^T          (TMEM, KV rows on lanes)
//     dP^T = V dO^T
//     P^T  = 2^(S^T*scale*log2e - LSE*log2e), masked           -> bf16, TMEM
//     dV  += P^T dO          (A operand from TMEM)
//     dS^T = P^T (dP^T - Delta)                                -> bf16, TMEM
//     dK  += dS^T Q
//   and at the end dK *= scale.  (forge flash_attention.metal,
//   flash_attn_bwd_dv / flash_attn_bwd_dk: one owner per key row summing over
//   the group's query heads; teeny-kernels flash_attn2.rs,
//   flash_attention2_backward_dkv: no atomics are needed.)
//
// dQ: one CTA per (b, h, 128-row query block); loops over the visible KV
//   blocks in a fixed order, so the result is bitwise reproducible.
//     S = Q K^T ; dP = dO V^T ; dS = P (dP - Delta) -> bf16, TMEM ; dQ += dS K
//   and at the end dQ *= scale.  (forge flash_attention.metal,
//   flash_attn_bwd_dq; teeny-kernels flash_attention2_backward_dq.)
//
// Warp roles in both kernels: warps 0-7 compute (warp w owns TMEM lanes
// 32*(w%4).. and the column half w/4), warp 8 TMA producer, warp 9 MMA issuer
// and TMEM owner.  Both compute halves write their bf16 results back into the
// columns they themselves read, so no half overwrites data the other half
// still has to load.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kCompute = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Ctl& ctl, unsigned code) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, ctl, code);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

__device__ __forceinline__ void reg_tie(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Named barrier over the 256 compute threads (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// TMEM column of the 16-wide K slice kk of a 128-wide bf16 operand written by
// the two compute halves: half 0 packs keys 0..63 into columns [0, 32), half 1
// packs keys 64..127 into columns [64, 96) of the same region.
__device__ __forceinline__ uint32_t packed_slice_col(int kk) { return (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8; }

// Store 64 values (this thread's half of a 128-wide row) as 32 packed bf16x2
// columns starting at taddr.
__device__ __forceinline__ void store_half_row_bf16(uint32_t taddr, const float (&v)[64]) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
  tmem_st16(taddr, pk);
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(v[32 + 2 * e], v[32 + 2 * e + 1]);
  tmem_st16(taddr + 16, pk);
}

__device__ __forceinline__ void load_half_row(uint32_t taddr, float (&v)[64]) {
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr, r0);
  tmem_ld32(taddr + 32, r1);
  tmem_ld_wait(r0);
  reg_tie(r1);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    v[c] = __uint_as_float(r0[c]);
    v[32 + c] = __uint_as_float(r1[c]);
  }
}

// Write `ncols` fp32 TMEM columns of this thread's lane, times `mul`, as bf16
// to global memory at dst (16-byte aligned, ncols a multiple of 32).
__device__ __forceinline__ void store_acc_row(uint32_t taddr, int ncols, float mul, __nv_bfloat16* dst,
                                              bool valid) {
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + c, r);
    tmem_ld_wait(r);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (valid) {
      uint4* d = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
      for (int v = 0; v < 4; ++v) d[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 64 * 2;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = 2;
  // dK/dV kernel: K, V resident; Q and dO streamed.
  // dQ kernel:    Q, dO resident; K and V streamed.
  static constexpr int kOffA = 0;                          // resident tile 1
  static constexpr int kOffB = kTileBytes;                 // resident tile 2
  static constexpr int kOffX = 2 * kTileBytes;             // streamed tile 1, kStages deep
  static constexpr int kOffY = kOffX + kStages * kTileBytes;  // streamed tile 2
  static constexpr int kOffBar = kOffY + kStages * kTileBytes;
  static constexpr int kOffRow = kOffBar + 512;            // per-stage LSE / Delta rows
  static constexpr int kSmemBytes = kOffRow + 2 * 2 * 128 * 4 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmS = 0;     // S or S^T, 128 columns
  static constexpr uint32_t kTmDP = 128;  // dP or dP^T, 128 columns
  static constexpr uint32_t kTmAcc = 256; // dV then dK (dK/dV kernel) or dQ
};

struct BwdBars {
  uint64_t res_full;     // resident tiles loaded
  uint64_t x_full[2];    // streamed stage loaded (both tiles)
  uint64_t x_empty[2];   // streamed stage consumed by the MMAs
  uint64_t s_full;       // S (S^T) in TMEM
  uint64_t dp_full;      // dP (dP^T) in TMEM
  uint64_t p_full;       // P^T written back (dK/dV kernel only)
  uint64_t ds_full;      // dS (dS^T) written back
  uint64_t acc_full;     // accumulators final
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// ============================================================== dK / dV

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                            const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  float* srow = reinterpret_cast<float*>(smem + C::kOffRow);  // [2 buffers][LSE 128 | Delta 128]

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kb = blockIdx.x;  // small kb sees the most query blocks: launched first
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int rep = s.H / s.HKV;
  int qlo, qhi;
  q_range_for_kv(s.T, kBM, kBN, s.causal, s.window, kb, qlo, qhi);
  const int nqb = qhi - qlo + 1;
  const int niter = rep * nqb;  // (head r, query block qb) pairs, r outer

  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->x_full[i], 1);
      mbar_init(&bars->x_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, kCompute);
    mbar_init(&bars->ds_full, kCompute);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Ctl ctl{&bars->abort, p.err, p.timeout_ns};
  constexpr unsigned kCode = 2u;  // FA_DEVERR_DKDV_TIMEOUT

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      mbar_arrive_expect_tx(&bars->res_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(&tmK, &bars->res_full, smem + C::kOffA + c * C::kChunkBytes, g * D + c * 64, kb * kBN, b);
        tma_load_3d(&tmV, &bars->res_full, smem + C::kOffB + c * C::kChunkBytes, g * D + c * 64, kb * kBN, b);
      }
      int issued = 0;
      for (int n = 0; n < niter; ++n) {
        const int st = n & 1;
        if (n >= 2 && !wait_bar(&bars->x_empty[st], ((n >> 1) - 1) & 1, ctl, kCode)) break;
        const int h = g * rep + n / nqb;
        const int qb = qlo + n % nqb;
        mbar_arrive_expect_tx(&bars->x_full[st], 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(&tmQ, &bars->x_full[st], smem + C::kOffX + st * C::kTileBytes + c * C::kChunkBytes,
                      h * D + c * 64, qb * kBM, b);
          tma_load_3d(&tmdO, &bars->x_full[st], smem + C::kOffY + st * C::kTileBytes + c * C::kChunkBytes,
                      h * D + c * 64, qb * kBM, b);
        }
        issued = n + 1;
      }
      if (bars->abort) {
        drain_bar(&bars->res_full, 0, p.timeout_ns);
        for (int n = imax(0, issued - 2); n < issued; ++n) drain_bar(&bars->x_full[n & 1], (n >> 1) & 1, p.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);  // K-major x K-major
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);   // TMEM A x MN-major B
      const uint32_t sK = sbase + C::kOffA;
      const uint32_t sV = sbase + C::kOffB;
      bool ok = wait_bar(&bars->res_full, 0, ctl, kCode);
      for (int n = 0; ok && n < niter; ++n) {
        const int st = n & 1;
        const uint32_t sQ = sbase + C::kOffX + st * C::kTileBytes;
        const uint32_t sdO = sbase + C::kOffY + st * C::kTileBytes;
        if (!(ok = wait_bar(&bars->x_full[st], (n >> 1) & 1, ctl, kCode))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // S^T = K Q^T
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kTmS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->s_full);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V dO^T
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kTmDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdO + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->dp_full);
        if (!(ok = wait_bar(&bars->p_full, n & 1, ctl, kCode))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)  // dV += P^T dO   (K = query rows)
          mma_ts(tmem + C::kTmAcc, tmem + C::kTmS + packed_slice_col(kk),
                 sdesc_sw128(sdO + kk * 2048, C::kChunkBytes, 1024), idesc_acc, (n > 0 || kk > 0));
        if (!(ok = wait_bar(&bars->ds_full, n & 1, ctl, kCode))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)  // dK += dS^T Q
          mma_ts(tmem + C::kTmAcc + D, tmem + C::kTmDP + packed_slice_col(kk),
                 sdesc_sw128(sQ + kk * 2048, C::kChunkBytes, 1024), idesc_acc, (n > 0 || kk > 0));
        mma_commit(&bars->x_empty[st]);
      }
      if (ok) mma_commit(&bars->acc_full);
      mma_commit(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- compute
    const int tid = threadIdx.x;        // 0..255
    const int quarter = warp & 3;       // TMEM lane quarter
    const int half = warp >> 2;         // column half
    const int jrow = quarter * 32 + lane;  // KV row within the block (TMEM lane)
    const int j = kb * kBN + jrow;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int n = 0; n < niter; ++n) {
      const int h = g * rep + n / nqb;
      const int qb = qlo + n % nqb;
      // stage LSE*log2e and Delta of the 128 query rows into shared memory
      float* buf = srow + (n & 1) * 256;
      {
        const int r = tid & 127;
        const int i = qb * kBM + r;
        const size_t idx = (static_cast<size_t>(b) * s.H + h) * s.T + i;
        float v = 0.f;
        if (i < s.T) v = (tid < 128) ? p.LSE[idx] * kLog2e : p.Delta[idx];
        buf[tid] = v;
      }
      compute_sync();
      if (!(ok = warp_wait(&bars->s_full, n & 1, ctl, kCode))) break;
      tc_fence_after();
      float pv[64];
      load_half_row(tmem + lane_addr + C::kTmS + half * 64, pv);
      const bool need_mask = block_needs_mask(s.T, kBM, kBN, s.causal, s.window, qb, kb);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int ic = half * 64 + c;  // query row within the block
        float e = ex2(fmaf(pv[c], sl2, -buf[ic]));
        if (need_mask && masked(s.T, s.causal, s.window, qb * kBM + ic, j)) e = 0.f;
        pv[c] = e;
      }
      store_half_row_bf16(tmem + lane_addr + C::kTmS + half * 64, pv);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      if (!(ok = warp_wait(&bars->dp_full, n & 1, ctl, kCode))) break;
      tc_fence_after();
      float dp[64];
      load_half_row(tmem + lane_addr + C::kTmDP + half * 64, dp);
#pragma unroll
      for (int c = 0; c < 64; ++c) dp[c] = pv[c] * (dp[c] - buf[128 + half * 64 + c]);
      store_half_row_bf16(tmem + lane_addr + C::kTmDP + half * 64, dp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    if (ok) ok = warp_wait(&bars->acc_full, 0, ctl, kCode);
    if (ok) {
      tc_fence_after();
      const size_t rowoff = ((static_cast<size_t>(b) * s.T + j) * s.HKV + g) * D + half * (D / 2);
      store_acc_row(tmem + lane_addr + C::kTmAcc + half * (D / 2), D / 2, 1.f,
                    static_cast<__nv_bfloat16*>(p.dV) + rowoff, j < s.T);
      store_acc_row(tmem + lane_addr + C::kTmAcc + D + half * (D / 2), D / 2, p.s.scale,
                    static_cast<__nv_bfloat16*>(p.dK) + rowoff, j < s.T);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================== dQ

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                          const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nq = ceil_div(s.T, kBM);
  const int qb = nq - 1 - static_cast<int>(blockIdx.x);  // longest causal tiles first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int g = h / (s.H / s.HKV);
  int kb_lo, kb_hi;
  kv_range_for_q(s.T, kBM, kBN, s.causal, s.window, qb, kb_lo, kb_hi);
  const int nblk = kb_hi - kb_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->x_full[i], 1);
      mbar_init(&bars->x_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, kCompute);
    mbar_init(&bars->ds_full, kCompute);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Ctl ctl{&bars->abort, p.err, p.timeout_ns};
  constexpr unsigned kCode = 4u;  // FA_DEVERR_DQ_TIMEOUT

  if (warp == 8) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
      mbar_arrive_expect_tx(&bars->res_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(&tmQ, &bars->res_full, smem + C::kOffA + c * C::kChunkBytes, h * D + c * 64, qb * kBM, b);
        tma_load_3d(&tmdO, &bars->res_full, smem + C::kOffB + c * C::kChunkBytes, h * D + c * 64, qb * kBM, b);
      }
      int issued = 0;
      for (int n = 0; n < nblk; ++n) {
        const int st = n & 1;
        if (n >= 2 && !wait_bar(&bars->x_empty[st], ((n >> 1) - 1) & 1, ctl, kCode)) break;
        const int kb = kb_lo + n;
        mbar_arrive_expect_tx(&bars->x_full[st], 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(&tmK, &bars->x_full[st], smem + C::kOffX + st * C::kTileBytes + c * C::kChunkBytes,
                      g * D + c * 64, kb * kBN, b);
          tma_load_3d(&tmV, &bars->x_full[st], smem + C::kOffY + st * C::kTileBytes + c * C::kChunkBytes,
                      g * D + c * 64, kb * kBN, b);
        }
        issued = n + 1;
      }
      if (bars->abort) {
        drain_bar(&bars->res_full, 0, p.timeout_ns);
        for (int n = imax(0, issued - 2); n < issued; ++n) drain_bar(&bars->x_full[n & 1], (n >> 1) & 1, p.timeout_ns);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQ = sbase + C::kOffA;
      const uint32_t sdO = sbase + C::kOffB;
      bool ok = wait_bar(&bars->res_full, 0, ctl, kCode);
      for (int n = 0; ok && n < nblk; ++n) {
        const int st = n & 1;
        const uint32_t sK = sbase + C::kOffX + st * C::kTileBytes;
        const uint32_t sV = sbase + C::kOffY + st * C::kTileBytes;
        if (!(ok = wait_bar(&bars->x_full[st], (n >> 1) & 1, ctl, kCode))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kTmS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->s_full);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO V^T
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kTmDP, sdesc_sw128(sdO + off, 16, 1024), sdesc_sw128(sV + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->dp_full);
        if (!(ok = wait_bar(&bars->ds_full, n & 1, ctl, kCode))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)  // dQ += dS K   (K = key rows)
          mma_ts(tmem + C::kTmAcc, tmem + C::kTmS + packed_slice_col(kk),
                 sdesc_sw128(sK + kk * 2048, C::kChunkBytes, 1024), idesc_acc, (n > 0 || kk > 0));
        mma_commit(&bars->x_empty[st]);
      }
      if (ok) mma_commit(&bars->acc_full);
      mma_commit(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int irow = quarter * 32 + lane;
    const int i = qb * kBM + irow;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    float lse2 = 0.f, delta = 0.f;
    if (i < s.T) {
      const size_t idx = (static_cast<size_t>(b) * s.H + h) * s.T + i;
      lse2 = p.LSE[idx] * kLog2e;
      delta = p.Delta[idx];
    }
    bool ok = true;
    for (int n = 0; n < nblk; ++n) {
      const int kb = kb_lo + n;
      if (!(ok = warp_wait(&bars->s_full, n & 1, ctl, kCode))) break;
      tc_fence_after();
      float pv[64];
      load_half_row(tmem + lane_addr + C::kTmS + half * 64, pv);
      const bool need_mask = block_needs_mask(s.T, kBM, kBN, s.causal, s.window, qb, kb);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float e = ex2(fmaf(pv[c], sl2, -lse2));
        if (need_mask && masked(s.T, s.causal, s.window, i, kb * kBN + half * 64 + c)) e = 0.f;
        pv[c] = e;
      }
      if (!(ok = warp_wait(&bars->dp_full, n & 1, ctl, kCode))) break;
      tc_fence_after();
      float dp[64];
      load_half_row(tmem + lane_addr + C::kTmDP + half * 64, dp);
#pragma unroll
      for (int c = 0; c < 64; ++c) dp[c] = pv[c] * (dp[c] - delta);
      store_half_row_bf16(tmem + lane_addr + C::kTmS + half * 64, dp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    if (ok) ok = warp_wait(&bars->acc_full, 0, ctl, kCode);
    if (ok) {
      tc_fence_after();
      const size_t rowoff = ((static_cast<size_t>(b) * s.T + i) * s.H + h) * D + half * (D / 2);
      store_acc_row(tmem + lane_addr + C::kTmAcc + half * (D / 2), D / 2, p.s.scale,
                    static_cast<__nv_bfloat16*>(p.dQ) + rowoff, i < s.T);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_dkdv_d(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkdv_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(ceil_div(p.s.T, kBN), p.s.HKV, p.s.B);
  fa_bwd_dkdv_bf16_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tm.q, tm.k, tm.v, tm.dO, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_d(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_dq_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(ceil_div(p.s.T, kBM), p.s.H, p.s.B);
  fa_bwd_dq_bf16_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tm.q, tm.k, tm.v, tm.dO, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  if (p.s.D == 64) return launch_dkdv_d<64>(tm, p, stream);
  if (p.s.D == 128) return launch_dkdv_d<128>(tm, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  if (p.s.D == 64) return launch_dq_d<64>(tm, p, stream);
  if (p.s.D == 128) return launch_dq_d<128>(tm, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
