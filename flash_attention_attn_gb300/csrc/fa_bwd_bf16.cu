// fa_bwd_bf16.cu -- attention backward for sm_103a (tcgen05 + TMA).
//
// Two kernels, each recomputing P block by block from the forward's LSE.
// Both are persistent (at most one CTA per SM, units of work handed out
// longest first, fa_sched.cuh):
//
// dK/dV: a unit is (b, kv head g, 128-row KV block).  K and V stay in
//   shared memory and dK, dV in TMEM for the whole unit while it visits
//   every query head of the group and every 128-row query block that sees the
//   KV block.  Accumulation is private to the unit: no atomics.
//     S^T  = K Q^T          (TMEM, KV rows on lanes)
//     dP^T = V dO^T
//     P^T  = 2^(S^T*scale*log2e - LSE*log2e), masked           -> bf16, TMEM
//     dS^T = P^T (dP^T - Delta)                                -> bf16, TMEM
//     dV  += P^T dO ;  dK += dS^T Q   (A operands from TMEM)
//   and at the end dK *= scale.  (forge flash_attention.metal,
//   flash_attn_bwd_dv / flash_attn_bwd_dk: one owner per key row summing over
//   the group's query heads; teeny-kernels flash_attn2.rs,
//   flash_attention2_backward_dkv: no atomics are needed.)
//
// dQ: a unit is (b, h, 128-row query block); it loops over the visible
//   128-row KV blocks in a fixed order, so the result is bitwise reproducible.
//     S = Q K^T ; dP = dO V^T ; dS = P (dP - Delta) -> bf16, TMEM ; dQ += dS K
//   and at the end dQ *= scale.  (forge flash_attention.metal,
//   flash_attn_bwd_dq; teeny-kernels flash_attention2_backward_dq.)
//
// Both kernels use 128 x 128 score tiles, so every MMA is [128 x 128 x 16] or
// wider: a tcgen05 MMA with N = 64 was measured on GB300 at 48 cycles
// against 64 for N = 128 (2/3 of the rate).  TMEM holds the fp32 score and
// dP tiles, the bf16 P and dS written back over them (the A operands of the
// accumulator MMAs) and the accumulators.  The per-row LSE and Delta of each
// streamed query block travel with its shared-memory stage (the producer
// warp loads them next to the TMA copies).
//
// Warp roles in both kernels: warps 0-7 compute (warp w owns TMEM lanes
// 32*(w%4).. and the 64-column half w/4 of each 128-column tile), warp 8 TMA
// producer, warp 9 MMA issuer and TMEM owner.  Each half writes its bf16
// results back into the first 32 columns of the 64 it read, so no half
// overwrites data the other still has to load.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kCompute = 256;
constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRowBytes = 128;  // one 64-element bf16 row of a swizzled chunk

__device__ __forceinline__ void reg_tie(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Two 32-column TMEM loads of this thread's lane, waited for together.
__device__ __forceinline__ void load_two_cols32(uint32_t a0, uint32_t a1, float (&v0)[32], float (&v1)[32]) {
  uint32_t r0[32], r1[32];
  tmem_ld32(a0, r0);
  tmem_ld32(a1, r1);
  tmem_ld_wait(r0);
  reg_tie(r1);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    v0[c] = __uint_as_float(r0[c]);
    v1[c] = __uint_as_float(r1[c]);
  }
}

// Write `ncols` fp32 TMEM columns of this thread's lane, times `mul`, as bf16
// to global memory at dst (16-byte aligned, ncols a multiple of 32).
// ncols accumulator columns of this thread's lane, scaled, as 16-bit values;
// only the first nvalid columns are stored (a head dim below the kernel's).
// st32: dst is 32-byte aligned and nvalid a multiple of 16, so the row
// leaves in whole 32-byte sectors.
template <bool F16>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, int ncols, int nvalid, float mul, uint16_t* dst,
                                              bool valid, bool st32) {
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + c, r);
    tmem_ld_wait(r);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack2<F16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (valid) {
      if (st32) {
#pragma unroll
        for (int v = 0; v < 2; ++v)
          if (c + v * 16 < nvalid) st_global_v8(dst + c + v * 16, pk + 8 * v);
      } else {
        uint4* d = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          if (c + v * 8 < nvalid) d[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
  }
}

struct BwdBars {
  uint64_t res_full;
  uint64_t res_empty;  // the unit's MMAs are done with the resident tiles
  uint64_t x_full[kStages];   // streamed stage loaded: Q (and dO, unless split) in dK/dV, K in dQ
  uint64_t x_empty[kStages];  // streamed stage free
  uint64_t v_full[kStages];   // second ring, stage loaded: dO in dK/dV (split rings), V in dQ
  uint64_t v_empty[kStages];  // second ring, stage free
  uint64_t s_full[2];
  uint64_t dp_full[2];
  uint64_t p_full[2];   // P written back (256 compute threads)
  uint64_t ds_full[2];  // dS (and P) written back (256 compute threads)
  uint64_t acc_full;
  uint64_t drain;
  SchedRing sched;  // units handed from the producer to the other roles
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(BwdBars) <= 512, "backward barriers exceed their shared-memory slot");

__device__ __forceinline__ void init_bars(BwdBars* bars, uint32_t x_full_count, uint32_t v_full_count,
                                          uint32_t v_empty_count) {
  mbar_init(&bars->res_full, 1);
  mbar_init(&bars->res_empty, 1);
  for (int i = 0; i < kStages; ++i) {
    mbar_init(&bars->x_full[i], x_full_count);
    mbar_init(&bars->x_empty[i], 1);
    mbar_init(&bars->v_full[i], v_full_count);
    mbar_init(&bars->v_empty[i], v_empty_count);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&bars->s_full[i], 1);
    mbar_init(&bars->dp_full[i], 1);
    mbar_init(&bars->p_full[i], kCompute / 32);  // one arrival per compute warp
    mbar_init(&bars->ds_full[i], kCompute / 32);
  }
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->drain, 1);
  sched_init(&bars->sched, 9);  // consumers: eight compute warps and the MMA warp
  bars->abort = 0;
  fence_mbar_init();
}

// The D/16 MMAs of one [128 x N] product, A and B both K-major in shared
// memory (A in a_chunk-byte chunks, B in b_chunk-byte chunks).  Descriptors
// are built once and stepped by adding (bytes >> 4) to the start address.
template <int D>
__device__ __forceinline__ void issue_kk(uint32_t d_tmem, uint32_t a_smem, int a_chunk, uint32_t b_smem, int b_chunk,
                                         uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(a_smem, 16, 1024);
  const uint64_t b0 = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t ao = (kk >> 2) * a_chunk + (kk & 3) * 32;
    const uint32_t bo = (kk >> 2) * b_chunk + (kk & 3) * 32;
    mma_ss_e(d_tmem, a0 + (ao >> 4), b0 + (bo >> 4), idesc, kk > 0 ? 1u : 0u);
  }
}

// TMEM column of 16-element slice kk (0..7) of a 128-element bf16 operand row
// that the two compute halves packed: half h writes elements [64h, 64h + 64)
// into columns [64h, 64h + 32).
__device__ __forceinline__ uint32_t packed_slice_col128(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// ============================================================== dK / dV

// dK/dV tiles: 128 key rows per unit (K, V resident), 128-row query blocks
// streamed, so every MMA runs at full rate (N = 128).  TMEM: S^T (128
// columns), dP^T (128), dV (D), dK (D): at D = 128 there is no room for a
// second score buffer, so the compute warps work in two passes per block
// (P^T from S^T, then dS^T from dP^T) and the MMA warp queues
//   dV(n) S^T(n+1) dK(n) dP^T(n+1) ...
// so that each pass overlaps the MMAs of the other buffer.
// At D = 128 the Q and dO blocks stream through rings of their own (kSplit):
// a dO stage is free once dV(n) and the dS pass that reads its Delta rows
// are done, a Q stage only after dK(n), and the Q ring has three stages, the
// dO ring two.  A clock64 trace of one CTA on GB300 showed S^T(n+1) waiting
// for its Q block with a shared two-stage ring (the block could only start
// loading after dK(n-1)); the split rings took the long causal workload's
// dK/dV 4 % faster.  They fill the 227 KB of shared memory exactly, so that
// layout needs the dynamic shared memory to start 1024-byte aligned, which
// the kernel checks.  At D = 64 a shared four-stage ring has room to spare
// and one barrier per stage costs less.
template <int D>
struct DkdvTiles {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunk = 128 * kRowBytes;  // [128][64] bf16 = 16 KB
  static constexpr int kTile = kChunks * kChunk;
  static constexpr bool kSplit = (D == 128);
  static constexpr int kQStages = (D == 64) ? 4 : 3;
  static constexpr int kOStages = (D == 64) ? 4 : 2;  // equal to kQStages when the rings are shared
  static constexpr int kOffRes0 = 0;                            // K
  static constexpr int kOffRes1 = kTile;                        // V
  static constexpr int kOffX = 2 * kTile;                       // Q stages
  static constexpr int kOffY = kOffX + kQStages * kTile;        // dO stages
  static constexpr int kOffLse = kOffY + kOStages * kTile;      // [Q stage][-LSE*log2e of 128 rows]
  static constexpr int kOffDel = kOffLse + kQStages * 128 * 4;  // [dO stage][Delta of 128 rows]
  static constexpr int kOffBar = kOffDel + kOStages * 128 * 4;
  static constexpr int kSlack = kSplit ? 0 : 1024;              // room to align the base (none when split)
  static constexpr int kSmemBytes = kOffBar + 512 + kSlack;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmS = 0;     // S^T, then P^T (bf16)
  static constexpr uint32_t kTmDP = 128;  // dP^T, then dS^T (bf16)
  static constexpr uint32_t kTmDV = 256;
  static constexpr uint32_t kTmDK = 256 + D;
  static_assert(kSplit || kQStages == kOStages, "a shared ring has one stage count");
};
static_assert(DkdvTiles<128>::kSmemBytes <= 232448, "dK/dV tiles exceed 227 KB of shared memory");

// Work units of the dK/dV kernel: (KV block kb, KV head g, batch b), numbered
// with kb fastest, ascending (under causal masking the first key blocks are
// seen by the most query blocks: longest first), then g, then b, so that the
// units in flight at any time share a KV head and re-read the same Q and dO
// blocks from L2.
__host__ __device__ __forceinline__ int dkdv_units(const Shape& s) { return ceil_div(s.Tk, 128) * s.HKV * s.B; }

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                            const BwdParams p) {
  using C = DkdvTiles<D>;
  constexpr int BQ = 128;  // query rows per streamed block
  constexpr int BK = 128;  // key rows per unit
  // the dQ kernel that follows inside one backward call reads nothing this
  // kernel writes: let its CTAs take the SMs this grid leaves idle
  grid_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::kSlack)) {
    // the layout does not fit: report it (FA_DEVERR_LAYOUT) and do nothing
    if (threadIdx.x == 0) {
      atomicOr(p.err, 8u);
      sched_exit(p.sched);
    }
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = smem_u32(smem);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  float* slse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sdel = reinterpret_cast<float*>(smem + C::kOffDel);
  // the barriers that guard a dO stage: the second ring's, or the Q stage's
  // own when the rings are shared
  uint64_t* const do_full = C::kSplit ? bars->v_full : bars->x_full;

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rep = s.H / s.HKV;
  const int nunits = dkdv_units(s);
  const int cta = static_cast<int>(blockIdx.x);
  // unit u -> (kb, g, b) and the query blocks [qlo, qlo + nqb) that see kb;
  // niter = rep * nqb (head r, query block) pairs, r outer
  struct Unit {
    int kb, g, b, qlo, nqb, niter;
  };
  auto unit = [&](int u) {
    Unit w;
    const int nkb = ceil_div(s.Tk, BK);
    w.kb = u % nkb;
    const int r = u / nkb;
    w.g = r % s.HKV;
    w.b = r / s.HKV;
    int qhi;
    q_range_for_kv(s.T, s.Tk, BQ, BK, s.causal, s.window, w.kb, w.qlo, qhi);
    w.nqb = qhi - w.qlo + 1;
    w.niter = rep * w.nqb;
    return w;
  };

  // Q (and dO) stages: the elected lane's expect-tx plus the 32 lanes that
  // write the stage's LSE and Delta rows; a split dO stage is freed by the
  // dV MMAs' commit and by the eight compute warps once they have read its
  // Delta rows
  if (threadIdx.x == 0) init_bars(bars, 1 + 32, 1 + 32, 1 + kCompute / 32);
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
    }
    int xc = 0, uc = 0;  // streamed stages and units issued by this CTA
    bool ok = true;
    int u = cta;  // the CTA's first unit; later ones are claimed from the counter
    for (int seq = 0; ok && !p.inject_stall; ++seq) {
      if (!(ok = sched_publish(&bars->sched, seq, u, ctl, kCode))) break;
      if (u >= nunits) break;  // the end marker has been handed on
      const Unit w = unit(u);
      // K and V of this unit once the previous unit's MMAs are done with them
      if (uc > 0 && !(ok = warp_wait(&bars->res_empty, (uc - 1) & 1, ctl, kCode))) break;
      mbar_arrive_expect_tx_e(&bars->res_full, 2 * C::kTile);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d_e(&tmK, &bars->res_full, smem + C::kOffRes0 + c * C::kChunk, c * 64, w.g, w.kb * BK, w.b);
        tma_load_4d_e(&tmV, &bars->res_full, smem + C::kOffRes1 + c * C::kChunk, c * 64, w.g, w.kb * BK, w.b);
      }
      ++uc;
      // -LSE (pre-scaled to base 2) and Delta of one block's 128 query rows,
      // four per lane; read one block ahead so that their latency overlaps the
      // waits for the stages
      float l2[4], dl[4];
      auto load_rows = [&](int n) {
        const int h = w.g * rep + n / w.nqb;
        const int qb = w.qlo + n % w.nqb;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int i = qb * BQ + lane + 32 * q4;
          l2[q4] = 0.f;
          dl[q4] = 0.f;
          if (i < s.T) {
            const size_t idx = (static_cast<size_t>(w.b) * s.H + h) * s.T + i;
            l2[q4] = -p.LSE[idx] * kLog2e;
            dl[q4] = p.Delta[idx];
          }
        }
      };
      if (w.niter > 0) load_rows(0);
      for (int n = 0; n < w.niter; ++n) {
        const int h = w.g * rep + n / w.nqb;
        const int qb = w.qlo + n % w.nqb;
        // Q block and its -LSE*log2e rows (one elected lane arms and copies)
        const int sq = xc % C::kQStages;
        if (xc >= C::kQStages && !(ok = warp_wait(&bars->x_empty[sq], ((xc / C::kQStages) - 1) & 1, ctl, kCode)))
          break;
        mbar_arrive_expect_tx_e(&bars->x_full[sq], (C::kSplit ? 1 : 2) * C::kTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmQ, &bars->x_full[sq], smem + C::kOffX + sq * C::kTile + c * C::kChunk, c * 64, h,
                        qb * BQ, w.b);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) slse[sq * 128 + lane + 32 * q4] = l2[q4];
        // dO block and its Delta rows: in the Q block's stage, or in a stage
        // of the dO ring
        const int sd = xc % C::kOStages;
        if (C::kSplit) {
          mbar_arrive(&bars->x_full[sq]);
          if (xc >= C::kOStages && !(ok = warp_wait(&bars->v_empty[sd], ((xc / C::kOStages) - 1) & 1, ctl, kCode)))
            break;
          mbar_arrive_expect_tx_e(&bars->v_full[sd], C::kTile);
        }
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmdO, &do_full[sd], smem + C::kOffY + sd * C::kTile + c * C::kChunk, c * 64, h, qb * BQ,
                        w.b);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) sdel[sd * 128 + lane + 32 * q4] = dl[q4];
        mbar_arrive(&do_full[sd]);
        ++xc;
        if (n + 1 < w.niter) load_rows(n + 1);
      }
      // claim the next unit only now, near the end of this one, so that the
      // CTAs that finish first take the next longest units
      int claimed = 0;
      if (lane == 0) claimed = sched_claim(p.sched);
      u = __shfl_sync(0xffffffffu, claimed, 0);
    }
    if (lane == 0 && bars->abort) {
      if (uc > 0) drain_bar(&bars->res_full, (uc - 1) & 1, p.timeout_ns);
      for (int n = imax(0, xc - C::kQStages); n < xc; ++n)
        drain_bar(&bars->x_full[n % C::kQStages], (n / C::kQStages) & 1, p.timeout_ns);
      if (C::kSplit)
        for (int n = imax(0, xc - C::kOStages); n < xc; ++n)
          drain_bar(&bars->v_full[n % C::kOStages], (n / C::kOStages) & 1, p.timeout_ns);
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    {  // the whole warp runs the loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_f32acc<F16>(128, BQ, false, false);  // K-major x K-major, N = 128
      constexpr uint32_t idesc_acc = idesc_f32acc<F16>(128, D, false, true);  // TMEM A x MN-major B, N = D
      const uint32_t sK = sbase + C::kOffRes0;
      const uint32_t sV = sbase + C::kOffRes1;
      int xc = 0, uc = 0;  // streamed stages and units consumed (x_full, p/ds phases run with xc)
      auto q_ready = [&](int xg) -> bool {  // Q block xg (and its dO, when the rings are shared) loaded
        const int sq = xg % C::kQStages;
        if (!warp_wait(&bars->x_full[sq], (xg / C::kQStages) & 1, ctl, kCode)) return false;
        tc_fence_after();
        return true;
      };
      auto issue_s = [&](int xg) {  // S^T = K Q^T of Q block xg (already waited for)
        const int sq = xg % C::kQStages;
        issue_kk<D>(tmem + C::kTmS, sK, C::kChunk, sbase + C::kOffX + sq * C::kTile, C::kChunk, idesc_s);
        mma_commit_e(&bars->s_full[0]);
      };
      auto issue_dp = [&](int xg) -> bool {  // dP^T = V dO^T of dO block xg
        const int sd = xg % C::kOStages;
        if (C::kSplit) {
          if (!warp_wait(&bars->v_full[sd], (xg / C::kOStages) & 1, ctl, kCode)) return false;
          tc_fence_after();
        }
        issue_kk<D>(tmem + C::kTmDP, sV, C::kChunk, sbase + C::kOffY + sd * C::kTile, C::kChunk, idesc_s);
        mma_commit_e(&bars->dp_full[0]);
        return true;
      };
      // acc (+)= A[TMEM, 128 packed query rows] x B[128 query rows][D] (MN-major)
      auto issue_acc128 = [&](uint32_t acc, uint32_t a_tmem, uint32_t b_smem, bool accumulate) {
        const uint64_t b0 = sdesc_sw128(b_smem, C::kChunk, 1024);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts_e(acc, a_tmem + packed_slice_col128(kk), b0 + ((kk * 16 * kRowBytes) >> 4), idesc_acc,
                   (accumulate || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int u = sched_next(&bars->sched, seq, ctl, kCode);
        if (u < 0) {
          ok = false;
          break;
        }
        if (u >= nunits) break;
        const Unit w = unit(u);
        if (!(ok = warp_wait(&bars->res_full, uc & 1, ctl, kCode))) break;
        tc_fence_after();
        ++uc;
        if (w.niter > 0) {
          if (!(ok = q_ready(xc))) break;
          issue_s(xc);
          if (!(ok = issue_dp(xc))) break;
        }
        if (w.niter <= 1) mma_commit_e(&bars->res_empty);  // every MMA reading K and V is issued
        for (int n = 0; ok && n < w.niter; ++n) {
          const int xg = xc + n;
          const int sq = xg % C::kQStages;
          const int sd = xg % C::kOStages;
          // the next Q block's wait while the compute warps still form P^T_n,
          // so that S^T_{n+1} follows the dV MMAs without a gap (the deeper
          // Q ring, or the shared four-stage one, has it loaded by then)
          if (n + 1 < w.niter && !(ok = q_ready(xg + 1))) break;
          if (!(ok = warp_wait(&bars->p_full[0], xg & 1, ctl, kCode))) break;
          tc_fence_after();
          issue_acc128(tmem + C::kTmDV, tmem + C::kTmS, sbase + C::kOffY + sd * C::kTile, n > 0);  // dV += P^T dO
          if (C::kSplit) mma_commit_e(&bars->v_empty[sd]);  // the dO stage, once its Delta rows are read too
          if (n + 1 < w.niter) issue_s(xg + 1);  // P^T_n is read by the dV MMAs queued above
          if (!(ok = warp_wait(&bars->ds_full[0], xg & 1, ctl, kCode))) break;
          tc_fence_after();
          issue_acc128(tmem + C::kTmDK, tmem + C::kTmDP, sbase + C::kOffX + sq * C::kTile, n > 0);  // dK += dS^T Q
          mma_commit_e(&bars->x_empty[sq]);
          if (n + 1 < w.niter) {
            if (!(ok = issue_dp(xg + 1))) break;  // dS^T_n is read by the dK MMAs queued above
            if (n + 2 == w.niter) mma_commit_e(&bars->res_empty);  // the unit's last MMAs reading K and V
          }
        }
        if (!ok) break;
        mma_commit_e(&bars->acc_full);
        xc += w.niter;
      }
      mma_commit_e(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- compute
    const int quarter = warp & 3;          // TMEM lane quarter
    const int half = warp >> 2;            // 64-column half of each 128-column tile
    const int jrow = quarter * 32 + lane;  // key row within the block (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + C::kTmS + half * 64;
    const uint32_t dp_addr = tmem + lane_addr + C::kTmDP + half * 64;
    const float sl2 = p.scale_log2;
    int xc = 0, uc = 0;
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int u = sched_next(&bars->sched, seq, ctl, kCode);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= nunits) break;
      const Unit w = unit(u);
      const int j = w.kb * BK + jrow;
      for (int n = 0; ok && n < w.niter; ++n) {
        const int xg = xc + n;
        const int sq = xg % C::kQStages;
        const int sd = xg % C::kOStages;
        const int qb = w.qlo + n % w.nqb;
        // pass 1: P^T = 2^(S^T*scale*log2e - LSE*log2e), masked -> bf16 over S^T.
        // The stage's LSE rows land long before the scores: wait for them
        // first, so that this wait stays off the chain from S^T to the dV MMAs.
        if (!(ok = warp_wait(&bars->x_full[sq], (xg / C::kQStages) & 1, ctl, kCode))) break;  // LSE rows visible
        if (!(ok = warp_wait(&bars->s_full[0], xg & 1, ctl, kCode))) break;
        tc_fence_after();
        const bool need_mask = block_needs_mask(s.T, s.Tk, BQ, BK, s.causal, s.window, qb, w.kb);
        float pv[64];
        {
          float lo[32], hi[32];
          load_two_cols32(s_addr, s_addr + 32, lo, hi);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            pv[c] = lo[c];
            pv[32 + c] = hi[c];
          }
        }
        const float4* lse4 = reinterpret_cast<const float4*>(slse + sq * 128 + half * 64);  // -LSE*log2e per query
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l = lse4[c4];
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 0], pv[4 * c4 + 1]), sl2x2, f2_pack(l.x, l.y)), x0, x1);
          f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]), sl2x2, f2_pack(l.z, l.w)), x2, x3);
          pv[4 * c4 + 0] = ex2(x0);
          pv[4 * c4 + 1] = ex2(x1);
          pv[4 * c4 + 2] = ex2(x2);
          pv[4 * c4 + 3] = ex2(x3);
        }
        if (need_mask) {
          // the visibility rule element by element (the [lo, hi] range form
          // the other kernels use measured 3 % slower here on the long causal
          // workload: it changed this kernel's register allocation)
          const int i0 = qb * BQ + half * 64;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int i = i0 + c;
            const bool hide = i >= s.T || j >= s.Tk || (s.causal && j > i) || (s.window > 0 && i - j >= s.window);
            pv[c] = hide ? 0.f : pv[c];
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = pack2<F16>(pv[2 * e], pv[2 * e + 1]);
          tmem_st32(s_addr, pk);  // 64 packed values into the first 32 columns of this half
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->p_full[0]);
        // pass 2: dS^T = P^T (dP^T - Delta) -> bf16 over dP^T (the Delta rows
        // came with the dO block, before dP^T)
        if (C::kSplit && !(ok = warp_wait(&bars->v_full[sd], (xg / C::kOStages) & 1, ctl, kCode))) break;
        if (!(ok = warp_wait(&bars->dp_full[0], xg & 1, ctl, kCode))) break;
        tc_fence_after();
        float dlo[32], dhi[32];
        load_two_cols32(dp_addr, dp_addr + 32, dlo, dhi);
        const float4* del4 = reinterpret_cast<const float4*>(sdel + sd * 128 + half * 64);
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d = del4[c4];
          const float4 e = del4[8 + c4];
          // dS = P (dP - Delta), paired
          f2_unpack(f2_mul(f2_pack(pv[4 * c4 + 0], pv[4 * c4 + 1]),
                           f2_sub(f2_pack(dlo[4 * c4 + 0], dlo[4 * c4 + 1]), f2_pack(d.x, d.y))),
                    dlo[4 * c4 + 0], dlo[4 * c4 + 1]);
          f2_unpack(f2_mul(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]),
                           f2_sub(f2_pack(dlo[4 * c4 + 2], dlo[4 * c4 + 3]), f2_pack(d.z, d.w))),
                    dlo[4 * c4 + 2], dlo[4 * c4 + 3]);
          f2_unpack(f2_mul(f2_pack(pv[32 + 4 * c4 + 0], pv[32 + 4 * c4 + 1]),
                           f2_sub(f2_pack(dhi[4 * c4 + 0], dhi[4 * c4 + 1]), f2_pack(e.x, e.y))),
                    dhi[4 * c4 + 0], dhi[4 * c4 + 1]);
          f2_unpack(f2_mul(f2_pack(pv[32 + 4 * c4 + 2], pv[32 + 4 * c4 + 3]),
                           f2_sub(f2_pack(dhi[4 * c4 + 2], dhi[4 * c4 + 3]), f2_pack(e.z, e.w))),
                    dhi[4 * c4 + 2], dhi[4 * c4 + 3]);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pk[e] = pack2<F16>(dlo[2 * e], dlo[2 * e + 1]);
          pk[16 + e] = pack2<F16>(dhi[2 * e], dhi[2 * e + 1]);
        }
        tmem_st32(dp_addr, pk);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->ds_full[0]);
        if (C::kSplit) warp_arrive(&bars->v_empty[sd]);  // its Delta rows are read
      }
      if (!ok) break;
      xc += w.niter;
      if (!(ok = warp_wait(&bars->acc_full, uc & 1, ctl, kCode))) break;
      ++uc;
      tc_fence_after();
      const size_t rowoff = ((static_cast<size_t>(w.b) * s.Tk + j) * s.HKV + w.g) * s.D + half * (D / 2);
      const int nvalid = s.D - half * (D / 2);  // columns of this half inside the head dim
      const bool st32 =
          ((reinterpret_cast<uintptr_t>(p.dK) | reinterpret_cast<uintptr_t>(p.dV)) & 31) == 0 && (s.D & 15) == 0;
      store_acc_row<F16>(tmem + lane_addr + C::kTmDV + half * (D / 2), D / 2, nvalid, 1.f,
                         static_cast<uint16_t*>(p.dV) + rowoff, j < s.Tk, st32);
      store_acc_row<F16>(tmem + lane_addr + C::kTmDK + half * (D / 2), D / 2, nvalid, s.scale,
                         static_cast<uint16_t*>(p.dK) + rowoff, j < s.Tk, st32);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) sched_exit(p.sched);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================== dQ

// dQ tiles: 128-row query tile (Q, dO resident), 128-row K/V blocks streamed,
// so every score MMA is [128 x 128 x 16] (a 64-wide one runs at 2/3 rate).
// TMEM: S double-buffered (2 x 128 columns), dP single (128), dQ (D).  dP of
// block n+1 is computed as soon as the compute warps have released block n.
template <int D>
struct DqTiles {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunk = 128 * kRowBytes;  // [128][64] bf16 = 16 KB
  static constexpr int kTile = kChunks * kChunk;
  // K is held from its S MMA to its dQ MMA, V only until its dP MMA: K gets
  // the deeper ring (3 + 2 stages = 224 KB of tiles at D = 128)
  static constexpr int kKStages = (D == 64) ? 4 : 3;
  static constexpr int kVStages = (D == 64) ? 4 : 2;
  static constexpr int kOffRes0 = 0;               // Q
  static constexpr int kOffRes1 = kTile;           // dO
  static constexpr int kOffK = 2 * kTile;          // K stages
  static constexpr int kOffV = kOffK + kKStages * kTile;  // V stages
  static constexpr int kOffBar = kOffV + kVStages * kTile;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmS = 0;     // 2 x 128 columns
  static constexpr uint32_t kTmDP = 256;  // 128 columns
  static constexpr uint32_t kTmDQ = 384;  // D columns
};

// Work units of the dQ kernel: (query block qb, head h, batch b), numbered
// with qb fastest from the end of the sequence (longest causal work first),
// then h, then b, so that the units in flight at any time share a KV head.
__host__ __device__ __forceinline__ int dq_units(const Shape& s) { return ceil_div(s.T, 128) * s.H * s.B; }

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                          const BwdParams p) {
  using C = DqTiles<D>;
  constexpr int BQ = 128;  // query rows per unit
  constexpr int BK = 128;  // key rows per streamed block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nq = ceil_div(s.T, BQ);
  const int nunits = dq_units(s);
  const int cta = static_cast<int>(blockIdx.x);
  // unit u -> (qb, h, b, g) and the visible KV blocks [kb_lo, kb_lo + nblk)
  struct Unit {
    int qb, h, b, g, kb_lo, nblk;
  };
  auto unit = [&](int u) {
    Unit w;
    const int x = u % nq;
    const int r = u / nq;
    w.qb = nq - 1 - x;
    w.h = r % s.H;
    w.b = r / s.H;
    w.g = w.h / (s.H / s.HKV);
    int kb_hi;
    kv_range_for_q(s.T, s.Tk, BQ, BK, s.causal, s.window, w.qb, w.kb_lo, kb_hi);
    w.nblk = kb_hi - w.kb_lo + 1;
    return w;
  };

  if (threadIdx.x == 0) init_bars(bars, 1, 1, 1);
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
    // the whole warp streams K and V through separate rings (a V stage is
    // freed after its dP MMA, a K stage only after its dQ MMA), in the order
    // the MMAs need them; one elected lane arms each barrier and issues each copy
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
    }
    int kc = 0, vc = 0, uc = 0;  // K blocks, V blocks and units issued by this CTA
    bool ok = true;
    int u = cta;  // the CTA's first unit; later ones are claimed from the counter
    for (int seq = 0; ok && !p.inject_stall; ++seq) {
      if (!(ok = sched_publish(&bars->sched, seq, u, ctl, kCode))) break;
      if (u >= nunits) break;  // the end marker has been handed on
      const Unit w = unit(u);
      // Q and dO of this unit once the previous unit's MMAs are done with them
      if (uc > 0 && !(ok = warp_wait(&bars->res_empty, (uc - 1) & 1, ctl, kCode))) break;
      mbar_arrive_expect_tx_e(&bars->res_full, 2 * C::kTile);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d_e(&tmQ, &bars->res_full, smem + C::kOffRes0 + c * C::kChunk, c * 64, w.h, w.qb * BQ, w.b);
        tma_load_4d_e(&tmdO, &bars->res_full, smem + C::kOffRes1 + c * C::kChunk, c * 64, w.h, w.qb * BQ, w.b);
      }
      ++uc;
      for (int n = 0; n < w.nblk; ++n) {
        const int sk = kc % C::kKStages;
        if (kc >= C::kKStages && !(ok = warp_wait(&bars->x_empty[sk], ((kc / C::kKStages) - 1) & 1, ctl, kCode)))
          break;
        mbar_arrive_expect_tx_e(&bars->x_full[sk], C::kTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmK, &bars->x_full[sk], smem + C::kOffK + sk * C::kTile + c * C::kChunk, c * 64, w.g,
                        (w.kb_lo + n) * BK, w.b);
        ++kc;
        const int sv = vc % C::kVStages;
        if (vc >= C::kVStages && !(ok = warp_wait(&bars->v_empty[sv], ((vc / C::kVStages) - 1) & 1, ctl, kCode)))
          break;
        mbar_arrive_expect_tx_e(&bars->v_full[sv], C::kTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmV, &bars->v_full[sv], smem + C::kOffV + sv * C::kTile + c * C::kChunk, c * 64, w.g,
                        (w.kb_lo + n) * BK, w.b);
        ++vc;
      }
      // claim the next unit only now, near the end of this one, so that the
      // CTAs that finish first take the next longest units
      int claimed = 0;
      if (lane == 0) claimed = sched_claim(p.sched);
      u = __shfl_sync(0xffffffffu, claimed, 0);
    }
    if (bars->abort) {
      if (uc > 0) drain_bar(&bars->res_full, (uc - 1) & 1, p.timeout_ns);
      for (int n = imax(0, kc - C::kKStages); n < kc; ++n)
        drain_bar(&bars->x_full[n % C::kKStages], (n / C::kKStages) & 1, p.timeout_ns);
      for (int n = imax(0, vc - C::kVStages); n < vc; ++n)
        drain_bar(&bars->v_full[n % C::kVStages], (n / C::kVStages) & 1, p.timeout_ns);
    }
  } else if (warp == 9) {
    {  // the whole warp runs the loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_f32acc<F16>(128, BK, false, false);  // K-major x K-major, N = 128
      constexpr uint32_t idesc_acc = idesc_f32acc<F16>(128, D, false, true);  // TMEM A x MN-major B, N = D
      const uint32_t sQ = sbase + C::kOffRes0;
      const uint32_t sdO = sbase + C::kOffRes1;
      // streamed blocks consumed by this CTA: block bg uses K stage
      // bg % kKStages, V stage bg % kVStages and S buffer bg & 1
      auto issue_s = [&](int bg) -> bool {  // S = Q K^T into buffer bg & 1
        const int st = bg % C::kKStages;
        if (!warp_wait(&bars->x_full[st], (bg / C::kKStages) & 1, ctl, kCode)) return false;
        tc_fence_after();
        issue_kk<D>(tmem + C::kTmS + (bg & 1) * 128, sQ, C::kChunk, sbase + C::kOffK + st * C::kTile, C::kChunk,
                    idesc_s);
        mma_commit_e(&bars->s_full[bg & 1]);
        return true;
      };
      auto v_ready = [&](int bg) -> bool {  // V block bg loaded
        const int st = bg % C::kVStages;
        if (!warp_wait(&bars->v_full[st], (bg / C::kVStages) & 1, ctl, kCode)) return false;
        tc_fence_after();
        return true;
      };
      auto issue_dp = [&](int bg) {  // dP = dO V^T (V already waited for); its V stage is free once this completes
        const int st = bg % C::kVStages;
        issue_kk<D>(tmem + C::kTmDP, sdO, C::kChunk, sbase + C::kOffV + st * C::kTile, C::kChunk, idesc_s);
        mma_commit_e(&bars->dp_full[0]);
        mma_commit_e(&bars->v_empty[st]);
      };
      int bc = 0, uc = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int u = sched_next(&bars->sched, seq, ctl, kCode);
        if (u < 0) {
          ok = false;
          break;
        }
        if (u >= nunits) break;
        const Unit w = unit(u);
        if (!(ok = warp_wait(&bars->res_full, uc & 1, ctl, kCode))) break;
        tc_fence_after();
        ++uc;
        if (w.nblk > 0) {
          if (!(ok = issue_s(bc))) break;
          if (!(ok = v_ready(bc))) break;
          issue_dp(bc);
        }
        if (w.nblk <= 1) mma_commit_e(&bars->res_empty);  // every MMA reading Q and dO is issued
        // queue order: S0 dP0 S1 | dP1 dQ0 S2 | dP2 dQ1 S3 ...
        for (int n = 0; ok && n < w.nblk; ++n) {
          const int bg = bc + n;
          if (n + 1 < w.nblk && !(ok = issue_s(bg + 1))) break;
          const int st = bg % C::kKStages;
          // the next V block's wait before the dS wait, so that dP_{n+1}
          // issues as soon as dS_n has been written
          if (n + 1 < w.nblk && !(ok = v_ready(bg + 1))) break;
          if (!(ok = warp_wait(&bars->ds_full[0], bg & 1, ctl, kCode))) break;
          tc_fence_after();
          if (n + 1 < w.nblk) {
            issue_dp(bg + 1);  // dP_n has been read: its columns are free
            if (n + 2 == w.nblk) mma_commit_e(&bars->res_empty);  // the unit's last MMAs reading Q and dO
          }
          // dQ += dS K   (K = the block's 128 key rows)
          const uint64_t b0 = sdesc_sw128(sbase + C::kOffK + st * C::kTile, C::kChunk, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ts_e(tmem + C::kTmDQ, tmem + C::kTmS + (bg & 1) * 128 + packed_slice_col128(kk),
                     b0 + ((kk * 16 * kRowBytes) >> 4), idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit_e(&bars->x_empty[st]);
        }
        if (!ok) break;
        mma_commit_e(&bars->acc_full);
        bc += w.nblk;
      }
      mma_commit_e(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    const int quarter = warp & 3;
    const int half = warp >> 2;  // 64-key half of each 128-key block
    const int irow = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    int bc = 0, uc = 0;
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int u = sched_next(&bars->sched, seq, ctl, kCode);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= nunits) break;
      const Unit w = unit(u);
      const int i = w.qb * BQ + irow;
      int vis_lo, vis_hi;  // keys row i sees
      visible_keys(s.T, s.Tk, s.causal, s.window, i, vis_lo, vis_hi);
      float lse2 = 0.f, delta = 0.f;
      if (i < s.T) {
        const size_t idx = (static_cast<size_t>(w.b) * s.H + w.h) * s.T + i;
        lse2 = p.LSE[idx] * kLog2e;
        delta = p.Delta[idx];
      }
      for (int n = 0; ok && n < w.nblk; ++n) {
        const int kb = w.kb_lo + n;
        const int bg = bc + n;
        const int bf = bg & 1;
        // pass 1 (overlaps the dP MMA of this block): P = 2^(S*scale*log2e - LSE*log2e), masked
        if (!(ok = warp_wait(&bars->s_full[bf], (bg >> 1) & 1, ctl, kCode))) break;
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_addr + C::kTmS + bf * 128 + half * 64;
        const uint32_t dp_addr = tmem + lane_addr + C::kTmDP + half * 64;
        float pv[64];
        {
          float lo[32], hi[32];
          load_two_cols32(s_addr, s_addr + 32, lo, hi);
          const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1, y0, y1;
            f2_unpack(f2_fma(f2_pack(lo[c], lo[c + 1]), sl2x2, nl2), x0, x1);
            f2_unpack(f2_fma(f2_pack(hi[c], hi[c + 1]), sl2x2, nl2), y0, y1);
            pv[c] = ex2(x0);
            pv[c + 1] = ex2(x1);
            pv[32 + c] = ex2(y0);
            pv[33 + c] = ex2(y1);
          }
        }
        if (block_needs_mask(s.T, s.Tk, BQ, BK, s.causal, s.window, w.qb, kb)) {
          // the keys this row sees, relative to the 64 columns
          const int a = vis_lo - (kb * BK + half * 64), z = vis_hi - (kb * BK + half * 64);
#pragma unroll
          for (int c = 0; c < 64; ++c) pv[c] = (c < a || c > z) ? 0.f : pv[c];
        }
        // pass 2: dS = P (dP - Delta) -> bf16 over the S columns this thread read
        if (!(ok = warp_wait(&bars->dp_full[0], bg & 1, ctl, kCode))) break;
        tc_fence_after();
        {
          float lo[32], hi[32];
          load_two_cols32(dp_addr, dp_addr + 32, lo, hi);
          uint32_t pk[32];
          const uint64_t dl2 = f2_pack(delta, delta);
#pragma unroll
          for (int e = 0; e < 16; ++e) {  // dS = P (dP - Delta), paired
            float a0, a1, b0, b1;
            f2_unpack(f2_mul(f2_pack(pv[2 * e], pv[2 * e + 1]), f2_sub(f2_pack(lo[2 * e], lo[2 * e + 1]), dl2)), a0,
                      a1);
            f2_unpack(f2_mul(f2_pack(pv[32 + 2 * e], pv[33 + 2 * e]), f2_sub(f2_pack(hi[2 * e], hi[2 * e + 1]), dl2)),
                      b0, b1);
            pk[e] = pack2<F16>(a0, a1);
            pk[16 + e] = pack2<F16>(b0, b1);
          }
          tmem_st32(s_addr, pk);  // dS of keys [64 half, 64 half + 64) -> columns [64 half, 64 half + 32)
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->ds_full[0]);
      }
      if (!ok) break;
      bc += w.nblk;
      if (!(ok = warp_wait(&bars->acc_full, uc & 1, ctl, kCode))) break;
      ++uc;
      tc_fence_after();
      const size_t rowoff = ((static_cast<size_t>(w.b) * s.T + i) * s.H + w.h) * s.D + half * (D / 2);
      const bool st32 = (reinterpret_cast<uintptr_t>(p.dQ) & 31) == 0 && (s.D & 15) == 0;
      store_acc_row<F16>(tmem + lane_addr + C::kTmDQ + half * (D / 2), D / 2, s.D - half * (D / 2), s.scale,
                         static_cast<uint16_t*>(p.dQ) + rowoff, i < s.T, st32);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) sched_exit(p.sched);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // launched as a dependent of the dK/dV kernel, this grid may not complete
  // before that one: work after the backward on the stream sees dK and dV
  if (threadIdx.x == 0) grid_dependency_wait();
}

template <int D, bool F16>
cudaError_t launch_dkdv_d(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  using C = DkdvTiles<D>;
  static std::atomic<unsigned long long> attr_set{0};
  const void* kfn = reinterpret_cast<const void*>(fa_bwd_dkdv_bf16_kernel<D, F16>);
  if (cudaError_t e = set_smem_once(kfn, C::kSmemBytes, attr_set); e != cudaSuccess) return e;
  const dim3 grid(imax(1, imin(p.ctas, dkdv_units(p.s))));
  fa_bwd_dkdv_bf16_kernel<D, F16><<<grid, kThreads, C::kSmemBytes, stream>>>(tm.q, tm.k, tm.v, tm.dO, p);
  return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_dq_d(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  using C = DqTiles<D>;
  static std::atomic<unsigned long long> attr_set{0};
  const void* kfn = reinterpret_cast<const void*>(fa_bwd_dq_bf16_kernel<D, F16>);
  if (cudaError_t e = set_smem_once(kfn, C::kSmemBytes, attr_set); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(imax(1, imin(p.ctas, dq_units(p.s))));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.after_dkdv ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fa_bwd_dq_bf16_kernel<D, F16>, tm.q, tm.k, tm.v, tm.dO, p);
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  if (p.s.D <= 64) return p.f16 ? launch_dkdv_d<64, true>(tm, p, stream) : launch_dkdv_d<64, false>(tm, p, stream);
  if (p.s.D <= 128) return p.f16 ? launch_dkdv_d<128, true>(tm, p, stream) : launch_dkdv_d<128, false>(tm, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream) {
  if (p.s.D <= 64) return p.f16 ? launch_dq_d<64, true>(tm, p, stream) : launch_dq_d<64, false>(tm, p, stream);
  if (p.s.D <= 128) return p.f16 ? launch_dq_d<128, true>(tm, p, stream) : launch_dq_d<128, false>(tm, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
