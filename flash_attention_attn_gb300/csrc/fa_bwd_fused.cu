// fa_bwd_fused.cu -- attention backward for head dims up to 64 under causal
// masking, without recomputing S and dP for dQ: one persistent kernel forms
// dK and dV (as the dK/dV kernel does) and, from the same dS tile, every dQ
// partial  dQ_i += dS_ij K_j, which it adds into an fp32 accumulator in a
// fixed order, so that the result is still bitwise reproducible.
//
// This follows the Graphcore flash_attention_qkv_packed.cpp backward
// (flashAttentionQKVPackedGrad): its loop over KV blocks writes dQ_i += dS K_j
// back in place, one KV block after the other, in the same pass that produces
// dK and dV.  Here the KV blocks of a query block are different work units,
// possibly on different SMs; the order is enforced by a turn counter per
// (batch, head, query block) in the workspace.
//
// Per streamed query block n of a unit (KV block kb, KV head g, batch b):
//   S^T = K Q^T, dP^T = V dO^T                          (TMEM)
//   P^T, dS^T from them (compute warps)                 -> bf16 in TMEM
//   dS (the same values) also into shared memory, laid out as the
//   MN-major A operand of  dQ_part = dS K  (M = 128 queries, N = 64, K = 128 keys)
//   dV += P^T dO ;  dK += dS^T Q ;  dQ_part = dS K      (tensor core)
//   dQ_part: TMEM -> registers -> shared memory (fp32), then the reducer warp
//   adds it into the fp32 accumulator tile of (b, h, query block) with a TMA
//   reduce-add (the first contribution stores instead), once every
//   contribution before it in the fixed order is in; the last one scales the
//   tile, rounds it to the element type and writes dQ.
//
// Fixed order of the contributions to query block qb: KV blocks kb_hi(qb),
// kb_hi - 1, ..., kb_lo(qb) (the diagonal block first).  Units are handed out
// with kb descending inside each (KV head, batch), and a unit visits its query
// blocks in ascending order, so the unit for kb + 1 reaches query block qb
// before the unit for kb does: a turn wait only waits when an earlier unit
// runs slower.  Every unit that a turn waits for was handed out earlier, so
// it is running on an SM of this launch (the launch is cooperative: all its
// CTAs are resident together) or already done; turn waits are bounded by the
// wait budget like every other wait.
//
// Warps: 0-7 compute (warp w: TMEM lanes 32*(w%4).., 64-column half w/4),
// 8 TMA producer, 9 MMA issuer and TMEM owner, 10 reducer.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kThreadsF = 352;
constexpr int kComputeF = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr int kRowB = 128;  // one 64-element 16-bit row of a swizzled chunk

struct FusedTiles {
  static constexpr int kChunk = 128 * kRowB;  // [128][64] 16-bit = 16 KB
  static constexpr int kStages = 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kChunk;
  static constexpr int kOffX = 2 * kChunk;                    // Q stages
  static constexpr int kOffY = kOffX + kStages * kChunk;      // dO stages
  static constexpr int kOffDS = kOffY + kStages * kChunk;     // dS: 2 chunks [128 keys][64 queries]
  static constexpr int kOffStg = kOffDS + 2 * kChunk;         // dQ partials: 2 buffers x 2 chunks [128 queries][32 fp32]
  static constexpr int kOffRows = kOffStg + 4 * kChunk;       // [stage][-LSE*log2e 128 | Delta 128]
  static constexpr int kOffBar = kOffRows + kStages * 256 * 4;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmS = 0;     // S^T, then P^T
  static constexpr uint32_t kTmDP = 128;  // dP^T, then dS^T
  static constexpr uint32_t kTmDV = 256;  // 64 columns
  static constexpr uint32_t kTmDK = 320;  // 64 columns
  static constexpr uint32_t kTmDQ = 384;  // 64 columns: the dQ partial
};

struct FusedBars {
  uint64_t res_full, res_empty;
  uint64_t x_full[FusedTiles::kStages];
  uint64_t x_empty[FusedTiles::kStages];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t acc_full;   // dK, dV of the unit complete
  uint64_t dq_full;    // the dQ partial of a block complete
  uint64_t stg_full[2];   // the compute warps have copied a partial to shared memory
  uint64_t stg_empty[2];  // the reducer has handed it to the TMA unit
  uint64_t drain;
  SchedRing sched;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FusedBars) <= 512, "fused-backward barriers exceed their shared-memory slot");

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// The 4-D TMA store / reduce-add of one [128 rows][32 fp32] chunk (128-byte
// swizzle) from shared memory into the accumulator; bulk-group completion.
__device__ __forceinline__ void tma_store_4d(const void* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_4d(const void* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::
                   "l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void reg_tie32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Two 32-column TMEM loads of this thread's lane, waited for together.
__device__ __forceinline__ void load2_cols32(uint32_t a0, uint32_t a1, float (&v0)[32], float (&v1)[32]) {
  uint32_t r0[32], r1[32];
  tmem_ld32(a0, r0);
  tmem_ld32(a1, r1);
  tmem_ld_wait(r0);
  reg_tie32(r1);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    v0[c] = __uint_as_float(r0[c]);
    v1[c] = __uint_as_float(r1[c]);
  }
}

// 128 bytes (eight 16-byte units) as row `row` of a 128-byte-swizzled chunk:
// logical unit u of the row sits at unit u ^ (row & 7).
__device__ __forceinline__ void store_row128_sw(uint8_t* chunk, int row, const uint32_t (&v)[32]) {
  uint8_t* rp = chunk + row * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<uint4*>(rp + ((u ^ (row & 7)) << 4)) = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}

// ncols accumulator columns of this thread's lane, scaled, as 16-bit values
// (only the first nvalid stored).
template <bool F16>
__device__ __forceinline__ void store_acc(uint32_t taddr, int ncols, int nvalid, float mul, uint16_t* dst, bool valid) {
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + c, r);
    tmem_ld_wait(r);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack2<F16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (valid) {
      uint4* d = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        if (c + v * 8 < nvalid) d[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

// Units: (KV block kb, KV head g, batch b), kb fastest and descending.
__host__ __device__ __forceinline__ int fused_units(const Shape& s) { return ceil_div(s.Tk, 128) * s.HKV * s.B; }

template <bool F16>
__global__ void __launch_bounds__(kThreadsF, 1)
    fa_bwd_fused_d64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                            const __grid_constant__ CUtensorMap tmAcc, const BwdParams p) {
  using C = FusedTiles;
  constexpr int D = 64;
  constexpr int BQ = 128, BK = 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  FusedBars* bars = reinterpret_cast<FusedBars*>(smem + C::kOffBar);
  float* srows = reinterpret_cast<float*>(smem + C::kOffRows);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rep = s.H / s.HKV;
  const int nq = ceil_div(s.T, BQ);
  const int nkb = ceil_div(s.Tk, BK);
  const int nunits = fused_units(s);
  const int cta = static_cast<int>(blockIdx.x);
  struct Unit {
    int kb, g, b, qlo, nqb, niter;
  };
  auto unit = [&](int u) {
    Unit w;
    w.kb = nkb - 1 - u % nkb;
    const int r = u / nkb;
    w.g = r % s.HKV;
    w.b = r / s.HKV;
    int qhi;
    q_range_for_kv(s.T, s.Tk, BQ, BK, s.causal, s.window, w.kb, w.qlo, qhi);
    w.nqb = qhi - w.qlo + 1;
    w.niter = rep * w.nqb;
    return w;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    mbar_init(&bars->res_empty, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->x_full[i], 1 + 32);  // expect-tx arrival + the 32 lanes writing the rows
      mbar_init(&bars->x_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, kComputeF / 32);
    mbar_init(&bars->ds_full, kComputeF / 32);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->dq_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->stg_full[i], kComputeF / 32);
      mbar_init(&bars->stg_empty[i], 1);
    }
    mbar_init(&bars->drain, 1);
    sched_init(&bars->sched, 10);  // compute warps, MMA warp, reducer
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
    }
    int xc = 0, uc = 0;
    bool ok = true;
    int u = cta;
    for (int seq = 0; ok && !p.inject_stall; ++seq) {
      if (!(ok = sched_publish(&bars->sched, seq, u, ctl, kCode))) break;
      if (u >= nunits) break;
      const Unit w = unit(u);
      // K and V once the previous unit's MMAs (its last dQ partial reads K)
      // are done with them
      if (uc > 0 && !(ok = warp_wait(&bars->res_empty, (uc - 1) & 1, ctl, kCode))) break;
      mbar_arrive_expect_tx_e(&bars->res_full, 2 * C::kChunk);
      tma_load_4d_e(&tmK, &bars->res_full, smem + C::kOffK, 0, w.g, w.kb * BK, w.b);
      tma_load_4d_e(&tmV, &bars->res_full, smem + C::kOffV, 0, w.g, w.kb * BK, w.b);
      ++uc;
      float l2[4], dl[4];
      auto load_rows = [&](int n) {
        const int h = w.g * rep + n / w.nqb;
        const int qb = w.qlo + n % w.nqb;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = qb * BQ + lane + 32 * k;
          l2[k] = 0.f;
          dl[k] = 0.f;
          if (i < s.T) {
            const size_t idx = (static_cast<size_t>(w.b) * s.H + h) * s.T + i;
            l2[k] = -p.LSE[idx] * kLog2eF;
            dl[k] = p.Delta[idx];
          }
        }
      };
      if (w.niter > 0) load_rows(0);
      for (int n = 0; n < w.niter; ++n) {
        const int st = xc % C::kStages;
        if (xc >= C::kStages && !(ok = warp_wait(&bars->x_empty[st], ((xc / C::kStages) - 1) & 1, ctl, kCode)))
          break;
        const int h = w.g * rep + n / w.nqb;
        const int qb = w.qlo + n % w.nqb;
        mbar_arrive_expect_tx_e(&bars->x_full[st], 2 * C::kChunk);
        tma_load_4d_e(&tmQ, &bars->x_full[st], smem + C::kOffX + st * C::kChunk, 0, h, qb * BQ, w.b);
        tma_load_4d_e(&tmdO, &bars->x_full[st], smem + C::kOffY + st * C::kChunk, 0, h, qb * BQ, w.b);
        float* rows = srows + st * 256;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          rows[lane + 32 * k] = l2[k];
          rows[128 + lane + 32 * k] = dl[k];
        }
        mbar_arrive(&bars->x_full[st]);
        ++xc;
        if (n + 1 < w.niter) load_rows(n + 1);
      }
      if (!ok) break;
      int claimed = 0;
      if (lane == 0) claimed = sched_claim(p.sched);
      u = __shfl_sync(0xffffffffu, claimed, 0);
    }
    if (lane == 0 && bars->abort) {
      if (uc > 0) drain_bar(&bars->res_full, (uc - 1) & 1, p.timeout_ns);
      for (int n = imax(0, xc - C::kStages); n < xc; ++n)
        drain_bar(&bars->x_full[n % C::kStages], (n / C::kStages) & 1, p.timeout_ns);
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_f32acc<F16>(128, BQ, false, false);   // K-major x K-major, N = 128
    constexpr uint32_t idesc_acc = idesc_f32acc<F16>(128, D, false, true);   // TMEM A x MN-major B, N = 64
    constexpr uint32_t idesc_dq = idesc_f32acc<F16>(128, D, true, true);     // MN-major A (dS) x MN-major B (K)
    const uint32_t sK = sbase + C::kOffK;
    const uint32_t sV = sbase + C::kOffV;
    int xc = 0, uc = 0;
    auto stage_ready = [&](int xg) -> bool {
      const int st = xg % C::kStages;
      if (!warp_wait(&bars->x_full[st], (xg / C::kStages) & 1, ctl, kCode)) return false;
      tc_fence_after();
      return true;
    };
    auto issue_kk = [&](uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {  // [128 x 128] = A B^T, K = 64
      const uint64_t a0 = sdesc_sw128(a_smem, 16, 1024);
      const uint64_t b0 = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) mma_ss_e(d_tmem, a0 + ((kk * 32) >> 4), b0 + ((kk * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
    };
    auto issue_acc = [&](uint32_t acc, uint32_t a_tmem, uint32_t b_smem, bool accumulate) {
      const uint64_t b0 = sdesc_sw128(b_smem, C::kChunk, 1024);
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk)
        mma_ts_e(acc, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8, b0 + ((kk * 16 * kRowB) >> 4), idesc_acc,
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
        if (!(ok = stage_ready(xc))) break;
        issue_kk(tmem + C::kTmS, sK, sbase + C::kOffX + (xc % C::kStages) * C::kChunk);
        mma_commit_e(&bars->s_full);
        issue_kk(tmem + C::kTmDP, sV, sbase + C::kOffY + (xc % C::kStages) * C::kChunk);
        mma_commit_e(&bars->dp_full);
      }
      for (int n = 0; ok && n < w.niter; ++n) {
        const int xg = xc + n;
        const int st = xg % C::kStages;
        if (n + 1 < w.niter && !(ok = stage_ready(xg + 1))) break;
        if (!(ok = warp_wait(&bars->p_full, xg & 1, ctl, kCode))) break;
        tc_fence_after();
        issue_acc(tmem + C::kTmDV, tmem + C::kTmS, sbase + C::kOffY + st * C::kChunk, n > 0);  // dV += P^T dO
        if (n + 1 < w.niter) {
          issue_kk(tmem + C::kTmS, sK, sbase + C::kOffX + ((xg + 1) % C::kStages) * C::kChunk);  // S^T_{n+1}
          mma_commit_e(&bars->s_full);
        }
        if (!(ok = warp_wait(&bars->ds_full, xg & 1, ctl, kCode))) break;
        tc_fence_after();
        issue_acc(tmem + C::kTmDK, tmem + C::kTmDP, sbase + C::kOffX + st * C::kChunk, n > 0);  // dK += dS^T Q
        {  // dQ partial = dS K: A = dS from shared memory (MN-major: queries contiguous), B = K (MN-major)
          const uint64_t a0 = sdesc_sw128(sbase + C::kOffDS, C::kChunk, 1024);
          const uint64_t b0 = sdesc_sw128(sK, C::kChunk, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss_e(tmem + C::kTmDQ, a0 + ((kk * 16 * kRowB) >> 4), b0 + ((kk * 16 * kRowB) >> 4), idesc_dq,
                     kk > 0 ? 1u : 0u);
          mma_commit_e(&bars->dq_full);
        }
        mma_commit_e(&bars->x_empty[st]);
        if (n + 1 == w.niter) mma_commit_e(&bars->res_empty);  // the unit's last MMAs reading K and V
        if (n + 1 < w.niter) {
          issue_kk(tmem + C::kTmDP, sV, sbase + C::kOffY + ((xg + 1) % C::kStages) * C::kChunk);  // dP^T_{n+1}
          mma_commit_e(&bars->dp_full);
        }
      }
      if (!ok) break;
      if (w.niter == 0) mma_commit_e(&bars->res_empty);
      mma_commit_e(&bars->acc_full);
      xc += w.niter;
    }
    mma_commit_e(&bars->drain);
    drain_bar(&bars->drain, 0, p.timeout_ns);
  } else if (warp == 10) {
    // -------------------------------------------------------------- reducer
    // Per streamed block: wait for the dQ partial in shared memory, then for
    // its turn, then store it (first contribution) or add it (the others)
    // into the fp32 accumulator tile with the TMA unit; the last contribution
    // also scales, rounds and writes dQ.
    unsigned* turns = p.turns;
    float* acc = p.dq_acc;
    int xc = 0;
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int u = sched_next(&bars->sched, seq, ctl, kCode);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= nunits) break;
      const Unit w = unit(u);
      for (int n = 0; ok && n < w.niter; ++n) {
        const int xg = xc + n;
        const int h = w.g * rep + n / w.nqb;
        const int qb = w.qlo + n % w.nqb;
        int kb_lo, kb_hi;
        kv_range_for_q(s.T, s.Tk, BQ, BK, s.causal, s.window, qb, kb_lo, kb_hi);
        const unsigned idx = static_cast<unsigned>(kb_hi - w.kb);
        unsigned* turn = turns + (static_cast<size_t>(w.b) * s.H + h) * nq + qb;
        const int sb = xg & 1;  // staging buffer of this partial
        if (!(ok = warp_wait(&bars->stg_full[sb], (xg >> 1) & 1, ctl, kCode))) break;
        if (idx > 0) {  // every contribution before this one must be in
          bool seen = false;
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
              if (ld_acquire(turn) == idx) {
                seen = true;
                break;
              }
              if (*ctl.abort) break;
              if (globaltimer_ns() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1;
                atomicOr(ctl.err, kCode);
                break;
              }
            }
          }
          if (!(ok = __shfl_sync(0xffffffffu, seen, 0))) break;
        }
        if (lane == 0) {
          fence_async_global();
          for (int c = 0; c < 2; ++c) {
            const void* src = smem + C::kOffStg + (2 * sb + c) * C::kChunk;
            if (idx == 0)
              tma_store_4d(&tmAcc, src, c * 32, h, qb * BQ, w.b);
            else
              tma_reduce_add_4d(&tmAcc, src, c * 32, h, qb * BQ, w.b);
          }
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&bars->stg_empty[sb]);  // the partial has been read out of shared memory
          bulk_wait0();                   // and added into the accumulator
          fence_async_global();
          __threadfence();
        }
        __syncwarp();
        if (w.kb == kb_lo) {
          // the last contribution: dQ = scale * accumulator, rounded to the
          // element type; rows past the sequence and columns past the head
          // dim stay untouched
#pragma unroll 1
          for (int rr = 0; rr < 4; ++rr) {
            const int row = qb * BQ + lane + 32 * rr;
            if (row >= s.T) continue;
            const size_t base = ((static_cast<size_t>(w.b) * s.T + row) * s.H + h) * s.D;
            const float4* src = reinterpret_cast<const float4*>(acc + base);
            uint32_t pk[32];
#pragma unroll
            for (int c4 = 0; c4 < D / 4; ++c4) {
              const float4 v = c4 * 4 < s.D ? __ldcg(src + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
              pk[2 * c4] = pack2<F16>(v.x * s.scale, v.y * s.scale);
              pk[2 * c4 + 1] = pack2<F16>(v.z * s.scale, v.w * s.scale);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dQ) + base);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (v * 8 < s.D) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
          if (lane == 0) *turn = 0u;  // ready for the next launch
        } else if (lane == 0) {
          st_release(turn, idx + 1);
        }
        __syncwarp();
      }
      if (!ok) break;
      xc += w.niter;
    }
    if (lane == 0) bulk_wait0();
  } else {
    // -------------------------------------------------------------- compute
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int jrow = quarter * 32 + lane;  // key row of the unit's block = TMEM lane; query row for dQ
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + C::kTmS + half * 64;
    const uint32_t dp_addr = tmem + lane_addr + C::kTmDP + half * 64;
    const float sl2 = p.scale_log2;
    uint8_t* ds_chunk = smem + C::kOffDS + half * C::kChunk;
    uint8_t* stg_chunk = smem + C::kOffStg + half * C::kChunk;  // + 2 chunks for the second buffer
    int xc = 0, uc = 0;
    // The dQ partial of block xg: TMEM -> shared memory for the reducer.  Run
    // in the next block's dS pass, after that block's dS is formed (its P
    // registers are dead by then) and before dS is released: releasing it
    // lets the MMA warp issue the next partial into the same TMEM columns.
    auto copy_dq = [&](int xg) -> bool {
      const int sb = xg & 1;
      if (!warp_wait(&bars->dq_full, xg & 1, ctl, kCode)) return false;
      // the buffer's previous partial (two blocks back) handed on
      if (xg >= 2 && !warp_wait(&bars->stg_empty[sb], ((xg >> 1) - 1) & 1, ctl, kCode)) return false;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tmem + lane_addr + C::kTmDQ + half * 32, r);
      tmem_ld_wait(r);
      store_row128_sw(stg_chunk + sb * 2 * C::kChunk, jrow, r);
      fence_async_smem();
      tc_fence_before();
      warp_arrive(&bars->stg_full[sb]);
      return true;
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
      const int j = w.kb * BK + jrow;
      for (int n = 0; ok && n < w.niter; ++n) {
        const int xg = xc + n;
        const int st = xg % C::kStages;
        const int qb = w.qlo + n % w.nqb;
        const float* rows = srows + st * 256 + half * 64;
        // pass 1: P^T
        if (!(ok = warp_wait(&bars->x_full[st], (xg / C::kStages) & 1, ctl, kCode))) break;
        if (!(ok = warp_wait(&bars->s_full, xg & 1, ctl, kCode))) break;
        tc_fence_after();
        const bool need_mask = block_needs_mask(s.T, s.Tk, BQ, BK, s.causal, s.window, qb, w.kb);
        float pv[64];
        {
          float lo[32], hi[32];
          load2_cols32(s_addr, s_addr + 32, lo, hi);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            pv[c] = lo[c];
            pv[32 + c] = hi[c];
          }
        }
        const float4* lse4 = reinterpret_cast<const float4*>(rows);
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
          tmem_st32(s_addr, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->p_full);
        // pass 2: dS^T = P^T (dP^T - Delta) -> bf16 into TMEM (A of dK) and,
        // as row j of the [keys][queries] tile, into shared memory (A of dQ)
        if (!(ok = warp_wait(&bars->dp_full, xg & 1, ctl, kCode))) break;
        tc_fence_after();
        float dlo[32], dhi[32];
        load2_cols32(dp_addr, dp_addr + 32, dlo, dhi);
        const float4* del4 = reinterpret_cast<const float4*>(rows + 128);
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d = del4[c4];
          const float4 e = del4[8 + c4];
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
        store_row128_sw(ds_chunk, jrow, pk);  // queries [64 half, 64 half + 64) of key row jrow
        fence_async_smem();
        tmem_st_wait();
        // the previous block's dQ partial is done by now: hand it on
        if (n > 0 && !(ok = copy_dq(xg - 1))) break;
        tc_fence_before();
        warp_arrive(&bars->ds_full);
      }
      if (!ok) break;
      if (w.niter > 0 && !(ok = copy_dq(xc + w.niter - 1))) break;
      xc += w.niter;
      if (!(ok = warp_wait(&bars->acc_full, uc & 1, ctl, kCode))) break;
      ++uc;
      tc_fence_after();
      const size_t rowoff = ((static_cast<size_t>(w.b) * s.Tk + j) * s.HKV + w.g) * s.D + half * (D / 2);
      const int nvalid = s.D - half * (D / 2);
      store_acc<F16>(tmem + lane_addr + C::kTmDV + half * (D / 2), D / 2, nvalid, 1.f,
                     static_cast<uint16_t*>(p.dV) + rowoff, j < s.Tk);
      store_acc<F16>(tmem + lane_addr + C::kTmDK + half * (D / 2), D / 2, nvalid, s.scale,
                     static_cast<uint16_t*>(p.dK) + rowoff, j < s.Tk);
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

template <bool F16>
cudaError_t launch_fused(const TensorMaps& tm, const CUtensorMap& acc_map, const BwdParams& p, cudaStream_t stream) {
  // the cooperative launch checks residency against the preferred carveout:
  // raise it too
  static std::atomic<unsigned long long> attr_set{0};
  if (cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fa_bwd_fused_d64_kernel<F16>),
                                    FusedTiles::kSmemBytes, attr_set, /*carveout=*/true);
      e != cudaSuccess)
    return e;
  const int units = fused_units(p.s);
  // cooperative: every CTA is resident at once, so every unit a turn waits
  // for is running or done
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(imax(1, imin(p.ctas, units)));
  cfg.blockDim = dim3(kThreadsF);
  cfg.dynamicSmemBytes = FusedTiles::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_bwd_fused_d64_kernel<F16>, tm.q, tm.k, tm.v, tm.dO, acc_map, p);
}

}  // namespace

bool fused_backward_applies(const Shape& s, int f16_or_bf16) {
  return f16_or_bf16 && s.D <= 64 && s.causal == 1 && s.Tk == s.T;
}

cudaError_t launch_bwd_fused(const TensorMaps& tm, const CUtensorMap& acc_map, const BwdParams& p,
                             cudaStream_t stream) {
  return p.f16 ? launch_fused<true>(tm, acc_map, p, stream) : launch_fused<false>(tm, acc_map, p, stream);
}

}  // namespace fa
