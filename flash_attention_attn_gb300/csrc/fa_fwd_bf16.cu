// fa_fwd_bf16.cu -- fused causal / sliding-window GQA attention forward for
// sm_103a: TMA -> shared memory -> tcgen05 MMA -> TMEM, online softmax in
// registers.  Two kernels: the two-tile kernel further down (two 128-row
// query tiles per CTA, used for almost every shape) and, first, the one-tile
// kernel (sequences of one query tile with an odd number of query heads per
// KV head, and the test hook).
//
// One-tile kernel: one CTA computes one 128-row query tile of one (b, h).
// Warp roles:
//   warps 0-3  softmax: thread t owns query row t of the tile (= TMEM lane t).
//   warp  4    TMA producer: the Q tile once, then K and V blocks through an
//              NS-stage ring guarded by full/empty mbarriers (a K stage is
//              released as soon as its S MMA is done, a V stage after PV).
//   warp  5    MMA issuer (one thread) and TMEM owner.
//
// Per visible KV block n (the loop skips blocks above the causal diagonal and
// before the window, and applies the per-element mask only on blocks that
// need it):
//   S_n = Q K_n^T          -> TMEM S[n % 2] (128 x 128 fp32)
//   softmax: m_new = max(m, rowmax S_n); P = 2^(S*scale*log2e - m); l += rowsum P;
//            P -> bf16 into the first 64 columns of S[n % 2]
//   O += P V_n             -> TMEM O (128 x D fp32), A operand read from TMEM
// S_{n+1} is computed while the softmax works on S_n.  O is rescaled only
// when a row's max grows by more than 2^8 (the rows keep a stale reference
// max otherwise, which is exact: numerator and denominator share it).
// The recurrence is the online softmax of the Graphcore flash-attention-ipu
// forward (flashAttentionQKVPackedWithStash: m_new, c = exp(m - m_new),
// l = l*c + rowsum, o = o*c + P V, o /= l, lse = m + log l at the end).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;              // 64-wide bf16 chunks per row
  static constexpr int kChunkBytes = 128 * 64 * 2;    // one [128][64] chunk
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (D == 64) ? 4 : 3;   // K/V ring depth (3 x 64 KB fits at D = 128)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmQ = 0;      // Q as bf16 A operand: D/2 columns
  static constexpr uint32_t kTmS = 128;    // S[0] at 128, S[1] at 256
  static constexpr uint32_t kTmO = 384;    // O: D columns
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 256 between rescales
constexpr int kThreads = 192;

struct Bars {
  uint64_t q_full;
  uint64_t q_tmem;  // Q copied into TMEM by the 128 softmax threads
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t k_empty[4];  // K stage free once its S MMA completed
  uint64_t v_empty[4];  // V stage free once its PV MMA completed
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "one-tile barriers exceed their shared-memory slot");

__device__ __forceinline__ void reg_tie(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nq = ceil_div(s.T, kBM);
  const int qb = nq - 1 - static_cast<int>(blockIdx.x);  // longest causal tiles first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int g = h / (s.H / s.HKV);
  int kb_lo, kb_hi;
  kv_range_for_q(s.T, s.Tk, kBM, kBN, s.causal, s.window, qb, kb_lo, kb_hi);
  const int nblk = kb_hi - kb_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_tmem, 4);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);  // one arrival per softmax warp
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Ctl ctl{&bars->abort, p.err, p.timeout_ns};
  constexpr unsigned kCode = 1u;  // FA_DEVERR_FWD_TIMEOUT

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop; one elected lane arms each barrier and
    // issues each copy
    if (!p.inject_stall) {
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
      }
      mbar_arrive_expect_tx_e(&bars->q_full, C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d_e(&tmQ, &bars->q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, h, qb * kBM, b);
      int issued = 0;
      for (int n = 0; n < nblk; ++n) {
        const int st = n % C::kStages;
        const int kb = kb_lo + n;
        uint8_t* sk = smem + C::kOffK + st * C::kTileBytes;
        uint8_t* sv = smem + C::kOffV + st * C::kTileBytes;
        if (n >= C::kStages && !warp_wait(&bars->k_empty[st], ((n / C::kStages) - 1) & 1, ctl, kCode)) break;
        mbar_arrive_expect_tx_e(&bars->k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmK, &bars->k_full[st], sk + c * C::kChunkBytes, c * 64, g, kb * kBN, b);
        if (n >= C::kStages && !warp_wait(&bars->v_empty[st], ((n / C::kStages) - 1) & 1, ctl, kCode)) {
          drain_bar(&bars->k_full[st], (n / C::kStages) & 1, p.timeout_ns);
          break;
        }
        mbar_arrive_expect_tx_e(&bars->v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_e(&tmV, &bars->v_full[st], sv + c * C::kChunkBytes, c * 64, g, kb * kBN, b);
        issued = n + 1;
      }
      if (bars->abort) {
        // let every copy already issued land before the CTA exits
        drain_bar(&bars->q_full, 0, p.timeout_ns);
        for (int n = imax(0, issued - C::kStages); n < issued; ++n) {
          drain_bar(&bars->k_full[n % C::kStages], (n / C::kStages) & 1, p.timeout_ns);
          drain_bar(&bars->v_full[n % C::kStages], (n / C::kStages) & 1, p.timeout_ns);
        }
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMA issuer
    {  // the whole warp runs the loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_f32acc<F16>(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_f32acc<F16>(128, D, false, true);
      bool ok = warp_wait(&bars->q_tmem, 0, ctl, kCode);
      for (int n = 0; ok && n <= nblk; ++n) {
        if (n < nblk) {
          const int st = n % C::kStages;
          const int sb = n & 1;
          if (!(ok = warp_wait(&bars->k_full[st], (n / C::kStages) & 1, ctl, kCode))) break;
          tc_fence_after();
          const uint32_t sk = sbase + C::kOffK + st * C::kTileBytes;
          // descriptors built once, stepped by (bytes >> 4) in the address field
          const uint64_t kdesc = sdesc_sw128(sk, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ts_e(tmem + C::kTmS + sb * 128, tmem + C::kTmQ + kk * 8, kdesc + off, idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit_e(&bars->s_full[sb]);
          mma_commit_e(&bars->k_empty[st]);
        }
        if (n >= 1) {
          const int m = n - 1;
          const int st = m % C::kStages;
          const int sb = m & 1;
          if (!(ok = warp_wait(&bars->p_full[sb], (m >> 1) & 1, ctl, kCode))) break;
          if (!(ok = warp_wait(&bars->v_full[st], (m / C::kStages) & 1, ctl, kCode))) break;
          tc_fence_after();
          const uint32_t sv = sbase + C::kOffV + st * C::kTileBytes;
          const uint64_t vdesc = sdesc_sw128(sv, C::kChunkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            // P: 16 bf16 keys per step = 8 TMEM columns; V: 16 key rows = 2048 bytes
            mma_ts_e(tmem + C::kTmO, tmem + C::kTmS + sb * 128 + kk * 8, vdesc + ((kk * 2048) >> 4), idesc_o,
                   (m > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_e(&bars->o_done);
          mma_commit_e(&bars->v_empty[st]);
        }
      }
      // every MMA this thread issued must finish before TMEM is released
      mma_commit_e(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = threadIdx.x;  // 0..127 = TMEM lane = tile row
    const int row = qb * kBM + t;
    int vis_lo, vis_hi;  // keys this row sees
    visible_keys(s.T, s.Tk, s.causal, s.window, row, vis_lo, vis_hi);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_run = -CUDART_INF_F;  // reference max, log2 domain
    float l_run = 0.f;
    // Q into TMEM (row t on lane t) as the A operand of every S MMA, so that
    // those MMAs read only K from shared memory
    bool ok = warp_wait(&bars->q_full, 0, ctl, kCode);
    if (ok) {
      tile_row_to_tmem<D>(smem + C::kOffQ, C::kChunkBytes, t, tmem + lane_addr + C::kTmQ);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bars->q_tmem);
    }
    for (int n = 0; ok && n < nblk; ++n) {
      const int kb = kb_lo + n;
      const int sb = n & 1;
      if (!(ok = warp_wait(&bars->s_full[sb], (n >> 1) & 1, ctl, kCode))) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + C::kTmS + sb * 128;
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(s_addr + 0, r0);
      tmem_ld32(s_addr + 32, r1);
      tmem_ld32(s_addr + 64, r2);
      tmem_ld32(s_addr + 96, r3);
      tmem_ld_wait(r0);
      reg_tie(r1);
      reg_tie(r2);
      reg_tie(r3);
      float sv[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        sv[c] = __uint_as_float(r0[c]);
        sv[32 + c] = __uint_as_float(r1[c]);
        sv[64 + c] = __uint_as_float(r2[c]);
        sv[96 + c] = __uint_as_float(r3[c]);
      }
      if (block_needs_mask(s.T, s.Tk, kBM, kBN, s.causal, s.window, qb, kb)) {
        // this row's visible keys, relative to the block
        const int a = vis_lo - kb * kBN, z = vis_hi - kb * kBN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < a || c > z) sv[c] = -CUDART_INF_F;
      }
      float mx = sv[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, sv[c]);
      mx *= sl2;  // scale > 0, so the max commutes with the scaling
      const float m_new = fmaxf(m_run, mx);
      const bool first = (n == 0);
      const bool resc = !first && (m_new - m_run > kRescaleThreshold);
      const float m_ref = (first || resc) ? m_new : m_run;
      const float m_use = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;
      float sum = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(sv[q4 * 32 + 2 * e], sl2, -m_use));
          const float p1 = ex2(fmaf(sv[q4 * 32 + 2 * e + 1], sl2, -m_use));
          sum += p0 + p1;
          pk[e] = pack2<F16>(p0, p1);
        }
        tmem_st16(s_addr + q4 * 16, pk);
      }
      tmem_st_wait();
      if (!first) {
        if (__any_sync(0xffffffffu, resc)) {
          // O holds P_0..P_{n-1} V; wait for the last of those MMAs, then rescale
          if (!(ok = warp_wait(&bars->o_done, (n - 1) & 1, ctl, kCode))) break;
          tc_fence_after();
          const float corr = resc ? ex2(m_run - m_new) : 1.f;
          const uint32_t o_addr = tmem + lane_addr + C::kTmO;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ro[32];
            tmem_ld32(o_addr + c * 32, ro);
            tmem_ld_wait(ro);
#pragma unroll
            for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * corr);
            tmem_st32(o_addr + c * 32, ro);
          }
          tmem_st_wait();
          if (resc) l_run *= corr;
        }
      }
      if (first || resc) m_run = m_new;
      l_run += sum;
      tc_fence_before();
      warp_arrive(&bars->p_full[sb]);
    }
    if (ok && nblk > 0) ok = warp_wait(&bars->o_done, (nblk - 1) & 1, ctl, kCode);
    if (ok) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const uint32_t o_addr = tmem + lane_addr + C::kTmO;
      uint16_t* orow = static_cast<uint16_t*>(p.O) + ((static_cast<size_t>(b) * s.T + row) * s.H + h) * s.D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ro[32];
        tmem_ld32(o_addr + c * 32, ro);
        tmem_ld_wait(ro);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<F16>(__uint_as_float(ro[2 * e]) * inv, __uint_as_float(ro[2 * e + 1]) * inv);
        if (row < s.T) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)  // columns past a head dim below D are not stored
            if (c * 32 + v * 8 < s.D) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row < s.T) {
        const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : 0.f;
        p.LSE[(static_cast<size_t>(b) * s.H + h) * s.T + row] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- two tiles
//
// Two 128-row query tiles A and B per work unit, sharing every K/V block the
// unit streams: one query block of two query heads that share a KV head
// (head pairs, when H/HKV is even; both tiles see the same key range) or
// query blocks 2j and 2j + 1 of one head (block pairs).  Each 64 KB K/V block
// (D = 128) feeds four 128x128 MMA groups instead of two, which halves the
// TMA traffic per MMA.  Measured on GB300, a K/V ring feeding one tile is
// bounded near 1600 cycles per block by the TMA stream itself against 1024
// cycles of MMAs.
//
// Persistent: at most one CTA per SM, each walking its share of the units
// (longest causal work first, snake order across CTAs).  Barriers, TMEM and
// the K/V rings live for the whole launch and their phases run on across
// units, so the next unit's Q and first K/V blocks load while the current
// unit finishes, and its first score MMAs run while the softmax warps store
// the current unit's O.
//   warps 0-3 softmax of tile A, warps 4-7 softmax of tile B (warp w owns
//             TMEM lanes 32*(w%4).. = rows of its tile)
//   warp  8   TMA producer: per unit Q_A, Q_B (once the previous unit's
//             score MMAs are done with them), then K and V blocks in the
//             order the MMAs need them
//   warp  9   MMA issuer and TMEM owner
// (both run converged; one elected lane issues each copy and each MMA)
// TMEM: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [256+D,256+2D).
// No S buffer is doubled; the tiles ping-pong instead.  Per streamed block n
// the MMA queue is  PV_A(n) S_A(n+1) PV_B(n) S_B(n+1), so the softmax of one
// tile runs while the tensor pipe works on the other's.  S_t(n+1) overwrites
// the P_t(n) that PV_t(n) reads; the tensor pipe executes in order.  For the
// same reason a completed S_t(n+1) implies a completed PV_t(n): the softmax
// may rescale O_t as soon as it sees its scores, and O_t's own barrier is
// committed only once per unit, after the tile's last PV.  The first PV of
// the next unit (which overwrites O_t) waits for P of that unit's first
// block, which the same softmax warps release only after they have read O_t
// out for the epilogue.
// A tile skips the streamed blocks outside its own visible range (with a
// window the first block may be A's only, with causal masking the last is
// B's only).
template <int D>
struct Fwd2Cfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 64 * 2;  // one [128][64] bf16 chunk
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // a K stage is held from S_A(n) to S_B(n), a V stage from PV_A(n) to PV_B(n)
  // one MMA iteration later, so V gets the deeper ring
  static constexpr int kKStages = (D == 64) ? 4 : 2;
  static constexpr int kVStages = (D == 64) ? 4 : 3;
  static constexpr int kOffQ = 0;  // Q_A, Q_B
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmS = 0;    // S_t at t * 128
  static constexpr uint32_t kTmO = 256;  // O_t at 256 + t * D
};

constexpr int kThreads2 = 320;

struct Bars2 {
  uint64_t q_full;
  uint64_t q_empty;     // the unit's score MMAs are done with Q_A, Q_B
  uint64_t k_full[4];
  uint64_t k_empty[4];  // K stage free once the S MMAs of both tiles completed
  uint64_t v_full[4];
  uint64_t v_empty[4];  // V stage free once the PV MMAs of both tiles completed
  uint64_t s_full[2];   // per tile
  uint64_t p_half[2];   // per tile: keys 0-63 of P stored (and O rescaled), one arrival per softmax warp
  uint64_t p_full[2];   // per tile: keys 64-127 of P stored, one arrival per softmax warp
  uint64_t o_done[2];   // per tile: all its PV MMAs of the unit completed (committed once per unit)
  uint64_t drain;
  SchedRing sched;      // units handed from the producer to the other roles
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Bars2) <= 512, "two-tile barriers exceed their shared-memory slot");

// One work unit of the two-tile forward: query blocks q_a, q_b of heads h_a,
// h_b in batch b, KV head g; the visible KV block range of each tile (B is
// empty past the end) and their union [lo, lo + nblk).
struct Fwd2Unit {
  int q_a, q_b, h_a, h_b, g, b;
  int lo_a, hi_a, lo_b, hi_b;
  bool has_b;
  int lo, nblk;
};

// Units numbered with x (the query block, or block pair, counted from the
// end of the sequence: longest causal work first) fastest, then head (pair),
// then batch, so that the units in flight at any time share a KV head and
// re-read its K/V blocks from L2 (measured on GB300: numbering x outermost,
// which spreads the units in flight over all KV heads, made the long causal
// workload's forward 2 % and its dK/dV 6.5 % slower).
__device__ __forceinline__ Fwd2Unit fwd2_unit(const Shape& s, bool pack_heads, int u) {
  const int nq = ceil_div(s.T, kBM);
  const int nx = pack_heads ? nq : ceil_div(nq, 2);
  const int ny = pack_heads ? s.H / 2 : s.H;
  const int x = u % nx;
  const int r = u / nx;
  const int y = r % ny;
  Fwd2Unit w;
  w.b = r / ny;
  // Block pairs: blocks 2j and 2j + 1 of one head; head pairs: one block of
  // heads 2j and 2j + 1, which share a KV head when H/HKV is even, so that
  // both tiles see the same key range.
  w.q_a = pack_heads ? nq - 1 - x : 2 * (ceil_div(nq, 2) - 1 - x);
  w.q_b = pack_heads ? w.q_a : w.q_a + 1;
  w.h_a = pack_heads ? 2 * y : y;
  w.h_b = pack_heads ? w.h_a + 1 : w.h_a;
  w.g = w.h_a / (s.H / s.HKV);
  w.lo_b = 1;
  w.hi_b = 0;
  kv_range_for_q(s.T, s.Tk, kBM, kBN, s.causal, s.window, w.q_a, w.lo_a, w.hi_a);
  if (w.q_b < nq) kv_range_for_q(s.T, s.Tk, kBM, kBN, s.causal, s.window, w.q_b, w.lo_b, w.hi_b);
  w.has_b = w.lo_b <= w.hi_b;
  w.lo = w.has_b ? imin(w.lo_a, w.lo_b) : w.lo_a;
  const int hi = w.has_b ? imax(w.hi_a, w.hi_b) : w.hi_a;
  w.nblk = hi - w.lo + 1;  // the adjacent tiles' ranges overlap or touch: the union is contiguous
  return w;
}

__host__ __device__ __forceinline__ int fwd2_units(const Shape& s, bool pack_heads) {
  const int nq = ceil_div(s.T, kBM);
  return pack_heads ? nq * (s.H / 2) * s.B : ceil_div(nq, 2) * s.H * s.B;
}

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads2, 1)
    fa_fwd2_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Fwd2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars2* bars = reinterpret_cast<Bars2*>(smem + C::kOffBar);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool pack = p.pack_heads != 0;
  const int nunits = fwd2_units(s, pack);
  const int cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_half[t], 4);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->o_done[t], 1);
    }
    mbar_init(&bars->drain, 1);
    sched_init(&bars->sched, 9);  // consumers: eight softmax warps and the MMA warp
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
  constexpr unsigned kCode = 1u;  // FA_DEVERR_FWD_TIMEOUT

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop; one elected lane arms each barrier and
    // issues each copy
    if (!p.inject_stall) {
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
      }
      int kc = 0, vc = 0, uc = 0;  // K blocks, V blocks and units issued by this CTA
      bool ok = true;
      int u = cta;  // the CTA's first unit; later ones are claimed from the counter
      for (int seq = 0; ok; ++seq) {
        if (!(ok = sched_publish(&bars->sched, seq, u, ctl, kCode))) break;
        if (u >= nunits) break;  // the end marker has been handed on
        const Fwd2Unit w = fwd2_unit(s, pack, u);
        // Q_A, Q_B of this unit once the previous unit's score MMAs are done
        auto load_q = [&]() -> bool {
          if (uc > 0 && !warp_wait(&bars->q_empty, (uc - 1) & 1, ctl, kCode)) return false;
          mbar_arrive_expect_tx_e(&bars->q_full, (w.has_b ? 2 : 1) * C::kTileBytes);
          for (int t = 0; t < (w.has_b ? 2 : 1); ++t)
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d_e(&tmQ, &bars->q_full, smem + C::kOffQ + t * C::kTileBytes + c * C::kChunkBytes, c * 64,
                            t ? w.h_b : w.h_a, (t ? w.q_b : w.q_a) * kBM, w.b);
          ++uc;
          return true;
        };
        // With the two-stage K ring (D = 128) the unit's first K block is
        // issued before Q: its slot frees before Q's buffer (the previous
        // unit's last score MMAs), so its latency overlaps that wait (the
        // windowed workload's forward 0.8 % faster); with the four-stage ring
        // (D = 64) that order measured 2 % slower.
        constexpr bool kKFirst = (C::kKStages == 2);
        if ((!kKFirst || w.nblk == 0) && !(ok = load_q())) break;
        for (int n = 0; n < w.nblk; ++n) {
          const int st = kc % C::kKStages;
          if (kc >= C::kKStages && !(ok = warp_wait(&bars->k_empty[st], ((kc / C::kKStages) - 1) & 1, ctl, kCode)))
            break;
          mbar_arrive_expect_tx_e(&bars->k_full[st], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d_e(&tmK, &bars->k_full[st], smem + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes,
                          c * 64, w.g, (w.lo + n) * kBN, w.b);
          ++kc;
          if (kKFirst && n == 0 && !(ok = load_q())) break;
          const int sv = vc % C::kVStages;
          if (vc >= C::kVStages && !(ok = warp_wait(&bars->v_empty[sv], ((vc / C::kVStages) - 1) & 1, ctl, kCode)))
            break;
          mbar_arrive_expect_tx_e(&bars->v_full[sv], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d_e(&tmV, &bars->v_full[sv], smem + C::kOffV + sv * C::kTileBytes + c * C::kChunkBytes,
                          c * 64, w.g, (w.lo + n) * kBN, w.b);
          ++vc;
        }
        // claim the next unit only now, near the end of this one, so that the
        // CTAs that finish first take the next longest units
        int claimed = 0;
        if (lane == 0) claimed = sched_claim(p.sched);
        u = __shfl_sync(0xffffffffu, claimed, 0);
      }
      if (bars->abort) {
        // let every copy already issued land before the CTA exits
        if (uc > 0) drain_bar(&bars->q_full, (uc - 1) & 1, p.timeout_ns);
        for (int n = imax(0, kc - C::kKStages); n < kc; ++n)
          drain_bar(&bars->k_full[n % C::kKStages], (n / C::kKStages) & 1, p.timeout_ns);
        for (int n = imax(0, vc - C::kVStages); n < vc; ++n)
          drain_bar(&bars->v_full[n % C::kVStages], (n / C::kVStages) & 1, p.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    {  // the whole warp runs the loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_f32acc<F16>(128, 128, false, false);  // Q x K^T, both K-major
      constexpr uint32_t idesc_o = idesc_f32acc<F16>(128, D, false, true);     // P (TMEM) x V (MN-major)
      int n_p[2] = {0, 0};  // PV MMAs issued per tile so far (p_half / p_full phases)
      int kc = 0, vc = 0, uc = 0;  // K blocks, V blocks and units consumed by this CTA
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int u = sched_next(&bars->sched, seq, ctl, kCode);
        if (u < 0) {
          ok = false;
          break;
        }
        if (u >= nunits) break;
        const Fwd2Unit w = fwd2_unit(s, pack, u);
        auto in_tile = [&](int t, int kb) {
          return t ? (w.lo_b <= kb && kb <= w.hi_b) : (w.lo_a <= kb && kb <= w.hi_a);
        };
        int k_seen = -1;  // last block of this unit whose K stage this thread waited for
        auto issue_s = [&](int t, int n) -> bool {  // S_t = Q_t K_n^T
          const int kg = kc + n;
          const int st = kg % C::kKStages;
          if (k_seen < n) {
            if (!warp_wait(&bars->k_full[st], (kg / C::kKStages) & 1, ctl, kCode)) return false;
            tc_fence_after();
            k_seen = n;
          }
          const uint64_t qdesc = sdesc_sw128(sbase + C::kOffQ + t * C::kTileBytes, 16, 1024);
          const uint64_t kdesc = sdesc_sw128(sbase + C::kOffK + st * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss_e(tmem + C::kTmS + t * 128, qdesc + off, kdesc + off, idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit_e(&bars->s_full[t]);
          return true;
        };
        if (!(ok = warp_wait(&bars->q_full, uc & 1, ctl, kCode))) break;
        tc_fence_after();
        ++uc;
        if (w.nblk > 0) {
          for (int t = 0; ok && t < 2; ++t)
            if (in_tile(t, w.lo)) ok = issue_s(t, 0);
          if (!ok) break;
          mma_commit_e(&bars->k_empty[kc % C::kKStages]);
        }
        if (w.nblk <= 1) mma_commit_e(&bars->q_empty);  // every score MMA of the unit is issued
        for (int n = 0; ok && n < w.nblk; ++n) {
          const int kb = w.lo + n;
          const int vg = vc + n;
          const int stv = vg % C::kVStages;
          if (!(ok = warp_wait(&bars->v_full[stv], (vg / C::kVStages) & 1, ctl, kCode))) break;
          const uint64_t vdesc = sdesc_sw128(sbase + C::kOffV + stv * C::kTileBytes, C::kChunkBytes, 1024);
          for (int t = 0; ok && t < 2; ++t) {
            if (in_tile(t, kb)) {
              // P arrives in two halves of 64 keys: the first half's MMAs run
              // while the softmax still forms the second
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                if (!(ok = warp_wait(hf ? &bars->p_full[t] : &bars->p_half[t], n_p[t] & 1, ctl, kCode))) break;
                tc_fence_after();
#pragma unroll
                for (int k4 = 0; k4 < kBN / 32; ++k4) {  // P: 16 bf16 keys = 8 TMEM columns; V: 16 rows = 2048 bytes
                  const int kk = hf * (kBN / 32) + k4;
                  mma_ts_e(tmem + C::kTmO + t * D, tmem + C::kTmS + t * 128 + kk * 8, vdesc + ((kk * 2048) >> 4),
                           idesc_o, (kb > (t ? w.lo_b : w.lo_a) || kk > 0) ? 1u : 0u);
                }
              }
              if (!ok) break;
              if (kb == (t ? w.hi_b : w.hi_a)) mma_commit_e(&bars->o_done[t]);  // the tile's last PV of the unit
              ++n_p[t];
            }
            if (n + 1 < w.nblk && in_tile(t, kb + 1)) ok = issue_s(t, n + 1);
          }
          if (!ok) break;
          if (n + 2 == w.nblk) mma_commit_e(&bars->q_empty);  // the unit's last score MMAs are issued
          mma_commit_e(&bars->v_empty[stv]);
          if (n + 1 < w.nblk) mma_commit_e(&bars->k_empty[(kc + n + 1) % C::kKStages]);
        }
        kc += w.nblk;
        vc += w.nblk;
      }
      // every MMA this thread issued must finish before TMEM is released
      mma_commit_e(&bars->drain);
      drain_bar(&bars->drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = warp >> 2;               // tile
    const int r = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + C::kTmS + t * 128;
    const uint32_t o_addr = tmem + lane_addr + C::kTmO + t * D;
    const float sl2 = p.scale_log2;
    // O rows start on 32-byte boundaries: whole-sector stores
    const bool o32 = (reinterpret_cast<uintptr_t>(p.O) & 31) == 0 && (s.D & 15) == 0;
    int sc = 0, oc = 0;  // s_full and o_done phases this tile has waited for
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int u = sched_next(&bars->sched, seq, ctl, kCode);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= nunits) break;
      const Fwd2Unit w = fwd2_unit(s, pack, u);
      const int q = t ? w.q_b : w.q_a;
      const int h = t ? w.h_b : w.h_a;
      const int row = q * kBM + r;
      int vis_lo, vis_hi;  // keys this row sees
      visible_keys(s.T, s.Tk, s.causal, s.window, row, vis_lo, vis_hi);
      const int lo_own = t ? w.lo_b : w.lo_a;
      const int nb = (t ? w.hi_b : w.hi_a) - lo_own + 1;  // 0 for a tile past the end
      float m_run = -CUDART_INF_F;  // reference max, log2 domain
      float l_run = 0.f;
      for (int j = 0; ok && j < nb; ++j) {
        const int kb = lo_own + j;
        if (!(ok = warp_wait(&bars->s_full[t], sc & 1, ctl, kCode))) break;
        ++sc;
        tc_fence_after();
        // The masking pre-pass stays rolled over 32-column chunks: unrolled with
        // everything else, this softmax did not fit the instruction cache next
        // to the other roles and ran several times slower.
        if (block_needs_mask(s.T, s.Tk, kBM, kBN, s.causal, s.window, q, kb)) {
          // rare (diagonal, window-edge and tail blocks): -inf over the masked
          // scores in TMEM, so that both passes below stay mask-free
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t ra[32];
            tmem_ld32(s_addr + c4 * 32, ra);
            tmem_ld_wait(ra);
            // this row's visible keys, relative to the chunk
            const int a = vis_lo - (kb * kBN + c4 * 32), z = vis_hi - (kb * kBN + c4 * 32);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < a || c > z) ra[c] = __float_as_uint(-CUDART_INF_F);
            tmem_st32(s_addr + c4 * 32, ra);
          }
          tmem_st_wait();
        }
        // One TMEM round trip per block: the row's 128 scores stay in registers
        // for both passes (re-reading them for pass 2 cost two more load
        // latencies on the softmax's critical path).
        // pass 1 rides on the loads: each 32-column load also returns the
        // maximum of its values (sm_103a load-with-reduction)
        uint32_t s0[32], s1[32], s2[32], s3[32];
        float m0, m1, m2, m3;
        tmem_ld32_max(s_addr, s0, m0);
        tmem_ld32_max(s_addr + 32, s1, m1);
        tmem_ld32_max(s_addr + 64, s2, m2);
        tmem_ld32_max(s_addr + 96, s3, m3);
        tmem_ld_wait(s0);
        reg_tie(s1);
        reg_tie(s2);
        reg_tie(s3);
        reg_tie4(m0, m1, m2, m3);
        float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        mx *= sl2;  // scale > 0, so the max commutes with the scaling
        const float m_new = fmaxf(m_run, mx);
        const bool first = (j == 0);
        const bool resc = !first && (m_new - m_run > kRescaleThreshold);
        const float m_ref = (first || resc) ? m_new : m_run;
        const float m_use = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;
        // pass 2: P = 2^(S*scale*log2e - m), row sum, bf16 pairs into the first
        // 64 columns of S_t.  Paired fp32: (x0, x1) = (s0, s1)*scale*log2e
        // - (m, m) in one instruction; the sum in two packed partials.
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t sum2[2] = {0ull, 0ull};
        // 32 scores -> 16 packed columns of P, stored as soon as they are formed
        // so that each quarter's registers free up for the next
        auto exp_quarter = [&](const uint32_t(&a)[32], uint32_t col) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x01 =
                f2_fma(f2_pack(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1])), sl2x2, negm2);
            float x0, x1;
            f2_unpack(x01, x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
            pk[e] = pack2<F16>(p0, p1);
          }
          tmem_st16(s_addr + col, pk);
        };
        exp_quarter(s0, 0);
        exp_quarter(s1, 16);
        if (!first && __any_sync(0xffffffffu, resc)) {
          // O_t holds P_0..P_{j-1} V, complete since S_t(j) is (in-order
          // pipe); rescaled before the first half of P is released to PV_t(j)
          const float corr = resc ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ro[32];
            tmem_ld32(o_addr + c * 32, ro);
            tmem_ld_wait(ro);
#pragma unroll
            for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * corr);
            tmem_st32(o_addr + c * 32, ro);
          }
          if (resc) l_run *= corr;
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->p_half[t]);
        exp_quarter(s2, 32);
        exp_quarter(s3, 48);
        tmem_st_wait();
        float a0, a1;
        f2_unpack(f2_add(sum2[0], sum2[1]), a0, a1);
        if (first || resc) m_run = m_new;
        l_run += a0 + a1;
        tc_fence_before();
        warp_arrive(&bars->p_full[t]);
      }
      if (!ok || nb == 0) continue;
      if (!(ok = warp_wait(&bars->o_done[t], oc & 1, ctl, kCode))) break;
      ++oc;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint16_t* orow = static_cast<uint16_t*>(p.O) + ((static_cast<size_t>(w.b) * s.T + row) * s.H + h) * s.D;
      // the whole O row in one TMEM round trip (the scores' registers are
      // free again), so that the next unit's softmax starts sooner
      uint32_t ro[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(o_addr + c * 32, ro[c]);
      tmem_ld_wait(ro[0]);
#pragma unroll
      for (int c = 1; c < D / 32; ++c) reg_tie(ro[c]);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<F16>(__uint_as_float(ro[c][2 * e]) * inv, __uint_as_float(ro[c][2 * e + 1]) * inv);
        if (row < s.T) {
          if (o32) {  // 32-byte stores: one whole sector per store
#pragma unroll
            for (int v = 0; v < 2; ++v)
              if (c * 32 + v * 16 < s.D) st_global_v8(orow + c * 32 + v * 16, pk + 8 * v);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)  // columns past a head dim below D are not stored
              if (c * 32 + v * 8 < s.D) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      if (row < s.T) {
        const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : 0.f;
        p.LSE[(static_cast<size_t>(w.b) * s.H + h) * s.T + row] = lse;
      }
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

template <int D, bool F16>
cudaError_t launch_fwd2_d(const TensorMaps& tm, const FwdParams& p, cudaStream_t stream) {
  using C = Fwd2Cfg<D>;
  static std::atomic<unsigned long long> attr_set{0};
  const void* kfn = reinterpret_cast<const void*>(fa_fwd2_bf16_kernel<D, F16>);
  if (cudaError_t e = set_smem_once(kfn, C::kSmemBytes, attr_set); e != cudaSuccess) return e;
  const int units = fwd2_units(p.s, p.pack_heads != 0);
  const dim3 grid(imax(1, imin(p.ctas, units)));
  fa_fwd2_bf16_kernel<D, F16><<<grid, kThreads2, C::kSmemBytes, stream>>>(tm.q, tm.k, tm.v, p);
  return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_fwd_d(const TensorMaps& tm, const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  static std::atomic<unsigned long long> attr_set{0};
  const void* kfn = reinterpret_cast<const void*>(fa_fwd_bf16_kernel<D, F16>);
  if (cudaError_t e = set_smem_once(kfn, C::kSmemBytes, attr_set); e != cudaSuccess) return e;
  dim3 grid(ceil_div(p.s.T, kBM), p.s.H, p.s.B);
  fa_fwd_bf16_kernel<D, F16><<<grid, kThreads, C::kSmemBytes, stream>>>(tm.q, tm.k, tm.v, p);
  return cudaGetLastError();
}

}  // namespace

template <bool F16>
cudaError_t launch_fwd_t(const TensorMaps& tm, const FwdParams& p0, cudaStream_t stream) {
  const int mode = fwd_mode(p0.s);
  const bool two = mode >= 2;
  FwdParams p = p0;
  p.pack_heads = mode == 3;
  // head dims up to 64 run the 64-wide kernels, up to 128 the 128-wide ones
  if (p.s.D <= 64) return two ? launch_fwd2_d<64, F16>(tm, p, stream) : launch_fwd_d<64, F16>(tm, p, stream);
  if (p.s.D <= 128) return two ? launch_fwd2_d<128, F16>(tm, p, stream) : launch_fwd_d<128, F16>(tm, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_bf16(const TensorMaps& tm, const FwdParams& p, cudaStream_t stream) {
  return p.f16 ? launch_fwd_t<true>(tm, p, stream) : launch_fwd_t<false>(tm, p, stream);
}

}  // namespace fa
