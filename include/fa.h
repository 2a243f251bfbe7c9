/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused causal / sliding-window GQA
 * flash-attention library (libfa_gb300.so).
 *
 * What it computes.  For every batch b, query head h and query row i, with
 * KV head g = h / (H / HKV) (consecutive query heads share a KV head: forge
 * flash_attention.metal, kernel flash_attn_fwd, the `hkv` index):
 *
 *   S_ij  = scale * Q[b,i,h,:] . K[b,j,g,:]
 *   Visible(i, j) = (!causal || j <= i) && (window == 0 || i - j < window)
 *   P_ij  = softmax_j of S_i. over visible j        (0 where not visible)
 *   O[b,i,h,:]   = sum_j P_ij V[b,j,g,:]
 *   LSE[b,h,i]   = log sum_j exp(S_ij)  over visible j  (natural log)
 *
 * `window` counts the keys a query keeps, itself included, 0 meaning no
 * window (forge flash_attention.metal, struct FlashParams).  The forward is
 * the online-softmax recurrence (running max m, running sum l, rescale of O,
 * LSE = m + log l; Graphcore flash_attention_qkv_packed.cpp,
 * flashAttentionQKVPackedWithStash) and writes nothing of size T x T.  The
 * backward recomputes P block by block from LSE (forge flash_attention.metal,
 * flash_attn_bwd_dq / _dv / _dk; teeny-kernels flash_attn2.rs,
 * flash_attention2_backward_dq / _dkv):
 *
 *   dP_ij = dO_i . V_j ;  Delta_i = dO_i . O_i ;  dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_{h in group} sum_i dS_ij Q_i
 *   dV_j  =       sum_{h in group} sum_i P_ij dO_i
 *
 * Layouts (all row-major and contiguous, element type `dtype` unless noted):
 *   Q, O, dO, dQ : [B, T, H,   head_dim]
 *   K, V, dK, dV : [B, T, HKV, head_dim]
 *   LSE          : [B, H, T] float32 (always fp32, whatever `dtype` is)
 *
 * Memory and ownership.  Every pointer argument except those of
 * fa_plan_* is a DEVICE pointer owned by the caller.  The library allocates
 * no device memory and keeps no per-call state; it caches only the driver's
 * tensor-map encoder and a few device attributes.  Outputs are overwritten,
 * never accumulated into, so they need no clearing.
 *
 * Workspace.  Each call takes a caller-owned device workspace of at least
 * fa_workspace_size() bytes, 256-byte aligned.  Its first 256 bytes must be
 * zero before the first call (allocate the workspace zero-filled): they hold
 * the device error word (the first 4 bytes), which fa_check_status() reads
 * and sets back to zero, and the work counters of the persistent kernels,
 * which every launch leaves at zero again.  The backward also keeps
 * Delta = rowsum(dO * O), [B, H, T] fp32, in the workspace.  Calls that share
 * a workspace must be ordered (same stream).
 *
 * Streams.  Every launch goes onto `stream` (a cudaStream_t; NULL = the
 * legacy default stream) and returns without synchronising.
 *
 * Errors.  Return values are fa_status codes.  A call that fails host-side
 * validation returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED and launches
 * nothing.  Launch failures return FA_ERR_CUDA.  Kernels never trap and never
 * wait without bound: a pipeline wait that exceeds its time budget makes the
 * kernel set the error word and exit, which fa_check_status() reports as
 * FA_ERR_TIMEOUT.
 *
 * Supported: dtype FA_DTYPE_BF16 or FA_DTYPE_FP16 (tcgen05 tensor-core
 * kernels, fp32 accumulation; P and dS are rounded to the input type before
 * their MMAs; head_dim 16 to 128 in steps of 8) or FA_DTYPE_FP32 (fp32
 * CUDA-core kernels; head_dim 64 or 128); any B, T, H, HKV >= 1 with
 * H % HKV == 0; scale > 0 and finite; window >= 0; 16-byte aligned tensor
 * pointers.  No fallback path exists: an unsupported shape is an error.
 *
 * Cross-attention (fa_fwd_cross, fa_bwd_cross): Tq query rows attend to Tk
 * key rows, Tk != Tq allowed, K/V/dK/dV then [B, Tk, HKV, head_dim] and
 * Q/O/dO/dQ/LSE sized by Tq.  Every key is visible to every query (the
 * teeny-kernels page's flash_attn2.rs forward takes n_ctx_q and n_ctx_k and
 * masks nothing); causal and window masking are defined here only for
 * Tq == Tk (fa_fwd, fa_bwd).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale */
  FA_ERR_UNSUPPORTED = 2,  /* valid but unsupported head_dim / dtype / device */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 4,      /* a kernel wait ran out of budget (device error word) */
  FA_ERR_WORKSPACE = 5     /* workspace missing, too small or misaligned */
} fa_status;

typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP32 = 1, FA_DTYPE_FP16 = 2 } fa_dtype;

typedef enum { FA_OP_FWD = 0, FA_OP_BWD = 1, FA_OP_BWD_FUSED = 2 } fa_op;

/*
 * Bytes of device workspace for this shape: fa_fwd (op = FA_OP_FWD) takes
 * 256 bytes, for the error word and the persistent kernels' work counters;
 * fa_bwd and its stages (FA_OP_BWD) also B*H*T floats of Delta (rounded up to
 * 256 bytes); the fused backward fa_bwd_dkdv_dq (FA_OP_BWD_FUSED, 16-bit
 * elements with head_dim <= 64 only, else 0) also its fp32 dQ accumulator
 * (B*T*H*head_dim floats) and turn counters (B*H*ceil(T/128) words), each
 * rounded up to 256 bytes.  A FA_OP_BWD_FUSED workspace serves every
 * backward entry point.  Returns 0 for sizes that are out of range.
 */
size_t fa_workspace_size(int op, int B, int T, int H, int HKV, int head_dim, int dtype);

/*
 * Forward: O and LSE from Q, K, V (see the top of this file).
 *   Q [B,T,H,D], K/V [B,T,HKV,D] in `dtype`; O [B,T,H,D] in `dtype`;
 *   LSE [B,H,T] fp32; workspace >= fa_workspace_size(FA_OP_FWD, ...).
 */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
           int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window,
           int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: dQ, dK, dV from Q, K, V, the forward's O and LSE, and dO.
 * Runs three kernels in stream order: Delta = rowsum(dO * O) into the
 * workspace, then dK/dV (every KV block accumulated privately by one unit of
 * work, no atomics), then dQ (every query block by one unit, fixed order, no
 * atomics), so the result is bitwise reproducible.  dQ reads nothing dK/dV
 * writes, so it is launched as a programmatic dependent of dK/dV (16-bit
 * types): its CTAs start on the SMs the dK/dV kernel leaves idle, and it
 * completes only after dK/dV has, so work queued after fa_bwd sees all three
 * gradients.  The results are the same bits as the three stage calls.
 * (fa_bwd_dkdv_dq is the alternative second stage that forms dQ without
 * recomputing S and dP.)
 *   O, LSE: exactly what fa_fwd produced for the same inputs.
 *   workspace >= fa_workspace_size(FA_OP_BWD, ...).
 */
int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
           const void* dO, void* dQ, void* dK, void* dV,
           int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window,
           int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages of fa_bwd, callable one by one (fa_bwd runs these kernels
 * in this order on `stream`, the dQ one as a programmatic dependent of the
 * dK/dV one; called one by one they run in plain stream order, with the same
 * results bit for bit).  Same arguments and layouts as
 * fa_bwd; the workspace carries Delta from the first stage to the other two,
 * so all three must get the same workspace and be stream-ordered.
 *   fa_bwd_preprocess: Delta = rowsum(dO * O) into the workspace (HBM-bound).
 *   fa_bwd_dkdv:       dK, dV (one unit of work per KV block, no atomics).
 *   fa_bwd_dq:         dQ (one unit of work per query block, fixed order, no atomics).
 */
int fa_bwd_preprocess(const void* O, const void* dO, int B, int T, int H, int HKV, int head_dim, int dtype,
                      void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_dkdv(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dK, void* dV,
                int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
                void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_dq(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ,
              int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The fused second stage of the backward (Graphcore
 * flash_attention_qkv_packed.cpp, flashAttentionQKVPackedGrad: dQ_i += dS K_j
 * written back in the same pass over KV blocks that produces dK and dV):
 * dK, dV and dQ in one persistent, cooperatively launched kernel, after
 * fa_bwd_preprocess.  Every (KV block, KV head, batch) unit forms, besides
 * its dK/dV contribution, the dQ partial dS K of each query block it sees and
 * adds it into the workspace's fp32 accumulator once the partials of the KV
 * blocks above it are in (a turn counter per query block; the diagonal block
 * first), so the sum has a fixed order; the last partial of a query block
 * writes dQ = scale * accumulator in the element type.
 *   Shapes: 16-bit elements, head_dim <= 64, causal = 1, any window; else
 *   FA_ERR_UNSUPPORTED.  workspace >= fa_workspace_size(FA_OP_BWD_FUSED,
 *   ...), else FA_ERR_WORKSPACE; its turn counters are cleared by a memset
 *   on `stream` before the launch.  A turn wait is bounded like every kernel
 *   wait (FA_ERR_TIMEOUT through fa_check_status, FA_DEVERR_DKDV_TIMEOUT in
 *   the error word).
 *   Speed: measured on GB300 it is slower than fa_bwd_dkdv + fa_bwd_dq (the
 *   recompute of S and dP costs less than handing every partial through
 *   memory in a fixed order, whose hops between SMs are serial per query
 *   block), so fa_bwd does not use it.
 */
int fa_bwd_dkdv_dq(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ, void* dK,
                   void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Cross-attention: fa_fwd / fa_bwd for Tq query rows over Tk key rows, no
 * mask (see the top of this file).
 *   Q, O, dO, dQ [B,Tq,H,D]; K, V, dK, dV [B,Tk,HKV,D]; LSE [B,H,Tq] fp32.
 *   Workspace: fa_workspace_size(op, B, Tq, H, HKV, head_dim, dtype) bytes
 *   (Delta has one row per query).  Tq = Tk gives exactly fa_fwd / fa_bwd
 *   with causal = 0, window = 0.  Same kernels, same errors and stream
 *   behaviour as fa_fwd / fa_bwd; Tq or Tk < 1 is FA_ERR_INVALID_ARG.
 */
int fa_fwd_cross(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int Tq, int Tk, int H, int HKV, int head_dim, float scale,
                 int dtype, void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_cross(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                 const void* dO, void* dQ, void* dK, void* dV,
                 int B, int Tq, int Tk, int H, int HKV, int head_dim, float scale,
                 int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_static_scratch: fa_bwd for callers that cannot allocate device
 * memory.  The source pages have no counterpart of this entry point; it
 * exists for the library's users.
 *
 * Who needs it: code that may not call cudaMalloc (or any allocating
 * routine) at the point where it runs the backward -- for example inside
 * another allocator's callback, in a plugin whose host program owns every
 * device allocation, or on a path that must not touch the allocator while a
 * CUDA graph is being built.  fa_bwd's workspace (the Delta rows and the
 * error word) is then out of reach, so this variant keeps that scratch in a
 * fixed device array inside the library itself.
 *
 *   Inputs and outputs: exactly those of fa_bwd, caller-owned device memory.
 *   Scratch: a static device array of 256 bytes plus
 *     FA_STATIC_SCRATCH_MAX_ROWS floats (16 MiB + 256 B).  Every GPU that
 *     loads the library holds these bytes until the process exits.
 *   Limit: B*H*T <= FA_STATIC_SCRATCH_MAX_ROWS; larger shapes return
 *     FA_ERR_WORKSPACE before anything is launched.
 *   err_word: optional caller-owned device pointer (4-byte aligned) that
 *     receives this call's device error word (0, or fa_device_error_bits
 *     when a kernel wait ran out of budget).  With NULL the word stays
 *     inside the library, where no caller can read it: a kernel that gave
 *     up on a wait then goes unreported and dQ, dK and dV may be partly
 *     unwritten.  Pass a word whenever the outputs matter.
 *   No allocation: the call makes no cudaMalloc/cudaFree or other allocating
 *     call; it only issues a 4-byte memset (clearing the error word, since
 *     the array keeps the previous call's contents), the three backward
 *     kernels, and, with err_word, a 4-byte device-to-device copy.
 *   Validation: every check of fa_bwd runs before anything is queued, so a
 *     call that fails it launches nothing.
 *   Set-up: the first call on each device looks the array's device address
 *     up with that device current (cudaGetSymbolAddress); make that first
 *     call before any stream capture.  The address is cached per device and
 *     context: after cudaDeviceReset (a new context, in which the array is
 *     loaded again) the next call looks it up afresh.
 *   Sharing: all calls share the one array per device, so calls whose work
 *     overlaps on the GPU (different streams, or threads racing on one
 *     device) race on it; order them on one stream.
 * Returns the same status codes as fa_bwd.
 */
#define FA_STATIC_SCRATCH_MAX_ROWS (4 * 1024 * 1024)
int fa_bwd_static_scratch(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                          const void* dO, void* dQ, void* dK, void* dV,
                          int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window,
                          int dtype, unsigned int* err_word, void* stream);

/*
 * Synchronises `stream`, reads the workspace's device error word, resets it
 * to zero and returns FA_OK, FA_ERR_TIMEOUT (a kernel gave up on a wait) or
 * FA_ERR_CUDA (the synchronisation itself failed).  If raw_word is not NULL
 * the word as read is stored there (bit flags, see fa_device_error_bits).
 */
int fa_check_status(void* workspace, void* stream, unsigned int* raw_word);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(int status);

/*
 * Host mirror of the kernels' tile scheduling, exported for tests.  For tile
 * sizes BM (query rows) x BN (key rows):
 *   fa_plan_kv_range: the KV blocks [*lo, *hi] query tile qb must visit
 *     (blocks wholly above the causal diagonal or wholly outside the window
 *     are skipped);
 *   fa_plan_q_range: the query tiles [*lo, *hi] that see KV block kb;
 *   fa_plan_block_mask: 1 if block (qb, kb) holds any element that is
 *     masked (not visible, or a row/key index >= T), so the per-element test
 *     must run; 0 if every element is visible; -1 for bad sizes.
 * The masked blocks of a causal schedule are the diagonal-crossing blocks of
 * the Graphcore page's triu-offset scheme (getTriuOffsetSequence); inside
 * block (qb, kb) element (r, c) is in the future iff c - r >= k with
 * k = qb*BM - kb*BN + 1.  The range functions return FA_ERR_INVALID_ARG
 * for bad sizes.
 */
int fa_plan_kv_range(int T, int BM, int BN, int causal, int window, int qb, int* lo, int* hi);
int fa_plan_q_range(int T, int BM, int BN, int causal, int window, int kb, int* lo, int* hi);
int fa_plan_block_mask(int T, int BM, int BN, int causal, int window, int qb, int kb);
/*
 * The per-element rule the kernels apply inside a block that needs a mask,
 * as index ranges (host memory outputs): fa_plan_row_keys gives the keys
 * [*lo, *hi] query row i sees, fa_plan_key_rows the query rows [*lo, *hi]
 * that see key j; empty (lo > hi) past the end of the sequence.  Tq query
 * rows, Tk key rows.  FA_ERR_INVALID_ARG for bad sizes.
 */
int fa_plan_row_keys(int Tq, int Tk, int causal, int window, int i, int* lo, int* hi);
int fa_plan_key_rows(int Tq, int Tk, int causal, int window, int j, int* lo, int* hi);

/*
 * Pre-attention prologue: RMS-norm of every query and key head vector of the
 * packed QK projection, then the rotary mix with per-position factors, as the
 * modded-nanogpt page qkv_rope.py defines it (`_qk_norm_rope_forward_kernel`,
 * without its paired-heads and key-offset options):
 *
 *   x = qk[t][c][:] ;  rstd = 1 / sqrt(mean_d x_d^2 + 2^-23) ;  n = rstd x
 *   y_d = f1[t][d] n_d + f2[t][d] n_(d xor 1)
 *
 * qk      [tokens][hq + hk][head_dim] 16-bit (dtype bf16 or fp16): heads
 *         c < hq are queries, the next hk are keys (hq = hk in the page; any
 *         hk >= 1 here, so that GQA keys can be produced).
 * f1, f2  [tokens][head_dim] fp32 rotary factors (cos / signed sin, or any).
 * q       [tokens][hq][head_dim], k [tokens][hk][head_dim], same dtype:
 *         with tokens = B*T these are the [B,T,H,D] / [B,T,HKV,D] tensors
 *         fa_fwd reads.
 * The backward (the norm/rotary part of the page's
 * `_qkv_norm_rope_pack_fp8_backward_kernel`, without the fp8 packing) takes
 * the gradients dq, dk of q and k and writes dqk, the gradient of qk:
 *   gn_e = f1[t][e] g_e + f2[t][e xor 1] g_(e xor 1)
 *   dx_e = rstd (gn_e - n_e mean_d(gn_d n_d))
 * head_dim 64 or 128; every pointer 16-byte aligned (else
 * FA_ERR_INVALID_ARG); fp32 arithmetic.  Asynchronous on `stream`; the
 * caller owns every buffer.
 */
int fa_qk_norm_rope_fwd(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens, int hq,
                        int hk, int head_dim, int dtype, void* stream);
int fa_qk_norm_rope_bwd(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2, void* dqk,
                        int tokens, int hq, int hk, int head_dim, int dtype, void* stream);

/*
 * The same prologue with its two options (the modded-nanogpt qkv_rope.py
 * page, `_qk_norm_rope_forward_kernel`, PAIRED and KEY_OFFSET branches, and
 * the norm/rotary part of `_qkv_norm_rope_pack_fp8_backward_kernel`), for a
 * projection with equally many query and key heads:
 *   qk [tokens][2*heads][head_dim]: heads 0..heads-1 are queries, the rest
 *   keys; logical head h = c mod heads.
 *   paired (heads even): f1, f2 [tokens][2*head_dim]; head h rotates with
 *     factor half h mod 2 and is written to token 2t + h / (heads/2), head
 *     h mod (heads/2) of q, k [2*tokens][heads/2][head_dim].
 *   key_offset: f1, f2 [tokens][head_dim]; q, k [tokens][heads][head_dim];
 *     a key row of token t > 0 takes dims d >= rotary_dim (even, 0..head_dim)
 *     from token t-1's normalised row of the same head, unrotated
 *     (y_d = x'_d / sqrt(mean(x'^2) + 2^-23)).  Token 0 and the queries are
 *     the plain prologue.
 *   Neither option: the plain prologue with hq = hk = heads (rotary_dim is
 *   ignored unless key_offset is set).
 * The backward is the exact gradient of this forward (for key offset, a key
 * row's stationary dims get the gradient of token t+1's key output, plus the
 * rotation term at t = 0); dq, dk have the forward's output shapes and dqk
 * the shape of qk.
 * Errors: both options, an odd head count with paired, or a bad rotary_dim
 * with key_offset: FA_ERR_INVALID_ARG; otherwise as fa_qk_norm_rope_fwd.
 */
int fa_qk_norm_rope_fwd_opt(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens,
                            int heads, int head_dim, int rotary_dim, int paired, int key_offset, int dtype,
                            void* stream);
int fa_qk_norm_rope_bwd_opt(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2,
                            void* dqk, int tokens, int heads, int head_dim, int rotary_dim, int paired, int key_offset,
                            int dtype, void* stream);

/* Tile sizes the bf16 kernels use (query rows, key rows per block). */
int fa_tile_m(void);
int fa_tile_n(void);

/*
 * Test hook.  wait_timeout_ns: budget of one pipeline wait inside a kernel
 * (0 = the default of 2 s).  inject_stall: 0 = none; 1, 2 or 3 = the next
 * launch of the 16-bit forward, dK/dV or dQ kernel withholds its first tile
 * loads, so that the kernel's waits run out of budget and it exits with the
 * device error word set (FA_DEVERR_FWD_TIMEOUT, _DKDV_ or _DQ_); the hook
 * clears itself at that launch.  FA_ERR_INVALID_ARG for other values.
 * Affects later calls of this process only.
 */
int fa_debug_config(unsigned long long wait_timeout_ns, int inject_stall);

/*
 * Test hook.  Query tiles per CTA of the 16-bit forward: 1 (one 128-row
 * tile), 2 (two 128-row tiles, adjacent query blocks of one head, sharing
 * every K/V block the CTA streams), 3 (two tiles, the same query block of
 * two query heads that share a KV head; needs an even H/HKV, else as 0) or 0
 * (automatic: 3 when H/HKV is even, else 2 when the sequence has at least
 * two query tiles, else 1).  All produce the same O and LSE up to fp32
 * rounding order.  Returns FA_ERR_INVALID_ARG for any other value.  Affects
 * later calls of this process only.
 */
int fa_debug_fwd_tiles(int tiles);

/*
 * Test hook.  The tensor-core forward (two-tile kernel) and both backward
 * kernels are persistent: they launch at most one CTA per SM and each CTA
 * walks a fixed share of the work units (query tiles, or KV blocks for
 * dK/dV), longest first.  ctas > 0 sets the CTAs launched (at most one per
 * work unit): fewer than the SMs sends several units through one CTA on
 * small shapes, more gives every unit a CTA of its own; 0 restores one per
 * SM.  Results do not depend on it.  FA_ERR_INVALID_ARG for ctas < 0.
 * Affects later calls of this process only.
 */
int fa_debug_max_ctas(int ctas);

/* Bit flags of the device error word (which wait gave up). */
typedef enum {
  FA_DEVERR_FWD_TIMEOUT = 1u << 0,
  FA_DEVERR_DKDV_TIMEOUT = 1u << 1,
  FA_DEVERR_DQ_TIMEOUT = 1u << 2,
  /* a kernel found its dynamic shared memory placed so that its tile layout
     does not fit, and did nothing (fa_check_status reports FA_ERR_TIMEOUT) */
  FA_DEVERR_LAYOUT = 1u << 3
} fa_device_error_bits;

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
