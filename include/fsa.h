/*
 * fsa.h -- frame-aligned block-sparse attention with a norm-bound softmax, for B300 (sm_103a).
 *
 * What it computes.  Tokens are F frames x T tokens per frame (N = F*T per head).
 * A query in frame f attends every key whose frame g satisfies |f - g| <= w, or
 * g == ref (one global reference frame); the window is clipped at the sequence
 * ends and the reference frame is counted once.  For every head h and query
 * row i the library returns
 *     out[h][i] = softmax_j( c <q_i, k_j> ) v_j   over the attended keys j,
 *     lse[h][i] = ln sum_j exp( c <q_i, k_j> ),   c = 1/sqrt(D),
 * which is exactly masked softmax attention over those frame pairs.
 * Source: "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU"
 * (aihot.vn), section "Xoa bo mat na" (window + reference frame, block size a
 * multiple of 16 that divides a frame, Fig. 3) and section "Giai phong Softmax"
 * (fixed per-row upper bound from precomputed norms instead of a running max,
 * per-head fallback to the running max inside the same kernel, optional mean-centred
 * keys, Fig. 4).  fsa_prep also prepares q, k, v from the hidden states in one fused
 * pass (section "Bo cuc la ABI", Fig. 5).
 *
 * Layouts (all row-major, contiguous, caller-owned device memory):
 *   q, k, v   bf16 [H][N][D], passed as 16-bit patterns (uint16_t), 16-byte aligned
 *   out       fp32 [H][N][D]
 *   lse       fp32 [H][N]   (natural log)
 *   qnorm     fp32 [H][N],  kmax fp32 [H][F],  bound fp32 [H][N],  eligible uint8 [H]
 *   x         bf16 [N][d_model] and w bf16 [3*H*D][d_model] (fsa_prep only)
 * D must be 64 or 128.  H*N must stay below 2^31.
 *
 * Streams: every device call is asynchronous on the given stream (a cudaStream_t
 * passed as void*; NULL = legacy default stream).  Nothing synchronises the host
 * except fsa_plan_destroy and the first device use of a plan (see fsa_plan).
 *
 * Errors: every call returns an int status (fsa_status) and never throws.  Invalid
 * arguments are rejected before any device work is enqueued.
 */
#ifndef FSA_H_
#define FSA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fsa_plan_s* fsa_plan_t; /* opaque, library-owned */

enum fsa_mode {
    FSA_MODE_NORM_BOUND = 0, /* fixed per-row bound; heads that fail eligibility fall back */
    FSA_MODE_ONLINE_MAX = 1  /* running max with accumulator rescale on every head */
};

enum fsa_status {
    FSA_OK = 0,
    FSA_ERR_INVALID_ARG = -1, /* bad shape, null pointer, block does not tile the frames */
    FSA_ERR_UNSUPPORTED = -2, /* D not in {64,128}, device is not sm_103, plan shape not handled */
    FSA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
    FSA_ERR_TIMEOUT = -4,     /* a bounded device-side wait gave up (reported via fsa_stats_t) */
    FSA_ERR_SCRATCH_LIMIT = -5 /* fsa_norms_noalloc: the problem needs more than its fixed scratch */
};

/* Device-side statistics, written by fsa_forward_ex and fsa_prep when the caller passes a
 * device pointer to one of these.  The call zeroes it first (on the stream). */
typedef struct fsa_stats {
    int32_t error;          /* 0, or FSA_ERR_TIMEOUT if a bounded wait inside a kernel gave up */
    int32_t timeout_site;   /* diagnostic: which wait gave up (0 if none) */
    int32_t fallback_heads; /* heads run with the running max although norm_bound was requested */
    int32_t items_done;     /* attention work items (128-row query tiles of one head) completed */
    int64_t underflow_rows; /* rows whose bound gap is >= 126 ln 2 (known only where the row max is
                               tracked and a bound is available) or whose row sum underflowed */
    int64_t pairs_visited;  /* coverage: sum over completed work items of (valid query rows) x
                               (keys the item's tiles consumed); a complete call visits every
                               active block pair once, H * nnz * block^2 */
} fsa_stats_t;

/*
 * fsa_plan -- build the frame-aligned active block list (host only, no device work).
 * Source: aihot.vn page above, section "Xoa bo mat na" and Fig. 3: with a block size
 * that is a multiple of 16 and divides T, every block pair is fully inside the mask
 * or fully outside it, so no tile needs a mask predicate or padding.
 *   F >= 1 frames, T >= 16 tokens per frame, w >= 0 window half-width in frames,
 *   0 <= ref < F reference frame, block: multiple of 16 dividing T.
 * The plan holds the block CSR (query blocks ascending, key blocks ascending within a
 * row) and the per-frame key runs the kernel walks.  *out receives a new plan on
 * FSA_OK and is untouched otherwise.  Device data (the work list and a workspace for
 * the norms) is created lazily by the first fsa_norms / fsa_forward* call on the
 * then-current device, which allocates device memory and therefore should come
 * before any stream capture.  A plan must not be used from two streams at once.
 * Errors: FSA_ERR_INVALID_ARG for out == NULL, a bad shape, or F*T >= 2^31.
 */
int fsa_plan(int F, int T, int w, int ref, int block, fsa_plan_t* out);

/* Free a plan and its device data (synchronises the device if it holds any). NULL is a no-op. */
void fsa_plan_destroy(fsa_plan_t plan);

/*
 * fsa_plan_export -- copy the block CSR to host memory.
 *   row_ptr: int32 [N/block + 1] or NULL;  col_idx: int32 [nnz] or NULL;  nnz: int64 out or NULL.
 * Call once with NULL arrays to learn nnz.  Host only.
 */
int fsa_plan_export(fsa_plan_t plan, int32_t* row_ptr, int32_t* col_idx, int64_t* nnz);

/*
 * fsa_plan_set_tau -- eligibility threshold (nats) on the per-head gap bound used by
 * norm_bound mode.  A head is eligible for the fixed bound iff for all its rows
 *     c ( ||q_i|| Kmax_S(f) - <q_i, kbar_S(f)> ) <= tau,
 * an upper bound on (bound - row max) because the max logit is at least the mean
 * logit.  The pages check eligibility per head but give no criterion or number;
 * the default is 64 (exp(-64) stays far above the fp32 normal range).  tau > 0.
 */
int fsa_plan_set_tau(fsa_plan_t plan, float tau);

/*
 * fsa_plan_set_key_tile -- keys per tensor-core tile: 0 = automatic (128, the kernel's
 * largest, the width of its S buffers in TMEM, and the fastest measured), else a multiple of
 * 16 in [16, 128].  Every key run (a whole number of frames) is cut into tiles of this many
 * keys and one last narrower tile of the rest (a multiple of 16, since T is); no tile is
 * partially masked.  Results are bitwise independent of `block`; they may change in the last
 * bits with the key tile (summation order).
 * Errors: FSA_ERR_INVALID_ARG for a NULL plan or a key tile outside that set.
 */
int fsa_plan_set_key_tile(fsa_plan_t plan, int key_tile);

/*
 * fsa_plan_set_center_keys -- mean-centred key norms in the bound (on = 1) or not (0, the
 * default).  Source: aihot.vn page above, "Giai phong Softmax": keys share a large common
 * component, so measuring their norms about the key mean tightens the bound, and the
 * softmax is invariant to the shift.  With on = 1, per head h
 *     mu_h         = mean of all N keys of head h
 *     kmax[h][g]   = max over keys n of frame g of ||k_{h,n} - mu_h||
 *     bound[h][n]  = c * (qnorm[h][n] * max_{g in S(frame(n))} kmax[h][g] + <q_{h,n}, mu_h>)
 * and the eligibility statistic is bound - c <q_i, kbar_S(f)> as without centring.  The
 * bound is still an upper bound on the uncentred logits, so out and lse mean the same in
 * both settings.  It costs a second read of K in fsa_norms / fsa_norms_noalloc.
 * Errors: FSA_ERR_INVALID_ARG for a NULL plan or on not in {0, 1}.
 */
int fsa_plan_set_center_keys(fsa_plan_t plan, int on);

/*
 * fsa_norms -- the precomputed norm arrays of the bound.
 * Source: aihot.vn page above, section "Giai phong Softmax": by Cauchy-Schwarz the
 * largest logit of a query is at most its norm times the largest key norm; a small
 * array of precomputed norms lets every row fix its bound when it starts.
 *   qnorm[h][n]  = ||q_{h,n}||                                (fp32 sum of bf16 squares)
 *   kmax[h][g]   = max over keys n of frame g of ||k_{h,n}||
 *   bound[h][n]  = c * qnorm[h][n] * max_{g in S(frame(n))} kmax[h][g]
 *   (kmax and bound take their centred forms when fsa_plan_set_center_keys is on)
 *   eligible[h]  = 1 iff the head passes the tau test of fsa_plan_set_tau
 * q, k: device bf16 [H][N][D].  Any output pointer may be NULL (the value is then kept
 * only in the plan's workspace).  Uses plan-owned workspace (per-frame key sums).
 * Errors: FSA_ERR_INVALID_ARG (q/k NULL, H < 0), FSA_ERR_UNSUPPORTED (D, device),
 * FSA_ERR_CUDA (launch or allocation failure).  H == 0 is a no-op.
 */
int fsa_norms(const uint16_t* q, const uint16_t* k, int H, int D, fsa_plan_t plan,
              float* qnorm, float* kmax, float* bound, uint8_t* eligible, void* stream);

/*
 * fsa_forward -- frame-aligned sparse attention, one pass over window + reference frame.
 * Source: aihot.vn page above, "Xoa bo mat na" (single pass, no masks, no merge) and
 * "Giai phong Softmax" (norm-bound softmax with per-head in-kernel fallback).
 *   mode FSA_MODE_NORM_BOUND: runs fsa_norms into the plan's workspace, then the
 *        attention kernel with p = exp(s - bound_i) (no running max, no rescale) on
 *        eligible heads and the running max on the others;
 *   mode FSA_MODE_ONLINE_MAX: the attention kernel with a running max on every head.
 * q, k, v device bf16 [H][N][D]; out device fp32 [H][N][D]; lse device fp32 [H][N].
 * Errors as fsa_norms, plus FSA_ERR_INVALID_ARG for a bad mode or NULL tensor.
 */
int fsa_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse,
                int H, int D, fsa_plan_t plan, int mode, void* stream);

/*
 * fsa_forward_ex -- fsa_forward with caller-supplied norms and optional diagnostics.
 *   bound, eligible: device arrays as produced by fsa_norms (both or neither).  When
 *        given, the norms pass is skipped and these are used as they are; when NULL in
 *        norm_bound mode, fsa_norms runs into the plan's workspace first.
 *   rowmax: optional device fp32 [H][N]; rows that ran with the running max receive
 *        their max logit c <q_i, k_j> (natural units), rows that ran with the fixed
 *        bound receive NaN (they never form the max).
 *   dev_stats: optional device fsa_stats_t, zeroed by this call, then filled by the
 *        kernels (timeouts, fallback heads, underflow rows).
 */
int fsa_forward_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse,
                   int H, int D, fsa_plan_t plan, int mode,
                   const float* bound, const uint8_t* eligible, float* rowmax,
                   fsa_stats_t* dev_stats, void* stream);

/*
 * fsa_forward_host -- fsa_forward on host tensors, with the copies overlapped.
 * The pages have no counterpart (their pipeline keeps activations on the accelerator); this
 * is the library's end-to-end entry for callers whose q, k, v live in host memory.  The
 * heads are split into chunks of heads_per_chunk heads (0 = automatic, about eight
 * chunks).  Chunk c is copied to the device on one stream, computed (fsa_norms in
 * norm_bound mode, then the attention) on a second, and its out and lse are copied back on
 * a third, so the host-to-device copy of chunk c+1, the compute of chunk c and the
 * device-to-host copy of chunk c-1 run at the same time.  Heads are independent, so the
 * results equal those of fsa_forward on device copies of the same tensors, bit for bit.
 *   q, k, v: host bf16 [H][N][D]; out: host fp32 [H][N][D]; lse: host fp32 [H][N].  Page-locked
 *   (pinned) host memory is needed for the copies to overlap; pageable memory works but
 *   serialises them.
 *   The pipeline starts after the work already queued on `stream` and `stream` waits for its
 *   end: synchronise `stream` before reading out and lse.  The host buffers must stay valid
 *   and unchanged until then.
 *   The plan keeps device copies of the whole problem (3 x H*N*D bf16 + H*N*D and H*N fp32),
 *   three streams and the events, grown on the first call for a given size (cudaMalloc: make
 *   that call before any stream capture) and freed by fsa_plan_destroy.
 * Errors as fsa_forward, plus FSA_ERR_INVALID_ARG for heads_per_chunk < 0.  A CUDA error in
 * the middle returns FSA_ERR_CUDA with earlier chunks possibly still in flight.
 */
int fsa_forward_host(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse,
                     int H, int D, fsa_plan_t plan, int mode, int heads_per_chunk, void* stream);

/*
 * fsa_forward_masked -- the same attention, computed the way a general block-sparse kernel
 * with a mask computes it: the comparison point for the frame-aligned layout.
 * Source: aihot.vn page above, section "Xoa bo mat na", and the bib.com.ua page "HeyGen
 * pryskoryla Avatar IV na TPU u 1,86 raza" (its section on the sparse-attention mask): they
 * describe the state the frame-aligned kernel replaced: blocks of a multiple of 128 tokens over a sequence padded
 * to a whole number of blocks, element-wise mask predicates on the blocks a frame boundary cuts,
 * and the window and the reference frame run as two passes whose partial results a third pass
 * merges.  This entry point does exactly that on B300:
 *   pass 0: query blocks and key blocks of `block` tokens; a query block visits every key block
 *     that meets the union of its rows' windows [f - w, f + w] (clipped to [0, F)); keys outside
 *     a row's own window are masked by predicate on the tiles the interval cuts;
 *   pass 1: the query blocks that hold a row whose window leaves out the reference frame visit
 *     the key blocks of the reference frame; rows whose window holds it see no key there;
 *   merge: rows whose window leaves out the reference frame combine the two softmax results
 *     through their log-sum-exps; pass 1 writes its fp32 partial out and lse to plan-owned
 *     buffers (H*N*D + H*N floats, grown on first use).
 * Both passes run the running-max softmax (the pages' comparison state has no norm bound), on
 * the same persistent tcgen05 kernel as fsa_forward (128-row query tiles, 128-key tiles).  The
 * result is the attention fsa_forward computes, up to rounding.
 *   q, k, v, out, lse, H, D, stream: as fsa_forward.  plan: its F, T, w and ref are used (its
 *   block size is not).  block: a multiple of 128 from 128 to 1024.  dev_stats: optional, as in
 *   fsa_forward_ex (items_done and pairs_visited count both passes, masked pairs included).
 *   The item tables of the last block size used are kept in the plan.
 * Errors as fsa_forward, plus FSA_ERR_INVALID_ARG for a block size outside that set.
 */
int fsa_forward_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse,
                       int H, int D, fsa_plan_t plan, int block, fsa_stats_t* dev_stats, void* stream);

/*
 * fsa_prep -- the attention's inputs from the hidden states, in one fused pass.
 * Source: aihot.vn page above, "Bo cuc la ABI", Fig. 5: normalisation, rotary embeddings,
 * projection and head packing fused into one kernel that writes exactly the layout the next
 * step reads (no repacking copies in between).  Readings of this library:
 *   xhat = x / sqrt(mean_c x_c^2 + 1e-6)            (RMS norm over d_model, no gain: fold a
 *                                                   gain into w)
 *   y    = xhat w^T                                 (w rows: q heads, then k, then v)
 *   q, k of every head rotated at position n (the token index): pairs (i, i + D/2) turned
 *        by n * 10000^(-2i/D); v not rotated
 *   q, k, v written as bf16 [H][N][D], the layout fsa_forward* read.
 * The projection's epilogue also produces the norms of fsa_norms for these q and k (from
 * the bf16 values written), so no separate pass re-reads them:
 *   qnorm[h][n], kmax[h][g], bound[h][n], eligible[h]   as in fsa_norms.
 *   x: device bf16 [N][d_model] (N = F*T of the plan), d_model a multiple of 64;
 *   w: device bf16 [3*H*D][d_model];  q, k, v: device bf16 [H][N][D] outputs;
 *   qnorm (may be NULL), kmax, bound, eligible: device outputs, or NULL to keep them in the
 *   plan's workspace;  dev_stats: optional, as in fsa_forward_ex (a bounded wait that gave
 *   up records FSA_ERR_TIMEOUT there).
 * All pointers 16-byte aligned.  Uses and may grow plan-owned workspace; the first call builds
 * the plan's rotary table (N*D/2 (cos, sin) pairs) on the host and uploads it (again if D changes).
 * Errors: FSA_ERR_INVALID_ARG (NULL or misaligned tensor, bad d_model), FSA_ERR_UNSUPPORTED
 * (D not 64 or 128, H*D not a multiple of 256, mean-centred keys on the plan, device),
 * FSA_ERR_CUDA.  H == 0 is a no-op.
 */
int fsa_prep(const uint16_t* x, const uint16_t* w, int d_model, int H, int D, fsa_plan_t plan,
             uint16_t* q, uint16_t* k, uint16_t* v, float* qnorm, float* kmax, float* bound,
             uint8_t* eligible, fsa_stats_t* dev_stats, void* stream);

/*
 * fsa_norms_noalloc -- fsa_norms for callers that cannot allocate device memory.
 * The pages have no counterpart; this is a service of the library.  fsa_norms keeps its
 * scratch (per-frame key sums, per-head maxima) in a plan workspace grown with cudaMalloc,
 * and its first call uploads the plan's work list.  Engines that hand out all device memory
 * themselves, and loops that cannot take the device synchronisation of cudaMalloc/cudaFree,
 * need a call that allocates nothing: this one keeps that scratch in a fixed 2 MiB device array
 * compiled into the library (every GPU that loads the library holds it until the process
 * exits).  On every call it zeroes the array's counters (a small memset on `stream`) and writes
 * the plan's key runs into it with a small kernel that takes them as launch arguments, so no
 * host buffer is read on the stream.
 *   Arguments and results are those of fsa_norms, except that kmax, bound and eligible are
 *   required (they are the outputs; qnorm may be NULL).
 *   Limit: with C = min(8, max(1, T/256)) key chunks per frame, (H*F + 2*H)*4 + F*5*4 + H*F*D*4 +
 *   H*F*C*D*4 + H*F*C*4 + H*4 + H*D*4 bytes (each part rounded up to 256) must fit in 2 MiB, e.g.
 *   H=24, F=24, T=1200, D=128 uses 1.4 MiB; larger problems return FSA_ERR_SCRATCH_LIMIT
 *   before any device work.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current and remembers it together with the device's CUDA context; a
 *   later call in a different context (after cudaDeviceReset, for instance) looks it up again.
 *   Every call shares the one array and overwrites what the previous call left there, so
 *   calls whose work overlaps on the GPU (different streams, or different host threads) race;
 *   serialise them.
 *   Calls no cudaMalloc, cudaFree or other allocating routine.
 */
int fsa_norms_noalloc(const uint16_t* q, const uint16_t* k, int H, int D, fsa_plan_t plan,
                      float* qnorm, float* kmax, float* bound, uint8_t* eligible, void* stream);

/*
 * fsa_last_cuda_error -- the code of the last CUDA call that failed inside this library on the
 * calling host thread (a cudaError_t value; driver CUresult values are returned plus 100000),
 * or 0; reading it clears it.  Diagnostic companion of FSA_ERR_CUDA.  Host only.
 */
int fsa_last_cuda_error(void);

/* Human-readable name of a status code (static storage). */
const char* fsa_status_string(int status);

/*
 * fsa_selftest_wait_timeout -- checks the bounded-wait path without faulting the GPU.
 * Launches one tiny kernel whose only thread waits, through the same bounded mbarrier
 * wait the attention kernel uses, on a barrier nothing arrives at, with a limit of
 * limit_cycles SM clock cycles.  *status receives the code the kernel reported
 * (FSA_ERR_TIMEOUT when the wait gave up as designed).  Synchronises the stream.
 */
int fsa_selftest_wait_timeout(long long limit_cycles, int32_t* status, void* stream);

/*
 * fsa_selftest_grid_timeout -- checks the bounded grid barrier of fsa_prep without faulting
 * the GPU.  Launches `ctas` CTAs of 256 threads (cooperatively, so all are resident; 1 <= ctas
 * <= the SM count) that meet at the same bounded grid barrier fsa_prep uses between its phases,
 * with a target of ctas + missing arrivals.
 *   missing = 0: the barrier opens; result = {0, 0, 0, ctas}.
 *   missing = 1: the barrier never opens; each CTA's waiting thread gives up after limit_cycles
 *   SM clock cycles and raises its CTA's abort flag, and the kernel reports
 *   result = {FSA_ERR_TIMEOUT, 16 (the grid-barrier site), ctas, ctas}.
 *   result (host, 4 int32): status reported by the kernel, wait site, CTAs whose abort flag was
 *   raised, arrivals counted at the barrier.  Synchronises the stream.
 *   Errors: FSA_ERR_INVALID_ARG for a NULL result, limit_cycles <= 0, missing not 0 or 1, or
 *   ctas out of range.
 */
int fsa_selftest_grid_timeout(long long limit_cycles, int ctas, int missing, int32_t* result, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FSA_H_ */
