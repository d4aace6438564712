/*
 * moe_reader.h -- C ABI of the GB300 (sm_103a) calibration-free channel
 * reader for Mixture-of-Experts decoding.
 *
 * The reader replaces the routed-expert gated-MLP step of a decode token
 * ("Channel Selection for Mixture-of-Experts Decoding Needs No Calibration
 * Data"; Chinese summary page, sections 核心方法 and 方法步骤详情; Korean
 * summary page, section 어떻게 쓰나):
 *
 *   prepare (load time, weights only)
 *     - rotate every gate/up row in 128-coordinate blocks with a randomized
 *       Hadamard matrix R and store a ternary sketch per block: 2-bit codes,
 *       an FP16 scale and the FP16 block mean-squared error rho_b;
 *     - precompute the down-column norms ||d_j||;
 *     - take the top-r left singular vectors U of the layer's stacked down
 *       columns and store b_j = U^T d_j;
 *     - transpose every down projection so a kept channel's down weights are
 *       one contiguous row.
 *   decode (per token)
 *     - rotate x once; per block screen only the c largest-|Rx| coordinates;
 *     - score s_j = w_j ||d_j|| |phi(ghat_j) vhat_j| for every routed channel
 *       and keep the exact top-k over all routed experts together;
 *     - y = sum_{j in K} w_j phi(g_j^T x)(v_j^T x) d_j      (native BF16 rows)
 *         + U sum_{j in S} w_j b_j phi(ghat_j) vhat_j       (rank-r recovery).
 *
 * Conventions shared by every entry point
 *   - Return value: MOE_READER_OK (0) or a negative MOE_READER_E* code.  No
 *     call traps, asserts, exits or throws across the ABI.
 *   - "dev" pointers are CUDA device pointers on the handle's device; "host"
 *     pointers are ordinary host memory.  `stream` is a cudaStream_t (NULL =
 *     the legacy default stream).
 *   - A handle is not safe for concurrent use from several host threads or
 *     streams: decode calls share one workspace.
 */
#ifndef MOE_READER_H
#define MOE_READER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_READER_ABI_VERSION 1

/* Status codes. */
#define MOE_READER_OK        0
#define MOE_READER_EINVAL   -1  /* bad config, shape, k, batch, pointer or alignment */
#define MOE_READER_ENOMEM   -2  /* device allocation failed */
#define MOE_READER_ECUDA    -3  /* a CUDA runtime call failed */
#define MOE_READER_ETIMEOUT -4  /* a device-side wait exceeded its bound (never hangs) */
#define MOE_READER_EDEVICE  -5  /* a device-side input check failed (see error bits) */
#define MOE_READER_ESTATE   -6  /* call needs a completed decode that does not exist */
#define MOE_READER_ETOOBIG  -7  /* request exceeds the fixed scratch of moe_reader_topk_noalloc */

/* Device error bits reported by moe_reader_status(). */
#define MOE_READER_ERR_EXPERT_RANGE  0x1u  /* expert id outside [0, E) (clamped) */
#define MOE_READER_ERR_EXPERT_DUP    0x2u  /* an expert id repeated within a token */
#define MOE_READER_ERR_WEIGHT        0x4u  /* routing weight negative or non-finite */
#define MOE_READER_ERR_X_NONFINITE   0x8u  /* x holds a NaN or an infinity */
#define MOE_READER_ERR_TIMEOUT      0x10u  /* a bounded device wait gave up */

typedef struct moe_reader moe_reader_t;   /* opaque handle */

/* Layer shape and limits.  All fields are required. */
typedef struct {
  int32_t hidden;             /* H: a multiple of 8, 8..65536; zero-padded to Hp = 128*ceil(H/128) */
  int32_t num_experts;        /* E >= 1 */
  int32_t experts_per_token;  /* topk, 1 <= topk <= min(E, 64) */
  int32_t inter;              /* I: channels per expert, a multiple of 64, <= 8192; topk*I <= 32768 */
  int32_t screen_coords;      /* c: coordinates screened per block, 1..128 (80 = partial screen) */
  int32_t rank;               /* r: recovery rank, 1 <= r <= min(H, 64) */
  int32_t max_batch;          /* B_max: 1..1024 tokens per decode (workspace sizing) */
  int32_t flags;              /* 0 or MOE_READER_FLAG_RHO_RANK | MOE_READER_FLAG_TRIT5 */
} moe_reader_config;

/* Full-screen ranking (Chinese summary page, 方法步骤详情 decode (2): from the
 * 28.7% budget the whole sketch is read and rho_b ranks channels by the
 * expected squared output error after skipping).  Needs screen_coords = 128.
 * The score of channel j becomes
 *   w_j^2 (p_j^2 max(||d_j||^2 - ||b_j||^2, 0) + var(a_j) ||d_j||^2),
 *   var(a_j) = (phi'(ghat_j) vhat_j)^2 var(g_j) + phi(ghat_j)^2 var(v_j),
 *   var(g_j) = sum_b rho^g_{j,b} ||(R x)_b||^2 (likewise var(v_j)),
 * the expected squared norm of what skipping leaves, w_j (a_j d_j - p_j U b_j),
 * to first order in the sketch errors; the top-k and everything after it are
 * unchanged. */
#define MOE_READER_FLAG_RHO_RANK 0x1

/* Five trits per byte (the Chinese summary page's ~30 bytes per 128-coordinate
 * block, 方法步骤详情 load-time (1) and 核心方法): the sketch codes of a
 * coordinate run are stored as ceil(I/5) bytes, byte j holding channels
 * 5j .. 5j+4 as sum_m digit(t_{5j+m}) 3^m with digit(0) = 0, digit(+1) = 1,
 * digit(-1) = 2, the run padded to 32-byte sectors (S = ceil(ceil(I/5)/32)*32
 * instead of ceil(ceil(I/4)/32)*32).  Every estimate, score, kept set and
 * output equals the 2-bit layout's; the screen reads and holds fewer bytes.
 * Combines with MOE_READER_FLAG_RHO_RANK. */
#define MOE_READER_FLAG_TRIT5 0x2

/* Read accounting of the last decode, in 32-byte sectors.  Every parameter
 * array starts on a 256-byte boundary; a count is the number of distinct
 * sectors read, a union over the tokens of the batch ("Channel Selection
 * for Mixture-of-Experts Decoding Needs No Calibration Data", Chinese summary
 * page, section 前置知识: reads are billed per 32-byte sector).             */
#define MOE_READER_ARR_CODES  0   /* ternary codes of the screened coordinates */
#define MOE_READER_ARR_SCALES 1   /* FP16 block scales of the routed experts */
#define MOE_READER_ARR_DNORM  2   /* ||d_j|| of the routed experts */
#define MOE_READER_ARR_G      3   /* native gate rows of kept channels (caller's array) */
#define MOE_READER_ARR_V      4   /* native up rows of kept channels (caller's array) */
#define MOE_READER_ARR_DT     5   /* transposed down rows of kept channels */
#define MOE_READER_ARR_B      6   /* b_j rows of skipped channels */
#define MOE_READER_ARR_U      7   /* U, read whole when any token skips a channel */
typedef struct {
  uint64_t sectors[8];          /* indexed by MOE_READER_ARR_* */
  uint64_t dense_sectors;       /* G, V and D of every routed expert (denominator) */
  uint64_t activation_bytes;    /* x, ids, w read and y written (not in the fraction) */
  int32_t batch;                /* B of the last decode */
  int32_t k;                    /* k of the last decode */
} moe_reader_stats;

/* Derived sizes of a prepared handle. */
typedef struct {
  int32_t hidden_padded;        /* Hp */
  int32_t num_blocks;           /* nb = Hp / 128 */
  int32_t routed_channels;      /* N = topk * I */
  int32_t run_stride;           /* S: bytes per coordinate run, ceil(ceil(I/4)/32)*32
                                   (ceil(ceil(I/5)/32)*32 with MOE_READER_FLAG_TRIT5) */
  uint64_t resident_bytes[9];   /* codes, scales, rho, dnorm, Dt, U (with its transpose), b,
                                   sigma, workspace */
} moe_reader_info;

/*
 * moe_reader_prepare -- build the reader for one MoE layer from its weights
 * alone (Chinese summary page, 方法步骤详情, load-time steps (1)-(4)).
 *
 *   cfg     host; the layer shape.
 *   gate    dev, BF16 [E][I][H] row-major (row j of G_e is channel j's gate row).
 *   up      dev, BF16 [E][I][H] row-major.
 *   down    dev, BF16 [E][H][I] row-major (column j of D_e is d_j).
 *   sigma   host, int8 [Hp], every entry +1 or -1: the sign vector of the
 *           randomized rotation R_b = H_128 diag(sigma_b) / sqrt(128).
 *   stream  work is enqueued on it; the call synchronizes it before returning.
 *   out     host; receives the handle.
 *
 * gate, up and down must be 256-byte aligned.  The handle keeps NON-OWNING
 * pointers to gate and up (the exact step reads their native rows), so those
 * two arrays must outlive it; `down` may be freed after the call returns
 * (the handle owns its transpose).  The handle owns everything else: codes
 * u8 [E][nb][128][2][S] (per block and coordinate, the gate run then the up
 * run of I 2-bit codes, 0b00 = 0, 0b01 = +1, 0b11 = -1, channel i in byte
 * i/4 at bits 2*(i%4)), scales and rho FP16 [E][nb][2][I], dnorm fp32 [E][I],
 * Dt BF16 [E][I][H], U FP16 [H][r], b FP16 [E][I][r] and the decode
 * workspace.  Errors: EINVAL, ENOMEM, ECUDA, ETIMEOUT; *out is NULL then.
 */
int moe_reader_prepare(const moe_reader_config* cfg, const void* gate, const void* up,
                       const void* down, const int8_t* sigma, void* stream,
                       moe_reader_t** out);

/*
 * moe_reader_decode -- one decode step of B tokens through the layer
 * (Chinese summary page, 方法步骤详情, decode steps (1)-(4); Korean summary
 * page, 어떻게 쓰나).  Asynchronous on `stream`.
 *
 *   x           dev, fp32 [B][H]: the tokens' hidden states.
 *   B           0 <= B <= max_batch (B = 0 enqueues nothing).
 *   expert_ids  dev, int32 [B][topk]: routed experts, distinct within a token.
 *   expert_w    dev, fp32 [B][topk]: routing weights (finite, >= 0).
 *               Routing itself (softmax, expert choice) is the caller's job.
 *   k           0 <= k <= N = topk*I exact channels per token; k = N gives
 *               the dense gated-MoE output, k = 0 recovery only.
 *   y           dev, fp32 [B][H]: overwritten with the routed-expert output.
 *
 * All four arrays must be 16-byte aligned and may not alias y.  Host-side
 * argument errors return EINVAL without enqueuing work.  Device-side input
 * errors (bad or repeated ids, bad weights, non-finite x) set error bits that
 * moe_reader_status() reports; the kernels then stay in bounds and y is
 * unspecified.
 */
int moe_reader_decode(moe_reader_t* h, const float* x, int32_t B, const int32_t* expert_ids,
                      const float* expert_w, int32_t k, float* y, void* stream);

/*
 * moe_reader_decode_shared -- one decode step of B tokens with ONE kept set
 * for the whole batch (batch-shared selection, the direction the Chinese
 * summary page's 未来方向 (1) names for keeping the gains at larger batches).
 * Arguments, alignment, errors and asynchrony as for moe_reader_decode.
 *
 * Every token is screened and scored as in moe_reader_decode.  The union of
 * the batch's routed channels (all I channels of each of the n_e distinct
 * routed experts) is ranked by the batch score S(e, i) = the sum of s_t(e, i)
 * over the tokens routed to e, in token order (fp32).  The top
 * K = round_half_up(k * n_e / topk) channels are kept (ties to the lower
 * global id e*I + i); each token computes its routed channels in that set
 * exactly, reading each kept gate/up row once for all its tokens, and
 * recovers its other routed channels with its own estimates.  At B = 1 this
 * is moe_reader_decode.  Needs B*topk + 16 and the selection's tables
 * (about 21 KB + E*I/8 bytes) to fit the decode's shared memory: EINVAL
 * otherwise.  After it, moe_reader_get_kept answers ESTATE; use
 * moe_reader_get_kept_shared.  Statistics count the union of the tokens'
 * reads as for moe_reader_decode.
 */
int moe_reader_decode_shared(moe_reader_t* h, const float* x, int32_t B, const int32_t* expert_ids,
                             const float* expert_w, int32_t k, float* y, void* stream);

/* moe_reader_get_kept_shared -- the kept set of the last shared decode:
 * host int32 [K] global ids e*I + i, ascending; *count (host, may be NULL)
 * receives K even when capacity < K (then EINVAL).  Synchronizes the
 * decode's stream.  ESTATE if the last decode was not a shared one. */
int moe_reader_get_kept_shared(moe_reader_t* h, int32_t* kept_host, int64_t capacity,
                               int32_t* count);

/*
 * moe_reader_decode_host -- the same decode with HOST buffers: copies x, ids
 * and w to the handle's device staging area, decodes, copies y back and
 * synchronizes `stream`.  Arguments as for moe_reader_decode but every array
 * is host memory (pinned memory gives the fastest copies).  Returns EDEVICE
 * if a device-side input check failed.
 */
int moe_reader_decode_host(moe_reader_t* h, const float* x_host, int32_t B,
                           const int32_t* ids_host, const float* w_host, int32_t k,
                           float* y_host, void* stream);

/*
 * moe_reader_decode_stack -- one decode step of B tokens through L stacked
 * layers with the residual stream carried on the device (Chinese summary
 * page, 局限与改进 (1) and 独立分析的弱点 (1): fixed per-launch costs dominate
 * small batches).  Asynchronous on `stream`.  With h_0 = h_in:
 *
 *   x_l     = h_l * f_l,  f_l = 1 / sqrt(mean_c h_l[c]^2 + 1e-6)
 *             (mean and root in fp64, f_l and the product in fp32)
 *   y_l     = moe_reader_decode(layers[l], x_l, ...)
 *   h_{l+1} = h_l + y_l                             (fp32)
 *   h_out   = h_L
 *
 * One small input kernel (the per-token scale of h_0) and one decode grid
 * per layer are enqueued in stream order.  Each layer's output blocks write
 * h_{l+1} and the next layer's input scale as they complete; the next layer
 * forms x_{l+1} in its screen.  No host work or separate residual kernel
 * sits between the layers.
 *
 *   layers      host array of L >= 1 distinct handles prepared with
 *               the same H, E, topk, I, c and r on the same device; a handle
 *               may not appear twice (each layer owns its counters).
 *   h_in        dev, fp32 [B][H]: the residual stream entering layer 0.
 *   B           0 <= B <= every handle's max_batch (B = 0 enqueues nothing).
 *   expert_ids  dev, int32 [L][B][topk]: layer l's routed experts.
 *   expert_w    dev, fp32 [L][B][topk]: layer l's routing weights.
 *   k           exact channels per token, the same in every layer.
 *   h_out       dev, fp32 [B][H]: overwritten with h_L.
 *   y_layers    dev, fp32 [L][B][H] or NULL: receives each y_l (NULL: the
 *               handles' own scratch holds them).
 *
 * Arrays must be 16-byte aligned; h_out may not overlap h_in, nor y_layers
 * either of them.  EINVAL for argument errors (nothing is enqueued).
 * Device-side errors land in the error word of the layer that met them;
 * a timeout in layer l also marks every later layer with the timeout bit,
 * so moe_reader_status() on each handle reports and clears it.
 * moe_reader_get_kept / get_stats / export on layers[l] then describe layer
 * l of this step.  Per-phase profiling covers moe_reader_decode only.
 * Each layer's y_l is as deterministic as moe_reader_decode's (fp32 atomic
 * adds of output chunks); h_{l+1} adds it to h_l once, in fp32.
 */
int moe_reader_decode_stack(moe_reader_t* const* layers, int32_t L, const float* h_in, int32_t B,
                            const int32_t* expert_ids, const float* expert_w, int32_t k,
                            float* h_out, float* y_layers, void* stream);

/*
 * moe_reader_set_wait_limit -- bound, in nanoseconds of the GPU's global
 * timer, of every device-side wait of this handle's later decode calls (a
 * wait for another CTA's hand-off: screen units, scores, the kept list,
 * exact items, a stacked layer's input).  0 restores the default of one
 * second.  When a wait runs out, the kernel sets MOE_READER_ERR_TIMEOUT and
 * an abort flag that ends every other wait of the launch, and returns;
 * moe_reader_status then answers ETIMEOUT and clears the handle's counters
 * so that the next decode runs normally.  Takes effect for decode calls
 * enqueued after it (a captured graph keeps the limit it was captured with).
 */
int moe_reader_set_wait_limit(moe_reader_t* h, uint64_t ns);

/*
 * moe_reader_inject_fault -- make one failure happen on purpose, for tests
 * of failure detection; nothing faults, traps or hangs the GPU:
 *   MOE_READER_INJECT_DECODE_STALL   (h required) the next decode call on h
 *       waits, in its score tasks, for one screen unit more than exist: the
 *       count is never reached, the wait runs out after the wait limit and
 *       the call ends with MOE_READER_ERR_TIMEOUT.  In a stack, later layers
 *       inherit the abort (see moe_reader_decode_stack).
 *   MOE_READER_INJECT_PREPARE_STALL  (h = NULL) the next moe_reader_prepare's
 *       cooperative tridiagonalisation waits at its grid barrier for one CTA
 *       more than it launched; the barrier's bound (about one second) runs
 *       out and prepare returns ETIMEOUT with nothing allocated.
 *   MOE_READER_INJECT_ALLOC_FAIL     (h = NULL) the library's next device
 *       allocation reports failure as if the device were out of memory; the
 *       call that made it returns ENOMEM after freeing what it holds.
 * Each injection fires once.  EINVAL for an unknown bit or a wrong h.
 */
#define MOE_READER_INJECT_DECODE_STALL  0x1u
#define MOE_READER_INJECT_PREPARE_STALL 0x2u
#define MOE_READER_INJECT_ALLOC_FAIL    0x4u
int moe_reader_inject_fault(moe_reader_t* h, uint32_t what);

/* moe_reader_status -- synchronize the stream of the last decode, read and
 * clear the device error word.  *bits (host, may be NULL) receives the
 * MOE_READER_ERR_* bits.  Returns OK, EDEVICE (input check) or ETIMEOUT. */
int moe_reader_status(moe_reader_t* h, uint32_t* bits);

/* moe_reader_get_stats -- read accounting of the last decode (synchronizes
 * its stream, computes the union counts on device).  ESTATE if no decode. */
int moe_reader_get_stats(moe_reader_t* h, moe_reader_stats* out);

/* moe_reader_get_kept -- kept global channel ids e*I + i of the last decode,
 * ascending per token: host int32 [B][k], `capacity` >= B*k entries.
 * Synchronizes the last decode's stream.  ESTATE if no decode or if the last
 * decode was a shared one (its tokens keep different counts). */
int moe_reader_get_kept(moe_reader_t* h, int32_t* kept_host, int64_t capacity);

/* Exportable arrays (moe_reader_export).  Prepared data: */
#define MOE_READER_EXPORT_CODES    0   /* u8   [E][nb][128][2][S] (2-bit or five-trit runs) */
#define MOE_READER_EXPORT_SCALES   1   /* f16  [E][nb][2][I] */
#define MOE_READER_EXPORT_RHO      2   /* f16  [E][nb][2][I] */
#define MOE_READER_EXPORT_DNORM    3   /* f32  [E][I] */
#define MOE_READER_EXPORT_DT       4   /* bf16 [E][I][H] */
#define MOE_READER_EXPORT_U        5   /* f16  [H][r] */
#define MOE_READER_EXPORT_B        6   /* f16  [E][I][r] */
#define MOE_READER_EXPORT_SIGMA    7   /* i8   [Hp] */
#define MOE_READER_EXPORT_EIGVALS  8   /* f64  [r]: top eigenvalues of sum_j d_j d_j^T */
/* Intermediates of the last decode (B = its batch): */
#define MOE_READER_EXPORT_MASK     9   /* u32  [B][nb][4]: screened coordinates, bit c%32 of word c/32 */
#define MOE_READER_EXPORT_GHAT    10   /* f32  [B][N]: sketch gate estimates, n = slot*I + i */
#define MOE_READER_EXPORT_VHAT    11   /* f32  [B][N]: sketch up estimates */
#define MOE_READER_EXPORT_SCORE   12   /* f32  [B][N]: output-unit scores s */

/* moe_reader_export_size -- bytes of an exportable array (negative error
 * code for a bad `which` or an intermediate before any decode). */
int64_t moe_reader_export_size(moe_reader_t* h, int32_t which);

/* moe_reader_export -- copy an array to host memory `dst` (`bytes` must
 * equal moe_reader_export_size).  Synchronizes the handle's device. */
int moe_reader_export(moe_reader_t* h, int32_t which, void* dst, int64_t bytes);

/* moe_reader_get_info -- derived sizes and resident bytes of a handle. */
int moe_reader_get_info(moe_reader_t* h, moe_reader_info* out);

/* Device timing of decode calls.  The decode is one persistent kernel; its
 * time comes from CUDA events recorded around it on the decode's stream (also
 * inside a captured CUDA graph), and its phases from globaltimer stamps every
 * CTA writes at the end of each phase.  Phase slots, in order:
 *   0 the whole kernel (events)
 *   1 rotation of x, coordinate selection and sketch screen  (to the last CTA's end)
 *   2 scores and global top-k                  (from the end of slot 1)
 *   3 exact kept channels and recovery vector  (from the end of slot 2)
 *   4 output                                   (from the end of slot 3)  */
#define MOE_READER_PHASES 5

/* moe_reader_set_profiling -- enable (1) or disable (0) recording; either
 * call empties the slots.  While enabled, decode call i records its events in
 * slot i % 64. */
int moe_reader_set_profiling(moe_reader_t* h, int32_t enable);

/* moe_reader_read_profile -- for each of the n = min(decodes recorded since
 * profiling was enabled, 64) slots, in slot order, wait for its events and
 * write the milliseconds of every phase to ms_out[slot][MOE_READER_PHASES]
 * (host, `capacity` >= n rows); *calls_out (host, may be NULL) = n.  A slot
 * recorded while a CUDA graph was captured holds the times of that graph's
 * latest replay; every slot must have been recorded (or replayed) before the
 * read.  Reading does not empty the slots. */
int moe_reader_read_profile(moe_reader_t* h, double* ms_out, int64_t capacity,
                            int64_t* calls_out);

/*
 * moe_reader_topk_noalloc -- exact top-k of every row of a score matrix,
 * with the decode's selection rule (larger score first; on equal scores the
 * lower id wins), using NO device allocation.  The pages have no counterpart
 * of this entry point: it exists for callers that cannot call cudaMalloc --
 * code running inside CUDA-graph stream capture, inference-engine plugins
 * that may only touch memory the engine hands them, and processes whose
 * allocator forbids device allocations after start-up.
 *
 *   scores  dev, fp32 [rows][cols].  Values are ordered as floats: -0 ties
 *           with +0, and every NaN (either sign, any payload) ranks above
 *           +infinity, NaNs tying with one another.
 *   ids     dev, int32 [rows][cols] tie-break ids, or NULL to use the column
 *           index (the decode passes global channel ids e*I + i).  Ids are
 *           compared as unsigned 32-bit values; entries equal in both score
 *           and id are taken in ascending column order.
 *   k       0 <= k <= cols kept entries per row.
 *   kept    dev, int32 [rows][k]: kept COLUMN indices, ascending per row.
 *
 * Scratch is one file-scope __device__ array of 2^18 elements x 9 bytes
 * (about 2.3 MiB), held by every GPU that loads the library until the
 * process exits; rows*cols above 2^18 returns MOE_READER_ETOOBIG and
 * enqueues nothing.  Each call rewrites the scratch it reads, so no state
 * carries over between calls, but every call shares the one array: calls
 * that can overlap on the GPU (different streams, or graphs replayed
 * concurrently) race and must be serialized by the caller.  The first call
 * on a device looks up the array's device address (once per device, under
 * a lock); make that first call before any stream capture.  Asynchronous
 * on `stream`; returns EINVAL for bad sizes or NULL pointers.
 */
int moe_reader_topk_noalloc(const float* scores, const int32_t* ids, int32_t rows, int32_t cols,
                            int32_t k, int32_t* kept, void* stream);

/* moe_reader_destroy -- free everything the handle owns (NULL is a no-op).
 * Synchronizes the handle's device first. */
void moe_reader_destroy(moe_reader_t* h);

/* moe_reader_strerror -- static text of a status code. */
const char* moe_reader_strerror(int code);

/* moe_reader_abi_version -- MOE_READER_ABI_VERSION of the built library. */
int moe_reader_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_READER_H */
