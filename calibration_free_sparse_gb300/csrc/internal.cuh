// Internal declarations shared by the reader's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_reader.h"

namespace mr {

constexpr int kBlock = 128;          // rotation block (coordinates)
constexpr int kSector = 32;          // DRAM sector bytes
constexpr int kMaxTopk = 64;
constexpr int kMaxRank = 64;
constexpr int kMaxBatch = 1024;
constexpr int kMaxInter = 8192;
constexpr int kPhases = 5;           // kernel, rotate, screen+top-k, exact, output
constexpr int kProfSlots = 64;       // decode calls recorded between two reads

// Device error word bits (mirror the public MOE_READER_ERR_* values).
constexpr uint32_t kErrExpertRange = MOE_READER_ERR_EXPERT_RANGE;
constexpr uint32_t kErrExpertDup = MOE_READER_ERR_EXPERT_DUP;
constexpr uint32_t kErrWeight = MOE_READER_ERR_WEIGHT;
constexpr uint32_t kErrXNonFinite = MOE_READER_ERR_X_NONFINITE;
constexpr uint32_t kErrTimeout = MOE_READER_ERR_TIMEOUT;

// Shapes derived from the public config.
struct Dims {
  int H, E, topk, I, c, r, Bmax;
  int Hp, nb, N;
  int S;            // bytes per coordinate run (multiple of 32), in the stored code layout
  int runW;         // 32-bit words of codes per run actually used (16 channels a word, 20 five-trit)
  int rho_rank;     // 1: full screen ranked by the expected skip error
  int trit5;        // 1: five trits per byte (else 2-bit codes)
  int S2b;          // the 2-bit layout's run stride (the sketch is built in it first)
};

// Decode workspace (device), sized for Bmax tokens.
struct Workspace {
  uint32_t* mask;       // [Bmax][nb][4]  screened coordinates
  int32_t* ids;         // [Bmax][topk]   sanitized expert ids
  float* w;             // [Bmax][topk]   routing weights
  float* partial;       // [Bmax][topk][nb][2][I]  alpha-scaled block partials
  float* ghat;          // [Bmax][N]
  float* vhat;          // [Bmax][N]
  float* p;             // [Bmax][N]      phi(ghat) vhat
  float* score;         // [Bmax][N]
  uint32_t* keptbits;   // [Bmax][N/32]   1 = kept
  int32_t* kept;        // [Bmax][N]      kept n = slot*I + i, ascending n (first k used)
  float* wa;            // [Bmax][N]      w * a for kept list entries
  float* cpart;         // [Bmax][r] recovery vector c = sum_S w_j p_j b_j
  // host-ABI staging
  float* x_stage;       // [Bmax][H]
  float* y_stage;       // [Bmax][H]
  float* h_stage;       // [Bmax][H]      residual stream entering this layer of a stack
  float* xscale;        // [Bmax]         1 / RMS of that residual, per token
  float* rn2;           // [Bmax][nb]     ||(R x)_b||^2 (the expected-error ranking)
  // batch-shared selection
  float* sscore;        // [E][I]         batch scores
  int32_t* skept;       // [E * I]        the batch's kept global ids, ascending
  uint32_t* sbits;      // [E][I / 32]    the batch's kept set
  int32_t* estart;      // [E + 1]        per expert: first entry in elist
  int32_t* elist;       // [Bmax*topk]    token slots routed to each expert, ascending
  int32_t* kcount;      // [Bmax]         kept channels per token
  int32_t* sK;          // [1]            the batch's kept count
  int32_t* sinfo;       // [E * I]        per kept channel: expert's elist start * 16384 + count
  int32_t* ids_stage;   // [Bmax][topk]
  float* w_stage;       // [Bmax][topk]
  // accounting scratch
  uint32_t* bm_codes;   // [E][nb][4]   coordinate-run bitmap (union)
  uint32_t* bm_kept;    // [E][I/32]
  uint32_t* bm_skip;    // [E][I/32]
  uint32_t* bm_expert;  // [E/32 + 1]
  unsigned long long* counters;  // [16]
  uint32_t* err;        // [1] device error word
  uint32_t* sync;       // counters and flags of the persistent decode (zero between calls)
};

struct Prepared {
  uint8_t* codes;       // [E][nb][128][2][S]
  __half* scales;       // [E][nb][2][I]
  __half* rho;          // [E][nb][2][I]
  float* dnorm;         // [E][I]
  __nv_bfloat16* Dt;    // [E][I][H]
  __half* U;            // [H][r]
  __half* Ut;           // [r][H]  U transposed: rank components as rows
  __half* b;            // [E][I][r]
  float* bnorm2;        // [E][I]  ||b_j||^2 of the stored FP16 b
  int8_t* sigma;        // [Hp]
  double* eigvals;      // [r]
};

}  // namespace mr

struct moe_reader {
  moe_reader_config cfg;
  mr::Dims d;
  int device;
  const __nv_bfloat16* G;   // caller-owned [E][I][H]
  const __nv_bfloat16* V;   // caller-owned [E][I][H]
  mr::Prepared p;
  mr::Workspace ws;
  uint64_t resident[9];
  int grid;                 // CTAs of the persistent decode (one per SM)
  // per-phase profiling (events around each decode kernel)
  int prof_on;
  int prof_used;
  int prof_created;
  cudaEvent_t prof_ev[mr::kProfSlots][2];
  unsigned long long* prof_stamps;      // device [kProfSlots][grid][5]
  // last decode
  uint64_t wait_ns;          // bound of every device-side wait (0: the default)
  uint32_t inject;           // MOE_READER_INJECT_DECODE_STALL pending for the next decode
  int has_decode;
  int last_B, last_k;
  int last_shared;          // the last decode used the batch-shared selection
  cudaStream_t last_stream;
};

namespace mr {

constexpr unsigned long long kDefaultWaitNs = 1000000000ull;   // one second

// Every device allocation of the library goes through here (api.cu), so a
// test can make one fail on purpose (MOE_READER_INJECT_ALLOC_FAIL).
cudaError_t device_alloc(void** p, size_t bytes);
// One-shot injection of a stall at the next prepare's grid barrier.
bool take_prepare_stall();

// ---- prepare launchers (prepare_sketch.cu / prepare_svd.cu) ----
cudaError_t launch_sketch(const Dims& d, const __nv_bfloat16* G, const __nv_bfloat16* V,
                          const int8_t* sigma, uint8_t* codes, __half* scales, __half* rho,
                          cudaStream_t s);
// Five-trit runs (stride d.S) from 2-bit runs (stride d.S2b), layout [E][nb][128][2][run].
cudaError_t launch_pack_trit5(const Dims& d, const uint8_t* codes2, uint8_t* codes5, cudaStream_t s);
cudaError_t launch_transpose_down(const Dims& d, const __nv_bfloat16* D, __nv_bfloat16* Dt,
                                  cudaStream_t s);
cudaError_t launch_dnorm(const Dims& d, const __nv_bfloat16* Dt, float* dnorm, cudaStream_t s);
// Recovery basis: U (fp16 [H][r]) and eigenvalues from Dt; OK, ENOMEM, ECUDA or
// ETIMEOUT (a grid barrier ran out; `stall` adds one CTA the barrier never sees).
int build_recovery_basis(const Dims& d, const __nv_bfloat16* Dt, __half* U, double* eigvals,
                         cudaStream_t s, bool stall = false);
cudaError_t launch_transpose_u(const Dims& d, const __half* U, __half* Ut, cudaStream_t s);
cudaError_t launch_bnorm2(const Dims& d, const __half* b, float* bnorm2, cudaStream_t s);
cudaError_t launch_project_b(const Dims& d, const __nv_bfloat16* Dt, const __half* U, __half* b,
                             cudaStream_t s);

// ---- decode launchers (decode.cu) ----
// `ev` (may be null): 2 events recorded around the kernel; `stamps` (may be
// null): [grid][5] globaltimer stamps of the phase ends.
// `shared`: the batch-shared selection kernel (one kept set for the batch).
cudaError_t launch_decode(const moe_reader& h, const float* x, int B, const int32_t* ids,
                          const float* w, int k, float* y, cudaStream_t s,
                          const cudaEvent_t* ev, unsigned long long* stamps, bool shared = false);
bool shared_supported(const Dims& d, int B);   // the shared kernel's tables fit at batch B
// A stack of L layers (distinct handles of equal shape), one launch per layer,
// with the residual stream h carried on the device: h_0 = h_in, layer l decodes
// x_l = h_l / RMS(h_l) (formed by layer l's screen into handle l's x_stage), h_{l+1} = h_l + y_l
// (handle l+1's h_stage; h_out for the last layer).  y_l goes to y_layers +
// l B H, or to handle l's y_stage when y_layers is null.
cudaError_t launch_decode_stack(moe_reader* const* hs, int L, const float* h_in, int B,
                                const int32_t* ids, const float* w, int k, float* h_out,
                                float* y_layers, cudaStream_t s);
cudaError_t configure_decode_kernels(const Dims& d);
int decode_grid(const Dims& d);          // 0 if the decode kernel cannot be co-resident
size_t sync_words(const Dims& d);        // uint32 words of the synchronisation area
cudaError_t launch_stats(const moe_reader& h, int B, int k, cudaStream_t s);
cudaError_t launch_gather_kept(const moe_reader& h, int B, int k, int32_t* out_dev,
                               cudaStream_t s);

}  // namespace mr
