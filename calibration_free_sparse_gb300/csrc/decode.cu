// Decode of the channel reader as ONE persistent cooperative kernel per call
// ("Channel Selection for Mixture-of-Experts Decoding Needs No Calibration
// Data", Chinese summary page, 方法步骤详情 decode steps (1)-(4) and 核心方法;
// Korean summary page, 어떻게 쓰나).
//
// One CTA per SM, all co-resident (cooperative launch).  The phases hand work
// to each other through counters and flags in global memory instead of
// kernel boundaries; every wait is bounded (one second of the global timer by
// default), after which the CTA raises the timeout bit and the abort flag and
// leaves.
//
//   phase 1a screen units per (token, expert slot, block), dealt to teams of
//            warps: the team's first warp rotates the unit's (token, block)
//            (fp32 Sylvester butterfly of sigma x), selects the c largest |Rx|
//            coordinates (ties -> lower index) and builds pair tables; the
//            team sums the ternary codes of the screened coordinates into
//            alpha-scaled block partials of ghat and vhat
//   phase 1b score task per (token, slot): the block partials summed in block
//            order, s = w ||d|| |phi(ghat) vhat|
//   phase 1c the CTA that scores a token's last slot runs the exact top-k
//            over the token's N channels (12-bit digit histogram, exact
//            ranking of the threshold digit, ties -> lower e*I + i) and
//            releases the token's flag
//   phase 2  warp items: kept channels (a_j = phi(g_j.x)(v_j.x) from native
//            BF16 rows, fp32 x) and 64-channel recovery chunks
//            (sum w_j p_j b_j over skipped channels)
//   phase 3  each CTA adds sum_K w_j a_j Dt_j over the kept rows of its own
//            items into y; recovery output chunks add U c
#include <algorithm>

#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// Shared-memory plan of the screen (host-computed, passed to the kernel).
constexpr size_t kSmemBudget = 226 * 1024 - 256;   // dynamic shared memory: 227 KB less static, slack
struct ScreenPlan {
  int wpt;           // 4-byte code words per thread (16 channels each)
  int tw;            // warps per team
  int nteams;        // teams side by side (at most 15: one named barrier each)
  int coord_off;     // within a unit buffer: the coordinates [128] u8 after the pair
                     // tables, then the screened Rx values [128] fp32
  int buf_bytes;     // one unit buffer
  int cc;            // list positions per copy chunk (even unless one chunk holds the list)
  int nch;           // chunks per unit
  int stage_bytes;   // one chunk stage: cc + 1 records (the spare slot of an odd count)
  int team_bytes;    // 256-byte flag area, two unit buffers, two chunk stages
  int e5_off;        // five-trit layout: the byte expansion table after the teams
  size_t bytes;      // shared memory of the screen; 0: the shape does not fit
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// warps: the warps that screen; budget: the shared memory they may use
ScreenPlan screen_plan(const Dims& d, int warps = kWarps, size_t budget = kSmemBudget) {
  ScreenPlan sp{};
  const int W4 = 2 * d.runW;                     // 4-byte words per coordinate record
  double best = 0.0;
  for (int wpt = 1; wpt <= 3; ++wpt) {           // most useful lanes per issue slot
    const int tw = (W4 + 32 * wpt - 1) / (32 * wpt);
    if (tw > warps) continue;
    const int nteams = std::min(15, warps / tw);
    const double score = (double)nteams / wpt;
    if (score > best + 1e-9) {
      best = score;
      sp.wpt = wpt;
      sp.tw = tw;
      sp.nteams = nteams;
    }
  }
  if (best == 0.0) return sp;
  // everything 256-byte aligned: four 64-byte pair tables share one 256-byte
  // block, whose base the table reads assemble byte-wise
  sp.coord_off = (int)round_up(64 * (size_t)((d.c + 1) / 2), 256);
  sp.buf_bytes = (int)round_up((size_t)sp.coord_off + 128 + 4 * kBlock, 256);   // + Rx in list order
  const size_t S2 = 2 * (size_t)d.S;
  const size_t per_team = (budget - (d.trit5 ? 1024 : 0)) / sp.nteams / 256 * 256;
  const size_t fixed = 256 + 2 * (size_t)sp.buf_bytes;
  for (int nch = 1; nch <= d.c && !sp.cc; ++nch) {
    int c1 = (d.c + nch - 1) / nch;
    if (nch > 1) c1 += c1 & 1;                  // chunks hold whole pairs
    if (fixed + 2 * round_up((size_t)(c1 + 1) * S2, 256) <= per_team) sp.cc = c1;
  }
  if (!sp.cc) return sp;
  sp.nch = (d.c + sp.cc - 1) / sp.cc;
  sp.stage_bytes = (int)round_up((size_t)(sp.cc + 1) * S2, 256);
  sp.team_bytes = (int)(fixed + 2 * (size_t)sp.stage_bytes);
  sp.bytes = (size_t)sp.nteams * sp.team_bytes;
  sp.e5_off = (int)sp.bytes;                      // five-trit byte -> 2-bit codes table
  if (d.trit5) sp.bytes += 1024;
  return sp;
}

struct Params {
  Dims d;
  int B, k;
  const float* x;
  const int32_t* ids_in;
  const float* w_in;
  float* y;
  const int8_t* sigma;
  const uint8_t* codes;
  const __half* scales;
  const float* dnorm;
  const __nv_bfloat16* G;
  const __nv_bfloat16* V;
  const __nv_bfloat16* Dt;
  const __half* U;
  const __half* Ut;
  const __half* bco;
  int32_t* ids_ws;
  float* w_ws;
  uint32_t* mask;
  float* partial;
  float* ghat;
  float* vhat;
  float* p;
  float* score;
  uint32_t* keptbits;
  int32_t* kept;
  float* wa;
  float* cvec;                  // [Bmax][r] recovery vectors, accumulated atomically
  unsigned long long* stamps;   // [grid][5] phase timestamps, or null
  uint32_t* sync;
  uint32_t* err;
  ScreenPlan sp;
  // a layer of a stack (hnext null: a lone layer).  Token t's input is
  // released on xwait[t] with its scale xscale[t] = 1 / RMS(hres[t]); the
  // screen forms x = hres * xscale and writes it to xfill for the rest of the
  // layer.  Each 256-column output block, once complete, writes hnext = hres
  // + y; the token's last block sets xscale_next (null: last layer) from the
  // blocks' fp64 sums of squares and releases xnext_ready.
  const uint32_t* xwait;
  const float* xscale;
  float* xfill;
  const float* hres;
  float* hnext;
  float* xscale_next;
  uint32_t* xnext_ready;
  uint32_t* next_abort;   // the next layer's abort flag and error word: an
  uint32_t* next_err;     // aborted layer aborts the next one too
  // batch-shared selection (the shared kernel only)
  float* sscore;          // [E][I]        batch scores of the routed experts
  int32_t* skept;         // [E * I]       the batch's kept global ids e*I + i, ascending
  uint32_t* sbits;        // [E][I / 32]   the batch's kept set (routed experts only)
  int32_t* estart;        // [E + 1]       per expert: its first entry in elist
  int32_t* elist;         // [Bmax*topk]   token slots routed to each expert, ascending
  int32_t* kcount;        // [Bmax]        kept channels of each token
  int32_t* sK;            // [1]           the batch's kept count
  int32_t* sinfo;         // [E * I]       per kept channel: its expert's first elist entry
                          //               * 16384 + the expert's token-slot count
  // the expected-error ranking (d.rho_rank)
  const __half* rho;      // [E][nb][2][I] block mean squared ternary error
  const float* bnorm2;    // [E][I]        ||b_j||^2
  float* rn2;             // [Bmax][nb]    ||(R x)_b||^2
  uint32_t* ecount;       // [E]           per expert: score tasks in (synchronisation)
  int smem_bytes;         // dynamic shared memory of a CTA (after alignment)
  unsigned long long wait_ns;   // bound of every wait (globaltimer nanoseconds)
  int stall;              // fault injection: score tasks wait for one screen unit too many
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Development trace: built with -DMR_TRACE, each CTA records the global timer
// at numbered points of the decode into g_trace[CTA][point] (the last time a
// point is passed); moe_reader_trace_read copies the table out.  Without the
// macro the points compile to nothing.
#ifdef MR_TRACE
constexpr int kTraceCtas = 256, kTracePoints = 32;
__device__ unsigned long long g_trace[kTraceCtas][kTracePoints];
#define TRACE_POINT(id)                                                            \
  do {                                                                             \
    if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x][(id)] = globaltimer();        \
  } while (0)
#else
#define TRACE_POINT(id) \
  do {                  \
  } while (0)
#endif

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// L2 eviction policy for rows read once: they go first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ldg_nc4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}
__device__ __forceinline__ uint4 ldcg4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ uint4 ldg_nc4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Hand-off primitives at GPU scope.  A block (or warp) barrier before a
// single thread's release makes the whole block's (warp's) earlier writes
// part of the release; an acquire-release add also orders the caller's
// later reads after every release it follows.
__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait (one thread) until *flag >= target, for at most P.wait_ns of the
// global timer.  false: timed out (the timeout bit and the launch's abort
// flag are raised) or another wait of the launch timed out first.
__device__ bool wait_at_least(const Params& P, const uint32_t* flag, uint32_t target);

// Offsets (in uint32) of the synchronisation area, fixed per handle.
// slot .. exact: the decode's own hand-offs; cbdone .. ssum: the residual
// hand-off of a stacked layer (ssum: fp64 [Bmax], 8-byte aligned).  Every
// group, and each single word below, starts a 128-byte line of its own, so
// that the words polled by many warps share no line with the counters that
// the hand-offs add to.
constexpr int kSyncLine = 32;
__host__ __device__ inline int sync_line(int w) { return (w + kSyncLine - 1) / kSyncLine * kSyncLine; }
struct SyncOff {
  int slot, tok, flag, exact, cbdone, tokdone, xready, ssum, ecount, total;
};
// The single words.  kSyncGen (64-bit, never reset but by the host) counts
// the CTAs of every launch of the handle; a launch's generation is its value
// at the launch's start divided by the grid (a CTA reads it with the add that
// counts it, so at most grid - 1 adds of its own launch precede the read).
// Token flags are released with generation + 1 and counters are zeroed by
// their last reader, so a launch leaves nothing to reset; kSyncTail counts
// the CTAs out for the end-of-launch reset of the words only the shared
// kernel uses.  Then the launch's abort flag, and the shared kernel's
// batch-wide hand-offs (routed experts scored, the batch's kept set
// released, shared kept items done).
constexpr int kSyncGen = 0, kSyncAbort = kSyncLine, kSyncBatch = 2 * kSyncLine,
              kSyncReady = 3 * kSyncLine, kSyncSdone = 4 * kSyncLine, kSyncTail = 5 * kSyncLine;
__host__ __device__ inline SyncOff sync_offsets(const Dims& d) {
  SyncOff o;
  o.slot = 6 * kSyncLine;
  o.tok = sync_line(o.slot + d.Bmax * d.topk);
  o.flag = sync_line(o.tok + d.Bmax);
  o.exact = sync_line(o.flag + d.Bmax);
  o.cbdone = sync_line(o.exact + d.Bmax);
  o.tokdone = sync_line(o.cbdone + d.Bmax * ((d.H + 255) / 256));
  o.xready = sync_line(o.tokdone + d.Bmax);
  o.ssum = sync_line(o.xready + d.Bmax);
  o.ecount = sync_line(o.ssum + 2 * d.Bmax);   // the shared kernel: score tasks in, per expert
  o.total = o.ecount + d.E;
  return o;
}

__device__ __forceinline__ bool reached(uint32_t v, uint32_t target) {
  return (int32_t)(v - target) >= 0;   // wrap-safe: flags carry a generation
}
__device__ bool wait_at_least(const Params& P, const uint32_t* flag, uint32_t target) {
  if (reached(ld_acquire(flag), target)) return true;
  uint32_t* abort_flag = P.sync + kSyncAbort;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    // poll without ordering; the acquire load orders what follows once it is met
    if (reached(ld_relaxed(flag), target) && reached(ld_acquire(flag), target)) return true;
    if ((it & 7u) == 0) {   // the abort flag and the clock every eighth poll
      if (ld_relaxed(abort_flag)) return false;
      if (globaltimer() - t0 > P.wait_ns) {
        atomicOr(P.err, kErrTimeout);
        atomicExch(abort_flag, 1u);
        return false;
      }
    }
    __nanosleep(64);
  }
}

// A warp's wait for a flag that several warps of the CTA wait for: the first
// warp to arrive polls global memory (wait_at_least) and leaves the outcome
// in shared memory (1 met, 2 given up); the others wait on that word, so the
// CTA has one poller per flag.  seen / claim: the flag's two shared words,
// zero before the first caller.  The fence pairs order the poller's acquire
// before the word and the waiters' later reads after it.
__device__ bool cta_wait(const Params& P, const uint32_t* flag, uint32_t target, int* seen, int* claim,
                         int lane) {
  int ok = 1;
  if (lane == 0) {
    volatile int* vs = seen;
    int v = *vs;
    if (v == 0) {
      if (atomicCAS(claim, 0, 1) == 0) {
        const bool met = wait_at_least(P, flag, target);
        __threadfence_block();
        *vs = met ? 1 : 2;
        v = met ? 1 : 2;
      } else {
        // the poller's wait is bounded; this bound only backs it up
        const unsigned long long t0 = globaltimer();
        while ((v = *vs) == 0) {
          if (globaltimer() - t0 > 2 * P.wait_ns) {
            v = 2;
            break;
          }
          __nanosleep(32);
        }
      }
    }
    __threadfence_block();
    ok = v == 1;
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// A group of warps of the CTA that works together: thread tid of nt, warp wid
// of nw, and the named barrier spanning the group (0: the whole CTA).
struct Grp {
  int tid, nt, wid, nw, bar;
  __device__ __forceinline__ void sync() const {
    if (bar == 0) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nt) : "memory");
  }
};
__device__ __forceinline__ Grp cta_group() {
  return Grp{(int)threadIdx.x, kThreads, (int)(threadIdx.x >> 5), kWarps, 0};
}

// ------------------- rotation and screen selection (phase 1a) --------------
// Rotation and screen selection of one (token, 128-block) by one warp: lane
// l ends with Rx of coordinates l + 32 s (s < 4) in u[s] and with word[s] =
// the selection bits of coordinates 32 s .. 32 s + 31 (the c largest |Rx|,
// ties to the lower coordinate).  UnitInput holds a unit's raw loads, issued
// by unit_issue one unit ahead and used by nothing until unit_finish forms
// sigma x, so that the loads land while the warp sums; rotate_select_loaded
// does the rest.
struct UnitInput {
  float x[4];       // x (a stacked layer: the residual h) of coordinates lane + 32 s
  int sg[4];        // their rotation signs
  float f;          // a stacked layer: the token's input scale
  int id[2];        // the token's expert ids of slots lane, lane + 32 (inputs)
  float w[2];       // their routing weights
};

template <bool STK>
__device__ __forceinline__ void unit_issue(const Params& P, int t, int b, int lane, UnitInput& in) {
  const Dims& d = P.d;
  const size_t row = (size_t)t * d.H;
  const float* src = STK ? P.hres : P.x;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int col = b * kBlock + lane + 32 * s;
    in.x[s] = col < d.H ? __ldcg(src + row + col) : 0.f;
    in.sg[s] = P.sigma[col];
  }
  in.f = STK ? __ldcg(P.xscale + t) : 1.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int sl = lane + 32 * h;
    in.id[h] = sl < d.topk ? __ldg(P.ids_in + t * d.topk + sl) : 0;
    in.w[h] = sl < d.topk ? __ldg(P.w_in + t * d.topk + sl) : 0.f;
  }
}

// sigma x into u; true: x held a NaN or an infinity.  A stacked layer's slot-0
// unit writes x = h * scale out for the rest of the layer.
template <bool STK>
__device__ __forceinline__ bool unit_finish(const Params& P, int t, int b, int slot, int lane,
                                            const UnitInput& in, float (&u)[4]) {
  const Dims& d = P.d;
  bool bad = false;
  const size_t row = (size_t)t * d.H;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int col = b * kBlock + lane + 32 * s;
    float xv = in.x[s];
    if (STK) {
      xv = col < d.H ? xv * in.f : 0.f;
      if (slot == 0 && col < d.H) P.xfill[row + col] = xv;
    }
    bad |= !isfinite(xv);
    u[s] = in.sg[s] < 0 ? -xv : xv;
  }
  return bad;
}

// u[s] = sigma x of coordinate lane + 32 s on entry (from unit_finish), Rx on exit.
__device__ void rotate_select_loaded(const Params& P, int lane, float (&u)[4], uint32_t (&word)[4]) {
  const Dims& d = P.d;
  // Sylvester butterfly, strides 1, 2, ..., 64; pair (i, i+h) -> (a + b, a - b) in fp32
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const float o = __shfl_xor_sync(0xffffffffu, u[s], h);
      u[s] = (lane & h) ? __fsub_rn(o, u[s]) : __fadd_rn(u[s], o);
    }
  }
  {
    float a0 = u[0], a1 = u[1], a2 = u[2], a3 = u[3];
    u[0] = __fadd_rn(a0, a1); u[1] = __fsub_rn(a0, a1);
    u[2] = __fadd_rn(a2, a3); u[3] = __fsub_rn(a2, a3);
    a0 = u[0]; a1 = u[1]; a2 = u[2]; a3 = u[3];
    u[0] = __fadd_rn(a0, a2); u[2] = __fsub_rn(a0, a2);
    u[1] = __fadd_rn(a1, a3); u[3] = __fsub_rn(a1, a3);
  }
  // the c-th largest |z|: T = the largest bit pattern with at least c
  // magnitudes >= T, searched two bits at a time from bit 30 (the sign bit of
  // a magnitude is 0), the three candidates of a step counted side by side;
  // then ties by index
  uint32_t m[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) m[s] = __float_as_uint(fabsf(u[s]));
  auto count_ge = [&](uint32_t v) {
    return (int)__reduce_add_sync(0xffffffffu, (unsigned)((m[0] >= v) + (m[1] >= v) + (m[2] >= v) +
                                                          (m[3] >= v)));
  };
  // A candidate with exactly c magnitudes at or above it ends the search:
  // those c are the selection (every magnitude equal to the c-th largest is
  // among them), the same set as the full search and its tie rule give.
  const float inv = 0.08838834764831845f;   // 1/sqrt(128) rounded to fp32
  uint32_t T = 0, Tx = 0xffffffffu;
  {
    const int n0 = count_ge(1u << 30);
    if (n0 == d.c) Tx = 1u << 30;
    if (n0 >= d.c) T = 1u << 30;
  }
#pragma unroll 1
  for (int bit = 28; bit >= 0 && Tx == 0xffffffffu; bit -= 2) {
    const uint32_t c1 = T | (1u << bit), c2 = T | (2u << bit), c3 = T | (3u << bit);
    const int n1 = count_ge(c1), n2 = count_ge(c2), n3 = count_ge(c3);
    Tx = n3 == d.c ? c3 : (n2 == d.c ? c2 : (n1 == d.c ? c1 : Tx));
    T = n3 >= d.c ? c3 : (n2 >= d.c ? c2 : (n1 >= d.c ? c1 : T));
  }
  if (Tx != 0xffffffffu) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      word[s] = __ballot_sync(0xffffffffu, m[s] >= Tx);
      u[s] *= inv;
    }
    return;
  }
  const int gt = (int)__reduce_add_sync(0xffffffffu, (unsigned)((m[0] > T) + (m[1] > T) + (m[2] > T) +
                                                                (m[3] > T)));
  const int need = d.c - gt;
  const uint32_t below = (1u << lane) - 1u;
  int before = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t eqb = __ballot_sync(0xffffffffu, m[s] == T);
    const bool sel = m[s] > T || (m[s] == T && before + __popc(eqb & below) < need);
    before += __popc(eqb);
    word[s] = __ballot_sync(0xffffffffu, sel);
    u[s] *= inv;
  }
}


// ------------------------------- top-k -------------------------------------
// k-th largest key among the entries keyfn accepts; per-warp histograms.
template <typename KeyFn>
__device__ uint32_t cta_radix_select(const Grp& g, int N, int kth, KeyFn keyfn, int* hist, int* sh,
                                     int* rem) {
  uint32_t prefix = 0, pmask = 0;
  int remaining = kth;
  const int warp = g.wid, lane = g.tid & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = g.tid; i < g.nw * 256; i += g.nt) hist[i] = 0;
    g.sync();
    for (int n = g.tid; n < N; n += g.nt) {
      uint32_t key;
      if (!keyfn(n, key)) continue;
      if ((key & pmask) == prefix) atomicAdd(&hist[warp * 256 + ((key >> shift) & 255u)], 1);
    }
    g.sync();
    for (int i = g.tid; i < 256; i += g.nt) {
      int tot = 0;
      for (int w = 0; w < g.nw; ++w) tot += hist[w * 256 + i];
      hist[g.nw * 256 + i] = tot;
    }
    g.sync();
    if (warp == 0) {
      const int* totals = hist + g.nw * 256;
      int local[8];
      int tot = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        local[u] = totals[255 - (lane * 8 + u)];
        tot += local[u];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int before = incl - tot, found = -1, r = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (found < 0 && before + local[u] >= remaining) {
          found = 255 - (lane * 8 + u);
          r = remaining - before;
        }
        before += local[u];
      }
      const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
      const int first = bal ? __ffs(bal) - 1 : 0;
      const int fd = __shfl_sync(0xffffffffu, found, first);
      const int fr = __shfl_sync(0xffffffffu, r, first);
      if (lane == 0) {
        sh[0] = fd < 0 ? 0 : fd;
        sh[1] = fr;
      }
    }
    g.sync();
    prefix |= (uint32_t)sh[0] << shift;
    pmask |= 255u << shift;
    remaining = sh[1];
    g.sync();
  }
  *rem = remaining;
  return prefix;
}

constexpr int kDigitBits = 12;               // first histogram: key bits 30..19
constexpr int kBins = 1 << kDigitBits;
constexpr int kCandMax = 1024;               // candidates ranked exactly; more -> radix

__device__ __forceinline__ int key_digit(uint32_t key) { return (int)((key >> 19) & (kBins - 1)); }

// Shared-memory layout of the top-k step (offsets in bytes from smem).
__host__ __device__ inline size_t topk_smem_bytes(int N) {
  return (size_t)4 * N                       // keys
         + (size_t)(kWarps + 1) * 256 * 4    // histogram (4096 bins, or the radix rows)
         + (size_t)N                         // keep flags
         + (size_t)kCandMax * 12             // candidate keys, ids, ranks
         + 512;                              // scalars, warp sums, expert ids
}

// Sum of wsum[0 .. wid) for the calling thread's warp, by a shuffle scan of
// the kWarps per-warp values (read after the barrier that follows their
// writes); *total (may be null) receives the sum of all of them.
__device__ __forceinline__ int warps_before(const int* wsum, int wid, int lane, int* total,
                                            int nw = kWarps) {
  const int v = lane < nw ? wsum[lane] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (total) *total = __shfl_sync(0xffffffffu, incl, 31);
  return __shfl_sync(0xffffffffu, incl - v, wid);
}

// The top-k's fallback when more than kCandMax keys share the threshold digit:
// a full radix select on the keys, ties by the lower global id.  Sets keep[].
__device__ __noinline__ void topk_radix_fallback(const Grp& g, const uint32_t* keys, uint8_t* keep,
                                                 const int* eid, int N, int k, int I, int* hist,
                                                 int* sh, int* wsum) {
  const int lane = g.tid & 31, wid = g.wid;
  int need2 = 0;
  const uint32_t T = cta_radix_select(
      g, N, k, [&](int n, uint32_t& key) { key = keys[n]; return true; }, hist, sh + 4, &need2);
  int eq = 0;
  for (int n = g.tid; n < N; n += g.nt) eq += keys[n] == T;
  eq = warp_sum_i(eq);
  if (lane == 0) wsum[wid] = eq;
  g.sync();
  int eq_total = 0;
  for (int w = 0; w < g.nw; ++w) eq_total += wsum[w];
  g.sync();
  uint32_t T2 = 0;
  if (need2 < eq_total) {
    int dummy = 0;
    T2 = cta_radix_select(
        g, N, need2,
        [&](int n, uint32_t& key) {
          if (keys[n] != T) return false;
          key = 0xffffffffu - (uint32_t)(eid[n / I] * I + n % I);
          return true;
        },
        hist, sh + 4, &dummy);
  }
  for (int n = g.tid; n < N; n += g.nt) {
    const uint32_t a = keys[n];
    keep[n] = a > T || (a == T && 0xffffffffu - (uint32_t)(eid[n / I] * I + n % I) >= T2);
  }
}

// ftag: the launch's flag value (generation + 1).
template <int NT>
__device__ void topk_token(const Params& P, const Grp& g, int t, unsigned char* smem, uint32_t ftag) {
  constexpr int NW = NT / 32;
  const Dims& d = P.d;
  const int N = d.N, k = P.k, I = d.I;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);                      // [N]
  int* hist = reinterpret_cast<int*>(keys + N);                             // [(kWarps+1)*256]
  uint8_t* keep = reinterpret_cast<uint8_t*>(hist + (kWarps + 1) * 256);    // [N]
  uint32_t* ckey = reinterpret_cast<uint32_t*>(keep + ((N + 15) & ~15));    // [kCandMax]
  uint32_t* cgid = ckey + kCandMax;                                         // [kCandMax]
  int* crank = reinterpret_cast<int*>(cgid + kCandMax);                     // [kCandMax]
  int* sh = crank + kCandMax;                                               // [8]
  int* wsum = sh + 8;                                                       // [kWarps]
  int* eid = wsum + kWarps;                                                 // [topk]
  const int lane = g.tid & 31, wid = g.wid;
  if (g.tid == 0) TRACE_POINT(8);
  {   // the token's N scores (N is a multiple of 64: whole float4 groups),
      // then its expert ids from the inputs, sanitised as the screen does
    const float4* s4 = reinterpret_cast<const float4*>(P.score + (size_t)t * N);
    uint4* k4 = reinterpret_cast<uint4*>(keys);
    const int e_in = g.tid < d.topk ? __ldg(P.ids_in + t * d.topk + g.tid) : 0;
    for (int q = g.tid; q < N / 4; q += NT) {
      const float4 v = __ldcg(s4 + q);
      k4[q] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                         __float_as_uint(v.w));
    }
    if (g.tid < d.topk) eid[g.tid] = (e_in < 0 || e_in >= d.E) ? 0 : e_in;
  }
  // the output adds into y[t]: start it from zero while the scores come in
  for (int h = 4 * g.tid; h < d.H; h += 4 * NT)
    *reinterpret_cast<float4*>(P.y + (size_t)t * d.H + h) = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = g.tid; i < kBins; i += NT) hist[i] = 0;
  if (g.tid == 0) sh[2] = 0;
  g.sync();
  if (g.tid == 0) TRACE_POINT(22);

  const bool all = k >= N, none = k <= 0;
  if (all || none) {
    for (int n = g.tid; n < N; n += NT) keep[n] = all;
  } else {
    // 1. histogram of the 12-bit digit (keys spread over hundreds of bins)
    for (int n = g.tid; n < N; n += NT) atomicAdd(&hist[key_digit(keys[n])], 1);
    g.sync();
    if (g.tid == 0) TRACE_POINT(9);
    // 2. the digit D holding the k-th largest key: 8 digits per thread, from the top
    constexpr int kPer = kBins / NT;
    int cnt[kPer], tot = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      cnt[u] = hist[kBins - 1 - (g.tid * kPer + u)];
      tot += cnt[u];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    g.sync();
    const int before = incl - tot + warps_before(wsum, wid, lane, nullptr, NW);
    if (before < k && before + tot >= k) {
      int above = before;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (above + cnt[u] >= k) {
          sh[0] = kBins - 1 - (g.tid * kPer + u);
          sh[1] = k - above;       // keys of digit D that are kept
          sh[3] = cnt[u];          // keys of digit D
          break;
        }
        above += cnt[u];
      }
    }
    g.sync();
    const int D = sh[0], need = sh[1], m = sh[3];
    if (g.tid == 0) TRACE_POINT(10);
    if (m <= kCandMax) {
      // 3. the candidates (digit D) ranked exactly: larger key, then lower global id
      for (int n = g.tid; n < N; n += NT) {
        const int dg = key_digit(keys[n]);
        keep[n] = dg > D;
        if (dg == D) {
          const int c = atomicAdd(&sh[2], 1);
          ckey[c] = keys[n] | 0u;
          cgid[c] = (uint32_t)(eid[n / I] * I + n % I);
          crank[c] = n;             // the channel for now; the rank below
        }
      }
      g.sync();
      if (g.tid == 0) TRACE_POINT(23);
      // a warp per candidate: its lanes count the candidates ahead of it
      for (int ci = wid; ci < m; ci += NW) {
        const uint32_t ki = ckey[ci], gi = cgid[ci];
        int ahead = 0;
        for (int cj = lane; cj < m; cj += 32) {
          const uint32_t kj = ckey[cj];
          ahead += kj > ki || (kj == ki && cgid[cj] < gi);
        }
        ahead = warp_sum_i(ahead);
        if (lane == 0) keep[crank[ci]] = ahead < need;
      }
    } else {
      // degenerate spread (too many keys in one digit): full radix select
      topk_radix_fallback(g, keys, keep, eid, N, k, I, hist, sh, wsum);
    }
  }
  g.sync();
  // 4. compaction in ascending n and the kept bitmap: warp w owns a contiguous
  if (g.tid == 0) TRACE_POINT(11);
  //    range of whole 32-channel words; one ballot per word
  const int words = N / 32;
  const int wper = (words + NW - 1) / NW;
  const int w0 = wid * wper, w1 = min(words, w0 + wper);
  int mine = 0;
  for (int wd = w0; wd < w1; ++wd) mine += __popc(__ballot_sync(0xffffffffu, keep[wd * 32 + lane]));
  if (lane == 0) wsum[wid] = mine;
  g.sync();
  int pos = warps_before(wsum, wid, lane, nullptr, NW);
  const uint32_t below = (1u << lane) - 1u;
  for (int wd = w0; wd < w1; ++wd) {
    const int n = wd * 32 + lane;
    const uint32_t bal = __ballot_sync(0xffffffffu, keep[n]);
    if (keep[n]) {
      const int at = pos + __popc(bal & below);
      if (at < N) P.kept[(size_t)t * N + at] = n;
    }
    if (lane == 0) P.keptbits[(size_t)t * words + wd] = bal;
    pos += __popc(bal);
  }
  if (g.tid == 0) TRACE_POINT(24);
  if (g.tid == 0) P.sync[sync_offsets(d).exact + t] = 0u;   // counted by items after the release
  g.sync();
  if (g.tid == 0) {
    st_release(&P.sync[sync_offsets(d).flag + t], ftag);
    TRACE_POINT(12);
  }
}

// ------------------------- batch-shared selection ---------------------------
// One kept set for the whole batch: the union of the routed experts' channels
// is ranked by the batch score (the routed tokens' scores summed in token
// order) and the top K = k n_e / topk (rounded half up, n_e routed experts)
// are kept; each token computes its share exactly and recovers the rest.

// In-place exclusive prefix sum of a[0..n) by the whole CTA (each thread a
// contiguous segment); returns the total.  wsum: [kWarps] scratch.
__device__ int block_exclusive_scan(int* a, int n, int* wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int per = (n + kThreads - 1) / kThreads;
  const int b0 = min(n, (int)threadIdx.x * per), b1 = min(n, b0 + per);
  int mine = 0;
  for (int q = b0; q < b1; ++q) mine += a[q];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  int before = incl - mine, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    before += w < wid ? wsum[w] : 0;
    total += wsum[w];
  }
  __syncthreads();   // every thread has read wsum
  for (int q = b0; q < b1; ++q) {
    const int v = a[q];
    a[q] = before;
    before += v;
  }
  __syncthreads();
  return total;
}

// The digit of a kBins histogram (counted from the top) holding the K-th
// largest key: sh[3] = digit, sh[4] = its keys to keep, sh[5] = its keys.
__device__ void digit_search(const int* hist, int K, int* wsum, int* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int kPer = kBins / kThreads;
  int c8[kPer], tot = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c8[q] = hist[kBins - 1 - (threadIdx.x * kPer + q)];
    tot += c8[q];
  }
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  int before = incl - tot;
  for (int w = 0; w < wid; ++w) before += wsum[w];
  if (before < K && before + tot >= K) {
    int above = before;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (above + c8[q] >= K) {
        sh[3] = kBins - 1 - (threadIdx.x * kPer + q);
        sh[4] = K - above;
        sh[5] = c8[q];
        break;
      }
      above += c8[q];
    }
  }
  __syncthreads();
}

// Shared-memory bytes of shared_select for a shape (0 if it does not fit the
// decode's dynamic shared memory).
__host__ __device__ inline size_t shared_select_bytes(const Dims& d) {
  return (size_t)(kWarps + 1) * 256 * 4 + (size_t)(3 * d.E + 2) * 4 + 64 + kWarps * 4 +
         (size_t)kCandMax * 12 + (size_t)d.E * (d.I / 32) * 4 + 256;
}

// The batch's kept set, by the CTA whose score task completed the last routed
// expert (all batch scores are in).
__device__ void shared_select(const Params& P, unsigned char* smem) {
  const Dims& d = P.d;
  const int BT = P.B * d.topk, E = d.E, I = d.I, IW = d.I / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  int* hist = reinterpret_cast<int*>(smem);            // [(kWarps + 1) * 256]
  int* cnt = hist + (kWarps + 1) * 256;                 // [E + 1] counts, then starts
  int* cur = cnt + (E + 1);                             // [E + 1] fill cursors
  int* uexp = cur + (E + 1);                            // [E] routed experts, ascending
  int* sh = uexp + E;                                   // [16]
  int* wsum = sh + 16;                                  // [kWarps]
  uint32_t* ckey = reinterpret_cast<uint32_t*>(wsum + kWarps);   // [kCandMax]
  uint32_t* cgid = ckey + kCandMax;                     // [kCandMax]
  int* cu = reinterpret_cast<int*>(cgid + kCandMax);    // [kCandMax]
  uint32_t* bits = reinterpret_cast<uint32_t*>(cu + kCandMax);   // [n_e][IW]
  uint32_t* kc = bits + (size_t)E * IW;   // the union's keys when they fit, else unused
  for (int e = threadIdx.x; e <= E; e += kThreads) cnt[e] = 0;
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
  if (threadIdx.x == 0) sh[2] = 0;
  __syncthreads();
  for (int ts = threadIdx.x; ts < BT; ts += kThreads) atomicAdd(&cnt[__ldcg(P.ids_ws + ts)], 1);
  __syncthreads();
  // routed-expert ranks (cur as scratch), then the starts of each expert's slots
  for (int e = threadIdx.x; e < E; e += kThreads) cur[e] = cnt[e] ? 1 : 0;
  __syncthreads();
  const int ne = block_exclusive_scan(cur, E, wsum);
  for (int e = threadIdx.x; e < E; e += kThreads)
    if (cnt[e]) uexp[cur[e]] = e;
  __syncthreads();
  block_exclusive_scan(cnt, E + 1, wsum);   // cnt[E] was 0: it becomes the total
  for (int e = threadIdx.x; e <= E; e += kThreads) {
    cur[e] = cnt[e];
    P.estart[e] = cnt[e];
  }
  const int K = (2 * P.k * ne + d.topk) / (2 * d.topk), U = ne * I;
  if (threadIdx.x == 0) *P.sK = K;
  __syncthreads();
  // the union's keys stay in shared memory when they fit; else their digits
  // (the second pass then reads only the threshold digit's keys again)
  const size_t room = (size_t)P.smem_bytes - (size_t)(reinterpret_cast<unsigned char*>(kc) - smem);
  const bool cached = (size_t)U * 4 <= room;
  const bool dcached = !cached && (size_t)U * 2 <= room;
  uint16_t* dc = reinterpret_cast<uint16_t*>(kc);
  // each expert's token slots in ascending order: one warp, 32 slots a step
  if (wid == 0) {
    for (int base = 0; base < BT; base += 32) {
      const int ts = base + lane;
      const int e = ts < BT ? __ldcg(P.ids_ws + ts) : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int at = ts < BT ? cur[e] + __popc(same & below) : 0;
      __syncwarp();
      if (ts < BT) {
        P.elist[at] = ts;
        if ((same & below) == 0) cur[e] += __popc(same);
      }
      __syncwarp();
    }
  }
  // 1. histogram of the batch scores' 12-bit digit over the union (the keys
  //    stay in shared memory when they fit)
  {
    constexpr int kV = 4;   // float4 loads in flight per thread
    const int U4 = U / 4;   // I is a multiple of 64: whole float4 groups of one expert
    for (int f0 = threadIdx.x; f0 < U4; f0 += kThreads * kV) {
      float4 kv[kV];
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const int f = f0 + v * kThreads;
        const int u = 4 * f, r = u / I;
        kv[v] = f < U4 ? __ldcg(reinterpret_cast<const float4*>(P.sscore + (size_t)uexp[r] * I +
                                                                 (u - r * I)))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const int f = f0 + v * kThreads;
        if (f >= U4) break;
        const uint32_t k4[4] = {__float_as_uint(kv[v].x), __float_as_uint(kv[v].y),
                                __float_as_uint(kv[v].z), __float_as_uint(kv[v].w)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (cached) kc[4 * f + c] = k4[c];
          if (dcached) dc[4 * f + c] = (uint16_t)key_digit(k4[c]);
          atomicAdd(&hist[key_digit(k4[c])], 1);
        }
      }
    }
  }
  __syncthreads();
  auto keyof = [&](int u) {
    if (cached) return kc[u];
    const int r = u / I, i = u - r * I;
    return __float_as_uint(__ldcg(P.sscore + (size_t)uexp[r] * I + i));
  };
  const bool all = K >= U, none = K <= 0;
  int D = -1, need = 0, m = 0;
  if (!all && !none) {
    // 2. the digit holding the K-th largest batch score
    digit_search(hist, K, wsum, sh);
    D = sh[3];
    need = sh[4];
    m = sh[5];
  }
  // the digit's members (u) when they fit the list after the key cache
  constexpr int kDl = 8192;
  const size_t used = cached ? (size_t)U * 4 : (dcached ? (size_t)U * 2 : 0);
  int* dl = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(kc) + ((used + 15) & ~(size_t)15));
  const bool listed = m > kCandMax && m <= kDl && ((used + 15) & ~(size_t)15) + (size_t)kDl * 4 <= room;
  // 3. kept bits above the digit (a ballot per 32 channels of one expert) and
  //    the digit's candidates
  for (int base = 32 * wid; base < U; base += kThreads) {
    const int u = base + lane, r = u / I, i = u - r * I;
    const int dg = dcached ? (int)dc[u] : key_digit(keyof(u));
    const unsigned keep = __ballot_sync(0xffffffffu, all || (!none && dg > D));
    if (lane == 0) bits[base >> 5] = keep;
    if (!all && !none && dg == D && m <= kCandMax) {
      const int c = atomicAdd(&sh[2], 1);
      cgid[c] = (uint32_t)(uexp[r] * I + i);
      cu[c] = u;
    } else if (listed && dg == D) {
      dl[atomicAdd(&sh[2], 1)] = u;
    }
  }
  __syncthreads();
  if (!all && !none && m <= kCandMax)   // the candidates' keys, all loads in flight together
    for (int c = threadIdx.x; c < m; c += kThreads) ckey[c] = keyof(cu[c]);
  __syncthreads();
  int mode = 0;   // 1: rank the candidates; 2: full radix select
  if (!all && !none) mode = m <= kCandMax ? 1 : 2;
  if (listed) {
    // a second 12-bit digit (key bits 18..7) inside digit D
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < m; c += kThreads) atomicAdd(&hist[(keyof(dl[c]) >> 7) & (kBins - 1)], 1);
    __syncthreads();
    digit_search(hist, need, wsum, sh);
    const int D2 = sh[3], need2 = sh[4], m2 = sh[5];
    if (threadIdx.x == 0) sh[2] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < m; c += kThreads) {
      const int u = dl[c];
      const uint32_t key = keyof(u);
      const int d2 = (int)((key >> 7) & (kBins - 1));
      if (d2 > D2) atomicOr(&bits[u >> 5], 1u << (u & 31));
      if (d2 == D2 && m2 <= kCandMax) {
        const int q = atomicAdd(&sh[2], 1);
        const int r = u / I;
        ckey[q] = key;
        cgid[q] = (uint32_t)(uexp[r] * I + (u - r * I));
        cu[q] = u;
      }
    }
    __syncthreads();
    if (m2 <= kCandMax) {   // D2's members ranked exactly
      m = m2;
      need = need2;
      mode = 1;
    }
  }
  {
    if (mode == 1) {
      // the candidates ranked exactly: larger score, then lower global id (a
      // warp per candidate)
      for (int ci = wid; ci < m; ci += kWarps) {
        const uint32_t ki = ckey[ci], gi = cgid[ci];
        int ahead = 0;
        for (int cj = lane; cj < m; cj += 32) {
          const uint32_t kj = ckey[cj];
          ahead += kj > ki || (kj == ki && cgid[cj] < gi);
        }
        ahead = warp_sum_i(ahead);
        if (lane == 0 && ahead < need) atomicOr(&bits[cu[ci] >> 5], 1u << (cu[ci] & 31));
      }
    } else if (mode == 2) {
      // degenerate spread: full radix select over the union, ties by id
      auto gidof = [&](int u) {
        const int r = u / I;
        return (uint32_t)(uexp[r] * I + (u - r * I));
      };
      int need2 = 0;
      const uint32_t T = cta_radix_select(
          cta_group(), U, K, [&](int u, uint32_t& key) { key = keyof(u); return true; }, hist, sh + 8,
          &need2);
      int eq = 0;
      for (int u = threadIdx.x; u < U; u += kThreads) eq += keyof(u) == T;
      eq = warp_sum_i(eq);
      if (lane == 0) wsum[wid] = eq;
      __syncthreads();
      int eq_total = 0;
      for (int w = 0; w < kWarps; ++w) eq_total += wsum[w];
      __syncthreads();
      uint32_t T2 = 0;
      if (need2 < eq_total) {
        int dummy = 0;
        T2 = cta_radix_select(
            cta_group(), U, need2,
            [&](int u, uint32_t& key) {
              if (keyof(u) != T) return false;
              key = 0xffffffffu - gidof(u);
              return true;
            },
            hist, sh + 8, &dummy);
      }
      for (int base = 32 * wid; base < U; base += kThreads) {
        const int u = base + lane;
        const uint32_t a = keyof(u);
        const bool kp = a > T || (a == T && 0xffffffffu - gidof(u) >= T2);
        const unsigned keep = __ballot_sync(0xffffffffu, kp);
        if (lane == 0) bits[base >> 5] = keep;
      }
    }
  }
  __syncthreads();
  // 4. the set per expert, and the kept global ids in ascending order
  const int words = ne * IW;
  for (int q = threadIdx.x; q < words; q += kThreads)
    P.sbits[(size_t)uexp[q / IW] * IW + q % IW] = bits[q];
  const int wper = (words + kWarps - 1) / kWarps;
  const int w0 = wid * wper, w1 = min(words, w0 + wper);
  int mine = 0;
  for (int wd = w0; wd < w1; ++wd) mine += __popc(bits[wd]);
  if (lane == 0) wsum[wid] = mine;
  __syncthreads();
  int pos = 0;
  for (int w = 0; w < wid; ++w) pos += wsum[w];
  {
    int r = w0 / IW, wr = w0 - r * IW;   // expert rank and word within it, advanced together
    for (int wd = w0; wd < w1; ++wd) {
      const uint32_t bw = bits[wd];
      if (bw) {
        if ((bw >> lane) & 1u) {
          const int e = uexp[r], at = pos + __popc(bw & below);
          P.skept[at] = e * I + wr * 32 + lane;
          P.sinfo[at] = cnt[e] * 16384 + (cnt[e + 1] - cnt[e]);
        }
        pos += __popc(bw);
      }
      if (++wr == IW) {
        wr = 0;
        ++r;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) st_release(P.sync + kSyncReady, 1u);
}

// The shared kernel's end of score task ts (expert e): the task that scores
// the last slot routed to e sums e's batch scores (token order), and the task
// that completes the last routed expert selects the batch's kept set.  The
// routing is read from the input (validated as the screen does), so no other
// task's writes are needed to know who routes where.
__device__ void shared_after_score(const Params& P, int e, unsigned char* smem, int* flag) {
  const Dims& d = P.d;
  const int BT = P.B * d.topk;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  int* lst = reinterpret_cast<int*>(smem);      // [BT] token slots routed to e, ascending
  int* cw = lst + BT;                           // [kWarps]
  int* seen = cw + kWarps;                      // [E] experts routed by the batch
  int* sh = seen + d.E;                         // [4]
  for (int q = threadIdx.x; q < d.E; q += kThreads) seen[q] = 0;
  __syncthreads();
  int n = 0;
  for (int base = 0; base < BT; base += kThreads) {
    const int ts = base + threadIdx.x;
    int ei = ts < BT ? P.ids_in[ts] : -1;
    if (ts < BT && (ei < 0 || ei >= d.E)) ei = 0;
    if (ts < BT) seen[ei] = 1;
    const bool hit = ts < BT && ei == e;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) cw[wid] = __popc(bal);
    __syncthreads();
    int before = n, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      before += w < wid ? cw[w] : 0;
      tot += cw[w];
    }
    if (hit) lst[before + __popc(bal & below)] = ts;
    n += tot;
    __syncthreads();
  }
  int ne = 0;
  for (int q0 = 0; q0 < d.E; q0 += kThreads) {
    const int q = q0 + threadIdx.x;
    ne += __syncthreads_count(q < d.E && seen[q]);
  }
  if (threadIdx.x == 0) {
    sh[0] = ne;
    // releases this slot's scores; the last of e's slots also acquires the others'
    sh[1] = atom_add_acq_rel(P.ecount + e, 1u) == (uint32_t)(n - 1);
  }
  __syncthreads();
  if (!sh[1]) return;
  for (int i = threadIdx.x; i < d.I; i += kThreads) {
    float sum = 0.f;
    for (int q0 = 0; q0 < n; q0 += 8) {   // eight loads in flight, added in token order
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = q0 + u < n ? __ldcg(P.score + (size_t)lst[q0 + u] * d.I + i) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (q0 + u < n) sum += v[u];
    }
    P.sscore[(size_t)e * d.I + i] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    *flag = atom_add_acq_rel(P.sync + kSyncBatch, 1u) == (uint32_t)(sh[0] - 1);
  __syncthreads();
  if (*flag) shared_select(P, smem);
  __syncthreads();
}

// Token t's share of the batch's set: its kept bitmap and ascending kept list
// (n = slot I + i) and their count; y[t] zeroed; then the token is released.
__device__ void shared_token(const Params& P, int t, unsigned char* smem, uint32_t ftag) {
  const Dims& d = P.d;
  const int IW = d.I / 32, words = d.N / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  int* wsum = reinterpret_cast<int*>(smem);   // [kWarps]
  uint32_t* tw = reinterpret_cast<uint32_t*>(wsum + kWarps);   // [words]
  for (int wd = threadIdx.x; wd < words; wd += kThreads) {
    const int slot = wd / IW;
    const int e = __ldcg(P.ids_ws + t * d.topk + slot);
    const uint32_t bw = __ldcg(P.sbits + (size_t)e * IW + (wd - slot * IW));
    tw[wd] = bw;
    P.keptbits[(size_t)t * words + wd] = bw;
  }
  __syncthreads();
  const int wper = (words + kWarps - 1) / kWarps;
  const int w0 = wid * wper, w1 = min(words, w0 + wper);
  int mine = 0;
  for (int wd = w0; wd < w1; ++wd) mine += __popc(tw[wd]);
  if (lane == 0) wsum[wid] = mine;
  __syncthreads();
  int pos = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    pos += w < wid ? wsum[w] : 0;
    total += wsum[w];
  }
  for (int wd = w0; wd < w1; ++wd) {
    const uint32_t bw = tw[wd];
    if ((bw >> lane) & 1u) P.kept[(size_t)t * d.N + pos + __popc(bw & below)] = wd * 32 + lane;
    pos += __popc(bw);
  }
  if (threadIdx.x == 0) {
    P.kcount[t] = total;
    P.sync[sync_offsets(d).exact + t] = 0u;   // counted by items after the release
  }
  __syncthreads();
  if (threadIdx.x == 0) st_release(&P.sync[sync_offsets(d).flag + t], ftag);
}

// ------------------------------- phase 1a ----------------------------------
// Screen units (token, slot, block) are dealt to the CTAs round-robin; all
// cost the same.  Inside a CTA the warps form teams that each compute whole
// units, several units side by side.  Shared memory per team: a flag area and
// two unit buffers, each the unit's pair tables [ceil(c/2)][16] fp32 (64-byte
// aligned) and its screened coordinates [128] u8.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void team_sync(int team, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(threads) : "memory");
}


// Publish a stored unit: the warp's partial stores, then (release add) its
// share of the (token, slot) counter (complete at nb * tw).
__device__ __forceinline__ void publish_unit(const Params& P, int ts, int lane) {
  __syncwarp();
  if (lane == 0) red_add_release(P.sync + sync_offsets(P.d).slot + ts, 1u);
}

// The first warp's part of screen unit uu: rotation and selection of the
// unit's (token, block) from its raw loads (in, issued by unit_issue), the
// side outputs (screened set, input checks, sanitised routing, zeroed
// recovery vector), and into `buf` the screened coordinate list, their Rx
// values and the pair tables.  Returns the unit's expert id, clamped into range.
template <bool STK>
__device__ int build_unit(const Params& P, unsigned char* buf, int uu, int lane, const UnitInput& in,
                          int team) {
  const Dims& d = P.d;
  uint8_t* cbuf = buf + P.sp.coord_off;
  float* rbuf = reinterpret_cast<float*>(cbuf + 128);
  const int b = uu % d.nb, ts = uu / d.nb, t = ts / d.topk, slot = ts % d.topk;
  float xu[4];
  const bool xbad = unit_finish<STK>(P, t, b, slot, lane, in, xu);
  // the slot's expert id and weight as given (lane-distributed loads)
  const int e_raw = __shfl_sync(0xffffffffu, slot < 32 ? in.id[0] : in.id[1], slot & 31);
  const float w_raw = __shfl_sync(0xffffffffu, slot < 32 ? in.w[0] : in.w[1], slot & 31);
  uint32_t word[4];
  rotate_select_loaded(P, lane, xu, word);
  if (lane == 0 && team == 0) TRACE_POINT(2);
  if (d.rho_rank) {   // ||(R x)_b||^2 for the expected-error ranking (every slot writes it)
    const float ss = warp_sum(xu[0] * xu[0] + xu[1] * xu[1] + xu[2] * xu[2] + xu[3] * xu[3]);
    if (lane == 0) P.rn2[(size_t)t * d.nb + b] = ss;
  }
  // the unit's side outputs: the block's screened set (the same from every
  // slot), the input checks, and at block 0 the slot's sanitised expert id
  // and weight (and, for slot 0, the token's zeroed recovery vector); the
  // warp's unit publication orders them before every later reader
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4)
    if (lane == s4) P.mask[((size_t)t * d.nb + b) * 4 + s4] = word[s4];
  if (slot == 0 && __any_sync(0xffffffffu, xbad) && lane == 0) atomicOr(P.err, kErrXNonFinite);
  if (b == 0) {
    // a repeated expert: an earlier slot of the token with the same id
    const bool dup = __any_sync(0xffffffffu, (lane < slot && in.id[0] == e_raw) ||
                                                  (lane + 32 < slot && in.id[1] == e_raw));
    if (lane == 0) {
      int e = e_raw;
      const float wv = w_raw;
      uint32_t bits = 0;
      if (e < 0 || e >= d.E) {
        bits |= kErrExpertRange;
        e = 0;
      }
      if (dup) bits |= kErrExpertDup;
      if (!(wv >= 0.f) || !isfinite(wv)) bits |= kErrWeight;
      if (bits) atomicOr(P.err, bits);
      P.ids_ws[ts] = e;
      P.w_ws[ts] = wv;
    }
    if (slot == 0)
      for (int j = lane; j < d.r; j += 32) P.cvec[(size_t)t * d.r + j] = 0.f;
  }
  // the screened list in ascending coordinate order; an odd count's spare
  // position repeats the last coordinate
  const uint32_t below = (1u << lane) - 1u;
  int listed = 0;
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4) {
    if ((word[s4] >> lane) & 1u) {
      const int pos = listed + __popc(word[s4] & below);
      cbuf[pos] = (uint8_t)(lane + 32 * s4);
      rbuf[pos] = xu[s4];
      if (pos == d.c - 1 && (d.c & 1)) cbuf[d.c] = (uint8_t)(lane + 32 * s4);
    }
    listed += __popc(word[s4]);
  }
  __syncwarp();
  float rv[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) rv[v] = 4 * lane + v < d.c ? rbuf[4 * lane + v] : 0.f;
  // pair tables: lane l holds list positions 4l .. 4l+3, i.e. pairs 2l, 2l+1
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int p = 4 * lane + 2 * h;
    if (p < d.c) {
      const float r0 = rv[2 * h], r1 = p + 1 < d.c ? rv[2 * h + 1] : 0.f;
      float4* tab = reinterpret_cast<float4*>(buf) + (p >> 1) * 4;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const float t1 = g4 == 1 ? r1 : (g4 == 3 ? -r1 : 0.f);   // code of the odd position
        tab[g4] = make_float4(t1, r0 + t1, t1, t1 - r0);         // even position 00 01 10 11
      }
    }
  }
  return (e_raw < 0 || e_raw >= d.E) ? 0 : e_raw;
}

// A team of tw warps owns whole units (team k takes the CTA's units k,
// k + nteams, ...).  Per unit the team's first warp writes the pair tables,
// the screened coordinates and the expert id into one of two unit buffers.
// The unit's coordinate records are copied into shared memory in chunks of
// cc positions with asynchronous 16-byte copies, chunk j + 1 in flight while
// chunk j is summed.  Thread tt owns WPT 4-byte code words of every record
// (16 channels each) and sums them in registers, two coordinates per table
// read.  A warp publishes a unit once the next one is computed, so the
// release finds the stores long done.
template <int WPT, bool T5, bool STK>
__device__ void screen_team(const Params& P, unsigned char* tsm, int team, int tt,
                            uint32_t e5_base) {
  const Dims& d = P.d;
  const ScreenPlan& sp = P.sp;
  const int lane = threadIdx.x & 31, tw_i = tt >> 5;
  constexpr int CPW = T5 ? 20 : 16;   // channels of a 4-byte code word
  const int TT = 32 * sp.tw, R16 = d.runW, W4 = 2 * R16;
  const int units = P.B * d.topk * d.nb, nctas = gridDim.x;
  const uint32_t S2 = 2u * (uint32_t)d.S;
  const int P16 = (int)(S2 / 16);                // 16-byte pieces per record
  volatile int* flag = reinterpret_cast<volatile int*>(tsm);   // [2 + n % 2] expert id of unit n
  unsigned char* ubuf = tsm + 256;                              // [2][buf_bytes]
  unsigned char* stage = ubuf + 2 * (size_t)sp.buf_bytes;       // [2][stage_bytes]
  uint32_t off[WPT];
  int gv[WPT], jw[WPT];
  bool has[WPT];
#pragma unroll
  for (int x = 0; x < WPT; ++x) {
    const int w = tt + TT * x;
    has[x] = w < W4;
    gv[x] = has[x] ? w / R16 : 0;
    jw[x] = has[x] ? w % R16 : 0;
    off[x] = (uint32_t)(gv[x] * d.S + jw[x] * 4);
  }
  auto unit_of = [&](int n) { return blockIdx.x + (team + n * sp.nteams) * nctas; };
  if (unit_of(0) >= units) return;               // no unit for this team
  // The first warp rotates and screens the unit's (token, block) itself, so
  // the team waits on no other CTA; it keeps the next unit's sigma x (and the
  // expert id) in registers until it writes that unit's buffer.
  UnitInput uin;
  auto load_list = [&](int uu) {
    const int b = uu % d.nb, ts = uu / d.nb, t = ts / d.topk;
    if (STK) {   // a stacked layer: token t's input comes from the layer before
      int ok = 1;
      if (lane == 0) ok = wait_at_least(P, P.xwait + t, 1u);
      __shfl_sync(0xffffffffu, ok, 0);   // on a timeout the abort flag ends the launch
      __syncwarp();
    }
    unit_issue<STK>(P, t, b, lane, uin);
    if (lane == 0 && team == 0) TRACE_POINT(1);
  };
  auto write_unit = [&](int n) {   // first warp: unit n's tables, coordinates and expert
    unsigned char* buf = ubuf + (size_t)(n & 1) * sp.buf_bytes;
    const int e = build_unit<STK>(P, buf, unit_of(n), lane, uin, team);
    if (lane == 0) flag[2 + (n & 1)] = e;
  };
  // asynchronous copies of chunk j (unit j / nch, chunk j % nch) into stage j % 2
  auto issue = [&](int j) {
    const int n = j / sp.nch, ch = j % sp.nch;
    const int u = unit_of(n);
    if (u < units) {
      const unsigned char* buf = ubuf + (size_t)(n & 1) * sp.buf_bytes;
      const uint8_t* coords = buf + sp.coord_off;
      const int b = u % d.nb, e = flag[2 + (n & 1)];
      const uint8_t* rec = P.codes + ((size_t)e * d.nb + b) * kBlock * S2;
      const int p0 = ch * sp.cc, npos = min(sp.cc, d.c - p0);
      const uint32_t dst0 = smem_addr(stage + (size_t)(j & 1) * sp.stage_bytes);
      if (TT % P16 == 0) {
        // every thread keeps one 16-byte piece offset: records tt / P16, + TT / P16, ...
        const int o = tt % P16, dp = TT / P16;
        const uint32_t dst_o = dst0 + 16u * (uint32_t)o;
        const uint8_t* src_o = rec + 16 * o;
        for (int p = tt / P16; p < npos; p += dp)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_o + (uint32_t)p * S2),
                       "l"(src_o + (size_t)coords[p0 + p] * S2)
                       : "memory");
      } else {
        const int pieces = npos * P16;
        int p = tt / P16, o = tt % P16;
        const int dp = TT / P16, dq = TT % P16;
        for (int q = tt; q < pieces; q += TT) {
          const uint8_t* src = rec + (size_t)coords[p0 + p] * S2 + 16 * o;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst0 + (uint32_t)p * S2 + 16u * o),
                       "l"(src)
                       : "memory");
          p += dp;
          o += dq;
          if (o >= P16) {
            o -= P16;
            ++p;
          }
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if (tw_i == 0) {
    load_list(unit_of(0));
    write_unit(0);
    if (lane == 0 && team == 0) TRACE_POINT(18);
    if (unit_of(1) < units) load_list(unit_of(1));
  }
  team_sync(team, TT);
  issue(0);
  if (tt == 0 && team == 0) TRACE_POINT(19);
  float acc[WPT][CPW];
  uint4 al[WPT][3];
  int pend = -1;
  for (int j = 0;; ++j) {
    const int n = j / sp.nch, ch = j % sp.nch;
    const int u = unit_of(n);
    if (u >= units) break;
    team_sync(team, TT);   // chunk j - 1 is summed by everyone: its stage and unit buffer are free
    // chunk j + 1 from this unit's buffer goes out before the next unit's
    // rotation and selection, which then run while it is in flight
    const bool early = ch + 1 < sp.nch;
    if (early) issue(j + 1);
    if (ch == 0 && tw_i == 0 && unit_of(n + 1) < units) {
      write_unit(n + 1);
      if (unit_of(n + 2) < units) load_list(unit_of(n + 2));   // in flight while unit n is summed
    }
    if (ch == 0) team_sync(team, TT);   // unit n + 1's buffer is written
    if (!early) issue(j + 1);
    if (tt == 0 && team == 0 && j == 0) TRACE_POINT(20);
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    team_sync(team, TT);   // every thread's copies of chunk j have landed
    if (tt == 0 && team == 0) TRACE_POINT(3);
    const int e = flag[2 + (n & 1)];
    const int ts = u / d.nb, b = u % d.nb;
    // alpha of the thread's channels: requested with the first chunk when
    // registers allow, else after the last
    constexpr bool kAlphaEarly = WPT < 3;
    auto load_alpha = [&]() {
#pragma unroll
      for (int x = 0; x < WPT; ++x) {
        const __half* a0 = P.scales + (((size_t)e * d.nb + b) * 2 + gv[x]) * d.I + CPW * jw[x];
        if (!T5) {
          const uint4* a4 = reinterpret_cast<const uint4*>(a0);
          al[x][0] = has[x] ? ldg_nc4(a4) : make_uint4(0u, 0u, 0u, 0u);
          al[x][1] = has[x] ? ldg_nc4(a4 + 1) : make_uint4(0u, 0u, 0u, 0u);
        } else {   // 20 halves: five 8-byte groups, those past I not read
          uint32_t h[10];
#pragma unroll
          for (int q = 0; q < 5; ++q) {
            const bool in = has[x] && CPW * jw[x] + 4 * q < d.I;
            const uint2 v = in ? ldg_stream2(reinterpret_cast<const uint2*>(a0 + 4 * q)) : make_uint2(0u, 0u);
            h[2 * q] = v.x;
            h[2 * q + 1] = v.y;
          }
          al[x][0] = make_uint4(h[0], h[1], h[2], h[3]);
          al[x][1] = make_uint4(h[4], h[5], h[6], h[7]);
          al[x][2] = make_uint4(h[8], h[9], 0u, 0u);
        }
      }
    };
    if (ch == 0) {
#pragma unroll
      for (int x = 0; x < WPT; ++x)
#pragma unroll
        for (int q = 0; q < CPW; ++q) acc[x][q] = 0.f;
      if (kAlphaEarly) load_alpha();
    }
    const uint32_t stg = smem_addr(stage + (size_t)(j & 1) * sp.stage_bytes);
    const uint32_t lut_base = smem_addr(ubuf + (size_t)(n & 1) * sp.buf_bytes);   // 256-aligned
    const int pbase = ch * sp.cc / 2;   // the chunk's first pair in the unit's list
    const int npos = min(sp.cc, d.c - ch * sp.cc), np = (npos + 1) >> 1;
    constexpr int kU = WPT == 3 ? 1 : 4;   // pairs per shared-memory load batch
    for (int pp0 = 0; pp0 < np; pp0 += kU) {
      uint32_t wa[kU][WPT], wb[kU][WPT];
#pragma unroll
      for (int v = 0; v < kU; ++v) {
        const int pp = pp0 + v;
#pragma unroll
        for (int x = 0; x < WPT; ++x) {
          // an odd count's last pair reads a spare record slot (its table ignores it)
          const bool in = pp < np && has[x];
          wa[v][x] = in ? lds_u32(stg + (uint32_t)(2 * pp) * S2 + off[x]) : 0u;
          wb[v][x] = in ? lds_u32(stg + (uint32_t)(2 * pp + 1) * S2 + off[x]) : 0u;
        }
      }
#pragma unroll
      for (int v = 0; v < kU; ++v) {
        // table of pair pg: 256-byte block pg / 4 (bytes 1-3 of the address),
        // 64 (pg % 4) + 4 index in the low byte; index 0 of a table is 0
        const int pg = pbase + min(pp0 + v, np - 1);
        const uint32_t blk = lut_base + 256u * (uint32_t)(pg >> 2);
        const uint32_t sub = (uint32_t)(pg & 3) * 0x40404040u;
#pragma unroll
        for (int x = 0; x < WPT; ++x) {
          if (T5) {
            // byte k of each word: five channels; the expansion table gives
            // their 2-bit codes a nibble apart, so that nibble m of
            // ea | eb << 2 is channel 5k + m's pair index
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t ba = __byte_perm(wa[v][x], 0u, 0x4440u + k);
              const uint32_t bb = __byte_perm(wb[v][x], 0u, 0x4440u + k);
              // (masked: the spare record slot of an odd count holds stale bytes)
              const uint32_t z = (lds_u32(e5_base + 4u * ba) & 0x33333u) |
                                 ((lds_u32(e5_base + 4u * bb) << 2) & 0xCCCCCu);
              const uint32_t we = ((z << 2) & 0x3C3C3C3Cu) | sub;   // channels 5k, 5k + 2, 5k + 4
              const uint32_t wo = ((z >> 2) & 0x3C3C3C3Cu) | sub;   // channels 5k + 1, 5k + 3
              acc[x][5 * k] += lds_f32(__byte_perm(we, blk, 0x7650u));
              acc[x][5 * k + 1] += lds_f32(__byte_perm(wo, blk, 0x7650u));
              acc[x][5 * k + 2] += lds_f32(__byte_perm(we, blk, 0x7651u));
              acc[x][5 * k + 3] += lds_f32(__byte_perm(wo, blk, 0x7651u));
              acc[x][5 * k + 4] += lds_f32(__byte_perm(we, blk, 0x7652u));
            }
            continue;
          }
          // nibble mm: (even-position code) | (odd-position code) << 2 of channel 2mm / 2mm+1
          const uint32_t ze = (wa[v][x] & 0x33333333u) | ((wb[v][x] << 2) & 0xCCCCCCCCu);
          const uint32_t zo = ((wa[v][x] >> 2) & 0x33333333u) | (wb[v][x] & 0xCCCCCCCCu);
          // byte k: 4 x (nibble 2k or 2k+1) + 64 (pg % 4), i.e. the address's low byte
          const uint32_t bee = ((ze << 2) & 0x3C3C3C3Cu) | sub;   // channels 4k
          const uint32_t beo = ((ze >> 2) & 0x3C3C3C3Cu) | sub;   // channels 4k + 2
          const uint32_t boe = ((zo << 2) & 0x3C3C3C3Cu) | sub;   // channels 4k + 1
          const uint32_t boo = ((zo >> 2) & 0x3C3C3C3Cu) | sub;   // channels 4k + 3
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t sel = 0x7650u + kb;   // low byte from the index word, the rest from blk
            acc[x][4 * kb] += lds_f32(__byte_perm(bee, blk, sel));
            acc[x][4 * kb + 1] += lds_f32(__byte_perm(boe, blk, sel));
            acc[x][4 * kb + 2] += lds_f32(__byte_perm(beo, blk, sel));
            acc[x][4 * kb + 3] += lds_f32(__byte_perm(boo, blk, sel));
          }
        }
      }
    }
    if (ch != sp.nch - 1) continue;
    if (!kAlphaEarly) load_alpha();
    if (pend >= 0) publish_unit(P, pend, lane);
#pragma unroll
    for (int x = 0; x < WPT; ++x) {
      if (!has[x]) continue;
      const uint32_t hw[12] = {al[x][0].x, al[x][0].y, al[x][0].z, al[x][0].w,
                               al[x][1].x, al[x][1].y, al[x][1].z, al[x][1].w,
                               al[x][2].x, al[x][2].y, al[x][2].z, al[x][2].w};
#pragma unroll
      for (int q = 0; q < CPW / 2; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[q]));
        acc[x][2 * q] *= f.x;
        acc[x][2 * q + 1] *= f.y;
      }
      float4* out = reinterpret_cast<float4*>(
          P.partial + (((size_t)ts * d.nb + b) * 2 + gv[x]) * d.I + CPW * jw[x]);
#pragma unroll
      for (int q = 0; q < CPW / 4; ++q)   // channels past I (the last five-trit word) are not stored
        if (!T5 || CPW * jw[x] + 4 * q < d.I)
          out[q] = make_float4(acc[x][4 * q], acc[x][4 * q + 1], acc[x][4 * q + 2], acc[x][4 * q + 3]);
    }
    pend = ts;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (pend >= 0) publish_unit(P, pend, lane);
  if (tt == 0) TRACE_POINT(4);
}

// Phase 1a of a CTA: its teams' screen units, WPT code words per thread.
// fg: the warps that screen (the table is built between its barriers).
template <int WPT, bool T5, bool STK>
__device__ void screen_compute(const Params& P, unsigned char* smem, int warp, const Grp& fg) {
  const ScreenPlan& sp = P.sp;
  const uint32_t e5_base = smem_addr(smem + sp.e5_off);
  if (T5) {   // the expansion table of a five-trit byte: its five 2-bit codes a nibble apart
    for (int v = fg.tid; v < 256; v += fg.nt) {   // bytes above 242 do not occur: 0
      uint32_t z = 0;
      int q = v < 243 ? v : 0;
#pragma unroll
      for (int m = 0; m < 5; ++m) {
        const int dg = q % 3;
        q /= 3;
        z |= (dg == 1 ? 1u : (dg == 2 ? 3u : 0u)) << (4 * m);
      }
      reinterpret_cast<uint32_t*>(smem + sp.e5_off)[v] = z;
    }
    fg.sync();
  }
  const int team = warp / sp.tw;
  if (team >= sp.nteams) return;   // warps left over by the team size
  const int tt = (warp % sp.tw) * 32 + (threadIdx.x & 31);
  screen_team<WPT, T5, STK>(P, smem + (size_t)team * sp.team_bytes, team, tt, e5_base);
}

// Score the channels of one (token, slot) once all its blocks are in: sum
// the block partials in block order, s = w ||d|| |phi(ghat) vhat|.  Returns
// -1 on abort, 1 when this was the token's last slot to be scored (the CTA
// then runs the token's top-k), else 0.
template <bool SH>
__device__ int score_task(const Params& P, const Grp& grp, int ts, int* flag, unsigned char* smem) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int t = ts / d.topk, slot = ts % d.topk, I = d.I;
  // the routing and the first channels' down norms are inputs: requested
  // before the wait for the slot's screen units
  int e = P.ids_in[ts];
  if (e < 0 || e >= d.E) e = 0;
  const float wv = P.w_in[ts];
  float dn0[2] = {0.f, 0.f};
  if (grp.tid < I) dn0[0] = __ldg(P.dnorm + (size_t)e * I + grp.tid);
  if (grp.tid + grp.nt < I) dn0[1] = __ldg(P.dnorm + (size_t)e * I + grp.tid + grp.nt);
  if (grp.tid == 0) {
    *flag = wait_at_least(P, P.sync + so.slot + ts, (uint32_t)(d.nb * P.sp.tw + P.stall));
    if (*flag) P.sync[so.slot + ts] = 0u;   // every unit is in: the count is not read again
  }
  grp.sync();
  if (!*flag) return -1;
  if (grp.tid == 0) TRACE_POINT(6);
  const float* pg0 = P.partial + ((size_t)ts * d.nb) * 2 * I;
  // channels i and i + grp.nt together: all their block loads first, then
  // the sums in block order
  for (int i = grp.tid; i < I; i += 2 * grp.nt) {
    const int i2 = i + grp.nt;
    const bool two = i2 < I;
    const bool first = i < grp.nt;
    const float dn[2] = {first ? dn0[0] : __ldg(P.dnorm + (size_t)e * I + i),
                         two ? (first ? dn0[1] : __ldg(P.dnorm + (size_t)e * I + i2)) : 0.f};
    float g[2] = {0.f, 0.f}, v[2] = {0.f, 0.f};
    int bb = 0;
    for (; bb + 16 <= d.nb; bb += 16) {
      float gg[2][16], vv[2][16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float* pb = pg0 + (size_t)(bb + u) * 2 * I;
        gg[0][u] = __ldcg(pb + i);
        vv[0][u] = __ldcg(pb + I + i);
        gg[1][u] = two ? __ldcg(pb + i2) : 0.f;
        vv[1][u] = two ? __ldcg(pb + I + i2) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          g[h] += gg[h][u];
          v[h] += vv[h][u];
        }
      }
    }
    for (; bb < d.nb; ++bb) {
      const float* pb = pg0 + (size_t)bb * 2 * I;
      g[0] += __ldcg(pb + i);
      v[0] += __ldcg(pb + I + i);
      if (two) {
        g[1] += __ldcg(pb + i2);
        v[1] += __ldcg(pb + I + i2);
      }
    }
    if (grp.tid == 0) TRACE_POINT(21);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h == 1 && !two) break;
      const int ii = h ? i2 : i;
      const float pv = silu_f(g[h]) * v[h];
      float sc = wv * dn[h] * fabsf(pv);
      if (d.rho_rank) {
        // the expected squared output error that skipping leaves:
        // w^2 (p^2 max(|d|^2 - |b|^2, 0) + var(a) |d|^2), var(a) to first order
        float var_g = 0.f, var_v = 0.f;
        for (int bb2 = 0; bb2 < d.nb; ++bb2) {
          const float r2 = __ldcg(P.rn2 + (size_t)t * d.nb + bb2);
          const __half* rb = P.rho + (((size_t)e * d.nb + bb2) * 2) * I + ii;
          var_g = fmaf(__half2float(rb[0]), r2, var_g);
          var_v = fmaf(__half2float(rb[I]), r2, var_v);
        }
        const float sg = 1.f / (1.f + expf(-g[h]));
        const float dphi = sg * (1.f + g[h] * (1.f - sg));
        const float phi = g[h] * sg;
        const float var_a = (dphi * v[h]) * (dphi * v[h]) * var_g + phi * phi * var_v;
        const float dn2 = dn[h] * dn[h];
        const float keep2 = fmaxf(dn2 - __ldg(P.bnorm2 + (size_t)e * I + ii), 0.f);
        sc = wv * wv * (pv * pv * keep2 + var_a * dn2);
      }
      const size_t o = (size_t)t * d.N + (size_t)slot * I + ii;
      P.ghat[o] = g[h];
      P.vhat[o] = v[h];
      P.p[o] = pv;
      P.score[o] = sc;
    }
  }
  grp.sync();
  if (SH) {
    // every output chunk of the batch adds into y[t]: start it from zero
    // before the batch's set is released
    if (slot == 0)
      for (int h = grp.tid; h < d.H; h += grp.nt) P.y[(size_t)t * d.H + h] = 0.f;
    shared_after_score(P, e, smem, flag);
    return 0;
  }
  if (grp.tid == 0) {
    // releases this slot's scores; the last slot in also acquires the others'
    const uint32_t prev = atom_add_acq_rel(P.sync + so.tok + t, 1u);
    *flag = prev == (uint32_t)(d.topk - 1);
    if (*flag) P.sync[so.tok + t] = 0u;   // the token's last slot: no more adds
    TRACE_POINT(7);
  }
  grp.sync();
  return *flag ? 1 : 0;
}

// ------------------------------- phase 2 -----------------------------------
__device__ __forceinline__ void dot8(const uint4& q, const float4& xa, const float4& xb, float& s) {
  s = fmaf(bf16_lo(q.x), xa.x, s); s = fmaf(bf16_hi(q.x), xa.y, s);
  s = fmaf(bf16_lo(q.y), xa.z, s); s = fmaf(bf16_hi(q.y), xa.w, s);
  s = fmaf(bf16_lo(q.z), xb.x, s); s = fmaf(bf16_hi(q.z), xb.y, s);
  s = fmaf(bf16_lo(q.w), xb.z, s); s = fmaf(bf16_hi(q.w), xb.w, s);
}


// Count `count` finished phase-2 items of token pt (pt < 0: none): a release
// add after the warp's barrier, so the items' stores come first.  Called
// right after the next item's first loads are issued.
__device__ __forceinline__ void publish_item(const Params& P, int pt, int count, int lane) {
  if (pt < 0) return;
  __syncwarp();
  if (lane == 0) red_add_release(P.sync + sync_offsets(P.d).exact + pt, (uint32_t)count);
}

// Slot s's sanitised expert id / weight of token t, lane-distributed (topk <= 64).
__device__ __forceinline__ int slot_expert(int e0, int e1, int slot) {
  const int a = __shfl_sync(0xffffffffu, e0, slot & 31);
  const int b = __shfl_sync(0xffffffffu, e1, slot & 31);
  return slot < 32 ? a : b;
}

struct TokenSlots {
  int e0, e1;
  float w0, w1;
};

// Token t's routing, lane-distributed, from the inputs, with the screen's
// sanitising (an expert id out of range reads as expert 0): independent of
// the decode's own writes, so it can be requested before any wait.
__device__ __forceinline__ TokenSlots input_token_slots(const Params& P, int t, int lane) {
  const Dims& d = P.d;
  TokenSlots ts;
  ts.e0 = lane < d.topk ? __ldg(P.ids_in + t * d.topk + lane) : 0;
  ts.e1 = lane + 32 < d.topk ? __ldg(P.ids_in + t * d.topk + lane + 32) : 0;
  ts.w0 = lane < d.topk ? __ldg(P.w_in + t * d.topk + lane) : 0.f;
  ts.w1 = lane + 32 < d.topk ? __ldg(P.w_in + t * d.topk + lane + 32) : 0.f;
  return ts;
}
__device__ __forceinline__ void sanitise_slots(const Dims& d, TokenSlots& ts) {
  if (ts.e0 < 0 || ts.e0 >= d.E) ts.e0 = 0;
  if (ts.e1 < 0 || ts.e1 >= d.E) ts.e1 = 0;
}

__device__ __forceinline__ TokenSlots load_token_slots(const Params& P, int t, int lane) {
  const Dims& d = P.d;
  TokenSlots ts;
  ts.e0 = lane < d.topk ? __ldcg(P.ids_ws + t * d.topk + lane) : 0;
  ts.e1 = lane + 32 < d.topk ? __ldcg(P.ids_ws + t * d.topk + lane + 32) : 0;
  ts.w0 = lane < d.topk ? __ldcg(P.w_ws + t * d.topk + lane) : 0.f;
  ts.w1 = lane + 32 < d.topk ? __ldcg(P.w_ws + t * d.topk + lane + 32) : 0.f;
  return ts;
}

// Kept channel q of the batch's set: its gate and up rows serve every token
// slot routed to its expert, four tokens per pass over the rows; w a lands in
// the token's dense [N] slot of wa.
// gid: the kept channel's global id; info: its expert's first elist entry *
// 16384 + the expert's token-slot count (read ahead by the caller).
__device__ void shared_kept_item(const Params& P, int gid, int info, int lane) {
  const Dims& d = P.d;
  const int e = gid / d.I, i = gid - e * d.I;
  const int l0 = info >> 14, l1 = l0 + (info & 16383);
  const size_t row = (size_t)e * d.I + i;
  const uint4* g4 = reinterpret_cast<const uint4*>(P.G + row * d.H);
  const uint4* v4 = reinterpret_cast<const uint4*>(P.V + row * d.H);
  const int n8 = d.H / 8;
  constexpr int kU = 8, kTG = 4;
  for (int g0 = l0; g0 < l1; g0 += kTG) {
    const int ng = min(kTG, l1 - g0);
    int tsl[kTG];
    float sg[kTG], sv[kTG];
#pragma unroll
    for (int u = 0; u < kTG; ++u) {   // independent of the rows' loads below
      tsl[u] = u < ng ? __ldcg(P.elist + g0 + u) : 0;
      sg[u] = 0.f;
      sv[u] = 0.f;
    }
    for (int h8 = lane; h8 < n8; h8 += 32 * kU) {
      uint4 gq[kU], vq[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const bool in = h8 + 32 * u < n8;
        gq[u] = in ? ldg_nc4(g4 + h8 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
        vq[u] = in ? ldg_nc4(v4 + h8 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int tg = 0; tg < kTG; ++tg) {
        if (tg >= ng) break;
        const float4* x4 = reinterpret_cast<const float4*>(P.x + (size_t)(tsl[tg] / d.topk) * d.H);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (h8 + 32 * u >= n8) break;
          const float4 xa = x4[2 * (h8 + 32 * u)], xb = x4[2 * (h8 + 32 * u) + 1];
          dot8(gq[u], xa, xb, sg[tg]);
          dot8(vq[u], xa, xb, sv[tg]);
        }
      }
    }
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg) {
      if (tg >= ng) break;
      const float a = warp_sum(sg[tg]), b = warp_sum(sv[tg]);
      if (lane == 0) {
        const int ts = tsl[tg], t = ts / d.topk, slot = ts - t * d.topk;
        P.wa[(size_t)t * d.N + (size_t)slot * d.I + i] = __ldcg(P.w_ws + ts) * silu_f(a) * b;
      }
    }
  }
}

__device__ void recovery_item(const Params& P, int t, int ch, int lane, int pend_t, int pend_n) {
  // 64 channels: lane l takes channels l and l + 32 (full b rows), then the
  // warp transposes and sums the 32 lane vectors; lane j ends with component j
  const Dims& d = P.d;
  const int n0 = ch * 64;
  const int slot = n0 / d.I;
  const int e = __ldcg(P.ids_ws + t * d.topk + slot);
  const float wv = __ldcg(P.w_ws + t * d.topk + slot);
  const uint32_t kb0 = __ldcg(P.keptbits + (size_t)t * (d.N / 32) + ch * 2);
  const uint32_t kb1 = __ldcg(P.keptbits + (size_t)t * (d.N / 32) + ch * 2 + 1);
  const bool s0 = !((kb0 >> lane) & 1u), s1 = !((kb1 >> lane) & 1u);
  const float c0 = s0 ? wv * __ldcg(P.p + (size_t)t * d.N + n0 + lane) : 0.f;
  const float c1 = s1 ? wv * __ldcg(P.p + (size_t)t * d.N + n0 + 32 + lane) : 0.f;
  publish_item(P, pend_t, pend_n, lane);
  const __half* b0 = P.bco + ((size_t)e * d.I + (n0 % d.I) + lane) * d.r;
  const __half* b1 = b0 + (size_t)32 * d.r;
  for (int j0 = 0; j0 < d.r; j0 += 32) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
    const int jn = min(32, d.r - j0);
    if ((d.r & 7) == 0) {
      // rows are 16-byte aligned: 8 components per load
      uint4 q0[4], q1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = 8 * u < jn;
        q0[u] = (in && s0) ? ldg_nc4(b0 + j0 + 8 * u) : make_uint4(0, 0, 0, 0);
        q1[u] = (in && s1) ? ldg_nc4(b1 + j0 + 8 * u) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w0[4] = {q0[u].x, q0[u].y, q0[u].z, q0[u].w};
        const uint32_t w1[4] = {q1[u].x, q1[u].y, q1[u].z, q1[u].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w0[h]));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w1[h]));
          v[8 * u + 2 * h] = fmaf(c1, f1.x, c0 * f0.x);
          v[8 * u + 2 * h + 1] = fmaf(c1, f1.y, c0 * f0.y);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < jn) {
          const float x0 = s0 ? c0 * __half2float(b0[j0 + j]) : 0.f;
          v[j] = s1 ? fmaf(c1, __half2float(b1[j0 + j]), x0) : x0;
        }
      }
    }
    // recursive halving: after 5 rounds lane l holds the warp sum of component l
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int j = 0; j < off; ++j) {
        const float send = upper ? v[j] : v[j + off];
        const float keep = upper ? v[j + off] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    if (lane < jn) atomicAdd(P.cvec + (size_t)t * d.r + j0 + lane, v[0]);
  }
}

// Count one output contribution to column block cb of token t in a stacked
// layer (a CTA's rows, or one recovery chunk of the block); true for the
// contribution that completes the block (`total` of them), whose warp then
// carries it.
__device__ __forceinline__ bool count_block(const Params& P, int t, int cb, int ncb, uint32_t total) {
  uint32_t* w = P.sync + sync_offsets(P.d).cbdone + t * ncb + cb;
  if (atom_add_acq_rel(w, 1u) + 1u != total) return false;
  *w = 0u;   // the block's last contribution: no more adds this launch
  return true;
}

// CTAs whose item ranges hold kept channels of token t (items are dealt in
// runs of ipw per warp, kWarps runs per CTA, token-major, kept items first).
__device__ __forceinline__ int kept_ctas(long long t, long long per_tok, int k, long long ipw) {
  if (k <= 0) return 0;
  const long long span = (long long)kWarps * ipw;
  return (int)((t * per_tok + k - 1) / span - (t * per_tok) / span + 1);
}

// ---------------- exact channels and their output, per CTA (per-token) ----------------
// Kept channel n (kept-list position qi) of token t: a = phi(g^T x)(v^T x)
// from the native rows.  w a and the channel's row go to the CTA's lists
// (wa_s, row_s; global wa when they do not fit), and the transposed down row
// heads for L2: the CTA adds every kept row's output once its channels are in.
__device__ void kept_item_cta(const Params& P, int t, int qi, int n, const TokenSlots& sl, int lane,
                              float* wa_s, int* row_s) {
  const Dims& d = P.d;
  const int slot = n / d.I, i = n % d.I;
  const int e = slot_expert(sl.e0, sl.e1, slot);
  const float wslot =
      __int_as_float(slot_expert(__float_as_int(sl.w0), __float_as_int(sl.w1), slot));
  const size_t row = (size_t)e * d.I + i;
  const uint64_t pol = policy_evict_first();
  const uint4* g4 = reinterpret_cast<const uint4*>(P.G + row * d.H);
  const uint4* v4 = reinterpret_cast<const uint4*>(P.V + row * d.H);
  const float4* x4 = reinterpret_cast<const float4*>(P.x + (size_t)t * d.H);
  const int n8 = d.H / 8;
  float sg = 0.f, sv = 0.f;
  int h8 = lane;
  constexpr int kU = 8;   // 16-byte loads per lane and row issued together
  for (; h8 + 32 * (kU - 1) < n8; h8 += 32 * kU) {
    uint4 gq[kU], vq[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      gq[u] = ldg_nc4_hint(g4 + h8 + 32 * u, pol);
      vq[u] = ldg_nc4_hint(v4 + h8 + 32 * u, pol);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float4 xa = x4[2 * (h8 + 32 * u)], xb = x4[2 * (h8 + 32 * u) + 1];
      dot8(gq[u], xa, xb, sg);
      dot8(vq[u], xa, xb, sv);
    }
  }
  for (; h8 < n8; h8 += 32) {
    const uint4 gq = ldg_nc4_hint(g4 + h8, pol), vq = ldg_nc4_hint(v4 + h8, pol);
    const float4 xa = x4[2 * h8], xb = x4[2 * h8 + 1];
    dot8(gq, xa, xb, sg);
    dot8(vq, xa, xb, sv);
  }
  sg = warp_sum(sg);
  sv = warp_sum(sv);
  if (lane == 0) {
    const float wa = wslot * silu_f(sg) * sv;
    if (wa_s) {
      wa_s[qi] = wa;
      row_s[qi] = (int)row;
    } else {
      P.wa[(size_t)t * d.N + qi] = wa;
    }
  }
}

// ------------------------------- output ------------------------------------
__device__ __forceinline__ void axpy8(float c, const uint4& v, float* acc) {
  acc[0] = fmaf(c, bf16_lo(v.x), acc[0]); acc[1] = fmaf(c, bf16_hi(v.x), acc[1]);
  acc[2] = fmaf(c, bf16_lo(v.y), acc[2]); acc[3] = fmaf(c, bf16_hi(v.y), acc[3]);
  acc[4] = fmaf(c, bf16_lo(v.z), acc[4]); acc[5] = fmaf(c, bf16_hi(v.z), acc[5]);
  acc[6] = fmaf(c, bf16_lo(v.w), acc[6]); acc[7] = fmaf(c, bf16_hi(v.w), acc[7]);
}

constexpr int kOutCols = 256;        // columns of an output block: 8 per lane
constexpr int kOutBatch = 12;        // kept rows whose loads a warp issues together

struct OutPlan {
  int ncb;   // output blocks
  int R;     // kept-row chunks per (token, block)
  int RC;    // kept rows per chunk
  int NR;    // chunks per (token, block): R, plus the recovery chunks of U c when k < N
};

__device__ __forceinline__ void axpy8h(float c, const uint4& v, float* acc) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
    acc[2 * h] = fmaf(c, f.x, acc[2 * h]);
    acc[2 * h + 1] = fmaf(c, f.y, acc[2 * h + 1]);
  }
}

// The CTA's output of token t's kept rows [q0, q1) of its kept list (their w a
// in wa_s / row_s at [s0, s0 + q1 - q0), or in global wa): 256-column chunks,
// 8 columns a lane, each chunk's rows split between kWarps / chunks warps; a
// warp loads its rows' 16-byte down pieces kO at a time, sums them in
// registers and adds its 8 columns into y once.
__device__ void cta_output(const Params& P, int t, int q0, int q1, const float* wa_s,
                           const int* row_s, int s0, const TokenSlots& sl, int warp, int lane,
                           int nw = kWarps) {
  const Dims& d = P.d;
  const int nchunk = (d.H + kOutCols - 1) / kOutCols;
  const int rsplit = max(1, nw / nchunk);              // warps per chunk
  const int nr = q1 - q0, per = (nr + rsplit - 1) / rsplit;
  const uint64_t pol = policy_evict_first();            // the last read of these rows
  constexpr int kO = 12;
  for (int wi = warp; wi < nchunk * rsplit; wi += nw) {
    const int ch = wi % nchunk, part = wi / nchunk;
    const int r_lo = q0 + part * per, r_hi = min(q1, r_lo + per);
    if (r_lo >= r_hi) continue;
    const int c0 = ch * kOutCols + 8 * lane;
    const bool on = c0 < d.H;                          // H is a multiple of 8
    float acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = 0.f;
    for (int r0 = r_lo; r0 < r_hi; r0 += kO) {
      uint4 v[kO];
      float c[kO];
#pragma unroll
      for (int u = 0; u < kO; ++u) {
        const int r = r0 + u;
        int row = 0;
        c[u] = 0.f;
        if (r < r_hi) {
          if (wa_s) {
            row = row_s[s0 + r - q0];
            c[u] = wa_s[s0 + r - q0];
          } else {
            const int n = __ldcg(P.kept + (size_t)t * d.N + r);
            const int slot = n / d.I;
            row = slot_expert(sl.e0, sl.e1, slot) * d.I + (n - slot * d.I);
            c[u] = __ldcg(P.wa + (size_t)t * d.N + r);
          }
        }
        v[u] = r < r_hi && on ? ldg_nc4_hint(P.Dt + (size_t)row * d.H + c0, pol)
                              : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kO; ++u) axpy8(c[u], v[u], acc);
    }
    if (on) {
      float4* yo = reinterpret_cast<float4*>(P.y + (size_t)t * d.H + c0);
      atomicAdd(yo, make_float4(acc[0], acc[1], acc[2], acc[3]));
      atomicAdd(yo + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
    }
  }
}

// ------------------------------ stack hand-off ------------------------------
// The warp that completes output block cb of token t: hnext = hres + y on the
// block's 256 columns (fp32), and, when a next layer reads it, the block's sum
// of squares (fp64) into the token's sum.  The token's last block sets the
// next layer's input scale 1 / sqrt(sum / H + 1e-6) and releases the token.
__device__ void carry_block(const Params& P, int t, int cb, int ncb, int lane) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const size_t row = (size_t)t * d.H;
  const int c0 = cb * kOutCols + lane * 8;
  double ss = 0.0;
  if (c0 < d.H) {
    const float4* h4 = reinterpret_cast<const float4*>(P.hres + row + c0);
    const float4* y4 = reinterpret_cast<const float4*>(P.y + row + c0);
    const float4 a0 = __ldcg(h4), a1 = __ldcg(h4 + 1), b0 = __ldcg(y4), b1 = __ldcg(y4 + 1);
    const float4 v0 = make_float4(a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w);
    const float4 v1 = make_float4(a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w);
    float4* o4 = reinterpret_cast<float4*>(P.hnext + row + c0);
    o4[0] = v0;
    o4[1] = v1;
    ss = (double)v0.x * v0.x + (double)v0.y * v0.y + (double)v0.z * v0.z + (double)v0.w * v0.w +
         (double)v1.x * v1.x + (double)v1.y * v1.y + (double)v1.z * v1.z + (double)v1.w * v1.w;
  }
  if (!P.xscale_next) return;   // the last layer: h_out only
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  double* sum = reinterpret_cast<double*>(P.sync + so.ssum) + t;
  __syncwarp();
  uint32_t prev = 0;
  if (lane == 0) {
    atomicAdd(sum, ss);
    prev = atom_add_acq_rel(P.sync + so.tokdone + t, 1u);
    if (prev == (uint32_t)(ncb - 1)) {
      const double tot = __ldcg(sum);
      // the token's last block: its count and sum are not read again this launch
      P.sync[so.tokdone + t] = 0u;
      *sum = 0.0;
      P.xscale_next[t] = (float)(1.0 / sqrt(tot / d.H + 1e-6));
      st_release(P.xnext_ready + t, 1u);
    }
  }
}

// One warp item: columns cb*256 + 8 lane .. +7 of token t over kept rows
// [rc RC, (rc+1) RC) of Dt, each row read as one coalesced 512-byte piece, or
// for rc = R the recovery U c as the r rows of U^T weighted by c.  The
// partial is added into y with fp32 atomics.
// The token's sanitised expert ids and weights, lane-distributed (topk <= 64).
// Wait state of a warp's output items: the token whose top-k it has seen
// (rows known) and the token whose phase-2 items it has seen counted (kept
// weights and the recovery vector known).
struct OutWait {
  uint32_t ftag = 1;   // the launch's flag value
  int flag_t = -1, count_t = -1;
  TokenSlots sl{};
  int kt = 0;          // the shared kernel: kept channels of token flag_t
  bool shared_in = false;   // the shared kernel: every kept item of the batch counted
};

__device__ bool out_wait(const Params& P, const uint32_t* word, uint32_t target, int lane) {
  int ok = 1;
  if (lane == 0) ok = wait_at_least(P, word, target);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

template <bool SH>
__device__ bool out_chunk(const Params& P, const OutPlan& op, int t, int cb, int rc, int lane,
                          int per_tok, OutWait& ow) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int c0 = cb * kOutCols + lane * 8;
  const bool on = c0 < d.H;                  // H is a multiple of 8
  int qb0 = rc * op.RC, qe = min(P.k, qb0 + op.RC);
  const uint64_t pol = policy_evict_first();  // the last read of these rows
  const float* wa_t = P.wa + (size_t)t * d.N;
  auto counted = [&]() {
    if (ow.count_t == t) return true;
    // the token's flag first: its count is zeroed before the flag's release
    if (!out_wait(P, P.sync + so.flag + t, ow.ftag, lane)) return false;
    if (!out_wait(P, P.sync + so.exact + t, (uint32_t)per_tok, lane)) return false;
    if (lane == 0) TRACE_POINT(15);
    if (SH && !ow.shared_in) {
      if (!out_wait(P, P.sync + kSyncSdone, (uint32_t)__ldcg(P.sK), lane)) return false;
      ow.shared_in = true;
    }
    ow.count_t = t;
    return true;
  };
  float acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = 0.f;
  if (rc >= op.R) {   // recovery chunk: rank components j0 .. j0 + nj - 1 of U c
    const int j0 = (rc - op.R) * kOutBatch, nj = min(kOutBatch, d.r - j0);
    if (SH) {   // the batch's kept rows are added by the shared chunks
      uint4 v[kOutBatch];
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u)
        v[u] = u < nj && on ? __ldg(reinterpret_cast<const uint4*>(P.Ut + (size_t)(j0 + u) * d.H + c0))
                            : make_uint4(0u, 0u, 0u, 0u);
      if (!out_wait(P, P.sync + so.flag + t, ow.ftag, lane)) return false;
      if (!out_wait(P, P.sync + so.exact + t, (uint32_t)per_tok, lane)) return false;
      const float cj_l = lane < nj ? __ldcg(P.cvec + (size_t)t * d.r + j0 + lane) : 0.f;
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u) {
        const float cw = __shfl_sync(0xffffffffu, cj_l, u);
        axpy8h(u < nj ? cw : 0.f, v[u], acc);
      }
      if (on) {
        float4* yo = reinterpret_cast<float4*>(P.y + (size_t)t * d.H + c0);
        atomicAdd(yo, make_float4(acc[0], acc[1], acc[2], acc[3]));
        atomicAdd(yo + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
      }
      return true;
    } else {
      uint4 v[kOutBatch];
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u)   // U^T rows do not depend on the token: load first
        v[u] = u < nj && on ? __ldg(reinterpret_cast<const uint4*>(P.Ut + (size_t)(j0 + u) * d.H + c0))
                            : make_uint4(0u, 0u, 0u, 0u);
      if (!counted()) return false;
      const float cj_l = lane < nj ? __ldcg(P.cvec + (size_t)t * d.r + j0 + lane) : 0.f;
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u) {
        const float cw = __shfl_sync(0xffffffffu, cj_l, u);
        axpy8h(u < nj ? cw : 0.f, v[u], acc);
      }
    }
  } else {
    // the rows come from the kept list and the expert ids alone (known at the
    // top-k): their loads go out before the token's phase-2 items are counted
    if (ow.flag_t != t) {
      if (!out_wait(P, P.sync + so.flag + t, ow.ftag, lane)) return false;
      ow.flag_t = t;
      ow.sl = load_token_slots(P, t, lane);
      if (SH) ow.kt = __ldcg(P.kcount + t);
    }
    if (SH) {   // the token's own kept count, in op.R chunks
      const int rct = (ow.kt + op.R - 1) / op.R;
      qb0 = rc * rct;
      qe = min(ow.kt, qb0 + rct);
    }
    for (int qb = qb0; qb < qe; qb += 32) {
      const int nq = min(32, qe - qb);
      int slot_l = 0, i_l = 0, n_l = 0;
      if (lane < nq) {
        n_l = __ldcg(P.kept + (size_t)t * d.N + qb + lane);
        slot_l = n_l / d.I;
        i_l = n_l - slot_l * d.I;
      }
      const int e_l = slot_expert(ow.sl.e0, ow.sl.e1, slot_l);   // every lane takes part
      const int row_l = e_l * d.I + i_l;
      // rows past the first load batch head for L2 now (4 lines of a 512-byte piece each)
      for (int p0 = kOutBatch * 4; p0 < nq * 4; p0 += 32) {
        const int pl = p0 + lane, i = pl >> 2;
        const int ro = __shfl_sync(0xffffffffu, row_l, i & 31);
        const int col = cb * kOutCols + (pl & 3) * 64;
        if (pl < nq * 4 && col < d.H)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(P.Dt + (size_t)ro * d.H + col));
      }
      float cw_l = 0.f;
      bool have_w = false;
      for (int i0 = 0; i0 < nq; i0 += kOutBatch) {
        uint4 v[kOutBatch];
        float c[kOutBatch];
#pragma unroll
        for (int u = 0; u < kOutBatch; ++u) {
          const int i = i0 + u;
          const int ro = __shfl_sync(0xffffffffu, row_l, i & 31);
          v[u] = i < nq && on ? ldcg4_hint(P.Dt + (size_t)ro * d.H + c0, pol)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
        if (!have_w) {   // with the first rows in flight
          if (!counted()) return false;
          cw_l = lane < nq ? __ldcg(wa_t + (SH ? n_l : qb + lane)) : 0.f;
          have_w = true;
        }
#pragma unroll
        for (int u = 0; u < kOutBatch; ++u) {
          const int i = i0 + u;
          const float cw = __shfl_sync(0xffffffffu, cw_l, i & 31);
          c[u] = i < nq ? cw : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kOutBatch; ++u) axpy8(c[u], v[u], acc);
      }
    }
  }
  // y was zeroed by the token's top-k; the chunks add in any order (fp32)
  if (on) {
    float4* yo = reinterpret_cast<float4*>(P.y + (size_t)t * d.H + c0);
    atomicAdd(yo, make_float4(acc[0], acc[1], acc[2], acc[3]));
    atomicAdd(yo + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  }
  return true;
}

// Output chunk c (rows c RCs .. of the batch's kept list) on column block cb:
// each kept down row piece is read once and added, weighed by w a, into every
// token routed to its expert (runs of one expert's rows, four tokens a pass).
__device__ bool shared_out_chunk(const Params& P, int c, int cb, int RCs, int K, int lane,
                                 OutWait& ow) {
  const Dims& d = P.d;
  if (!ow.shared_in) {
    if (!out_wait(P, P.sync + kSyncSdone, (uint32_t)K, lane)) return false;
    ow.shared_in = true;
  }
  const int c0 = cb * kOutCols + lane * 8;
  const bool on = c0 < d.H;
  const int q0 = c * RCs, q1 = min(K, q0 + RCs);
  const uint64_t pol = policy_evict_first();
  constexpr int kTG = 2, kSB = 8;   // tokens a pass, rows a load batch
  for (int q = q0; q < q1;) {
    // the next run of rows of one expert (at most 32)
    const int nq = min(32, q1 - q);
    const int info_l = lane < nq ? __ldcg(P.sinfo + q + lane) : -1;
    const int gid_l = lane < nq ? __ldcg(P.skept + q + lane) : 0;
    const int info = __shfl_sync(0xffffffffu, info_l, 0);
    const unsigned other = __ballot_sync(0xffffffffu, lane < nq && info_l != info);
    const int nr = other ? __ffs(other) - 1 : nq;
    const int l0 = info >> 14, nt = info & 16383;
    const int e = __shfl_sync(0xffffffffu, gid_l, 0) / d.I;
    const int i_l = gid_l - e * d.I;
    for (int g0 = 0; g0 < nt; g0 += kTG) {
      const int ng = min(kTG, nt - g0);
      float acc[kTG][8];
      float cw_l[kTG];
      int tt[kTG];
#pragma unroll
      for (int tg = 0; tg < kTG; ++tg) {
        const int ts = tg < ng ? __ldcg(P.elist + l0 + g0 + tg) : 0;
        const int t = ts / d.topk, slot = ts - t * d.topk;
        tt[tg] = t;
        cw_l[tg] = tg < ng && lane < nr ? __ldcg(P.wa + (size_t)t * d.N + (size_t)slot * d.I + i_l) : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[tg][u] = 0.f;
      }
      for (int i0 = 0; i0 < nr; i0 += kSB) {
        uint4 v[kSB];
#pragma unroll
        for (int u = 0; u < kSB; ++u) {
          const int ii = i0 + u;
          const int iro = __shfl_sync(0xffffffffu, i_l, ii & 31);
          v[u] = ii < nr && on ? ldcg4_hint(P.Dt + ((size_t)e * d.I + iro) * d.H + c0, pol)
                               : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int tg = 0; tg < kTG; ++tg) {
          if (tg >= ng) break;
#pragma unroll
          for (int u = 0; u < kSB; ++u) {
            const int ii = i0 + u;
            const float cw = __shfl_sync(0xffffffffu, cw_l[tg], ii & 31);
            axpy8(ii < nr ? cw : 0.f, v[u], acc[tg]);
          }
        }
      }
      if (on) {
#pragma unroll
        for (int tg = 0; tg < kTG; ++tg) {
          if (tg >= ng) break;
          float4* yo = reinterpret_cast<float4*>(P.y + (size_t)tt[tg] * d.H + c0);
          atomicAdd(yo, make_float4(acc[tg][0], acc[tg][1], acc[tg][2], acc[tg][3]));
          atomicAdd(yo + 1, make_float4(acc[tg][4], acc[tg][5], acc[tg][6], acc[tg][7]));
        }
      }
    }
    q += nr;
  }
  return true;
}

// Recovery output chunk rc of token t on column block cb (the per-token
// kernel): y += rank components rc*kOutBatch .. of U c, the U^T rows weighted
// by c, once the token's recovery chunks are counted; the U^T rows load first.
__device__ bool uc_item(const Params& P, int t, int cb, int rc, int lane, uint32_t ftag) {
  const Dims& d = P.d;
  const int c0 = cb * kOutCols + lane * 8;
  const bool on = c0 < d.H;                  // H is a multiple of 8
  const int j0 = rc * kOutBatch, nj = min(kOutBatch, d.r - j0);
  uint4 v[kOutBatch];
#pragma unroll
  for (int u = 0; u < kOutBatch; ++u)
    v[u] = u < nj && on ? __ldg(reinterpret_cast<const uint4*>(P.Ut + (size_t)(j0 + u) * d.H + c0))
                        : make_uint4(0u, 0u, 0u, 0u);
  // the token's flag first: its recovery count is zeroed before the flag's release
  if (!out_wait(P, P.sync + sync_offsets(d).flag + t, ftag, lane)) return false;
  if (!out_wait(P, P.sync + sync_offsets(d).exact + t, (uint32_t)(d.N / 64), lane)) return false;
  if (lane == 0) TRACE_POINT(15);
  const float cj_l = lane < nj ? __ldcg(P.cvec + (size_t)t * d.r + j0 + lane) : 0.f;
  float acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#pragma unroll
  for (int u = 0; u < kOutBatch; ++u) {
    const float cw = __shfl_sync(0xffffffffu, cj_l, u);
    axpy8h(u < nj ? cw : 0.f, v[u], acc);
  }
  if (on) {
    float4* yo = reinterpret_cast<float4*>(P.y + (size_t)t * d.H + c0);
    atomicAdd(yo, make_float4(acc[0], acc[1], acc[2], acc[3]));
    atomicAdd(yo + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  }
  return true;
}

// ------------------------------- the kernel --------------------------------
// One layer's decode by every CTA of the grid.  false: the launch is aborting.
// The end of a shared-selection decode by a CTA: the last CTA out resets the
// words only that kernel uses (the others need no reset: see kSyncGen; a
// stacked layer's words are zeroed by their last readers).  Every thread of
// the CTA calls it.
__device__ void decode_tail(const Params& P, int* ctl) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int nctas = gridDim.x;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    ctl[0] = atomicAdd(P.sync + kSyncTail, 1u) == (uint32_t)(nctas - 1);
  }
  __syncthreads();
  if (ctl[0] && threadIdx.x == 0) {
    for (int q = 0; q < d.E; ++q) P.sync[so.ecount + q] = 0u;
    P.sync[kSyncBatch] = 0u;
    P.sync[kSyncReady] = 0u;
    P.sync[kSyncSdone] = 0u;
    P.sync[kSyncTail] = 0u;
  }
  __syncthreads();
}

// Static shared control words of a CTA: [0] the last-CTA test, [1] a
// broadcast flag, then the shared waits of phase 2 for the first kTokWait
// tokens of the CTA's item range (seen words, then claim words), then the
// launch's flag value (generation + 1).
constexpr int kTokWait = 8, kCtlFtag = 2 + 2 * kTokWait, kCtlWords = kCtlFtag + 1;

__device__ __forceinline__ unsigned long long atom_add_u64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// STK: a layer of a stack (its input and residual come from the layer before).
template <bool SH, int WPT, bool T5, bool STK>
__device__ __forceinline__ bool decode_layer(const Params& P, unsigned char* smem, int* ctl) {
  if (threadIdx.x == 0) ctl[0] = 0;
  if (threadIdx.x < 2 * kTokWait) ctl[2 + threadIdx.x] = 0;   // ordered by the barrier after the screen
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nctas = gridDim.x;
  unsigned long long* stamp = P.stamps ? P.stamps + (size_t)blockIdx.x * 5 : nullptr;
  if (stamp && threadIdx.x == 0) stamp[0] = globaltimer();
  if (threadIdx.x == 0) TRACE_POINT(0);
  // the launch's generation: requested now, first needed after the screen
  unsigned long long gen_in = 0;
  if (threadIdx.x == 0) gen_in = atom_add_u64(reinterpret_cast<unsigned long long*>(P.sync + kSyncGen), 1ull);

  // phase 1a: screen units (rotation, selection and sketch sums), computed by teams of warps
  screen_compute<WPT, T5, STK>(P, smem, warp, cta_group());
  if (threadIdx.x == 0) ctl[kCtlFtag] = (int)(uint32_t)(gen_in / (unsigned long long)nctas + 1ull);
  __syncthreads();
  const uint32_t ftag = (uint32_t)ctl[kCtlFtag];
  if (stamp && threadIdx.x == 0) stamp[1] = globaltimer();
  if (threadIdx.x == 0) TRACE_POINT(5);
  // phase 1b: scoring tasks spread over the CTAs; the CTA that scores a
  // token's last slot runs the token's top-k (1c) at once
  {
    int* flag = &ctl[1];   // static shared memory: the top-k's working area starts at smem
    for (int ts = blockIdx.x; ts < P.B * d.topk; ts += nctas) {
      const int r = score_task<SH>(P, cta_group(), ts, flag, smem);
      if (r < 0) return false;
      if (!SH && r > 0) {
        topk_token<kThreads>(P, cta_group(), ts / d.topk, smem, ftag);
        // a stacked layer: every screen unit of the token has passed its
        // wait for the token's input, which the layer before sets again
        if (STK && threadIdx.x == 0) P.sync[so.xready + ts / d.topk] = 0u;
      }
      __syncthreads();
    }
    if (SH) {
      // 1c: each token's share of the batch's kept set (selected by the
      // score task that completed the last routed expert)
      for (int t = blockIdx.x; t < P.B; t += nctas) {
        if (threadIdx.x == 0)
          *flag = wait_at_least(P, P.sync + kSyncReady, 1u);
        __syncthreads();
        if (!*flag) return false;
        shared_token(P, t, smem, ftag);
        __syncthreads();
      }
    }
  }
  if (stamp && threadIdx.x == 0) stamp[2] = globaltimer();
  // phase 2: kept channels and recovery chunks, one warp each
  const int per_tok = SH ? d.N / 64 : P.k + d.N / 64;   // items counted per token
  if (SH) {
    // the batch's kept channels first (each serving all its tokens), then
    // every token's recovery chunks
    if (threadIdx.x == 0) ctl[1] = wait_at_least(P, P.sync + kSyncReady, 1u);
    __syncthreads();
    if (!ctl[1]) return false;
    const long long K = __ldcg(P.sK);
    const long long M = K + (long long)P.B * per_tok;
    const long long wtot = (long long)nctas * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long ipw = (M + wtot - 1) / wtot;
    const long long q0 = gw * ipw, q1 = min(M, q0 + ipw);
    int cur_t = -1, pend_t = -1, pend_n = 0, nk = 0;
    bool ok = true;
    long long kb = -64;
    int gid_l = 0, info_l = 0;   // lane j: kept channel kb + j
    for (long long q = q0; q < q1; ++q) {
      if (q < K) {
        if (q - kb >= 32) {
          kb = q;
          gid_l = kb + lane < K ? __ldcg(P.skept + kb + lane) : 0;
          info_l = kb + lane < K ? __ldcg(P.sinfo + kb + lane) : 0;
        }
        const int j = (int)(q - kb);
        shared_kept_item(P, __shfl_sync(0xffffffffu, gid_l, j), __shfl_sync(0xffffffffu, info_l, j),
                         lane);
        ++nk;
        continue;
      }
      const long long r = q - K;
      const int t = (int)(r / per_tok), ch = (int)(r % per_tok);
      if (t != cur_t) {
        int w_ok = 1;
        if (lane == 0) w_ok = wait_at_least(P, P.sync + so.flag + t, ftag);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        __syncwarp();
        cur_t = t;
      }
      const bool flush = pend_t >= 0 && pend_t != t;
      recovery_item(P, t, ch, lane, flush ? pend_t : -1, pend_n);
      if (flush) pend_n = 0;
      pend_t = t;
      ++pend_n;
    }
    if (ok) publish_item(P, pend_t, pend_n, lane);
    if (nk) {
      __syncwarp();
      if (lane == 0) red_add_release(P.sync + kSyncSdone, (uint32_t)nk);
    }
  } else {
    // kept channels and recovery chunks in contiguous runs of items per warp;
    // a warp meets one or two tokens and counts its recovery chunks of a token
    // when it leaves the token.  Each CTA then adds the output of the kept
    // rows of its range (register sums over the rows, one vector add per lane
    // and column chunk): no hand-off between CTAs on the way to y.
    const long long M = (long long)P.B * per_tok;
    const long long wtot = (long long)nctas * kWarps;
    const long long ipw = (M + wtot - 1) / wtot;
    const long long cq0 = min(M, (long long)blockIdx.x * kWarps * ipw);
    const long long cq1 = min(M, cq0 + (long long)kWarps * ipw);
    const int nitems = (int)(cq1 - cq0);
    // the CTA's lists of w a and rows when they fit (else global wa), then a
    // flag per (token, column block) of the range
    const int ncb_s = (d.H + kOutCols - 1) / kOutCols;
    const bool use_s = (size_t)nitems * 8 + (size_t)(nitems + 1) * ncb_s * 4 <= (size_t)P.smem_bytes;
    float* wa_s = use_s ? reinterpret_cast<float*>(smem) : nullptr;
    int* row_s = use_s ? reinterpret_cast<int*>(smem) + nitems : nullptr;
    int* done_s = reinterpret_cast<int*>(smem) + (use_s ? 2 * nitems : 0);
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long q0 = gw * ipw, q1 = min(M, q0 + ipw);
    int cur_t = -1, rec_t = -1, rec_n = 0;
    int kbase = 0, kn_l = 0;   // lane j: kept index at list position kbase + j
    TokenSlots sl{};
    bool ok = true;
    const int tf_cta = (int)(cq0 / per_tok);   // the first token of the CTA's range
    for (long long q = q0; q < q1; ++q) {
      const int t = (int)(q / per_tok), local = (int)(q % per_tok);
      if (t != cur_t) {
        if (rec_n) publish_item(P, rec_t, rec_n, lane);
        rec_n = 0;
        TokenSlots nsl = input_token_slots(P, t, lane);   // in flight during the wait
        bool w_ok;
        const int ti = t - tf_cta;
        if (ti < kTokWait) {
          w_ok = cta_wait(P, P.sync + so.flag + t, ftag, &ctl[2 + ti], &ctl[2 + kTokWait + ti], lane);
        } else {
          int o = 1;
          if (lane == 0) o = wait_at_least(P, P.sync + so.flag + t, ftag);
          w_ok = __shfl_sync(0xffffffffu, o, 0) != 0;
          __syncwarp();
        }
        if (!w_ok) {
          ok = false;
          break;
        }
        cur_t = t;
        sanitise_slots(d, nsl);
        sl = nsl;
        if (lane == 0 && warp == 0) TRACE_POINT(13);
        kbase = -64;
      }
      if (local < P.k) {
        if (local - kbase >= 32) {   // the next 32 kept indices in one read
          kbase = local;
          kn_l = kbase + lane < P.k ? __ldcg(P.kept + (size_t)t * d.N + kbase + lane) : 0;
        }
        const int n = __shfl_sync(0xffffffffu, kn_l, local - kbase);
        kept_item_cta(P, t, use_s ? (int)(q - cq0) : local, n, sl, lane, wa_s, row_s);
      } else {
        recovery_item(P, t, local - P.k, lane, -1, 0);
        rec_t = t;
        ++rec_n;
      }
    }
    if (ok && rec_n) publish_item(P, rec_t, rec_n, lane);
    if (lane == 0 && rec_n) TRACE_POINT(30);
    if (lane == 0) TRACE_POINT(14);
    if (threadIdx.x == 0) ctl[1] = 0;
    __syncthreads();
    if (!ok && lane == 0) ctl[1] = 1;   // this warp left its items: the launch is aborting
    __syncthreads();   // the CTA's kept channels are in
    if (stamp && threadIdx.x == 0) stamp[3] = globaltimer();
    if (ctl[1]) return false;   // a list entry may be missing: read no row
    const int ncb = (d.H + kOutCols - 1) / kOutCols;
    const int rec = P.k < d.N ? (d.r + kOutBatch - 1) / kOutBatch : 0;
    // the output of the kept rows of each token of the range
    if (cq0 < cq1) {
      const int tf = (int)(cq0 / per_tok), tl = (int)((cq1 - 1) / per_tok);
      for (int t = tf; t <= tl; ++t) {
        const long long a = max(cq0, (long long)t * per_tok);
        const long long b = min(cq1, (long long)t * per_tok + P.k);
        if (a >= b) continue;
        const TokenSlots tsl = use_s ? TokenSlots{} : load_token_slots(P, t, lane);
        cta_output(P, t, (int)(a - (long long)t * per_tok), (int)(b - (long long)t * per_tok), wa_s,
                   row_s, (int)(a - cq0), tsl, warp, lane);
      }
      if (lane == 0) TRACE_POINT(29);
      if (STK) {   // a stacked layer: each column block the CTA completes is carried
        __syncthreads();   // every output add of the CTA precedes the counts
        const int nr = (tl - tf + 1) * ncb;
        for (int r = threadIdx.x; r < nr; r += kThreads) {
          const int t = tf + r / ncb, cb = r % ncb;
          const long long a = max(cq0, (long long)t * per_tok);
          const long long b = min(cq1, (long long)t * per_tok + P.k);
          const uint32_t total = (uint32_t)(kept_ctas(t, per_tok, P.k, ipw) + rec);
          done_s[r] = a < b && count_block(P, t, cb, ncb, total);
        }
        __syncthreads();
        for (int r = warp; r < nr; r += kWarps)
          if (done_s[r]) carry_block(P, tf + r / ncb, r % ncb, ncb, lane);
      }
    }
    // recovery output chunks, dealt from the last warp down so that warps
    // without kept channels take them first
    const int nwarps = nctas * kWarps;
    const int items = P.B * ncb * rec;
    for (int it = nwarps - 1 - (int)gw; it < items; it += nwarps) {
      const int t = it / (ncb * rec);
      const int cb = (it / rec) % ncb;
      if (!uc_item(P, t, cb, it % rec, lane, ftag)) break;
      if (STK) {   // a stacked layer: the block's last contribution carries it
        __syncwarp();
        int last = 0;
        if (lane == 0)
          last = count_block(P, t, cb, ncb, (uint32_t)(kept_ctas(t, per_tok, P.k, ipw) + rec));
        if (__shfl_sync(0xffffffffu, last, 0)) carry_block(P, t, cb, ncb, lane);
      }
    }
  }
  if (SH) {
    if (lane == 0) TRACE_POINT(14);
    if (stamp) {
      __syncthreads();
      if (threadIdx.x == 0) stamp[3] = globaltimer();
    }
    // phase 3: output warp items, dealt from the last warp down so that warps
    // without phase-2 work take them first
    // the batch's kept rows in chunks of RCs rows per column block, then each
    // token's recovery chunks
    const int nwarps = nctas * kWarps;
    const int K = __ldcg(P.sK);
    const int ncb = (d.H + kOutCols - 1) / kOutCols;
    const int rec = P.k < d.N ? (d.r + kOutBatch - 1) / kOutBatch : 0;
    const int RCs = max(1, (int)(((long long)K * ncb + nwarps - 1) / nwarps));
    const int C = (K + RCs - 1) / RCs;
    const int items = C * ncb + P.B * ncb * rec;
    const int gw = blockIdx.x * kWarps + warp;
    OutPlan op;
    op.ncb = ncb;
    op.R = 0;
    op.RC = 0;
    op.NR = rec;
    OutWait ow;
    ow.ftag = ftag;
    for (int it = nwarps - 1 - gw; it < items; it += nwarps) {
      if (it < C * ncb) {
        if (!shared_out_chunk(P, it / ncb, it % ncb, RCs, K, lane, ow)) break;
      } else {
        const int r = it - C * ncb, t = r / (ncb * rec);
        if (!out_chunk<SH>(P, op, t, (r / rec) % ncb, r % rec, lane, per_tok, ow)) break;
      }
    }
  }
  if (stamp && threadIdx.x == 0) stamp[4] = globaltimer();
  if (threadIdx.x == 0) TRACE_POINT(16);
  if (SH) decode_tail(P, ctl);
  return true;
}

// the pair tables are addressed by assembling a 256-byte aligned block base
// with a low byte: align the working area to 256 bytes whatever the window offset
__device__ __forceinline__ unsigned char* aligned_smem(unsigned char* raw) {
  return raw + ((256u - (smem_addr(raw) & 255u)) & 255u);
}

// The batch-shared selection variant: one kept set for the whole batch.
// Kernels are specialised on the screen's code words per thread (WPT), so
// that each holds only the code it runs.
template <int WPT, bool T5>
__global__ void __launch_bounds__(kThreads, 1) decode_shared_kernel(const Params P) {
  extern __shared__ __align__(256) unsigned char smem_raw[];
  __shared__ int ctl[kCtlWords];
  decode_layer<true, WPT, T5, false>(P, aligned_smem(smem_raw), ctl);
}

template <int WPT, bool T5, bool STK>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const Params P) {
  extern __shared__ __align__(256) unsigned char smem_raw[];
  __shared__ int ctl[kCtlWords];
  decode_layer<false, WPT, T5, STK>(P, aligned_smem(smem_raw), ctl);
  if (threadIdx.x == 0) TRACE_POINT(17);
  if (STK && P.next_abort && threadIdx.x == 0 && ld_acquire(P.sync + kSyncAbort)) {
    // the next layer would wait for inputs that never come
    atomicOr(P.next_err, kErrTimeout);
    atomicExch(P.next_abort, 1u);
  }
}

using KernelFn = void (*)(const Params);

template <bool T5>
KernelFn pick_kernel_t(bool shared, int wpt, bool stack) {
  if (shared)
    return wpt == 1 ? decode_shared_kernel<1, T5> : wpt == 2 ? decode_shared_kernel<2, T5> : decode_shared_kernel<3, T5>;
  if (stack)
    return wpt == 1 ? decode_kernel<1, T5, true> : wpt == 2 ? decode_kernel<2, T5, true> : decode_kernel<3, T5, true>;
  return wpt == 1 ? decode_kernel<1, T5, false> : wpt == 2 ? decode_kernel<2, T5, false> : decode_kernel<3, T5, false>;
}

// The kernel for a decode: shared selection or not, a stacked layer or not,
// the screen's code words per thread and the code layout (2-bit or five
// trits per byte).
KernelFn pick_kernel(bool shared, int wpt, bool t5, bool stack = false) {
  return t5 ? pick_kernel_t<true>(shared, wpt, stack) : pick_kernel_t<false>(shared, wpt, stack);
}

size_t decode_smem_bytes(const Dims& d) {
  const size_t screen = screen_plan(d).bytes;
  const size_t topk = topk_smem_bytes(d.N);
  const size_t m = screen > topk ? screen : topk;
  return m + 256;   // + alignment slack of the working area
}

}  // namespace

size_t sync_words(const Dims& d) { return (size_t)sync_offsets(d).total; }

#ifdef MR_TRACE
}  // namespace mr
extern "C" int moe_reader_trace_read(unsigned long long* host, int clear) {
  if (cudaMemcpyFromSymbol(host, mr::g_trace, sizeof(mr::g_trace)) != cudaSuccess) return -3;
  if (clear) {
    static unsigned long long zero[mr::kTraceCtas][mr::kTracePoints];
    if (cudaMemcpyToSymbol(mr::g_trace, zero, sizeof(zero)) != cudaSuccess) return -3;
  }
  return 0;
}
namespace mr {
#endif

bool shared_supported(const Dims& d, int B) {
  // the selection CTA's tables and the score tasks' slot lists fit the
  // decode's shared memory; the elist packing holds 8192 token slots
  return shared_select_bytes(d) <= decode_smem_bytes(d) - 256 &&
         (size_t)(B * d.topk + kWarps + d.E + 4) * 4 <= decode_smem_bytes(d) - 256 &&
         B * d.topk <= 8192;
}

cudaError_t configure_decode_kernels(const Dims& d) {
  const ScreenPlan sp = screen_plan(d);
  if (sp.bytes == 0) return cudaErrorInvalidValue;
  const size_t smem = decode_smem_bytes(d);
  for (int v = 0; v < 3; ++v) {   // the shape's kernels: per-token, shared, stacked layer
    const KernelFn fn = pick_kernel(v == 1, sp.wpt, d.trit5 != 0, v == 2);
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, fn);
    if (err != cudaSuccess) return err;
    if ((size_t)fa.maxDynamicSharedSizeBytes < smem &&
        (err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
      return err;
  }
  return cudaSuccess;
}

int decode_grid(const Dims& d) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pick_kernel(false, screen_plan(d).wpt, d.trit5 != 0),
                                                    kThreads, decode_smem_bytes(d)) != cudaSuccess)
    return 0;
  return per_sm >= 1 ? sms : 0;   // one CTA per SM, all co-resident
}

static Params make_params(const moe_reader& h, const float* x, int B, const int32_t* ids, const float* w,
                   int k, float* y, unsigned long long* stamps) {
  const Dims& d = h.d;
  const Workspace& ws = h.ws;
  Params P;
  P.d = d;
  P.B = B;
  P.k = k;
  P.x = x;
  P.ids_in = ids;
  P.w_in = w;
  P.y = y;
  P.sigma = h.p.sigma;
  P.codes = h.p.codes;
  P.scales = h.p.scales;
  P.dnorm = h.p.dnorm;
  P.G = h.G;
  P.V = h.V;
  P.Dt = h.p.Dt;
  P.U = h.p.U;
  P.Ut = h.p.Ut;
  P.bco = h.p.b;
  P.ids_ws = ws.ids;
  P.w_ws = ws.w;
  P.mask = ws.mask;
  P.partial = ws.partial;
  P.ghat = ws.ghat;
  P.vhat = ws.vhat;
  P.p = ws.p;
  P.score = ws.score;
  P.keptbits = ws.keptbits;
  P.kept = ws.kept;
  P.wa = ws.wa;
  P.cvec = ws.cpart;
  P.stamps = stamps;
  P.sync = ws.sync;
  P.err = ws.err;
  P.sp = screen_plan(d);
  P.xwait = nullptr;
  P.xscale = nullptr;
  P.xfill = nullptr;
  P.hres = nullptr;
  P.hnext = nullptr;
  P.xscale_next = nullptr;
  P.xnext_ready = nullptr;
  P.next_abort = nullptr;
  P.next_err = nullptr;
  P.sscore = ws.sscore;
  P.skept = ws.skept;
  P.sbits = ws.sbits;
  P.estart = ws.estart;
  P.elist = ws.elist;
  P.kcount = ws.kcount;
  P.sK = ws.sK;
  P.sinfo = ws.sinfo;
  P.rho = h.p.rho;
  P.bnorm2 = h.p.bnorm2;
  P.rn2 = ws.rn2;
  P.ecount = ws.sync + sync_offsets(d).ecount;
  P.smem_bytes = (int)decode_smem_bytes(d) - 256;
  P.wait_ns = h.wait_ns ? (unsigned long long)h.wait_ns : kDefaultWaitNs;
  P.stall = (h.inject & MOE_READER_INJECT_DECODE_STALL) ? 1 : 0;
  return P;
}

// The first layer's input scale 1 / RMS(h_0[t]), one CTA per token (fp64
// sum of squares), each token released on `ready` for the decode that follows.
__global__ void __launch_bounds__(kThreads) stack_input_kernel(const float* h, float* scale,
                                                             uint32_t* ready, int H) {
  __shared__ double part[kWarps];
  const int t = blockIdx.x;
  double ss = 0.0;
  for (int c = 4 * threadIdx.x; c < H; c += 4 * kThreads) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(h + (size_t)t * H + c));
    ss += (double)v.x * v.x + (double)v.y * v.y + (double)v.z * v.z + (double)v.w * v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < kWarps; ++w) tot += part[w];
    scale[t] = (float)(1.0 / sqrt(tot / H + 1e-6));
    st_release(ready + t, 1u);
  }
}

static cudaError_t launch_params(const moe_reader& h, const Params& P, cudaStream_t s,
                                 bool shared = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = decode_smem_bytes(h.d);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pick_kernel(shared, P.sp.wpt, h.d.trit5 != 0, P.hnext != nullptr), P);
}

cudaError_t launch_decode(const moe_reader& h, const float* x, int B, const int32_t* ids,
                          const float* w, int k, float* y, cudaStream_t s, const cudaEvent_t* ev,
                          unsigned long long* stamps, bool shared) {
  cudaError_t err;
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev) {
    // inside stream capture a plain record is only a dependency marker; the
    // External flag makes it an event-record node of the graph
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((err = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return err;
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
    if ((err = cudaEventRecordWithFlags(ev[0], s, rec_flags)) != cudaSuccess) return err;
  }
  const Params P = make_params(h, x, B, ids, w, k, y, stamps);
  if ((err = launch_params(h, P, s, shared)) != cudaSuccess) return err;
  if (ev && (err = cudaEventRecordWithFlags(ev[1], s, rec_flags)) != cudaSuccess) return err;
  return cudaSuccess;
}

cudaError_t launch_decode_stack(moe_reader* const* hs, int L, const float* h_in, int B,
                                const int32_t* ids, const float* w, int k, float* h_out,
                                float* y_layers, cudaStream_t s) {
  if (L < 1) return cudaErrorInvalidValue;
  const Dims& d = hs[0]->d;
  const size_t tok = (size_t)B * d.topk, act = (size_t)B * d.H;
  stack_input_kernel<<<B, kThreads, 0, s>>>(h_in, hs[0]->ws.xscale,
                                             hs[0]->ws.sync + sync_offsets(d).xready, d.H);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  for (int l = 0; l < L; ++l) {
    const moe_reader& h = *hs[l];
    float* yl = y_layers ? y_layers + l * act : h.ws.y_stage;
    Params P = make_params(h, h.ws.x_stage, B, ids + l * tok, w + l * tok, k, yl, nullptr);
    P.xwait = h.ws.sync + sync_offsets(h.d).xready;
    P.xscale = h.ws.xscale;
    P.xfill = h.ws.x_stage;
    P.hres = l == 0 ? h_in : h.ws.h_stage;
    P.hnext = l + 1 < L ? hs[l + 1]->ws.h_stage : h_out;
    P.xscale_next = l + 1 < L ? hs[l + 1]->ws.xscale : nullptr;
    P.xnext_ready = l + 1 < L ? hs[l + 1]->ws.sync + sync_offsets(hs[l + 1]->d).xready : nullptr;
    P.next_abort = l + 1 < L ? hs[l + 1]->ws.sync + kSyncAbort : nullptr;
    P.next_err = l + 1 < L ? hs[l + 1]->ws.err : nullptr;
    // stream order: a layer's grid starts once the grid before has finished
    // (a grid allowed to start early, by programmatic serialization, parks
    // CTAs that would take SMs the layer before still needs, and was
    // measured slower); the per-token release on xwait keeps the hand-off
    // valid under any launch order
    if ((err = launch_params(h, P, s)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace mr
